// sgemm_ffma.cu -- FP32 SIMT GEMM on the FFMA pipe, C = A * B^T, C row-major.
//
// Design follows the CuTe DSL Ampere SGEMM example (SGemm.__call__ / kernel)
// re-done by hand for sm_103a:
//   * CTA tile 128 x 128 x BK, 256 threads, each thread owning an 8 x 8 block
//     of C as four 4 x 4 quadrants (4 consecutive rows x 4 consecutive columns
//     in each 64 x 64 sub-tile), so fragments load with 128-bit LDS;
//   * A and B tiles always stored MN-major in shared memory (k-rows of 128
//     floats, padded by 4 floats) so the fragment loads vectorise whatever
//     the global major; a K-major operand is transposed on the way in with
//     4-byte cp.async (conflict-free thanks to the pad), an MN-major operand
//     is copied with 16-byte cp.async when its base and leading dimension are
//     16-byte aligned (4-byte otherwise);
//   * a STAGES-deep cp.async ring (one barrier per k-tile; the wait allows
//     STAGES-2 groups in flight) and a register double buffer over k inside a
//     tile;
//   * every copy is predicated with zero fill on the M/N/K bounds, so ragged
//     shapes need no separate residue pass (the CuTe example shifts the
//     ragged k-tile to the front instead; predicating every copy costs a few
//     integer compares per k-tile here and keeps one code path);
//   * predicated epilogue with 128-bit stores when C allows them.
#include <cstdint>

#include "internal.h"

namespace libgemm {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 16;
constexpr int STAGES = 4;
constexpr int THREADS = 256;
constexpr int PAD = 4;
constexpr int LDS = BM + PAD;  // floats per k-row in shared memory (BM == BN)
constexpr int OPERAND_FLOATS = BK * LDS;
constexpr int STAGE_FLOATS = 2 * OPERAND_FLOATS;
constexpr int SMEM_BYTES = STAGES * STAGE_FLOATS * 4;
constexpr int BAND = 16;  // tile rows per raster band (L2 locality)

static_assert(BM == BN, "one shared-memory row stride serves both operands");
static_assert(BK == 16, "the K-major copy mapping below assumes BK == 16");

struct SgemmParams {
    const float* A;
    const float* B;
    float* C;
    int64_t lda, ldb, ldc;
    int M, N, K;
    int tiles_m, tiles_n;
    int c_vec;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, bool pred) {
    const int n = pred ? 4 : 0;  // src-size 0: zero fill, nothing read
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" :: "r"(dst), "l"(src), "r"(n)
                 : "memory");
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src),
                 "r"(bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

// Copy one BK-deep tile of an operand (rows r0.., k0..) into shared memory
// laid out [k][r] with row stride LDS floats.
template <bool KMAJOR, int VEC>
__device__ __forceinline__ void load_tile(uint32_t s, const float* __restrict__ X, int64_t ld,
                                          int R, int K, int r0, int k0, int tid) {
    if constexpr (KMAJOR) {
        // 2048 elements; a warp covers 4 rows x 8 consecutive k (32-byte
        // segments); smem bank = (4k + r) mod 32 is distinct within the warp.
#pragma unroll
        for (int i = 0; i < (BM * BK) / THREADS; ++i) {
            const int e = tid + i * THREADS;
            const int h = e >> 10;
            const int rr = (e & 1023) >> 3;
            const int kk = (h << 3) | (e & 7);
            const int gr = r0 + rr, gk = k0 + kk;
            const bool ok = gr < R && gk < K;
            const float* src = ok ? X + (int64_t)gr * ld + gk : X;
            cp_async_4(s + (uint32_t)(kk * LDS + rr) * 4u, src, ok);
        }
    } else if constexpr (VEC == 4) {
        // 512 float4 along r; a warp copies one 512-byte k-row.
#pragma unroll
        for (int i = 0; i < (BM * BK) / (4 * THREADS); ++i) {
            const int idx = tid + i * THREADS;
            const int kk = idx >> 5;
            const int rr = (idx & 31) << 2;
            const int gr = r0 + rr, gk = k0 + kk;
            int bytes = 0;
            if (gk < K && gr < R) bytes = (R - gr >= 4 ? 4 : R - gr) * 4;
            const float* src = bytes ? X + (int64_t)gk * ld + gr : X;
            cp_async_16(s + (uint32_t)(kk * LDS + rr) * 4u, src, bytes);
        }
    } else {
        // MN-major but not 16-byte aligned: coalesced 4-byte copies along r.
#pragma unroll
        for (int i = 0; i < (BM * BK) / THREADS; ++i) {
            const int e = tid + i * THREADS;
            const int kk = e >> 7;
            const int rr = e & 127;
            const int gr = r0 + rr, gk = k0 + kk;
            const bool ok = gr < R && gk < K;
            const float* src = ok ? X + (int64_t)gk * ld + gr : X;
            cp_async_4(s + (uint32_t)(kk * LDS + rr) * 4u, src, ok);
        }
    }
}

template <bool A_K, int A_VEC, bool B_K, int B_VEC>
__global__ void __launch_bounds__(THREADS, 2) sgemm_ffma_kernel(const SgemmParams p) {
    extern __shared__ __align__(16) float smem[];
    const int tid = threadIdx.x;

    // Raster: bands of BAND tile-rows, walking down M inside a band first.
    const int t = blockIdx.x;
    const int band_tiles = BAND * p.tiles_n;
    const int band = t / band_tiles;
    const int within = t - band * band_tiles;
    const int m_lo = band * BAND;
    const int rows_in_band = min(BAND, p.tiles_m - m_lo);
    const int tm = m_lo + within % rows_in_band;
    const int tn = within / rows_in_band;
    const int m0 = tm * BM, n0 = tn * BN;

    // Thread -> C block: warp (wy, wx) = (w / 2, w % 2), lane (ly, lx) =
    // (l / 8, l % 8); ty in 0..15, tx in 0..15.
    const int w = tid >> 5, l = tid & 31;
    const int ty = (w >> 1) * 4 + (l >> 3);
    const int tx = (w & 1) * 8 + (l & 7);

    const uint32_t s0 = smem_addr(smem);
    const int nkt = (p.K + BK - 1) / BK;

    auto load_stage = [&](int stage, int kt) {
        const uint32_t sa = s0 + (uint32_t)(stage * STAGE_FLOATS) * 4u;
        const uint32_t sb = sa + (uint32_t)OPERAND_FLOATS * 4u;
        load_tile<A_K, A_VEC>(sa, p.A, p.lda, p.M, p.K, m0, kt * BK, tid);
        load_tile<B_K, B_VEC>(sb, p.B, p.ldb, p.N, p.K, n0, kt * BK, tid);
    };

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < nkt) load_stage(s, s);
        cp_async_commit();
    }

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    float a[2][8], b[2][8];

    for (int kt = 0; kt < nkt; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();  // tile kt landed; every thread is done with tile kt-1

        const int nt = kt + STAGES - 1;
        if (nt < nkt) load_stage(nt % STAGES, nt);
        cp_async_commit();

        const float* sA = smem + (kt % STAGES) * STAGE_FLOATS;
        const float* sB = sA + OPERAND_FLOATS;

        auto load_frag = [&](int buf, int k) {
            const float4* pa = reinterpret_cast<const float4*>(sA + k * LDS + ty * 4);
            const float4* pb = reinterpret_cast<const float4*>(sB + k * LDS + tx * 4);
            const float4 a0 = pa[0], a1 = pa[16], b0 = pb[0], b1 = pb[16];
            a[buf][0] = a0.x; a[buf][1] = a0.y; a[buf][2] = a0.z; a[buf][3] = a0.w;
            a[buf][4] = a1.x; a[buf][5] = a1.y; a[buf][6] = a1.z; a[buf][7] = a1.w;
            b[buf][0] = b0.x; b[buf][1] = b0.y; b[buf][2] = b0.z; b[buf][3] = b0.w;
            b[buf][4] = b1.x; b[buf][5] = b1.y; b[buf][6] = b1.z; b[buf][7] = b1.w;
        };

        load_frag(0, 0);
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            if (k + 1 < BK) load_frag((k + 1) & 1, k + 1);
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    acc[i][j] = fmaf(a[k & 1][i], b[k & 1][j], acc[i][j]);
        }
    }
    cp_async_wait<0>();

    // Epilogue: rows ty*4 + (i & 3) + (i >> 2) * 64, cols tx*4 + (j & 3) + (j >> 2) * 64.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + ty * 4 + (i & 3) + (i >> 2) * 64;
        if (row >= p.M) continue;
        float* crow = p.C + (int64_t)row * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = n0 + tx * 4 + h * 64;
            if (p.c_vec && col + 3 < p.N) {
                *reinterpret_cast<float4*>(crow + col) =
                    make_float4(acc[i][h * 4 + 0], acc[i][h * 4 + 1], acc[i][h * 4 + 2],
                                acc[i][h * 4 + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < p.N) crow[col + j] = acc[i][h * 4 + j];
            }
        }
    }
}

template <bool A_K, int A_VEC, bool B_K, int B_VEC>
int launch_variant(const SgemmParams& sp, cudaStream_t stream) {
    auto kern = sgemm_ffma_kernel<A_K, A_VEC, B_K, B_VEC>;
    static bool configured = false;  // attribute is per function, set once
    if (!configured) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess)
            return kCuda;
        configured = true;
    }
    const int64_t tiles = (int64_t)sp.tiles_m * sp.tiles_n;
    kern<<<dim3((unsigned)tiles), dim3(THREADS), SMEM_BYTES, stream>>>(sp);
    if (cudaGetLastError() != cudaSuccess) return kCuda;
    note_launch();
    return kOk;
}

bool aligned16(const void* p, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && (ld & 3) == 0;
}

}  // namespace

int launch_sgemm_f32(const Problem& pr, const DeviceInfo&, cudaStream_t stream) {
    SgemmParams sp;
    sp.A = static_cast<const float*>(pr.A);
    sp.B = static_cast<const float*>(pr.B);
    sp.C = static_cast<float*>(pr.C);
    sp.lda = pr.lda;
    sp.ldb = pr.ldb;
    sp.ldc = pr.ldc;
    sp.M = (int)pr.M;
    sp.N = (int)pr.N;
    sp.K = (int)pr.K;
    sp.tiles_m = (int)((pr.M + BM - 1) / BM);
    sp.tiles_n = (int)((pr.N + BN - 1) / BN);
    sp.c_vec = aligned16(pr.C, pr.ldc) ? 1 : 0;
    if ((int64_t)sp.tiles_m * sp.tiles_n > 0x7fffffffLL) return kUnsupported;

    // A/B variant: K-major (4-byte transposing copies), MN-major 16-byte or 4-byte.
    const int av = pr.a_kmajor ? 0 : (aligned16(pr.A, pr.lda) ? 4 : 1);
    const int bv = pr.b_kmajor ? 0 : (aligned16(pr.B, pr.ldb) ? 4 : 1);
#define SG_CASE(AV, BV, AK, AVEC, BK_, BVEC) \
    if (av == AV && bv == BV) return launch_variant<AK, AVEC, BK_, BVEC>(sp, stream);
    SG_CASE(0, 0, true, 1, true, 1)
    SG_CASE(0, 4, true, 1, false, 4)
    SG_CASE(0, 1, true, 1, false, 1)
    SG_CASE(4, 0, false, 4, true, 1)
    SG_CASE(4, 4, false, 4, false, 4)
    SG_CASE(4, 1, false, 4, false, 1)
    SG_CASE(1, 0, false, 1, true, 1)
    SG_CASE(1, 4, false, 1, false, 4)
    SG_CASE(1, 1, false, 1, false, 1)
#undef SG_CASE
    return kInvalidArg;
}

}  // namespace libgemm
