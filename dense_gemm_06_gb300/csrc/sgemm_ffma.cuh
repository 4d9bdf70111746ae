// sgemm_ffma.cuh -- the FP32 SIMT GEMM kernel templates (see sgemm_ffma.cu
// for the design). Each tile configuration is instantiated in a translation
// unit of its own (sgemm_cfg<N>.cu) so the library compiles in parallel; the
// templates sit in an anonymous namespace, so every unit keeps private copies.
#pragma once

#include <atomic>
#include <cstdint>

#include "epilogue.cuh"
#include "internal.h"

namespace libgemm {

struct SgemmParams {
    const float* A;
    const float* B;
    float* C;
    int64_t lda, ldb, ldc;
    int M, N, K;
    int tiles_m, tiles_n;
    int c_vec;
    EpiParams epi;  // fused epilogue (inactive for a plain GEMM)
    int dp_tiles;   // tiles 0 .. dp_tiles-1 (raster order) are computed whole
    int splits;     // K-slices of each later tile (one CTA per slice)
    int kt_slice;   // k-tiles per slice
    float* ws;      // raw partial tiles of the slices: [unit][128 * 128 / 4] float4
    unsigned long long* check;  // device-check word (debug build; see internal.h)
};

// Launches configuration N (1..8, as GEMM_OPT_SIMT_CONFIG numbers them) for
// the operand variants av / bv (0 K-major, 4 MN-major 16-byte, 1 MN-major
// 4-byte); defined in sgemm_cfg<N>.cu.
int launch_sgemm_cfg1(const SgemmParams& sp, int av, int bv, int device, int sm_count,
                      int split_mode, Scratch* scratch, cudaStream_t s);
int launch_sgemm_cfg2(const SgemmParams& sp, int av, int bv, int device, int sm_count,
                      int split_mode, Scratch* scratch, cudaStream_t s);
int launch_sgemm_cfg3(const SgemmParams& sp, int av, int bv, int device, int sm_count,
                      int split_mode, Scratch* scratch, cudaStream_t s);
int launch_sgemm_cfg4(const SgemmParams& sp, int av, int bv, int device, int sm_count,
                      int split_mode, Scratch* scratch, cudaStream_t s);
int launch_sgemm_cfg5(const SgemmParams& sp, int av, int bv, int device, int sm_count,
                      int split_mode, Scratch* scratch, cudaStream_t s);
int launch_sgemm_cfg6(const SgemmParams& sp, int av, int bv, int device, int sm_count,
                      int split_mode, Scratch* scratch, cudaStream_t s);
int launch_sgemm_cfg7(const SgemmParams& sp, int av, int bv, int device, int sm_count,
                      int split_mode, Scratch* scratch, cudaStream_t s);
int launch_sgemm_cfg8(const SgemmParams& sp, int av, int bv, int device, int sm_count,
                      int split_mode, Scratch* scratch, cudaStream_t s);

// Chooses the K-split of the tail tiles (defined in sgemm_ffma.cu, with the
// model it uses); fills sp.dp_tiles, sp.splits and sp.kt_slice.
// Plans the tail split (K-slices) of a launch; with sk_ctas non-null (the
// TMA-fed kernel) it may instead plan stream-K and return its CTA count there
// (0: none).
void plan_split(SgemmParams& sp, int slots, int sm_count, int nkt, int split_mode,
                int* sk_ctas = nullptr);

namespace {


constexpr int BM = 128;
constexpr int BN = 128;
constexpr int PAD = 4;
constexpr int LDS = BM + PAD;  // floats per k-row in shared memory (BM == BN)
constexpr int BAND = 16;       // tile rows per raster band (L2 locality)

static_assert(BM == BN, "one shared-memory row stride serves both operands");

// Tile configurations (k-depth, ring depth, packed FMA, CTAs/SM, columns per
// thread). The CuTe Ampere SGEMM example's default is 128 x 128 x 8 with 3
// stages (and 8 x 8 per thread).
template <int BK_, int STAGES_, bool FMA2_, int MINB_, int TN_ = 8>
struct SgCfg {
    static constexpr int BK = BK_;
    static constexpr int STAGES = STAGES_;
    static constexpr bool FMA2 = FMA2_;
    static constexpr int MINB = MINB_;  // CTAs per SM the register budget is sized for
    static constexpr int TN = TN_;      // C columns per thread (8 or 16); rows: 8
    static constexpr int THREADS = BM * BN / (8 * TN_);
    static_assert(TN_ == 8 || TN_ == 16, "8 x 8 or 8 x 16 outputs per thread");
    static constexpr int OPERAND_FLOATS = BK * LDS;
    static constexpr int STAGE_FLOATS = 2 * OPERAND_FLOATS;
    static constexpr int SMEM_BYTES = STAGES * STAGE_FLOATS * 4;
    static_assert(BK % 8 == 0 && BK >= 8, "copy mappings assume BK multiple of 8");
};


// Raster: bands of BAND tile-rows, walking down M inside a band first.
__device__ __forceinline__ void tile_origin(const SgemmParams& p, int t, int& m0, int& n0) {
    const int band_tiles = BAND * p.tiles_n;
    const int band = t / band_tiles;
    const int within = t - band * band_tiles;
    const int m_lo = band * BAND;
    const int rows_in_band = min(BAND, p.tiles_m - m_lo);
    m0 = (m_lo + within % rows_in_band) * BM;
    n0 = (within / rows_in_band) * BN;
}

// Thread -> C block. A warp always spans 4 values of ty and 8 of tx (lane
// (l / 8, l % 8)), so a fragment load reads 4 or 8 consecutive 16-byte units.
// TN = 8: warp (wy, wx) = (w / 2, w % 2), ty in 0..15, tx in 0..15; the
// thread owns rows ty*4 + (i & 3) + (i >> 2) * 64, columns
// tx*4 + (c & 3) + (c >> 2) * 64. TN = 16: warp w covers ty = 4w .. 4w+3,
// tx in 0..7; columns tx*4 + (c & 3) + (c >> 2) * 32.
template <int TN>
__device__ __forceinline__ void thread_block(int tid, int& ty, int& tx) {
    const int w = tid >> 5, l = tid & 31;
    if constexpr (TN == 8) {
        ty = (w >> 1) * 4 + (l >> 3);
        tx = (w & 1) * 8 + (l & 7);
    } else {
        ty = w * 4 + (l >> 3);
        tx = l & 7;
    }
}

// Debug build: true when element (row, col) lies inside C, else records the
// failed check; always true in the default build.
__device__ __forceinline__ bool sg_inside(const SgemmParams& p, int row, int col) {
    return device_check(p.check, row >= 0 && row < p.M && col >= 0 && col < p.N, kCheckSgStore,
                        ((unsigned long long)(uint32_t)row << 24) | (uint32_t)col);
}

// Debug build: checks a CTA's tile origin and K-slice (kt0 .. kt0 + nkt of
// total k-tiles) against the problem.
__device__ __forceinline__ void sg_check_tile(const SgemmParams& p, int m0, int n0, int kt0,
                                              int nkt, int total) {
    device_check(p.check,
                 m0 >= 0 && m0 < p.M && n0 >= 0 && n0 < p.N && kt0 >= 0 && nkt >= 0 &&
                     kt0 + nkt <= total,
                 kCheckSgTile, (unsigned long long)blockIdx.x);
}

// Stores the thread's 8 x TN block of the tile at (m0, n0), applying the
// fused epilogue when one is active; predicated on M and N.
template <int TN>
__device__ __forceinline__ void store_block(const SgemmParams& p, const float2 (&acc)[8][TN / 2],
                                            int m0, int n0, int ty, int tx) {
    constexpr int CSTRIDE = BN / (TN / 4);  // columns between a thread's 4-column groups
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + ty * 4 + (i & 3) + (i >> 2) * 64;
        if (row >= p.M) continue;
        float* crow = p.C + (int64_t)row * p.ldc;
#pragma unroll
        for (int h = 0; h < TN / 4; ++h) {
            const int col = n0 + tx * 4 + h * CSTRIDE;
            float v[4] = {acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x,
                          acc[i][2 * h + 1].y};
            if (p.epi.active) {  // D = act(alpha * acc + beta * C_old + bias)
                float old[4] = {0.f, 0.f, 0.f, 0.f};
                if (p.epi.beta != 0.f) {
                    if (p.c_vec && col + 3 < p.N) {
                        const float4 o = *reinterpret_cast<const float4*>(crow + col);
                        old[0] = o.x; old[1] = o.y; old[2] = o.z; old[3] = o.w;
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (col + j < p.N) old[j] = crow[col + j];
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < p.N) v[j] = epilogue_value<float>(p.epi, v[j], old[j], row, col + j);
            }
            if (p.c_vec && col + 3 < p.N) {
                if (sg_inside(p, row, col + 3))
                    *reinterpret_cast<float4*>(crow + col) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < p.N && sg_inside(p, row, col + j)) crow[col + j] = v[j];
            }
        }
    }
}

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

// Copies BK-deep tiles of one operand (rows r0 .. r0+127) into shared memory
// laid out [k][r] with row stride LDS floats. Each thread keeps one pointer
// that advances by one k-tile per call, a count of the k it has left and a
// mask of its valid rows, so few registers stay live across the main loop.
template <int BK, bool KMAJOR, int VEC, int T>
struct TileLoader {
    static constexpr int KROWS = T / 8;  // K-major: rows one pass covers (8 k each)
    const float* ptr;    // this thread's first element of the next k-tile
    int64_t ld;
    int k_left;          // K minus this thread's first k of the next tile
    int rows_ok;         // K-major: bit q = row q*KROWS valid; MN 16B: valid rows of
                         // the vector; MN 4B: 1 if the row is valid
    uint32_t s_off;      // byte offset of its first element inside a stage

    // k0: first k of the first tile this CTA loads (a multiple of BK).
    __device__ __forceinline__ void init(const float* X, int64_t ld_, int R, int K, int r0,
                                         int k0, int tid) {
        ld = ld_;
        rows_ok = 0;
        if constexpr (KMAJOR) {
            // element e = tid + T i: k-group h = e / 1024, row = (e % 1024) / 8,
            // k = 8 h + e % 8; a thread's rows are tid / 8 + KROWS q.
            const int rr = tid >> 3, kk = tid & 7;
            ptr = X + (int64_t)(r0 + rr) * ld + k0 + kk;
            k_left = K - k0 - kk;
            s_off = (uint32_t)(kk * LDS + rr) * 4u;
#pragma unroll
            for (int q = 0; q < BM / KROWS; ++q) rows_ok |= (r0 + rr + KROWS * q < R) << q;
        } else if constexpr (VEC == 4) {
            // float4 idx = tid + T i: k = tid / 32 + (T / 32) i, rows 4 (tid % 32) ..
            const int rr = (tid & 31) << 2, kk = tid >> 5;
            ptr = X + (int64_t)(k0 + kk) * ld + r0 + rr;
            k_left = K - k0 - kk;
            s_off = (uint32_t)(kk * LDS + rr) * 4u;
            const int v = R - (r0 + rr);
            rows_ok = v >= 4 ? 4 : (v > 0 ? v : 0);
        } else {
            // element e = tid + T i: k = tid / 128 + (T / 128) i, row = tid % 128
            const int rr = tid & 127, kk = tid >> 7;
            ptr = X + (int64_t)(k0 + kk) * ld + r0 + rr;
            k_left = K - k0 - kk;
            s_off = (uint32_t)(kk * LDS + rr) * 4u;
            rows_ok = (r0 + rr < R) ? 1 : 0;
        }
    }

    // Issue the copies of the next k-tile into the stage at byte address s.
    __device__ __forceinline__ void load_next(uint32_t s) {
        if constexpr (KMAJOR) {
            const int64_t ldq = ld * KROWS;
#pragma unroll
            for (int h = 0; h < BK / 8; ++h) {
                const bool k_ok = 8 * h < k_left;
#pragma unroll
                for (int q = 0; q < BM / KROWS; ++q) {
                    const bool ok = k_ok && ((rows_ok >> q) & 1);
                    cp_async_4(s + s_off + (uint32_t)(8 * h * LDS + KROWS * q) * 4u,
                               ptr + q * ldq + 8 * h, ok);
                }
            }
            ptr += BK;
        } else if constexpr (VEC == 4) {
            constexpr int KS = T / 32;  // k-rows one pass covers
#pragma unroll
            for (int i = 0; i < BK / KS; ++i) {
                const bool ok = rows_ok > 0 && KS * i < k_left;
                cp_async_16(s + s_off + (uint32_t)(KS * i * LDS) * 4u, ptr + KS * i * ld,
                            ok ? rows_ok * 4 : 0);
            }
            ptr += BK * ld;
        } else {
            constexpr int KS = T / 128;
#pragma unroll
            for (int i = 0; i < BK / KS; ++i) {
                const bool ok = rows_ok && KS * i < k_left;
                cp_async_4(s + s_off + (uint32_t)(KS * i * LDS) * 4u, ptr + KS * i * ld, ok);
            }
            ptr += BK * ld;
        }
        k_left -= BK;
    }
};

template <class Cfg, bool A_K, int A_VEC, bool B_K, int B_VEC>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MINB) sgemm_ffma_kernel(const SgemmParams p) {
    constexpr int BK = Cfg::BK;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int T = Cfg::THREADS;
    constexpr int TN = Cfg::TN;
    constexpr int NB = TN / 4;           // 4-column groups per thread
    constexpr int CSTEP = BN / NB / 4;   // float4s between a thread's groups
    extern __shared__ __align__(16) float smem[];
    const int tid = threadIdx.x;

    // CTA -> tile (and K-slice for the split tail).
    int t = blockIdx.x, kt0 = 0;
    int nkt = (p.K + BK - 1) / BK;
    if (t >= p.dp_tiles) {
        const int unit = t - p.dp_tiles;
        t = p.dp_tiles + unit / p.splits;
        kt0 = (unit % p.splits) * p.kt_slice;
        nkt = max(0, min(nkt, kt0 + p.kt_slice) - kt0);
    }
    int m0, n0, ty, tx;
    tile_origin(p, t, m0, n0);
    sg_check_tile(p, m0, n0, kt0, nkt, (p.K + BK - 1) / BK);
    thread_block<TN>(tid, ty, tx);

    const uint32_t s0 = smem_addr(smem);

    TileLoader<BK, A_K, A_VEC, T> la;
    TileLoader<BK, B_K, B_VEC, T> lb;
    la.init(p.A, p.lda, p.M, p.K, m0, kt0 * BK, tid);
    lb.init(p.B, p.ldb, p.N, p.K, n0, kt0 * BK, tid);
    // Tiles are issued strictly in order kt = 0, 1, 2, ...
    auto load_stage = [&](int stage) {
        const uint32_t sa = s0 + (uint32_t)(stage * Cfg::STAGE_FLOATS) * 4u;
        la.load_next(sa);
        lb.load_next(sa + (uint32_t)Cfg::OPERAND_FLOATS * 4u);
    };

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < nkt) load_stage(s);
        cp_async_commit();
    }

    // acc[i][jj] holds the C columns (2 jj, 2 jj + 1) of b-index space of
    // row i: packed pairs for the two-lane FMA (fma.rn.f32x2 on sm_100+), or
    // two scalar FMAs; both round each product-sum once (IEEE fma).
    float2 acc[8][TN / 2];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);

    for (int kt = 0; kt < nkt; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();  // tile kt landed; every thread is done with tile kt-1

        const int nt = kt + STAGES - 1;
        if (nt < nkt) load_stage(nt % STAGES);
        cp_async_commit();

        const float* sA = smem + (kt % STAGES) * Cfg::STAGE_FLOATS;
        const float* sB = sA + Cfg::OPERAND_FLOATS;

        // Fully unrolled over the tile's k: the compiler hoists the 128-bit
        // fragment loads of step k+1 above the FMAs of step k as registers
        // allow (an explicit second fragment buffer does not fit next to
        // the accumulators).
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            const float4* pa = reinterpret_cast<const float4*>(sA + k * LDS + ty * 4);
            const float4* pb = reinterpret_cast<const float4*>(sB + k * LDS + tx * 4);
            const float4 a0 = pa[0], a1 = pa[16];
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            float2 b[TN / 2];
#pragma unroll
            for (int g = 0; g < NB; ++g) {
                const float4 q = pb[g * CSTEP];
                b[2 * g] = make_float2(q.x, q.y);
                b[2 * g + 1] = make_float2(q.z, q.w);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
#pragma unroll
                for (int j = 0; j < TN / 2; ++j) {
                    if constexpr (Cfg::FMA2) {
                        acc[i][j] = __ffma2_rn(make_float2(a[i], a[i]), b[j], acc[i][j]);
                    } else {
                        acc[i][j].x = fmaf(a[i], b[j].x, acc[i][j].x);
                        acc[i][j].y = fmaf(a[i], b[j].y, acc[i][j].y);
                    }
                }
            }
        }
    }
    cp_async_wait<0>();

    if ((int)blockIdx.x >= p.dp_tiles) {  // a K-slice of a tail tile: raw partial sums
        const int unit = (int)blockIdx.x - p.dp_tiles;
        float4* wsp = reinterpret_cast<float4*>(p.ws) + (size_t)unit * (BM * BN / 4) + tid;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int h = 0; h < NB; ++h)
                wsp[(NB * i + h) * T] = make_float4(acc[i][2 * h].x, acc[i][2 * h].y,
                                                    acc[i][2 * h + 1].x, acc[i][2 * h + 1].y);
        return;
    }
    store_block<TN>(p, acc, m0, n0, ty, tx);
}

// Tail fixup: tile dp_tiles + blockIdx.x = the sum of its K-slices' partial
// tiles, added in slice order, then the normal epilogue (same thread -> C
// mapping as the main kernel of this TN).
template <int TN>
__global__ void __launch_bounds__(BM * BN / (8 * TN)) sgemm_split_fixup_kernel(
    const SgemmParams p) {
    constexpr int T = BM * BN / (8 * TN);
    constexpr int NB = TN / 4;
    const int tid = threadIdx.x;
    int m0, n0, ty, tx;
    tile_origin(p, p.dp_tiles + blockIdx.x, m0, n0);
    sg_check_tile(p, m0, n0, 0, 0, 0);
    thread_block<TN>(tid, ty, tx);
    const float4* wsp = reinterpret_cast<const float4*>(p.ws) +
                        (size_t)blockIdx.x * p.splits * (BM * BN / 4) + tid;
    float2 acc[8][TN / 2];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int h = 0; h < NB; ++h) {
            const float4 q = wsp[(NB * i + h) * T];
            acc[i][2 * h] = make_float2(q.x, q.y);
            acc[i][2 * h + 1] = make_float2(q.z, q.w);
        }
    for (int sl = 1; sl < p.splits; ++sl) {
        const float4* w = wsp + (size_t)sl * (BM * BN / 4);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int h = 0; h < NB; ++h) {
                const float4 q = w[(NB * i + h) * T];
                acc[i][2 * h].x += q.x;
                acc[i][2 * h].y += q.y;
                acc[i][2 * h + 1].x += q.z;
                acc[i][2 * h + 1].y += q.w;
            }
    }
    store_block<TN>(p, acc, m0, n0, ty, tx);
}

// Sets the dynamic shared-memory limit of `kern` once per device; `done` is
// the calling variant's own flag word (one bit per device).
template <class Kern>
bool configure_once(Kern kern, std::atomic<uint64_t>& done, int device, int smem_bytes) {
    const uint64_t bit = 1ull << (device & 63);
    if (done.load() & bit) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
        cudaSuccess)
        return false;
    done.fetch_or(bit);
    return true;
}

template <class Cfg, bool A_K, int A_VEC, bool B_K, int B_VEC>
int launch_variant(SgemmParams sp, int device, int sm_count, int split_mode, Scratch* scratch,
                   cudaStream_t stream) {
    auto kern = sgemm_ffma_kernel<Cfg, A_K, A_VEC, B_K, B_VEC>;
    static std::atomic<uint64_t> configured{0};  // per kernel variant
    static std::atomic<int> per_sm[64];           // resident CTAs per SM, per device
    if (!configure_once(kern, configured, device, Cfg::SMEM_BYTES)) return kCuda;
    int occ = per_sm[device & 63].load();
    if (occ == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Cfg::THREADS,
                                                          Cfg::SMEM_BYTES) != cudaSuccess) {
            cudaGetLastError();
            occ = -1;
        }
        per_sm[device & 63].store(occ);
    }
    plan_split(sp, occ > 0 ? occ * sm_count : 0, sm_count, (sp.K + Cfg::BK - 1) / Cfg::BK,
               split_mode);
    const int64_t tail = (int64_t)sp.tiles_m * sp.tiles_n - sp.dp_tiles;
    if (tail > 0) {
        const size_t bytes = (size_t)tail * sp.splits * BM * BN * sizeof(float);
        sp.ws = scratch ? static_cast<float*>(scratch->get(bytes)) : nullptr;
        if (!sp.ws) {  // no scratch: compute every tile whole
            sp.dp_tiles = sp.tiles_m * sp.tiles_n;
            sp.splits = 1;
        }
    }
    const int64_t units = sp.dp_tiles + ((int64_t)sp.tiles_m * sp.tiles_n - sp.dp_tiles) * sp.splits;
    kern<<<dim3((unsigned)units), dim3(Cfg::THREADS), Cfg::SMEM_BYTES, stream>>>(sp);
    if (cudaGetLastError() != cudaSuccess) return kCuda;
    note_launch();
    const int64_t fix = (int64_t)sp.tiles_m * sp.tiles_n - sp.dp_tiles;
    if (fix > 0) {
        sgemm_split_fixup_kernel<Cfg::TN>
            <<<dim3((unsigned)fix), dim3(Cfg::THREADS), 0, stream>>>(sp);
        if (cudaGetLastError() != cudaSuccess) return kCuda;
        note_launch();
    }
    return kOk;
}

template <class Cfg>
int launch_layout(const SgemmParams& sp, int av, int bv, int device, int sm_count, int split_mode,
                  Scratch* scratch, cudaStream_t s) {
#define SG_CASE(AV, BV, AK, AVEC, BK_, BVEC)                                                   \
    if (av == AV && bv == BV)                                                                  \
        return launch_variant<Cfg, AK, AVEC, BK_, BVEC>(sp, device, sm_count, split_mode,      \
                                                        scratch, s);
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

}  // namespace
}  // namespace libgemm
