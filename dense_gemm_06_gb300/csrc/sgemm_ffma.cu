// sgemm_ffma.cu -- FP32 SIMT GEMM on the FFMA pipe, C = A * B^T, C row-major.
//
// Design follows the CuTe DSL Ampere SGEMM example (SGemm.__call__ / kernel)
// re-done by hand for sm_103a:
//   * CTA tile 128 x 128 x BK, 256 threads, each thread owning an 8 x 8 block
//     of C as four 4 x 4 quadrants (4 consecutive rows x 4 consecutive columns
//     in each 64 x 64 sub-tile), so fragments load with 128-bit LDS; or 128
//     threads owning 8 x 16 blocks (rows as above, columns in four groups of
//     4 spaced 32 apart), which loads 24 fragment values per 128 FMAs
//     instead of 16 per 64 and so needs a third fewer shared-memory reads;
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
//   * predicated epilogue with 128-bit stores when C allows them;
//   * wave tail: when the last wave of CTAs would leave at least half of the
//     CTA slots idle, the tiles of that wave are split along K into `splits`
//     slices computed by separate CTAs, which store raw partial sums in pool
//     scratch; a fixup kernel adds the slices in slice order and runs the
//     normal epilogue, so the last wave takes 1/splits of the time.
#include <cstdint>

#include "policy.h"
#include "sgemm_ffma.cuh"

namespace libgemm {
namespace {

// dst[c * ldd + r] = src[r * lds + c] for r < rows, c < cols: turns a K-major
// fp32 operand into an MN-major copy (32 x 32 tiles through padded shared
// memory; every warp reads and writes 128 contiguous bytes).
__global__ void __launch_bounds__(256) transpose_f32_kernel(const float* __restrict__ src,
                                                            int64_t lds, float* __restrict__ dst,
                                                            int64_t ldd, int rows, int cols) {
    __shared__ float t[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int tiles_c = (cols + 31) >> 5;
    const int64_t tiles = (int64_t)((rows + 31) >> 5) * tiles_c;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int r0 = (int)(tile / tiles_c) * 32, c0 = (int)(tile % tiles_c) * 32;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = r0 + ty + 8 * j, c = c0 + tx;
            if (r < rows && c < cols) t[ty + 8 * j][tx] = src[(int64_t)r * lds + c];
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + ty + 8 * j, r = r0 + tx;
            if (r < rows && c < cols) dst[(int64_t)c * ldd + r] = t[tx][ty + 8 * j];
        }
        __syncthreads();
    }
}

bool aligned16(const void* p, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && (ld & 3) == 0;
}

}  // namespace

// Chooses the K-split of the tail tiles, or (kernels that support it) a
// stream-K share of them (the models are plan_tail_split's and
// plan_stream_k's, in policy.h).
void plan_split(SgemmParams& sp, int slots, int sm_count, int nkt, int split_mode,
                int* sk_ctas) {
    const int64_t T = (int64_t)sp.tiles_m * sp.tiles_n;
    if (sk_ctas) {
        *sk_ctas = 0;
        const StreamK s = plan_stream_k(T, slots, sm_count, nkt, split_mode);
        if (s.sk_ctas > 0) {
            sp.dp_tiles = s.dp_tiles;
            sp.splits = 1;
            sp.kt_slice = nkt;
            *sk_ctas = s.sk_ctas;
            return;
        }
    }
    const TailSplit t = plan_tail_split(T, slots, sm_count, nkt, split_mode == 3 ? 1 : split_mode);
    sp.dp_tiles = t.dp_tiles;
    sp.splits = t.splits;
    sp.kt_slice = t.kt_slice;
}

int launch_transpose_f32(const float* src, int64_t lds, float* dst, int64_t ldd, int64_t rows,
                         int64_t cols, const DeviceInfo& dev, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return kOk;
    if (rows > 0x7fffffffLL || cols > 0x7fffffffLL) return kUnsupported;
    const int64_t tiles = ((rows + 31) / 32) * ((cols + 31) / 32);
    const int64_t cap = (int64_t)dev.sm_count * 8;
    const int grid = (int)(tiles < cap ? tiles : cap);
    transpose_f32_kernel<<<grid, 256, 0, stream>>>(src, lds, dst, ldd, (int)rows, (int)cols);
    if (cudaGetLastError() != cudaSuccess) return kCuda;
    note_launch();
    return kOk;
}

// Configuration 9: configuration 7's tile with TMA-fed shared memory when
// both operands are MN-major and 16-byte aligned (sgemm_cfg9.cu).
int launch_sgemm_cfg9(const SgemmParams& sp, int av, int bv, const DeviceInfo& dev,
                      int split_mode, Scratch* scratch, uint64_t wait_limit_ns, int fault_inject,
                      cudaStream_t s);

int launch_sgemm_f32(const Problem& pr, const DeviceInfo& dev, int config, int split_mode,
                     Scratch* scratch, uint64_t wait_limit_ns, int fault_inject,
                     cudaStream_t stream) {
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
    sp.epi = pr.epi;
    sp.dp_tiles = 0;
    sp.splits = 1;
    sp.kt_slice = 0;
    sp.ws = nullptr;
    sp.check = dev.check_word;
    if ((int64_t)sp.tiles_m * sp.tiles_n > 0x3fffffffLL) return kUnsupported;

    // A/B variant: K-major (4-byte transposing copies), MN-major 16-byte or 4-byte.
    const int av = pr.a_kmajor ? 0 : (aligned16(pr.A, pr.lda) ? 4 : 1);
    const int bv = pr.b_kmajor ? 0 : (aligned16(pr.B, pr.ldb) ? 4 : 1);
    const int d = dev.device, n = dev.sm_count;
    if (config != 9)
        dispatch_log("FFMA SGEMM (cp.async) %dx%dx%d: configuration %d, %d x %d tiles of 128 x 128, "
                     "A %s, B %s",
                     sp.M, sp.N, sp.K, config < 1 || config > 8 ? 1 : config, sp.tiles_m,
                     sp.tiles_n, av == 0 ? "K-major" : "MN-major",
                     bv == 0 ? "K-major" : "MN-major");
    switch (config) {
        case 2: return launch_sgemm_cfg2(sp, av, bv, d, n, split_mode, scratch, stream);
        case 3: return launch_sgemm_cfg3(sp, av, bv, d, n, split_mode, scratch, stream);
        case 4: return launch_sgemm_cfg4(sp, av, bv, d, n, split_mode, scratch, stream);
        case 5: return launch_sgemm_cfg5(sp, av, bv, d, n, split_mode, scratch, stream);
        case 6: return launch_sgemm_cfg6(sp, av, bv, d, n, split_mode, scratch, stream);
        case 7: return launch_sgemm_cfg7(sp, av, bv, d, n, split_mode, scratch, stream);
        case 8: return launch_sgemm_cfg8(sp, av, bv, d, n, split_mode, scratch, stream);
        case 9:
            return launch_sgemm_cfg9(sp, av, bv, dev, split_mode, scratch, wait_limit_ns,
                                     fault_inject, stream);
        default: return launch_sgemm_cfg1(sp, av, bv, d, n, split_mode, scratch, stream);
    }
}

}  // namespace libgemm
