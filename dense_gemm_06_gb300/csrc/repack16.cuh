// repack16.cuh -- copies rows of 16-bit elements whose starts have any 2-byte
// alignment into rows that start on 16-byte boundaries (what TMA needs), for
// the tensor-core path's misaligned operands (gemm_api.cu into pool scratch,
// gemm_noalloc.cu into the library's fixed array).
//
// A warp copies one row at a time. Each lane builds 16-byte groups of 8
// elements: it loads the two aligned 16-byte source chunks that hold the
// group (aligned vector loads, so a group costs two loads instead of eight
// 2-byte ones), shifts them by the row's byte offset and stores the group
// with one 16-byte store. Both chunks always hold at least one byte of the
// row, so no load touches an aligned 16-byte block the row does not reach.
// The last inner % 8 elements of a row are copied one by one.
#pragma once

#include <cstdint>

#include "ptx_sm100.cuh"

namespace libgemm {
namespace {

// One operand: `outer` rows of `inner` elements, row pitch `lds` elements in
// src and `ldd` in dst (dst rows 16-byte aligned: ldd a multiple of 8 and dst
// 16-byte aligned). outer == 0: nothing to copy.
struct Repack16 {
    const uint16_t* src;
    uint16_t* dst;
    int64_t lds, ldd, outer, inner;
};

// Bytes [off, off + 16) of the 32 bytes lo | hi (off even, 0..14, the same
// for every lane of the warp).
__device__ __forceinline__ uint4 shift_bytes(const uint4& lo, const uint4& hi, uint32_t off) {
    uint32_t w[5];
    switch (off >> 2) {
        case 0: w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w; w[4] = hi.x; break;
        case 1: w[0] = lo.y; w[1] = lo.z; w[2] = lo.w; w[3] = hi.x; w[4] = hi.y; break;
        case 2: w[0] = lo.z; w[1] = lo.w; w[2] = hi.x; w[3] = hi.y; w[4] = hi.z; break;
        default: w[0] = lo.w; w[1] = hi.x; w[2] = hi.y; w[3] = hi.z; w[4] = hi.w; break;
    }
    const uint32_t sh = (off & 3u) * 8u;  // 0 or 16
    return make_uint4(__funnelshift_r(w[0], w[1], sh), __funnelshift_r(w[1], w[2], sh),
                      __funnelshift_r(w[2], w[3], sh), __funnelshift_r(w[3], w[4], sh));
}

__device__ __forceinline__ void repack16_row(const uint16_t* __restrict__ src,
                                             uint16_t* __restrict__ dst, int64_t inner, int lane) {
    const uintptr_t s = reinterpret_cast<uintptr_t>(src);
    const uint4* __restrict__ chunk = reinterpret_cast<const uint4*>(s & ~(uintptr_t)15);
    const uint32_t off = (uint32_t)(s & 15u);  // even
    const int64_t groups = inner / 8;
    constexpr int U = 4;  // groups per lane in flight
    int64_t g = lane;
    for (; g + 32 * (U - 1) < groups; g += 32 * U) {
        uint4 lo[U], hi[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            lo[i] = chunk[g + 32 * i];
            // the group's bytes reach into the next chunk only when off > 0
            hi[i] = off ? chunk[g + 32 * i + 1] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < U; ++i)
            *reinterpret_cast<uint4*>(dst + 8 * (g + 32 * i)) = shift_bytes(lo[i], hi[i], off);
    }
    for (; g < groups; g += 32) {
        const uint4 lo = chunk[g];
        const uint4 hi = off ? chunk[g + 1] : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(dst + 8 * g) = shift_bytes(lo, hi, off);
    }
    for (int64_t c = 8 * groups + lane; c < inner; c += 32) dst[c] = src[c];
}

// Repacks up to two operands in one launch: warp w of the grid takes rows w,
// w + (warps in the grid), ... of a's rows followed by b's.
__global__ void __launch_bounds__(256) repack16_kernel(const Repack16 a, const Repack16 b) {
    // the GEMM launched after this may set itself up meanwhile (it waits for
    // this grid to complete before it reads the repacked rows)
    gemm_ptx::pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    const int64_t rows = a.outer + b.outer;
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < rows;
         r += warps) {
        const bool in_a = r < a.outer;
        const Repack16& j = in_a ? a : b;
        const int64_t rr = in_a ? r : r - a.outer;
        repack16_row(j.src + rr * j.lds, j.dst + rr * j.ldd, j.inner, lane);
    }
}

// Blocks of 256 threads for `rows` rows (a warp per row), at most 8 per SM.
inline int repack16_blocks(int64_t rows, int sm_count) {
    const int64_t want = (rows + 7) / 8, cap = (int64_t)sm_count * 8;
    return (int)(want < 1 ? 1 : (want > cap ? cap : want));
}

}  // namespace
}  // namespace libgemm
