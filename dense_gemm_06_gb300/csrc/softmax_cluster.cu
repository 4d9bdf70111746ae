// softmax_cluster.cu -- numerically stable row softmax, one row per thread-block
// cluster: y = exp(x - max(x)) / sum(exp(x - max(x))).
//
// After the Gluon Multi-CTA tutorial's multi-CTA softmax, which shards a row
// over up to 16 CTAs and lets the layout system insert the cross-CTA max and
// sum: here the row is split into CS contiguous slices (CS = cluster size, a
// power of two up to 16; one CTA holds up to 32768 columns), each CTA keeps its
// slice in registers (EPT values
// per thread, one read of x), reduces max and sum across its warps through
// shared memory, and the CTAs exchange their partial max and sum through
// distributed shared memory (mapa + ld.shared::cluster) between cluster
// barriers. Memory traffic is one read of x and one write of y.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx_sm100.cuh"

namespace libgemm {
namespace {

using namespace gemm_ptx;

constexpr int MAX_CLUSTER = 16;
constexpr int MAX_THREADS = 512;   // per CTA of a one-CTA row
constexpr int MAX_EPT = 32;        // values per thread of a one-CTA row
constexpr int CL_THREADS = 512;    // per CTA of a long row (one CTA up to 32768 columns,
constexpr int CL_EPT = 64;         // then a cluster): 64 values per thread
constexpr int WARP_ROWS_MAX_N = 1024;  // rows up to this length: one warp per row

struct SoftmaxParams {
    const float* x;
    float* y;
    int64_t ldx, ldy;
    int M, N;
    int cta_cols;  // columns per CTA (a multiple of 4)
    int cs;        // CTAs per row (cluster size)
    unsigned int* err;             // device error word (persistent kernel's waits)
    unsigned long long wait_limit_ns;
    int nbuf;                      // persistent kernel: ring slots of cta_cols floats
};

constexpr int PC_THREADS = 512;   // persistent cluster kernel: CTA size
constexpr int PC_MAX_NBUF = 8;    // shared-memory ring: this row and up to 7 ahead
constexpr int PC_MIN_N = 32769;   // rows at least this long take the persistent kernel
// Its two shapes: 8192 columns per CTA (16 per thread, <= 64 registers and a
// 96 KB ring, two CTAs per SM), or 16384 (32 per thread, a 192 KB ring, one
// CTA per SM) for rows that 16 CTAs of 8192 columns do not cover.
template <int EPT>
struct PcShape {
    static constexpr int COLS = PC_THREADS * EPT;
    static constexpr int MINB = EPT <= 16 ? 2 : 1;
    static constexpr int RING_BYTES = (MINB == 2 ? 96 : 192) * 1024;
};

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide reduction into *out (max or sum), using red[] as scratch.
template <bool MAX>
__device__ __forceinline__ void block_reduce(float v, float* red, float* out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = (blockDim.x + 31) >> 5;
    v = MAX ? warp_max(v) : warp_sum(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float t = lane < nw ? red[lane] : (MAX ? -INFINITY : 0.f);
        t = MAX ? warp_max(t) : warp_sum(t);
        if (lane == 0) *out = t;
    }
}

// Combine one partial per CTA of the cluster (the `slot` variable of every
// CTA) into *out: lanes of warp 0 read the peers' slots through distributed
// shared memory. Must follow a cluster barrier that published the slots.
template <bool MAX>
__device__ __forceinline__ void cluster_combine(const float* slot, int cs, float* out) {
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        float t = MAX ? -INFINITY : 0.f;
        if (lane < cs) t = ld_cluster_f32(mapa_shared(smem_u32(slot), (uint32_t)lane));
        t = MAX ? warp_max(t) : warp_sum(t);
        if (lane == 0) *out = t;
    }
    __syncthreads();
}

// Short rows: one warp per row, 8 rows per CTA, reductions by shuffles only.
template <int EPT, bool VEC>
__global__ void __launch_bounds__(256) softmax_warp_rows_kernel(const SoftmaxParams p) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= p.M) return;
    const float* xr = p.x + (int64_t)row * p.ldx;
    float* yr = p.y + (int64_t)row * p.ldy;
    float v[EPT];
#pragma unroll
    for (int j = 0; j < EPT / 4; ++j) {
        const int col = 4 * (lane + 32 * j);
        if (VEC && col + 3 < p.N) {
            const float4 q = *reinterpret_cast<const float4*>(xr + col);
            v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[4 * j + e] = col + e < p.N ? xr[col + e] : -INFINITY;
        }
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPT; ++i) m = fmaxf(m, v[i]);
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
        v[i] = expf(v[i] - m);
        s += v[i];
    }
    const float inv = 1.f / warp_sum(s);
#pragma unroll
    for (int j = 0; j < EPT / 4; ++j) {
        const int col = 4 * (lane + 32 * j);
        if (VEC && col + 3 < p.N) {
            *reinterpret_cast<float4*>(yr + col) =
                make_float4(v[4 * j] * inv, v[4 * j + 1] * inv, v[4 * j + 2] * inv,
                            v[4 * j + 3] * inv);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (col + e < p.N) yr[col + e] = v[4 * j + e] * inv;
        }
    }
}

template <int EPT, bool VEC>
__global__ void __launch_bounds__(MAX_THREADS) softmax_rows_kernel(const SoftmaxParams p) {
    __shared__ float red[32];
    __shared__ float cta_max, cta_sum, row_max, row_sum;
    const int cs = p.cs;
    const uint32_t crank = cs > 1 ? cluster_ctarank() : 0u;
    const int row = cs > 1 ? (int)cluster_id_x() : (int)blockIdx.x;
    const int c0 = (int)crank * p.cta_cols;
    const int c1 = min(p.N, c0 + p.cta_cols);
    const float* xr = p.x + (int64_t)row * p.ldx;
    float* yr = p.y + (int64_t)row * p.ldy;
    const int T = blockDim.x;

    // this thread's values: 16-byte chunks t, t + T, ... of the slice
    float v[EPT];
#pragma unroll
    for (int j = 0; j < EPT / 4; ++j) {
        const int col = c0 + 4 * ((int)threadIdx.x + j * T);
        if (VEC && col + 3 < c1) {
            const float4 q = *reinterpret_cast<const float4*>(xr + col);
            v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[4 * j + e] = col + e < c1 ? xr[col + e] : -INFINITY;
        }
    }

    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPT; ++i) m = fmaxf(m, v[i]);
    block_reduce<true>(m, red, &cta_max);
    if (cs > 1) cluster_sync_all(); else __syncthreads();
    if (cs > 1) cluster_combine<true>(&cta_max, cs, &row_max);
    const float mx = cs > 1 ? row_max : cta_max;

    float s = 0.f;
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
        v[i] = expf(v[i] - mx);  // masked entries: exp(-inf) = 0
        s += v[i];
    }
    block_reduce<false>(s, red, &cta_sum);
    if (cs > 1) cluster_sync_all(); else __syncthreads();
    if (cs > 1) cluster_combine<false>(&cta_sum, cs, &row_sum);
    const float inv = 1.f / (cs > 1 ? row_sum : cta_sum);

#pragma unroll
    for (int j = 0; j < EPT / 4; ++j) {
        const int col = c0 + 4 * ((int)threadIdx.x + j * T);
        if (VEC && col + 3 < c1) {
            *reinterpret_cast<float4*>(yr + col) =
                make_float4(v[4 * j] * inv, v[4 * j + 1] * inv, v[4 * j + 2] * inv,
                            v[4 * j + 3] * inv);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (col + e < c1) yr[col + e] = v[4 * j + e] * inv;
        }
    }
    // peers may still be reading this CTA's partials
    if (cs > 1) cluster_sync_all();
}

// Merges the softmax partial (m2, s2) into (m, s): m is a maximum, s a sum
// of exp(x - m) over the same values; an empty partial is (-inf, 0).
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2) {
    const float mx = fmaxf(m, m2);
    s = mx == -INFINITY ? 0.f : s * expf(m - mx) + s2 * expf(m2 - mx);
    m = mx;
}

__device__ __forceinline__ void warp_ms(float& m, float& s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        ms_merge(m, s, m2, s2);
    }
}

// Long rows, persistent: a cluster of `cs` CTAs walks the rows cid, cid +
// #clusters, ...; CTA k owns columns [k * cta_cols, (k+1) * cta_cols).
//  - Loads: one thread issues 1-D TMA bulk copies of the CTA's slices of the
//    next nbuf - 1 rows into an nbuf-slot shared-memory ring, so HBM reads
//    stay in flight across rows.
//  - Reduction: each warp reduces its values to a (max, sum of exp(x - max))
//    pair, the CTA merges its warps' pairs (rescaling each sum to the common
//    maximum), and pushes the result into every peer's exchange slot with
//    st.async, which completes on the peer's own mbarrier. No cluster barrier
//    (whose release would wait for the previous row's stores of y) sits on
//    the per-row path. The exponentials held in registers are then scaled by
//    exp(m_warp - m_row) / s_row and stored.
// Exchange slots and barriers are double-buffered by row parity: a CTA
// pushes row i + 2's pair only after its peers have all pushed row i + 1's,
// which each of them does after reading its slots of row i.
template <int EPT>
__global__ void __launch_bounds__(PC_THREADS, PcShape<EPT>::MINB)
    softmax_cluster_persistent_kernel(const SoftmaxParams p) {
    extern __shared__ __align__(128) float sbuf[];  // [nbuf][cta_cols]
    __shared__ __align__(8) uint64_t bars[PC_MAX_NBUF];
    __shared__ __align__(8) uint64_t xbars[2];
    __shared__ __align__(8) float2 xslot[2][MAX_CLUSTER];
    __shared__ float red_m[PC_THREADS / 32], red_s[PC_THREADS / 32];
    __shared__ float row_m_s, row_s_s;
    __shared__ int xfail_s;
    const int cs = p.cs, nbuf = p.nbuf;
    const int crank = (int)cluster_ctarank();
    const int cid = (int)cluster_id_x(), ncl = (int)num_clusters_x();
    const int c0 = crank * p.cta_cols;
    const int c1 = min(p.N, c0 + p.cta_cols);
    const int nbulk = c1 > c0 ? (c1 - c0) / 4 * 4 : 0;  // bulk-copied part (x 4 bytes % 16)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t bar0 = smem_u32(&bars[0]);
    const uint32_t xbar0 = smem_u32(&xbars[0]);
    const uint32_t buf0 = smem_u32(sbuf);

    if (tid == 0) {
        for (int k = 0; k < nbuf; ++k) mbar_init(bar0 + 8u * k, 1);
        mbar_init(xbar0, 1);
        mbar_init(xbar0 + 8u, 1);
        fence_mbarrier_init_cluster();
    }
    cluster_sync_all();  // peers' exchange barriers are initialised before any push

    // Bounded wait on an mbarrier phase: false once the limit passes or
    // another kernel has already reported an error.
    auto wait_bar = [&](uint32_t bar, uint32_t parity) {
        uint32_t n = 0;
        uint64_t t0 = 0;
        while (!mbar_try_wait(bar, parity)) {
            if ((++n & 31u) == 0) {
                if (t0 == 0) t0 = globaltimer_ns();
                if (*reinterpret_cast<volatile unsigned int*>(p.err) != kDevErrNone ||
                    globaltimer_ns() - t0 > p.wait_limit_ns)
                    return false;
            }
        }
        return true;
    };
    // Thread 0 only: ring slots holding a copy not yet waited for.
    bool pend[PC_MAX_NBUF] = {};
    uint32_t pend_parity[PC_MAX_NBUF] = {};
    bool failed = false;
    // Iteration `it` uses ring slot it % nbuf; its (it / nbuf)-th fill
    // completes that phase of the slot's barrier.
    auto issue = [&](int row, int it) {
        const int k = it % nbuf;
        if (tid == 0 && nbulk > 0 && !failed) {
            fence_proxy_async_smem();  // the generic-proxy reads of the slot come first
            mbar_arrive_expect_tx(bar0 + 8u * k, (uint32_t)nbulk * 4u);
            bulk_load_1d(buf0 + (uint32_t)(k * p.cta_cols) * 4u, p.x + (int64_t)row * p.ldx + c0,
                         (uint32_t)nbulk * 4u, bar0 + 8u * k);
            pend[k] = true;
            pend_parity[k] = (uint32_t)((it / nbuf) & 1);
        }
    };

    for (int d = 0; d < nbuf - 1; ++d)
        if (cid + d * ncl < p.M) issue(cid + d * ncl, d);
    int i = 0;
    for (int row = cid; row < p.M; row += ncl, ++i) {
        const int k = i % nbuf;
        // the slot of iteration i + nbuf - 1 was released in iteration i - 1
        if (row + (nbuf - 1) * ncl < p.M) issue(row + (nbuf - 1) * ncl, i + nbuf - 1);
        if (nbulk > 0 && !failed) {
            if (wait_bar(bar0 + 8u * k, (uint32_t)((i / nbuf) & 1))) {
                if (tid == 0) pend[k] = false;
            } else {
                atomicCAS(p.err, kDevErrNone, kDevErrTimeout);
                failed = true;
            }
        }
        // every thread takes the same path; a failed CTA reads x directly
        failed = __syncthreads_or(failed);
        float v[EPT];
        const float* sb = sbuf + k * p.cta_cols;
        const float* xr = p.x + (int64_t)row * p.ldx;
#pragma unroll
        for (int j = 0; j < EPT / 4; ++j) {
            const int off = 4 * (tid + j * PC_THREADS);  // column c0 + off
            if (!failed && off + 3 < nbulk) {
                const float4 q = *reinterpret_cast<const float4*>(sb + off);
                v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    v[4 * j + e] = c0 + off + e < c1 ? xr[c0 + off + e] : -INFINITY;
            }
        }

        float mw = -INFINITY;
#pragma unroll
        for (int e = 0; e < EPT; ++e) mw = fmaxf(mw, v[e]);
        mw = warp_max(mw);
        const float shift = mw == -INFINITY ? 0.f : mw;  // all-padding warp: exp(-inf) = 0
        float st = 0.f;
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
            v[e] = expf(v[e] - shift);
            st += v[e];
        }
        float m = mw, s = warp_sum(st);
        if (lane == 0) {
            red_m[warp] = m;
            red_s[warp] = s;
        }
        __syncthreads();  // also releases ring slot k for refilling
        if (warp == 0) {
            m = lane < PC_THREADS / 32 ? red_m[lane] : -INFINITY;
            s = lane < PC_THREADS / 32 ? red_s[lane] : 0.f;
            warp_ms(m, s);
            bool ok = true;
            if (cs > 1) {
                const int b = i & 1;
                const uint32_t xb = xbar0 + 8u * b;
                if (lane < cs)
                    st_async_v2_f32(mapa_shared(smem_u32(&xslot[b][crank]), (uint32_t)lane), m, s,
                                    mapa_shared(xb, (uint32_t)lane));
                if (lane == 0) mbar_arrive_expect_tx(xb, (uint32_t)cs * 8u);
                ok = __all_sync(0xffffffffu, wait_bar(xb, (uint32_t)((i >> 1) & 1)));
                m = -INFINITY;
                s = 0.f;
                if (lane < cs) {
                    const float2 q = xslot[b][lane];
                    m = q.x;
                    s = q.y;
                }
                warp_ms(m, s);
            }
            if (lane == 0) {
                row_m_s = m;
                row_s_s = s;
                xfail_s = ok ? 0 : 1;
                if (!ok) atomicCAS(p.err, kDevErrNone, kDevErrTimeout);
            }
        }
        __syncthreads();
        if (xfail_s) break;  // a peer stopped answering: give up on the remaining rows
        const float f = mw == -INFINITY ? 0.f : expf(mw - row_m_s) / row_s_s;
        float* yr = p.y + (int64_t)row * p.ldy;
#pragma unroll
        for (int j = 0; j < EPT / 4; ++j) {
            const int col = c0 + 4 * (tid + j * PC_THREADS);
            if (col + 3 < c1) {
                *reinterpret_cast<float4*>(yr + col) =
                    make_float4(v[4 * j] * f, v[4 * j + 1] * f, v[4 * j + 2] * f,
                                v[4 * j + 3] * f);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (col + e < c1) yr[col + e] = v[4 * j + e] * f;
            }
        }
    }
    if (tid == 0) {  // after a failure, let copies still in flight land before the CTA exits
        for (int k = 0; k < nbuf; ++k)
            if (pend[k]) wait_bar(bar0 + 8u * k, pend_parity[k]);
    }
    cluster_sync_all();  // no CTA leaves while a peer may still push into it
}

template <int EPT>
int launch_persistent(SoftmaxParams sp, int device, int sm_count, cudaStream_t stream) {
    using S = PcShape<EPT>;
    auto kern = softmax_cluster_persistent_kernel<EPT>;
    const int smem = sp.nbuf * sp.cta_cols * 4;
    static std::mutex mu;
    static uint64_t configured = 0;
    static int max_clusters[64][MAX_CLUSTER + 1];
    int nclusters;
    {
        std::lock_guard<std::mutex> lock(mu);
        const uint64_t bit = 1ull << (device & 63);
        if (!(configured & bit)) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     S::RING_BYTES) != cudaSuccess ||
                cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                    cudaSuccess) {
                cudaGetLastError();
                return kCuda;
            }
            for (int c = 0; c <= MAX_CLUSTER; ++c) max_clusters[device & 63][c] = 0;
            configured |= bit;
        }
        int& mc = max_clusters[device & 63][sp.cs];
        if (mc == 0) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = sp.cs;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(sp.cs * (sm_count * S::MINB / sp.cs));
            cfg.blockDim = dim3(PC_THREADS);
            cfg.dynamicSmemBytes = S::RING_BYTES;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int q = 0;
            if (cudaOccupancyMaxActiveClusters(&q, kern, &cfg) != cudaSuccess || q < 1) {
                cudaGetLastError();
                q = sm_count / sp.cs;
            }
            mc = q > 0 ? q : 1;
        }
        nclusters = mc;
    }
    if (nclusters > sp.M) nclusters = sp.M;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sp.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(sp.cs * nclusters);
    cfg.blockDim = dim3(PC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, sp) != cudaSuccess) {
        cudaGetLastError();
        return kCuda;
    }
    note_launch();
    return kOk;
}

// Chooses the persistent kernel's shape for rows of N columns (N <= 16 *
// 16384): the smallest cluster of 8192-column CTAs, else of 16384-column CTAs.
int launch_persistent_rows(SoftmaxParams sp, int device, int sm_count, cudaStream_t stream) {
    const int64_t N = sp.N;
    int cs = 1;
    while ((int64_t)cs * PcShape<16>::COLS < N) cs *= 2;
    const bool small = cs <= MAX_CLUSTER;
    if (!small) {
        cs = 1;
        while ((int64_t)cs * PcShape<32>::COLS < N) cs *= 2;
    }
    sp.cs = cs;
    sp.cta_cols = (int)(((N + cs - 1) / cs + 3) / 4 * 4);
    const int ring = small ? PcShape<16>::RING_BYTES : PcShape<32>::RING_BYTES;
    sp.nbuf = std::min(PC_MAX_NBUF, ring / (sp.cta_cols * 4));
    return small ? launch_persistent<16>(sp, device, sm_count, stream)
                 : launch_persistent<32>(sp, device, sm_count, stream);
}

template <int EPT, bool VEC>
int launch_cfg(const SoftmaxParams& sp, int threads, cudaStream_t stream) {
    auto kern = softmax_rows_kernel<EPT, VEC>;
    static std::once_flag once;
    static bool ok = true;
    std::call_once(once, [&] {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
            cudaGetLastError();
            ok = false;
        }
    });
    if (!ok && sp.cs > 8) return kUnsupported;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sp.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)((int64_t)sp.M * sp.cs));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = sp.cs > 1 ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, sp) != cudaSuccess) {
        cudaGetLastError();
        return kCuda;
    }
    note_launch();
    return kOk;
}

template <int EPT, bool VEC>
int launch_warp_rows(const SoftmaxParams& sp, cudaStream_t stream) {
    softmax_warp_rows_kernel<EPT, VEC><<<(unsigned)((sp.M + 7) / 8), 256, 0, stream>>>(sp);
    if (cudaGetLastError() != cudaSuccess) return kCuda;
    note_launch();
    return kOk;
}

template <bool VEC>
int launch_any(const SoftmaxParams& sp, int ept, int threads, bool warp_rows, cudaStream_t s) {
    if (warp_rows) {
        switch (ept) {
            case 4: return launch_warp_rows<4, VEC>(sp, s);
            case 8: return launch_warp_rows<8, VEC>(sp, s);
            case 16: return launch_warp_rows<16, VEC>(sp, s);
            default: return launch_warp_rows<32, VEC>(sp, s);
        }
    }
    if (ept == 16) return launch_cfg<16, VEC>(sp, threads, s);
    if (ept == 32) return launch_cfg<32, VEC>(sp, threads, s);
    return launch_cfg<64, VEC>(sp, threads, s);
}

}  // namespace

int64_t softmax_max_cols() { return (int64_t)MAX_CLUSTER * CL_THREADS * CL_EPT; }

int launch_softmax_rows(int64_t M, int64_t N, const float* x, int64_t ldx, float* y, int64_t ldy,
                        const DeviceInfo& dev, uint64_t wait_limit_ns, cudaStream_t stream) {
    if (N > softmax_max_cols()) return kUnsupported;
    // Bytes in flight per SM decide the bandwidth: every thread holds 4..32
    // values; short rows run one warp each, medium rows one CTA of <= 512
    // threads x 16-32 values, long rows a cluster of such CTAs.
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(y) & 15u) == 0 && (ldx & 3) == 0 &&
                     (ldy & 3) == 0;
    SoftmaxParams sp{x, y, ldx, ldy, (int)M, (int)N, 0, 1, dev.err_word, wait_limit_ns};
    if (vec && N >= PC_MIN_N && N <= (int64_t)MAX_CLUSTER * PcShape<32>::COLS)
        return launch_persistent_rows(sp, dev.device, dev.sm_count, stream);
    if (N <= WARP_ROWS_MAX_N) {
        int ept = 4;
        while (ept * 32 < N) ept *= 2;
        sp.cta_cols = (int)N;
        return vec ? launch_any<true>(sp, ept, 32, true, stream)
                   : launch_any<false>(sp, ept, 32, true, stream);
    }
    int cs = 1;
    while ((int64_t)cs * CL_THREADS * CL_EPT < N) cs *= 2;
    if ((int64_t)M * cs > 0x7fffffffLL) return kUnsupported;
    sp.cs = cs;
    sp.cta_cols = (int)(((N + cs - 1) / cs + 3) / 4 * 4);
    const int ept = sp.cta_cols <= 16 * MAX_THREADS ? 16
                    : (sp.cta_cols <= 32 * MAX_THREADS ? 32 : CL_EPT);
    int threads = (sp.cta_cols + ept - 1) / ept;
    threads = (threads + 31) / 32 * 32;
    return vec ? launch_any<true>(sp, ept, threads, false, stream)
               : launch_any<false>(sp, ept, threads, false, stream);
}

}  // namespace libgemm
