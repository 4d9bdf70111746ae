// softmax_cluster.cu -- numerically stable row softmax, a row per warp, CTA
// or thread-block cluster: y = exp(x - max(x)) / sum(exp(x - max(x))).
//
// After the Gluon Multi-CTA tutorial's multi-CTA softmax, which shards a row
// over up to 16 CTAs and lets the layout system insert the cross-CTA max and
// sum. Every thread keeps its values in registers (one read of x, one write
// of y), so the bandwidth is decided by the bytes each SM keeps in flight:
//  - rows up to 1024 columns: one warp per row, shuffles only;
//  - rows up to 16384 columns (and unaligned rows up to 32768): one CTA of
//    up to 512 threads x 16-64 values, max and sum through shared memory;
//  - longer 16-byte-aligned rows (up to 262144): a cluster of CTAs of 512
//    threads x 32 values (16384 columns, two CTAs per SM); each CTA reduces
//    its slice to a (max, sum of exp(x - max)) pair and pushes it into every
//    peer's shared memory with st.async, completing on the peer's mbarrier,
//    so the row needs one exchange and no cluster barrier after the loads;
//  - other long rows: a cluster of CTAs of 512 threads x 64 values that
//    exchange max, then sum, through distributed shared memory (mapa +
//    ld.shared::cluster) between cluster barriers.
#include <cuda_runtime.h>

#include <atomic>
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
    ErrWord* err;                  // device error word (bounded waits)
    ErrWord gen;                   // this launch's generation (see internal.h)
    unsigned long long wait_limit_ns;
    int fault_inject;              // test hook: row 0's first CTA withholds its partial
};

constexpr int PUSH_MIN_N = 16385;  // aligned rows at least this long: a cluster per row
constexpr int PUSH_THREADS = 512;  // ... of CTAs of PUSH_THREADS threads
constexpr int PUSH_COLS = 16384;   // and up to PUSH_COLS columns

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

// Long aligned rows, one cluster per row: the row is split into cs slices
// of up to PUSH_COLS columns, one per CTA of PUSH_THREADS threads that each
// hold PUSH_COLS / PUSH_THREADS values in registers (all loads issued at
// once, so a CTA keeps its whole slice in flight). Each warp reduces its
// values to a (max, sum of exp(x - max)) pair, the CTA merges its warps'
// pairs, and the CTAs exchange their pairs once: every CTA pushes its pair
// into each peer's slot with st.async, which completes on the peer's
// mbarrier. The only cluster barrier sits before the first push (the peers'
// mbarriers must be initialised) and is split so the loads overlap it.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) softmax_cluster_push_kernel(const SoftmaxParams p) {
    constexpr int EPT = PUSH_COLS / THREADS;
    __shared__ __align__(8) uint64_t xbar;
    __shared__ __align__(8) float2 xslot[MAX_CLUSTER];
    __shared__ float red_m[THREADS / 32], red_s[THREADS / 32];
    __shared__ float row_m_s, row_s_s;
    const int cs = p.cs;
    const int crank = (int)cluster_ctarank();
    const int row = (int)cluster_id_x();
    const int c0 = crank * p.cta_cols;
    const int c1 = min(p.N, c0 + p.cta_cols);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t xb = smem_u32(&xbar);
    if (tid == 0) {
        mbar_init(xb, 1);
        fence_mbarrier_init_cluster();
    }
    cluster_arrive_relaxed();

    const float* xr = p.x + (int64_t)row * p.ldx;
    float v[EPT];
#pragma unroll
    for (int j = 0; j < EPT / 4; ++j) {
        const int col = c0 + 4 * (tid + j * THREADS);
        if (col + 3 < c1) {
            const float4 q = *reinterpret_cast<const float4*>(xr + col);
            v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[4 * j + e] = col + e < c1 ? xr[col + e] : -INFINITY;
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
    st = warp_sum(st);
    if (lane == 0) {
        red_m[warp] = mw;
        red_s[warp] = st;
    }
    __syncthreads();
    cluster_wait();  // every peer's mbarrier is initialised
    if (warp == 0) {
        float m = lane < THREADS / 32 ? red_m[lane] : -INFINITY;
        float s = lane < THREADS / 32 ? red_s[lane] : 0.f;
        warp_ms(m, s);
        bool ok = true;
        if (cs > 1) {
            const bool withhold = p.fault_inject && row == 0 && crank == 0;
            if (lane < cs && !withhold)
                st_async_v2_f32(mapa_shared(smem_u32(&xslot[crank]), (uint32_t)lane), m, s,
                                mapa_shared(xb, (uint32_t)lane));
            if (lane == 0) mbar_arrive_expect_tx(xb, (uint32_t)cs * 8u);
            // bounded wait for every peer's pair
            bool done = false;
            uint32_t n = 0;
            uint64_t t0 = 0;
            while (!(done = mbar_try_wait(xb, 0u))) {
                if ((++n & 31u) == 0) {
                    if (t0 == 0) t0 = globaltimer_ns();
                    if (gen_failed(p.err, p.gen) ||
                        globaltimer_ns() - t0 > p.wait_limit_ns)
                        break;
                }
            }
            ok = __all_sync(0xffffffffu, done);
            m = -INFINITY;
            s = 0.f;
            if (lane < cs) {
                const float2 q = xslot[lane];
                m = q.x;
                s = q.y;
            }
            warp_ms(m, s);
        }
        if (lane == 0) {
            row_m_s = m;
            row_s_s = s;
            if (!ok) gen_record_timeout(p.err, p.gen);
        }
    }
    __syncthreads();
    const float f = mw == -INFINITY ? 0.f : expf(mw - row_m_s) / row_s_s;
    float* yr = p.y + (int64_t)row * p.ldy;
#pragma unroll
    for (int j = 0; j < EPT / 4; ++j) {
        const int col = c0 + 4 * (tid + j * THREADS);
        if (col + 3 < c1) {
            *reinterpret_cast<float4*>(yr + col) =
                make_float4(v[4 * j] * f, v[4 * j + 1] * f, v[4 * j + 2] * f, v[4 * j + 3] * f);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (col + e < c1) yr[col + e] = v[4 * j + e] * f;
        }
    }
}

int launch_push_rows(SoftmaxParams sp, int device, cudaStream_t stream) {
    auto kern = softmax_cluster_push_kernel<PUSH_THREADS>;
    static std::mutex mu;
    static uint64_t configured = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        const uint64_t bit = 1ull << (device & 63);
        if (!(configured & bit)) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                cudaSuccess) {
                cudaGetLastError();
                return kCuda;
            }
            configured |= bit;
        }
    }
    int cs = 1;
    while ((int64_t)cs * PUSH_COLS < sp.N) cs *= 2;
    if ((int64_t)sp.M * cs > 0x7fffffffLL) return kUnsupported;
    sp.cs = cs;
    sp.cta_cols = (int)(((sp.N + cs - 1) / cs + 3) / 4 * 4);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)((int64_t)sp.M * cs));
    cfg.blockDim = dim3(PUSH_THREADS);
    cfg.dynamicSmemBytes = 0;
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

template <int EPT, bool VEC>
int launch_cfg(const SoftmaxParams& sp, int threads, int device, cudaStream_t stream) {
    auto kern = softmax_rows_kernel<EPT, VEC>;
    // The cluster-size attribute belongs to the current device: set it once
    // per device (bit d of `tried`; bit d of `failed` if it was refused).
    static std::atomic<uint64_t> tried{0}, failed{0};
    const uint64_t bit = 1ull << (device & 63);
    if (!(tried.load() & bit)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
            cudaGetLastError();
            failed.fetch_or(bit);
        }
        tried.fetch_or(bit);
    }
    if ((failed.load() & bit) && sp.cs > 8) return kUnsupported;
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
int launch_any(const SoftmaxParams& sp, int ept, int threads, bool warp_rows, int device,
               cudaStream_t s) {
    if (warp_rows) {
        switch (ept) {
            case 4: return launch_warp_rows<4, VEC>(sp, s);
            case 8: return launch_warp_rows<8, VEC>(sp, s);
            case 16: return launch_warp_rows<16, VEC>(sp, s);
            default: return launch_warp_rows<32, VEC>(sp, s);
        }
    }
    if (ept == 16) return launch_cfg<16, VEC>(sp, threads, device, s);
    if (ept == 32) return launch_cfg<32, VEC>(sp, threads, device, s);
    return launch_cfg<64, VEC>(sp, threads, device, s);
}

}  // namespace

int64_t softmax_max_cols() { return (int64_t)MAX_CLUSTER * CL_THREADS * CL_EPT; }

int launch_softmax_rows(int64_t M, int64_t N, const float* x, int64_t ldx, float* y, int64_t ldy,
                        const DeviceInfo& dev, uint64_t wait_limit_ns, int fault_inject,
                        cudaStream_t stream) {
    if (N > softmax_max_cols()) return kUnsupported;
    // Bytes in flight per SM decide the bandwidth: every thread holds 4..64
    // values; short rows run one warp each, medium rows one CTA, long rows a
    // cluster of CTAs (see the top of this file).
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(y) & 15u) == 0 && (ldx & 3) == 0 &&
                     (ldy & 3) == 0;
    SoftmaxParams sp{x, y, ldx, ldy, (int)M, (int)N, 0, 1, dev.err_word, next_generation(),
                     wait_limit_ns, fault_inject};
    if (vec && N >= PUSH_MIN_N && N <= (int64_t)MAX_CLUSTER * PUSH_COLS)
        return launch_push_rows(sp, dev.device, stream);
    if (N <= WARP_ROWS_MAX_N) {
        int ept = 4;
        while (ept * 32 < N) ept *= 2;
        sp.cta_cols = (int)N;
        return vec ? launch_any<true>(sp, ept, 32, true, dev.device, stream)
                   : launch_any<false>(sp, ept, 32, true, dev.device, stream);
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
    return vec ? launch_any<true>(sp, ept, threads, false, dev.device, stream)
               : launch_any<false>(sp, ept, threads, false, dev.device, stream);
}

}  // namespace libgemm
