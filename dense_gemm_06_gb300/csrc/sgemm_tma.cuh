// sgemm_tma.cuh -- the TMA-fed FFMA kernel template (tile configuration 9;
// its launch is in sgemm_cfg9.cu): configuration 7's 128 x 128 tile (128
// threads, 8 x 16 outputs each, packed fma.rn.f32x2, two CTAs per SM) with
// shared memory filled by TMA instead of per-thread cp.async, for operands
// that are MN-major with 16-byte aligned bases and row pitches.
//
//   * one thread (thread 0) issues two 2-D tensor copies per k-tile (A and B
//     boxes of 128 x 16 fp32, rows of 512 bytes, zero fill past M, N and K)
//     into a 6-stage ring; they complete on the stage's `full` mbarrier;
//   * every thread arrives on the stage's `empty` mbarrier once it has read
//     the stage; thread 0 waits for that before refilling it. While the CTA
//     reads k-tile kt, thread 0 loads k-tile kt + 3 into the stage of
//     k-tile kt - 3: three tiles are in flight ahead, and the two stages in
//     between leave slack, so the warp that hosts the producer rarely waits
//     for the slowest warp;
//   * there is no CTA-wide barrier in the main loop: each warp only waits for
//     its data, so the four warps of a CTA may drift apart by up to two
//     k-tiles (measured at 8192^3: 5 stages with one of slack ran 0.8%
//     slower, 7 stages with two or three 1.5% slower, 12 stages of 8-deep
//     k-tiles 7% slower, three CTAs per SM, which spills, 1.5% slower);
//   * every wait is bounded (GEMM_OPT_WAIT_LIMIT_NS): one that runs out
//     records a timeout in the device error word and the thread stops; thread
//     0 then lets its copies in flight land (bounded) before the CTA exits;
//   * sgemm_sk.cuh holds its stream-K variant.
#pragma once

#include <cuda.h>

#include "ptx_sm100.cuh"
#include "sgemm_ffma.cuh"

namespace libgemm {
namespace {

using namespace gemm_ptx;

// A TMA-fed configuration: the tile shape of Cfg, LAG stages of slack
// before a stage is refilled.
template <class Cfg_, int LAG_>
struct TmaCfg {
    using Cfg = Cfg_;
    static constexpr int LAG = LAG_;
    static constexpr int BK = Cfg::BK;
    static constexpr int STAGES = Cfg::STAGES;
    static constexpr int TILE_FLOATS = BK * BM;                 // one operand's k-tile
    static constexpr uint32_t STAGE_BYTES = 2u * TILE_FLOATS * 4u;  // A and B
    static constexpr int SMEM = STAGES * (int)STAGE_BYTES + 2 * STAGES * 8 + 128;
    static_assert(STAGES - 1 - LAG >= 1, "at least one k-tile in flight ahead");
};

struct TmaArgs {
    ErrWord* err;              // device error word
    ErrWord gen;               // this launch's generation (see internal.h)
    unsigned long long limit;  // wait limit, ns
    int fault;                 // test hook: CTA 0 never loads its k-tile 1
};

// Bounded wait on a phase: true when it completed, false on timeout (or when
// another wait of the same launch, generation `gen`, has already failed).
__device__ __noinline__ bool sg_wait_slow(uint32_t bar, uint32_t parity, ErrWord* err,
                                          ErrWord gen, unsigned long long limit) {
    const uint64_t t0 = globaltimer_ns();
    uint32_t n = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++n & 31u) == 0) {
            if (gen_failed(err, gen)) return false;
            if (globaltimer_ns() - t0 > limit) {
                gen_record_timeout(err, gen);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool sg_wait(uint32_t bar, uint32_t parity, const TmaArgs& x) {
    if (mbar_try_wait(bar, parity)) return true;
    return sg_wait_slow(bar, parity, x.err, x.gen, x.limit);
}

// After a failed wait: thread 0 waits (bounded, ignoring the error word) for
// the copies of k-tiles [from, to) it issued, so none lands after the CTA
// has exited.
__device__ __noinline__ void sg_drain(uint32_t full0, int stages, int from, int to, int skipped,
                                      unsigned long long limit) {
    const uint64_t t0 = globaltimer_ns();
    for (int j = from; j < to; ++j) {
        if (j == skipped) continue;  // never issued (test hook)
        const uint32_t bar = full0 + 8u * (uint32_t)(j % stages);
        const uint32_t par = (uint32_t)(j / stages) & 1u;
        while (!mbar_try_wait(bar, par))
            if (globaltimer_ns() - t0 > limit) return;
    }
}

template <class TC>
__global__ void __launch_bounds__(TC::Cfg::THREADS, TC::Cfg::MINB)
    sgemm_ffma_tma_kernel(const SgemmParams p, const __grid_constant__ CUtensorMap tmap_a,
                          const __grid_constant__ CUtensorMap tmap_b, const TmaArgs x) {
    using Cfg = typename TC::Cfg;
    constexpr int TN = Cfg::TN;
    constexpr int NB = TN / 4;           // 4-column groups per thread
    constexpr int CSTEP = BN / NB / 4;   // float4s between a thread's groups
    constexpr int S = TC::STAGES;
    constexpr int LAG = TC::LAG;         // stages of slack before a refill
    constexpr int kTmaBK = TC::BK;
    constexpr int kTileFloats = TC::TILE_FLOATS;
    constexpr uint32_t kStageBytes = TC::STAGE_BYTES;
    extern __shared__ unsigned char smem_raw[];
    const int tid = threadIdx.x;

    // 128-byte aligned ring, then the full and empty barriers.
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 127u) & ~127u;
    const float* ring = reinterpret_cast<const float*>(smem_raw + (base - raw));
    const uint32_t full0 = base + S * kStageBytes, empty0 = full0 + 8u * S;

    // CTA -> tile (and K-slice for the split tail).
    int t = blockIdx.x, kt0 = 0;
    int nkt = (p.K + kTmaBK - 1) / kTmaBK;
    if (t >= p.dp_tiles) {
        const int unit = t - p.dp_tiles;
        t = p.dp_tiles + unit / p.splits;
        kt0 = (unit % p.splits) * p.kt_slice;
        nkt = max(0, min(nkt, kt0 + p.kt_slice) - kt0);
    }
    int m0, n0, ty, tx;
    tile_origin(p, t, m0, n0);
    sg_check_tile(p, m0, n0, kt0, nkt, (p.K + kTmaBK - 1) / kTmaBK);
    thread_block<TN>(tid, ty, tx);

    if (tid == 0) {
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, Cfg::THREADS);
        }
        fence_mbarrier_init_cluster();
        fence_proxy_async_smem();
    }
    __syncthreads();

    // Producer (thread 0): k-tile j of this CTA's range into stage j % S.
    const bool skip_tile1 = x.fault && blockIdx.x == 0;
    auto issue = [&](int j) {
        if (skip_tile1 && j == 1) return;
        const uint32_t s = (uint32_t)(j % S);
        const uint32_t bar = full0 + 8u * s;
        const uint32_t dst = base + s * kStageBytes;
        const int k = (kt0 + j) * kTmaBK;
        mbar_arrive_expect_tx(bar, kStageBytes);
        tma_load_2d<1>(dst, &tmap_a, bar, m0, k);
        tma_load_2d<1>(dst + (uint32_t)kTileFloats * 4u, &tmap_b, bar, n0, k);
    };
    int issued = 0;  // thread 0: k-tiles issued so far
    if (tid == 0) {
        for (; issued < S - 1 - LAG && issued < nkt; ++issued) issue(issued);
    }

    float2 acc[8][TN / 2];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);

    bool ok = true;
    int kt = 0;
    uint32_t s = 0, phase = 0;  // stage and parity of k-tile kt
    for (; kt < nkt; ++kt) {
        if (tid == 0 && issued < nkt) {
            // Refill the stage of k-tile issued - S once every thread has read it.
            if (issued >= S &&
                !sg_wait(empty0 + 8u * (uint32_t)(issued % S),
                         (uint32_t)(issued / S - 1) & 1u, x)) {
                ok = false;
                break;
            }
            issue(issued);
            ++issued;
        }
        if (!sg_wait(full0 + 8u * s, phase, x)) {
            ok = false;
            break;
        }
        const float* sA = ring + s * (2 * kTileFloats);
        const float* sB = sA + kTileFloats;
#pragma unroll
        for (int k = 0; k < kTmaBK; ++k) {
            const float4* pa = reinterpret_cast<const float4*>(sA + k * BM + ty * 4);
            const float4* pb = reinterpret_cast<const float4*>(sB + k * BN + tx * 4);
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
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < TN / 2; ++j)
                    acc[i][j] = __ffma2_rn(make_float2(a[i], a[i]), b[j], acc[i][j]);
        }
        mbar_arrive_local(empty0 + 8u * s);  // this thread is done with the stage
        if (++s == (uint32_t)S) {
            s = 0;
            phase ^= 1u;
        }
    }
    if (!ok) {
        // Thread 0's copies of k-tiles it has issued but not seen land.
        if (tid == 0) sg_drain(full0, S, kt, issued, skip_tile1 ? 1 : -1, x.limit);
        return;
    }

    if ((int)blockIdx.x >= p.dp_tiles) {  // a K-slice of a tail tile: raw partial sums
        const int unit = (int)blockIdx.x - p.dp_tiles;
        float4* wsp = reinterpret_cast<float4*>(p.ws) + (size_t)unit * (BM * BN / 4) + tid;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int h = 0; h < NB; ++h)
                wsp[(NB * i + h) * Cfg::THREADS] =
                    make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x,
                                acc[i][2 * h + 1].y);
        return;
    }
    store_block<TN>(p, acc, m0, n0, ty, tx);
}

}  // namespace
}  // namespace libgemm
