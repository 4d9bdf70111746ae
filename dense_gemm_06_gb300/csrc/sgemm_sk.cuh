// sgemm_sk.cuh -- the stream-K variant of the TMA-fed FFMA kernel (its
// launch is in sgemm_cfg9.cu; the plan is plan_stream_k in policy.h).
//
// Stream-K shares the k-iterations of tiles evenly over the CTAs instead of
// giving each CTA whole tiles, so every SM gets the same work when the tiles
// do not divide evenly over them (fp32 2048^3: 256 tiles on 152 SMs).
//
//   * iteration (tile t, k-tile k) = (t - dp_tiles) * nkt + k; stream-K CTA g
//     takes iterations [g I / G, (g + 1) I / G) of the I iterations, at most
//     one tile's worth: the end of one tile and, when the range runs on, the
//     head of the next;
//   * it computes the head first and publishes it: raw partial sums in its
//     workspace slot, then a flag (release, gpu scope) holding a token of the
//     launch's generation;
//   * the CTA whose range reaches a tile's last k-tile owns the tile: after
//     its own k-tiles it waits (acquire, bounded by GEMM_OPT_WAIT_LIMIT_NS)
//     for the flags of the lower-index CTAs that cover the tile's earlier
//     k-tiles, adds their partial sums to its accumulators and runs the normal
//     epilogue -- no separate fixup kernel. An owner only waits for CTAs with
//     lower indices, which publish before they wait on anything, so the waits
//     end as long as CTAs are started in index order.
//
// It is a kernel of its own because folding the segment logic into the
// whole-tile kernel measured 1.2% slower at 8192^3 even where it was compiled
// out.
#pragma once

#include "sgemm_tma.cuh"

namespace libgemm {
namespace {

// Stream-K arguments: the CTAs sharing the iterations, and their flags (a
// u64 each, in the workspace after the partial tiles).
struct SkArgs {
    int ctas;
    unsigned long long* flags;
};

// Stream-K flags: CTA c of launch `gen` has published its partial tile when
// its flag holds sk_token(gen). Generations never repeat, so flags left over
// from earlier launches (or whatever the pool memory held) never match
// except by a 2^-64 coincidence of the mixed value.
__device__ __forceinline__ unsigned long long sk_token(ErrWord gen) {
    return (unsigned long long)gen ^ 0x5bd1e9955bd1e995ull;
}

__device__ __forceinline__ void sk_publish(unsigned long long* flag, ErrWord gen) {
    __threadfence();  // the CTA's partial sums (ordered by the barrier before) first
    asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(flag), "l"(sk_token(gen))
                 : "memory");
}

// Bounded wait for a flag (thread 0 of the owner): true when it was set;
// false when the wait ran out (recorded in the error word) or another wait of
// the launch already failed.
__device__ __forceinline__ bool sk_wait(const unsigned long long* flag, ErrWord gen,
                                     const TmaArgs& x) {
    const unsigned long long want = sk_token(gen);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(flag) : "memory");
        if (v == want) return true;
        if ((n & 31u) == 0) {
            if (gen_failed(x.err, gen)) return false;
            if (globaltimer_ns() - t0 > x.limit) {
                gen_record_timeout(x.err, gen);
                return false;
            }
        }
    }
}

// The stream-K variant of sgemm_ffma_tma_kernel (the same tile, ring and
// waits): CTAs 0 .. dp_tiles-1 compute whole tiles; the others share the
// later tiles' k-iterations evenly, each taking one contiguous range of at
// most one tile's worth.
template <class TC>
__global__ void __launch_bounds__(TC::Cfg::THREADS, TC::Cfg::MINB)
    sgemm_ffma_tma_sk_kernel(const SgemmParams p, const __grid_constant__ CUtensorMap tmap_a,
                             const __grid_constant__ CUtensorMap tmap_b, const TmaArgs x,
                             const SkArgs k) {
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

    // CTA -> tile, or stream-K range.
    int t = blockIdx.x, kt0 = 0;
    const int nkt_tile = (p.K + kTmaBK - 1) / kTmaBK;
    int nkt = nkt_tile;  // k-tiles this CTA computes (over all its segments)
    const bool sk = (int)blockIdx.x >= p.dp_tiles;
    // stream-K: this CTA's iterations [it0, it0 + nkt) of the stream-K tiles
    // (tile t, k-tile k = iteration (t - dp_tiles) * nkt_tile + k, relative),
    // split evenly over the stream-K CTAs: at most one tile's worth. It covers
    // the end of tile t from k-tile kt0 (n_in_t k-tiles) and, when it runs on,
    // the head of tile t + 1 (n_head k-tiles).
    int n_head = 0;
    const int skg = (int)blockIdx.x - p.dp_tiles;  // stream-K CTA index
    int64_t I = 0;                                // stream-K iterations in all
    if (sk) {
        I = ((int64_t)p.tiles_m * p.tiles_n - p.dp_tiles) * nkt_tile;
        const int64_t it0 = (int64_t)skg * I / k.ctas;
        nkt = (int)((int64_t)(skg + 1) * I / k.ctas - it0);
        t = p.dp_tiles + (int)(it0 / nkt_tile);
        kt0 = (int)(it0 % nkt_tile);
        n_head = max(0, kt0 + nkt - nkt_tile);
    }
    int m0, n0, ty, tx;
    tile_origin(p, t, m0, n0);
    thread_block<TN>(tid, ty, tx);
    // stream-K order: the head of tile t + 1 first (it belongs to a later CTA,
    // which waits for it), then the part of tile t
    int mh = 0, nh = 0;
    if (n_head > 0) tile_origin(p, t + 1, mh, nh);
    sg_check_tile(p, m0, n0, kt0, nkt - n_head, nkt_tile);
    if (n_head > 0) sg_check_tile(p, mh, nh, 0, n_head, nkt_tile);

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

    // Producer (thread 0): k-tile j of this CTA's range into stage j % S
    // (stream-K: the range may continue into the next tile).
    const bool skip_tile1 = x.fault && blockIdx.x == 0;
    auto issue = [&](int j) {
        if (skip_tile1 && j == 1) return;
        const uint32_t s = (uint32_t)(j % S);
        const uint32_t bar = full0 + 8u * s;
        const uint32_t dst = base + s * kStageBytes;
        int mj = m0, nj = n0, kj = kt0 + j;
        if (j < n_head) {  // stream-K: the head of tile t + 1 comes first
            mj = mh;
            nj = nh;
            kj = j;
        } else {
            kj -= n_head;
        }
        const int k = kj * kTmaBK;
        mbar_arrive_expect_tx(bar, kStageBytes);
        tma_load_2d<1>(dst, &tmap_a, bar, mj, k);
        tma_load_2d<1>(dst + (uint32_t)kTileFloats * 4u, &tmap_b, bar, nj, k);
    };
    int issued = 0;  // thread 0: k-tiles issued so far
    if (tid == 0) {
        for (; issued < S - 1 - LAG && issued < nkt; ++issued) issue(issued);
    }

    float2 acc[8][TN / 2];
    bool ok = true;
    int kt = 0;
    uint32_t s = 0, phase = 0;  // stage and parity of k-tile kt
    // Segments: one (a whole tile or a K-slice), or for stream-K the head of
    // tile t + 1 (published) then the part of tile t.
    int seg_end = n_head > 0 ? n_head : nkt;
    for (int seg = 0;; ++seg) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);
    const int seg_begin = kt;
    for (; kt < seg_end; ++kt) {
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
    if (!sk) break;  // a whole tile: the epilogue below
    // stream-K. The CTA whose range reaches the end of a tile owns it: the
    // CTAs before it that cover the tile's earlier k-tiles publish their raw
    // partial sums (workspace slot g) and a flag; the owner waits for those
    // flags -- only lower-index CTAs, which publish before they wait on
    // anything -- adds their partials to its own and runs the epilogue.
    const bool head = seg == 0 && n_head > 0;
    const bool owner = !head && kt0 + (kt - seg_begin) == nkt_tile;
    if (!owner) {
        float4* wsp = reinterpret_cast<float4*>(p.ws) + (size_t)skg * (BM * BN / 4) + tid;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int h = 0; h < NB; ++h)
                wsp[(NB * i + h) * Cfg::THREADS] =
                    make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x,
                                acc[i][2 * h + 1].y);
        __syncthreads();  // every thread's partial sums are written
        if (tid == 0) sk_publish(k.flags + skg, x.gen);
        if (kt >= nkt) return;
        seg_end = nkt;  // after the head: the part of tile t
        continue;
    }
    {
        if (kt0 > 0) {  // earlier k-tiles of tile t are other CTAs' partials
            // relative first iteration of tile t; the CTA holding relative
            // iteration r is the last c with c * I / sk_ctas <= r
            const int64_t first = (int64_t)(t - p.dp_tiles) * nkt_tile;
            const int g0 = (int)(((first + 1) * k.ctas - 1) / I);
            if (tid == 0)
                for (int c = g0; c < skg && ok; ++c)
                    ok = sk_wait(k.flags + c, x.gen, x);
            ok = __syncthreads_and(ok);
            if (!ok) return;  // a wait ran out (recorded in the error word)
            for (int c = g0; c < skg; ++c) {
                const float4* w = reinterpret_cast<const float4*>(p.ws) +
                                  (size_t)c * (BM * BN / 4) + tid;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float4 q[NB];
#pragma unroll
                    for (int h = 0; h < NB; ++h) q[h] = __ldcg(w + (NB * i + h) * Cfg::THREADS);
#pragma unroll
                    for (int h = 0; h < NB; ++h) {
                        acc[i][2 * h].x += q[h].x;
                        acc[i][2 * h].y += q[h].y;
                        acc[i][2 * h + 1].x += q[h].z;
                        acc[i][2 * h + 1].y += q[h].w;
                    }
                    // keeps the loads of the next row group after these adds,
                    // so only NB loaded vectors are live next to the accumulators
                    __syncwarp();
                }
            }
        }
        break;  // the owner's tile, complete: the epilogue below (its last segment)
    }
    }

    // a whole tile, or a stream-K tile its owner has completed
    store_block<TN>(p, acc, m0, n0, ty, tx);
}

}  // namespace
}  // namespace libgemm
