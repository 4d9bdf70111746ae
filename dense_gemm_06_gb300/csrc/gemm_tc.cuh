// gemm_tc.cuh -- the tcgen05 GEMM kernel templates (see gemm_tc.cu for the
// design). Each element type is instantiated in a translation unit of its
// own (gemm_tc_<in>_<out>.cu) so the library compiles in parallel; the
// templates sit in an anonymous namespace, so every unit keeps private copies.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "epilogue.cuh"
#include "internal.h"
#include "policy.h"
#include "ptx_sm100.cuh"

namespace libgemm {

struct TcParams {
    CUtensorMap tmap_a;
    CUtensorMap tmap_b;        // K-major B: a CTA's whole share of a tile per box;
                               // N-major B: 64-column boxes
    CUtensorMap tmap_b_half;   // K-major B: the share of a half-width unit
    CUtensorMap tmap_c;        // valid when c_tma
    int c_tma;                 // C stored with TMA (16-byte aligned base and rows)
    void* C;
    int64_t ldc;
    int M, N, K;
    int tiles_m, tiles_n, num_kb;
    int tile_n;                // columns of a tile: 256, 128 or 64 (>= 64 * CG)
    int split_from;            // tiles from this raster index on run as two half-width
                               // units (== tiles_m * tiles_n: none)
    int split_mode;            // host only: GEMM_OPT_TC_SPLIT_TAIL, resolved at launch
    int pdl;                   // host only: launched as a programmatic dependent of the
                               // kernel before it on the stream
    int c_vec;                 // C base / ldc allow 16-byte stores
    ErrWord* err;              // device error word
    unsigned long long* check; // device-check word (debug build; see internal.h)
    ErrWord gen;               // this launch's generation (see internal.h)
    unsigned long long wait_limit_ns;
    int fault_inject;          // test hook: 1 = epilogue waits on a barrier nobody arrives at
    int clc;                   // 1: one cluster per tile, later tiles taken by try_cancel
    EpiParams epi;             // fused epilogue (inactive for a plain GEMM)
#ifdef LIBGEMM_TC_TRACE
    unsigned long long* trace;  // debug build: per-CTA phase timestamps (64 per CTA)
#endif
};

// Phase timestamps of the debug build (-DLIBGEMM_TC_TRACE): %globaltimer at
// fixed points of every role, 64 slots per CTA, for reading the kernel's
// timeline on the host. Compiled out of the library.
#ifdef LIBGEMM_TC_TRACE
#define TC_TRACE(p, slot)                                                              \
    do {                                                                               \
        if ((p).trace && (slot) < 64)                                                  \
            (p).trace[(size_t)blockIdx.x * 64 + (slot)] = gemm_ptx::globaltimer_ns();  \
    } while (0)
#else
#define TC_TRACE(p, slot) \
    do {                  \
    } while (0)
#endif

// Launches the kernel variant for CTA group cg (1 or 2), operand multicast mc
// and the operand majors; defined in gemm_tc_<in>_<out>.cu.
int launch_gemm_tc_f16_f32(TcParams& tp, int cg, bool mc, bool a_mn, bool b_mn,
                       const DeviceInfo& dev, cudaStream_t s);
int launch_gemm_tc_bf16_f32(TcParams& tp, int cg, bool mc, bool a_mn, bool b_mn,
                       const DeviceInfo& dev, cudaStream_t s);
int launch_gemm_tc_f16_f16(TcParams& tp, int cg, bool mc, bool a_mn, bool b_mn,
                       const DeviceInfo& dev, cudaStream_t s);
int launch_gemm_tc_bf16_bf16(TcParams& tp, int cg, bool mc, bool a_mn, bool b_mn,
                       const DeviceInfo& dev, cudaStream_t s);

namespace {


using namespace gemm_ptx;

constexpr int BK = 64;           // k per stage: 64 x 16-bit = one 128-byte swizzle row
constexpr int UMMA_K = 16;       // k per tcgen05.mma (kind::f16)
constexpr int TILE_N = 256;      // widest tile (per CTA pair when CG == 2): sizes the smem ring
constexpr int ROWS_A = 128;      // A rows per CTA (= TMEM lanes)
constexpr int ACC_COLS = 256;    // TMEM columns per accumulator
constexpr int TMEM_COLS = 512;   // two accumulators
constexpr int EPI_WARP0 = 4;     // epilogue warps 4..11 (warp % 4 == TMEM lane quarter)
constexpr int EPI_WARPS = 8;     // two per TMEM lane quarter, each storing half the chunks
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
constexpr int BAND = 8;          // tile rows per raster band
constexpr int CLC_SLOTS = 3;     // cluster-launch-control responses in flight

template <int CG> struct Cfg {
    static constexpr int B_ROWS = TILE_N / CG;            // B rows (N) held per CTA
    static constexpr int A_BYTES = ROWS_A * BK * 2;       // 16 KB
    static constexpr int B_BYTES = B_ROWS * BK * 2;       // 16 KB (CG 2) / 32 KB (CG 1)
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = CG == 2 ? 6 : 4;
    static constexpr int TILE_M = ROWS_A * CG;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    // barriers: full[S], empty[S], acc_full[2], acc_empty[2], drain, never,
    // clc_ready[CLC_SLOTS], clc_consumed[CLC_SLOTS], then the TMEM address
    // slot, padding, and the 16-byte CLC responses
    static constexpr int NUM_BARS = 2 * STAGES + 6 + 2 * CLC_SLOTS;
    static constexpr int RESP_OFFSET = (NUM_BARS * 8 + 8 + 15) / 16 * 16;
    static constexpr int BAR_BYTES = RESP_OFFSET + 16 * CLC_SLOTS;
    // epilogue staging: one 32 x 128-byte tile per epilogue warp
    static constexpr int EPI_BYTES = EPI_WARPS * 32 * 128;
    static constexpr int SMEM_BYTES = RING_BYTES + EPI_BYTES + BAR_BYTES + 1024;  // + align slack
    static_assert(SMEM_BYTES <= 232448, "over the 227 KB of shared memory a CTA may use");
};


struct TileCoord {
    int tm, tn;
};

__device__ __forceinline__ TileCoord raster(int t, int tiles_m, int tiles_n) {
    const int band_tiles = BAND * tiles_n;
    const int band = t / band_tiles;
    const int within = t - band * band_tiles;
    const int m_lo = band * BAND;
    const int rows = min(BAND, tiles_m - m_lo);
    TileCoord c;
    c.tm = m_lo + within % rows;
    c.tn = within / rows;
    if (band & 1) c.tn = tiles_n - 1 - c.tn;
    return c;
}

// Bounded wait: true when the phase completed, false on timeout, or when
// another wait of the same launch (generation `gen`) has already run out.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, ErrWord* err, ErrWord gen,
                                       unsigned long long limit) {
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

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const TcParams& p) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, p.err, p.gen, p.wait_limit_ns);
}

// One lane of the (converged) warp: the issuing lane of the producer and MMA
// roles, whose loops the whole warp runs so that their state stays
// warp-uniform (TMA and MMA operands are taken from uniform registers).
__device__ __forceinline__ bool elect_one() {
    uint32_t e;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(e));
    return e != 0;
}

// Bounded wait taken by every lane of a warp; the outcome is warp-uniform.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const TcParams& p) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, p));
}

// Spin (bounded by time, no barrier) to let in-flight async copies land.
__device__ __noinline__ void grace_period_ns(uint64_t ns) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < ns) {
    }
}

// Debug build: true when element (row, col) lies inside C, else records the
// failed check; always true in the default build.
__device__ __forceinline__ bool c_inside(const TcParams& p, int row, int col) {
    return device_check(p.check, row >= 0 && row < p.M && col >= 0 && col < p.N, kCheckTcStore,
                        ((unsigned long long)(uint32_t)row << 24) | (uint32_t)col);
}

// Shared-memory helpers for the epilogue staging tile.
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(a), "r"(x), "r"(y), "r"(z),
                 "r"(w) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
    return v;
}

// Epilogue staging tile of one warp: 32 rows of 32 elements, ROW_BYTES =
// 32 * sizeof(OutT) bytes each; 16-byte unit u of row r sits at unit
// u ^ swz(r). swz is the TMA swizzle pattern of the row width -- 128-byte
// swizzle (r & 7) for fp32 rows, 64-byte swizzle ((r >> 1) & 3) for 16-bit
// rows -- so the tile can be TMA-stored as is, and with it the row-wise
// writes (a quarter-warp = 8 rows, one unit each) and the column-wise reads
// of the st.global path are free of bank conflicts.
template <int ESIZE>
__device__ __forceinline__ int swz(int r) {
    if constexpr (ESIZE == 4) return r & 7;
    else return (r >> 1) & 3;
}

// The chunk with the fused epilogue: the fp32 accumulators are staged as is
// (128-byte rows, 128-byte swizzle pattern) and the epilogue is applied while
// reading the tile back row-wise, so C_old, bias and the store are coalesced
// and a 16-bit C is rounded once, after the epilogue.
template <typename OutT>
__device__ __forceinline__ void store_chunk_epi(const TcParams& p, uint32_t stage, int lane,
                                                int row0, int col0, const uint32_t (&v)[32]) {
    const uint32_t my_row = stage + (uint32_t)lane * 128u;
#pragma unroll
    for (int u = 0; u < 8; ++u)
        sts128(my_row + (uint32_t)((u ^ (lane & 7)) * 16), v[4 * u], v[4 * u + 1], v[4 * u + 2],
               v[4 * u + 3]);
    __syncwarp();
    const int u = lane & 7;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int r = 4 * j + (lane >> 3);
        const uint4 raw = lds128(stage + (uint32_t)r * 128u + (uint32_t)((u ^ (r & 7)) * 16));
        float f[4] = {__uint_as_float(raw.x), __uint_as_float(raw.y), __uint_as_float(raw.z),
                      __uint_as_float(raw.w)};
        const int grow = row0 + r, gcol = col0 + 4 * u;
        if (grow >= p.M) continue;
        OutT* dst = static_cast<OutT*>(p.C) + (int64_t)grow * p.ldc + gcol;
        if (p.c_vec && gcol + 3 < p.N) {
            if (!c_inside(p, grow, gcol + 3)) continue;
            float old[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (sizeof(OutT) == 4) {
                if (p.epi.beta != 0.f) {
                    const float4 o = *reinterpret_cast<const float4*>(dst);
                    old[0] = o.x; old[1] = o.y; old[2] = o.z; old[3] = o.w;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    f[e] = epilogue_value<OutT>(p.epi, f[e], old[e], grow, gcol + e);
                *reinterpret_cast<float4*>(dst) = make_float4(f[0], f[1], f[2], f[3]);
            } else {
                if (p.epi.beta != 0.f) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) old[e] = to_f32(dst[e]);
                }
                OutT o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = from_f32<OutT>(epilogue_value<OutT>(p.epi, f[e], old[e], grow, gcol + e));
                uint2 pk;
                pk.x = (uint32_t)(*reinterpret_cast<uint16_t*>(&o[0])) |
                       ((uint32_t)(*reinterpret_cast<uint16_t*>(&o[1])) << 16);
                pk.y = (uint32_t)(*reinterpret_cast<uint16_t*>(&o[2])) |
                       ((uint32_t)(*reinterpret_cast<uint16_t*>(&o[3])) << 16);
                *reinterpret_cast<uint2*>(dst) = pk;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (gcol + e >= p.N || !c_inside(p, grow, gcol + e)) continue;
                const float old = p.epi.beta != 0.f ? to_f32(dst[e]) : 0.f;
                dst[e] = from_f32<OutT>(epilogue_value<OutT>(p.epi, f[e], old, grow, gcol + e));
            }
        }
    }
    __syncwarp();  // the tile is rewritten by the next chunk
}

// Writes one 32 x 32 chunk of C: thread `lane` holds row (row0 + lane),
// columns col0 .. col0+31 in v[]. The chunk goes through the warp's staging
// tile and leaves it either by one TMA store (C rows 16-byte aligned and the
// chunk entirely inside C) or row by row with st.global (16-byte vectors when
// C's rows allow, coalesced predicated scalars otherwise), so every store
// writes whole row segments of C.
template <typename OutT>
__device__ __forceinline__ void store_chunk(const TcParams& p, uint32_t stage, int lane, int row0,
                                            int col0, const uint32_t (&v)[32]) {
    constexpr int ES = (int)sizeof(OutT);
    constexpr int ROW_BYTES = 32 * ES;
    if (p.epi.active) {
        store_chunk_epi<OutT>(p, stage, lane, row0, col0, v);
        return;
    }
    if (p.c_tma) {
        // the previous chunk's TMA store must have finished reading the tile
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
    }
    const uint32_t my_row = stage + (uint32_t)(lane * ROW_BYTES);
    if constexpr (ES == 4) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
            sts128(my_row + (uint32_t)((u ^ swz<4>(lane)) * 16), v[4 * u], v[4 * u + 1],
                   v[4 * u + 2], v[4 * u + 3]);
    } else {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float lo = __uint_as_float(v[2 * i]), hi = __uint_as_float(v[2 * i + 1]);
            if constexpr (std::is_same<OutT, __nv_bfloat16>::value) {
                __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
                pk[i] = *reinterpret_cast<uint32_t*>(&h2);
            } else {
                __half2 h2 = __floats2half2_rn(lo, hi);
                pk[i] = *reinterpret_cast<uint32_t*>(&h2);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            sts128(my_row + (uint32_t)((u ^ swz<2>(lane)) * 16), pk[4 * u], pk[4 * u + 1],
                   pk[4 * u + 2], pk[4 * u + 3]);
    }
    // TMA only for chunks entirely inside C; edge chunks take the st.global
    // path below, so no store ever relies on clipping at the edges of C.
    if (p.c_tma && row0 + 32 <= p.M && col0 + 32 <= p.N &&
        device_check(p.check, (col0 * ES) % 16 == 0 && row0 >= 0, kCheckTcTmaX,
                     (unsigned long long)(uint32_t)col0)) {
        fence_proxy_async_smem();  // make the tile visible to the TMA engine
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(&p.tmap_c, stage, col0, row0);
            bulk_commit_group();
        }
        return;
    }
    __syncwarp();
    constexpr int PER_UNIT = 16 / ES;           // elements per 16-byte unit
    constexpr int UNITS = 32 / PER_UNIT;        // 16-byte units per row
    constexpr int ROWS_PER_PASS = 32 / UNITS;
    // Rows of this chunk inside C, and the chunk's first row in C (as bytes).
    const int rows = min(32, p.M - row0);
    const int64_t step = p.ldc * ES;
    if (p.c_vec && col0 + 32 <= p.N) {
        const int u = lane % UNITS;
        char* dst = reinterpret_cast<char*>(p.C) +
                    ((int64_t)(row0 + lane / UNITS) * p.ldc + col0 + u * PER_UNIT) * ES;
#pragma unroll
        for (int j = 0; j < 32 / ROWS_PER_PASS; ++j) {
            const int r = j * ROWS_PER_PASS + lane / UNITS;
            const uint4 val =
                lds128(stage + (uint32_t)(r * ROW_BYTES) + (uint32_t)((u ^ swz<ES>(r)) * 16));
            if (r < rows && c_inside(p, row0 + r, col0 + u * PER_UNIT + PER_UNIT - 1))
                *reinterpret_cast<uint4*>(dst) = val;
            dst += ROWS_PER_PASS * step;
        }
    } else {
        // Lane = column; one coalesced row segment per store. Everything that
        // does not change from row to row is computed once: the lane's shared
        // offset for each of the 8 swizzle phases, the row pointer (advanced
        // by the row pitch) and the row bound. The shared loads of 8 rows are
        // issued together before their stores, so their latencies overlap.
        const int col = col0 + lane;
        const bool col_ok = col < p.N;
        const int u = lane / PER_UNIT, e = lane % PER_UNIT;
        uint32_t xs[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) xs[k] = stage + (uint32_t)(((u ^ k) * 16) + e * ES);
        char* dst = reinterpret_cast<char*>(p.C) + ((int64_t)row0 * p.ldc + col) * ES;
#pragma unroll
        for (int rb = 0; rb < 32; rb += 8) {
            uint32_t val[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t a = xs[swz<ES>(rb + i)] + (uint32_t)((rb + i) * ROW_BYTES);
                if constexpr (ES == 4) val[i] = lds32(a);
                else val[i] = lds16(a);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (rb + i < rows && col_ok && c_inside(p, row0 + rb + i, col)) {
                    if constexpr (ES == 4) *reinterpret_cast<uint32_t*>(dst) = val[i];
                    else *reinterpret_cast<uint16_t*>(dst) = (uint16_t)val[i];
                }
                dst += step;
            }
        }
    }
    __syncwarp();  // the tile is rewritten by the next chunk
}

template <int CG, bool MC, bool A_MN, bool B_MN, bool BF16, typename OutT>
__global__ void __launch_bounds__(THREADS, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
    using C_ = Cfg<CG>;
    // MC: a cluster holds two CTA pairs computing vertically adjacent tiles
    // that share their B columns; the rank-h CTA of each pair loads half of
    // B-half h and multicasts it to the rank-h CTAs of both pairs.
    static_assert(!MC || CG == 2, "operand multicast runs on CTA pairs");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 128-byte swizzle atoms must sit on 1024-byte boundaries.
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);

    const uint32_t sA0 = base;
    const uint32_t sB0 = base + C_::STAGES * C_::A_BYTES;
    const uint32_t epi0 = base + C_::RING_BYTES;
    const uint32_t bar0 = epi0 + C_::EPI_BYTES;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C_::STAGES + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * C_::STAGES + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * C_::STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * C_::STAGES + 4);
    const uint32_t never_bar = bar0 + 8u * (2 * C_::STAGES + 5);  // nothing ever arrives
    auto ready_bar = [&](int s) { return bar0 + 8u * (2 * C_::STAGES + 6 + s); };
    auto cons_bar = [&](int s) { return bar0 + 8u * (2 * C_::STAGES + 6 + CLC_SLOTS + s); };
    auto resp_addr = [&](int s) { return bar0 + (uint32_t)(C_::RESP_OFFSET + 16 * s); };
    uint32_t* tmem_slot =
        reinterpret_cast<uint32_t*>(smem + C_::RING_BYTES + C_::EPI_BYTES + 8 * C_::NUM_BARS);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) TC_TRACE(p, 0);
    // The next launch on the stream may set itself up meanwhile; it waits
    // for this grid to complete before it touches global memory.
    pdl_launch_dependents();
    const uint32_t crank = CG == 2 ? cluster_ctarank() : 0u;  // rank in the cluster
    const uint32_t rank = crank & (uint32_t)(CG - 1);          // rank in the CTA pair
    const int pair = MC ? (int)(crank >> 1) : 0;               // pair in the cluster
    const uint32_t lead = crank & ~(uint32_t)(CG - 1);         // cluster rank of the pair leader
    const bool leader = rank == 0;
    const int cluster = CG == 2 ? (int)cluster_id_x() : (int)blockIdx.x;
    const int nclusters = CG == 2 ? (int)num_clusters_x() : (int)gridDim.x;
    // Tiles (or, MC, pairs of vertically adjacent tiles) in raster order; the
    // tiles from split_from on are each run as two work units of half the
    // width, so a last, partial round of tiles takes half as long.
    const int unit_rows = MC ? (p.tiles_m + 1) / 2 : p.tiles_m;
    const int total_tiles = unit_rows * p.tiles_n;
    const int total_units = p.split_from + 2 * (total_tiles - p.split_from);
    struct Unit {
        int tm;     // tile row
        int col0;   // first column of C
        int width;  // columns (a multiple of 64 * CG)
    };
    auto unit_of = [&](int u) {
        int t = u, off = 0, w = p.tile_n;
        if (u >= p.split_from) {
            const int v = u - p.split_from;
            t = p.split_from + (v >> 1);
            w = p.tile_n >> 1;
            off = (v & 1) * w;
        }
        const TileCoord tc = raster(t, unit_rows, p.tiles_n);
        Unit un;
        un.tm = MC ? tc.tm * 2 + pair : tc.tm;  // MC: may be past the last tile row (all OOB)
        un.col0 = tc.tn * p.tile_n + off;
        un.width = w;
        device_check(p.check,
                     un.tm >= 0 && un.tm < (MC ? 2 * unit_rows : p.tiles_m) && un.col0 >= 0 &&
                         un.col0 % 64 == 0 && un.col0 + un.width <= p.tiles_n * p.tile_n,
                     kCheckTcUnit, (unsigned long long)u);
        return un;
    };
    // Next unit of a role (t = total_units: no more work). Static schedule:
    // every nclusters-th unit. CLC: the j-th response of the scheduler ring
    // (the unit of a cluster it cancelled), which the role then releases to
    // the pair leader's consumed barrier. warp_wide: all lanes of the warp
    // call it and one arrives. False when a wait ran out.
    auto advance = [&](int& t, int& j, bool warp_wide) -> bool {
        if (!p.clc) {
            t += nclusters;
            return true;
        }
        const int s = j % CLC_SLOTS;
        bool ok = wait_bar(ready_bar(s), (uint32_t)((j / CLC_SLOTS) & 1), p);
        if (warp_wide) ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        int x = 0;
        const bool more = clc_query(resp_addr(s), &x);
        if (warp_wide) __syncwarp();
        if (!warp_wide || (threadIdx.x & 31) == 0) {
            if constexpr (CG == 2) mbar_arrive_cluster(mapa_shared(cons_bar(s), lead));
            else mbar_arrive_local(cons_bar(s));
        }
        ++j;
        t = more ? x / CG : total_units;
        return true;
    };

    if (threadIdx.x == 0) {
        tma_prefetch_desc(&p.tmap_a);
        tma_prefetch_desc(&p.tmap_b);
        if (!B_MN && p.split_from < total_tiles) tma_prefetch_desc(&p.tmap_b_half);
        for (int s = 0; s < C_::STAGES; ++s) {
            mbar_init(full_bar(s), 1);   // leader's producer arms it for both CTAs
            mbar_init(empty_bar(s), MC ? 2 : 1);  // MMA commits of every pair using the stage
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), CG * EPI_WARPS);  // every epilogue warp of the pair
        }
        mbar_init(drain_bar, 1);
        mbar_init(never_bar, 1);
        for (int s = 0; s < CLC_SLOTS; ++s) {
            mbar_init(ready_bar(s), 1);  // this CTA's scheduler thread arms it
            // consumers of the pair: producers, the MMA thread, epilogue warps
            mbar_init(cons_bar(s), CG * (1 + EPI_WARPS) + 1);
        }
        fence_mbarrier_init_cluster();
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync_all(); else __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    if (threadIdx.x == 0) TC_TRACE(p, 1);

    bool aborted = false;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        // The warp runs the loop; one elected lane issues the copies.
        {
            pdl_wait();  // operands written by the kernel before this one (repack)
            int stage = 0;
            uint32_t phase = 0;
            int j = 0;
            for (int t = cluster; t < total_units && !aborted;) {
                const Unit un = unit_of(t);
                const int a_row = un.tm * C_::TILE_M + (int)rank * ROWS_A;
                const int b_rows = un.width / CG;  // B rows (N) this CTA holds
                const int b_row = un.col0 + (int)rank * b_rows;
                // bytes both CTAs of the pair load per stage (OOB fill included)
                const uint32_t bytes = (uint32_t)(CG * (C_::A_BYTES + b_rows * BK * 2));
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar_warp(empty_bar(stage), phase ^ 1u, p)) { aborted = true; break; }
                    const uint32_t fb =
                        CG == 2 ? mapa_shared(full_bar(stage), lead) : full_bar(stage);
                    const uint32_t sa = sA0 + stage * C_::A_BYTES;
                    const uint32_t sb = sB0 + stage * C_::B_BYTES;
                    const int k0 = kb * BK;
                    // every innermost TMA coordinate below is k0, a_row + 64 j or
                    // b_row + 64 j: 16-byte aligned when all three are multiples of 8
                    const bool x_ok = device_check(p.check, ((k0 | a_row | b_row) & 7) == 0,
                                                   kCheckTcTmaX, (unsigned long long)k0);
                    if (x_ok && elect_one()) {
                        if (leader) mbar_arrive_expect_tx(full_bar(stage), bytes);
                        if (kb == 0 && t == cluster) TC_TRACE(p, 2);
                        if constexpr (!A_MN) {
                            tma_load_2d<CG>(sa, &p.tmap_a, fb, k0, a_row);
                        } else {
#pragma unroll
                            for (int j = 0; j < ROWS_A / 64; ++j)
                                tma_load_2d<CG>(sa + j * 64 * BK * 2, &p.tmap_a, fb,
                                                a_row + 64 * j, k0);
                        }
                        if constexpr (MC) {
                            // this pair's 64-row piece of B-half `rank`, to both pairs
                            const uint16_t mask =
                                (uint16_t)((1u << rank) | (1u << (rank + 2)));
                            const uint32_t dst = sb + (uint32_t)(pair * 64 * BK * 2);
                            if constexpr (!B_MN)
                                tma_load_2d_mc_pair(dst, &p.tmap_b, fb, k0, b_row + 64 * pair,
                                                    mask);
                            else
                                tma_load_2d_mc_pair(dst, &p.tmap_b, fb, b_row + 64 * pair, k0,
                                                    mask);
                        } else if constexpr (!B_MN) {
                            // the CTA's rows of B in one box (fewer, larger boxes
                            // measured faster: two 64-row boxes cost 4% at 8192^3)
                            tma_load_2d<CG>(sb,
                                            un.width == p.tile_n ? &p.tmap_b : &p.tmap_b_half,
                                            fb, k0, b_row);
                        } else {
                            // 64-column boxes (the width of the 128-byte swizzle)
                            for (int j = 0; j < b_rows / 64; ++j)
                                tma_load_2d<CG>(sb + j * 64 * BK * 2, &p.tmap_b, fb,
                                                b_row + 64 * j, k0);
                        }
                    }
                    __syncwarp();
                    if (++stage == C_::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (aborted || !advance(t, j, true)) { aborted = true; break; }
            }
            if (aborted) grace_period_ns(200000);  // let issued copies land
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer --
        // The leader's warp runs the loop; one elected lane issues the MMAs
        // and the commits.
        if (leader) {
            // instruction descriptor without N (bits 17-22 = N >> 3, per unit)
            constexpr uint32_t idesc0 =
                make_idesc_f16(BF16, A_MN, B_MN, (uint32_t)C_::TILE_M, 0u);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int j = 0;
            int nt = 0;  // units issued (trace slots)
            // Shared-memory descriptors of stage 0 (128-byte swizzle) and the
            // step between the 16-deep k-slices of one MMA each: K-major
            // +32 bytes inside the swizzled 128-byte rows, MN-major +16
            // k-rows of 128 bytes (two 8-row atoms).
            const uint64_t a_desc0 = A_MN ? make_sdesc_sw128(sA0, 64 * BK * 2, 1024)
                                          : make_sdesc_sw128(sA0, 16, 1024);
            const uint64_t b_desc0 = B_MN ? make_sdesc_sw128(sB0, 64 * BK * 2, 1024)
                                          : make_sdesc_sw128(sB0, 16, 1024);
            constexpr int A_STEP = A_MN ? UMMA_K * 128 : UMMA_K * 2;
            constexpr int B_STEP = B_MN ? UMMA_K * 128 : UMMA_K * 2;
            for (int t = cluster; t < total_units && !aborted;) {
                const uint32_t idesc = idesc0 | ((uint32_t)(unit_of(t).width >> 3) << 17);
                if (!wait_bar_warp(acce_bar(acc), acc_phase ^ 1u, p)) { aborted = true; break; }
                tc_fence_after_sync();
                if (lane == 0) TC_TRACE(p, 4 + 4 * nt);
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar_warp(full_bar(stage), phase, p)) { aborted = true; break; }
                    tc_fence_after_sync();
                    if (kb == 0 && nt == 0 && lane == 0) TC_TRACE(p, 3);
                    // the stage's descriptors: the ring's first ones plus the
                    // stage offset (the address field counts 16-byte units)
                    const uint64_t ad = a_desc0 + (uint64_t)(stage * (C_::A_BYTES >> 4));
                    const uint64_t bd = b_desc0 + (uint64_t)(stage * (C_::B_BYTES >> 4));
                    if (elect_one()) {
#pragma unroll
                        for (int j = 0; j < BK / UMMA_K; ++j)
                            mma_f16<CG>(d_tmem, ad + (uint64_t)(j * (A_STEP >> 4)),
                                        bd + (uint64_t)(j * (B_STEP >> 4)), idesc,
                                        (kb | j) != 0 ? 1u : 0u);
                        if constexpr (MC) mma_commit_pair(empty_bar(stage), (uint16_t)0xF);
                        else mma_commit<CG>(empty_bar(stage));
                    }
                    __syncwarp();
                    if (++stage == C_::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (aborted) break;
                if (elect_one()) {
                    if constexpr (MC) mma_commit_pair(accf_bar(acc), (uint16_t)(0x3u << (2 * pair)));
                    else mma_commit<CG>(accf_bar(acc));
                }
                __syncwarp();
                if (lane == 0) TC_TRACE(p, 5 + 4 * nt);
                ++nt;
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
                if (!advance(t, j, true)) { aborted = true; break; }
            }
            // Drain: wait (bounded) until every MMA issued above has completed.
            if (elect_one()) {
                if constexpr (CG == 2) mma_commit_pair(drain_bar, (uint16_t)(1u << crank));
                else mma_commit_local(drain_bar);
            }
            __syncwarp();
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(drain_bar, 0) && globaltimer_ns() - t0 < 1000000000ull) {
            }
        }
        __syncwarp();
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------------ epilogue --
        // TMEM lane quarter of this warp (hardware: warp % 4) and its half of
        // the 32-column chunks (even or odd)
        const int q = (warp - EPI_WARP0) & 3;
        const int half = (warp - EPI_WARP0) >> 2;
        int acc = 0;
        uint32_t acc_phase = 0;
        pdl_wait();  // C may be read (fused epilogue) or written only after earlier kernels
        // Every lane waits; the decision to go on is taken warp-uniformly
        // (__all_sync) because tcgen05.ld below is a .sync.aligned warp op.
        if (p.fault_inject == 1) {
            // Test hook: a wait that nothing completes must time out cleanly.
            if (!__all_sync(0xffffffffu, wait_bar(never_bar, 0u, p))) aborted = true;
        }
        int j = 0;
        int nt = 0;  // units stored (trace slots)
        for (int t = cluster; t < total_units && !aborted;) {
            const Unit un = unit_of(t);
            if (!__all_sync(0xffffffffu, wait_bar(accf_bar(acc), acc_phase, p))) {
                aborted = true;
                break;
            }
            tc_fence_after_sync();
            if (warp == EPI_WARP0 && lane == 0) TC_TRACE(p, 6 + 4 * nt);
            const int row0 = un.tm * C_::TILE_M + (int)rank * ROWS_A + q * 32;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
            const uint32_t stage = epi0 + (uint32_t)((warp - EPI_WARP0) * 32 * 128);
#pragma unroll 1
            for (int c = half; c < un.width / 32; c += 2) {
                uint32_t v[32];
                if (nt == 0 && warp == EPI_WARP0 && lane == 0) TC_TRACE(p, 20 + 4 * c);
                tmem_ld_32x32b_x32(taddr + (uint32_t)(c * 32), v);
                tmem_wait_ld();
                if (nt == 0 && warp == EPI_WARP0 && lane == 0) TC_TRACE(p, 21 + 4 * c);
                store_chunk<OutT>(p, stage, lane, row0, un.col0 + c * 32, v);
                if (nt == 0 && warp == EPI_WARP0 && lane == 0) TC_TRACE(p, 22 + 4 * c);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 2) mbar_arrive_cluster(mapa_shared(acce_bar(acc), lead));
                else mbar_arrive_local(acce_bar(acc));
            }
            if (warp == EPI_WARP0 && lane == 0) TC_TRACE(p, 7 + 4 * nt);
            ++nt;
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            if (!advance(t, j, true)) { aborted = true; break; }
        }
        if (p.c_tma && lane == 0) bulk_wait_all();  // stores done before the CTA exits
        __syncwarp();
        if (warp == EPI_WARP0 && lane == 0) TC_TRACE(p, 62);
    } else if (warp == 2) {
        // --------------------------------------- tile scheduler (CLC) --
        // Each CTA arms its own ready barrier for every response; the pair
        // leader issues the requests (multicast to both CTAs), each one into
        // a slot that every consumer of the pair has released, and stops
        // after the first response that cancelled nothing.
        if (p.clc && lane == 0) {
            bool in_flight = false;
            for (int j = 0;; ++j) {
                const int s = j % CLC_SLOTS;
                const uint32_t round = (uint32_t)(j / CLC_SLOTS);
                if (leader && j >= CLC_SLOTS && !wait_bar(cons_bar(s), (round - 1u) & 1u, p))
                    break;
                mbar_arrive_expect_tx(ready_bar(s), 16);
                if (leader) {
                    fence_proxy_async_smem();  // consumers' reads of the slot come first
                    clc_try_cancel<CG == 2>(resp_addr(s), ready_bar(s));
                }
                in_flight = true;
                if (!wait_bar(ready_bar(s), round & 1u, p)) break;
                in_flight = false;
                int x = 0;
                if (!clc_query(resp_addr(s), &x)) break;
            }
            if (in_flight) grace_period_ns(200000);  // let a pending response land
        }
        __syncwarp();
    }

    // ------------------------------------------------------------ teardown --
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync_all(); else __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem_base, TMEM_COLS);
        if (lane == 0) TC_TRACE(p, 63);
    }
}

template <int CG, bool MC, bool A_MN, bool B_MN, bool BF16, typename OutT>
int launch_variant(TcParams& tp, const DeviceInfo& dev, cudaStream_t stream) {
    using C_ = Cfg<CG>;
    constexpr int CLUSTER = MC ? 2 * CG : CG;
    auto kern = gemm_tc_kernel<CG, MC, A_MN, B_MN, BF16, OutT>;
    static std::mutex mu;
    static uint64_t configured = 0;   // bit per device
    static int max_clusters[64];
    auto cluster_cfg = [&](cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, int nclusters) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CLUSTER;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(CLUSTER * nclusters);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = C_::SMEM_BYTES;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    };
    {
        std::lock_guard<std::mutex> lock(mu);
        const uint64_t bit = 1ull << (dev.device & 63);
        if (!(configured & bit)) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C_::SMEM_BYTES) != cudaSuccess)
                return kCuda;
            int n = dev.sm_count / CLUSTER;
            if (CLUSTER > 1) {
                cudaLaunchConfig_t cfg = {};
                cudaLaunchAttribute attr[1];
                cluster_cfg(cfg, attr, n);
                int q = 0;
                if (cudaOccupancyMaxActiveClusters(&q, kern, &cfg) == cudaSuccess && q > 0)
                    n = q;
                else
                    cudaGetLastError();
            }
            max_clusters[dev.device & 63] = n;
            configured |= bit;
        }
    }
    const int unit_rows = MC ? (tp.tiles_m + 1) / 2 : tp.tiles_m;
    const int tiles = unit_rows * tp.tiles_n;
    tp.split_from = (int)plan_tc_split(tiles, max_clusters[dev.device & 63], tp.tile_n, CG, MC,
                                       tp.split_mode);
    const int total = tp.split_from + 2 * (tiles - tp.split_from);  // work units
    // persistent: as many clusters as fit at once; CLC: one cluster per unit
    int nclusters = tp.clc ? total : max_clusters[dev.device & 63];
    if (nclusters > total) nclusters = total;
    if (nclusters < 1) nclusters = 1;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cluster_cfg(cfg, attr, nclusters);
    if (tp.pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    cfg.stream = stream;
    if (cudaLaunchKernelEx(&cfg, kern, tp) != cudaSuccess) return kCuda;
    note_launch();
    return kOk;
}

template <int CG, bool MC, bool BF16, typename OutT>
int dispatch_majors(TcParams& tp, bool a_mn, bool b_mn, const DeviceInfo& dev,
                    cudaStream_t s) {
    if (!a_mn && !b_mn) return launch_variant<CG, MC, false, false, BF16, OutT>(tp, dev, s);
    if (!a_mn && b_mn) return launch_variant<CG, MC, false, true, BF16, OutT>(tp, dev, s);
    if (a_mn && !b_mn) return launch_variant<CG, MC, true, false, BF16, OutT>(tp, dev, s);
    return launch_variant<CG, MC, true, true, BF16, OutT>(tp, dev, s);
}

}  // namespace
}  // namespace libgemm
