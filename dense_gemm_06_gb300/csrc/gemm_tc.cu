// gemm_tc.cu -- fp16/bf16 GEMM on the 5th-generation tensor cores (tcgen05),
// C = A * B^T with fp32 accumulation in tensor memory (TMEM).
//
// Structure (after the Gluon Multi-CTA tutorial's "fast matmul kernel" and its
// sections on 2-CTA tcgen05 MMA and TMA in a loop, re-designed for sm_103a in
// CUDA C++ with hand-written PTX):
//
//   * persistent (default): one CTA per SM (CG == 1) or one CTA pair per two SMs
//     (CG == 2, a cluster of 2 issuing cta_group::2 MMAs); every CTA walks the
//     same static tile sequence (cluster c takes tiles c, c + #clusters, ...),
//     rasterised in bands of BAND tile-rows with the column direction
//     alternating between bands (a serpentine in the spirit of the tutorial's
//     planar snake), so concurrently running tiles share A and B panels in L2;
//   * warp 0 = TMA producer, warp 1 = MMA issuer (+ TMEM allocation), warps
//     4..7 = epilogue; warp 2 = tile scheduler when cluster launch control is
//     on (one cluster per tile; running clusters take over unstarted ones);
//     warp 3 idle;
//   * an STAGES-deep smem ring of (A, B) k-tiles with full/empty mbarriers:
//     the producer waits `empty`, arms `full` with the expected bytes and
//     issues TMA loads (128-byte swizzle); the MMA warp waits `full`, issues
//     BK/16 MMAs and commits to `empty`;
//   * CG == 2: each CTA loads its own 128 rows of A and its own half of the
//     256-wide B tile; both CTAs' loads complete on the leader's `full`
//     barrier (armed by the leader for both), the leader issues M=256 x N=256
//     MMAs over both CTAs' smem, and its commits are multicast to both CTAs'
//     `empty` / `acc_full` barriers;
//   * TMEM holds two 256-column fp32 accumulators (double buffer) so the
//     epilogue of tile i overlaps the MMAs of tile i+1 (`acc_full` /
//     `acc_empty` barriers; `acc_empty` lives in the leader and counts the
//     epilogue warps of both CTAs);
//   * epilogue: each warp reads its 32 TMEM lanes (= 32 rows of C) in 32-column
//     chunks with tcgen05.ld, converts (fp32 as is, fp16/bf16 round to nearest
//     even), transposes the chunk through a swizzled shared-memory tile and
//     stores it row by row -- 16-byte vectors where C's rows allow, coalesced
//     predicated scalars at ragged edges or misaligned leading dimensions;
//   * every mbarrier wait is bounded: past `wait_limit_ns` (or once another
//     wait has failed) the thread records a timeout in the device error word
//     and its role stops; the CTA drains in-flight copies and MMAs before
//     releasing TMEM and exiting.
#include <cstring>
#include <mutex>

#include "gemm_tc.cuh"
#include "policy.h"

namespace libgemm {
namespace {

// ------------------------------------------------------------------ host --

// Signature of the driver's cuTensorMapEncodeTiled (resolved at run time, so
// the library does not link libcuda directly).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;
#ifdef LIBGEMM_TC_TRACE
unsigned long long* g_trace = nullptr;  // debug build: the phase-timestamp buffer
#endif

bool get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode != nullptr;
}

// The arguments of one 2-D tiled tensor map (zero fill outside the matrix).
struct MapArgs {
    const void* ptr;
    uint64_t inner, outer, stride_bytes;
    uint32_t box_inner, box_outer;
    int32_t dtype, swizzle, promotion, pad;
};

// An encoded tensor map is a pure function of its arguments, so a map made for
// one call serves every later call with the same arguments. A direct-mapped
// cache of kMapSlots maps (indexed by a hash of the arguments, replaced on a
// collision) lets a repeated problem -- the same buffers step after step --
// skip the driver's encoder (about 0.8 us per map on the GB300 host).
constexpr int kMapSlots = 256;
struct MapSlot {
    CUtensorMap map;
    MapArgs args;
    bool used;
};
std::mutex g_map_mu;
MapSlot g_maps[kMapSlots];

uint64_t hash_args(const MapArgs& a) {
    const uint64_t w[6] = {(uint64_t)(uintptr_t)a.ptr, a.inner, a.outer, a.stride_bytes,
                           ((uint64_t)a.box_inner << 32) | a.box_outer,
                           ((uint64_t)(uint32_t)a.dtype << 40) ^ ((uint64_t)(uint32_t)a.swizzle << 20) ^
                               (uint64_t)(uint32_t)a.promotion};
    uint64_t h = 0x9e3779b97f4a7c15ull;
    for (uint64_t x : w) {
        h ^= x + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
        h *= 0xff51afd7ed558ccdull;
    }
    return h ^ (h >> 33);
}

bool encode_cached(CUtensorMap* out, const MapArgs& a) {
    if (!get_encoder()) return false;
    MapSlot& slot = g_maps[hash_args(a) % kMapSlots];
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        if (slot.used && std::memcmp(&slot.args, &a, sizeof(a)) == 0) {
            *out = slot.map;
            return true;
        }
    }
    const cuuint64_t dims[2] = {a.inner, a.outer};
    const cuuint64_t strides[1] = {a.stride_bytes};
    const cuuint32_t box[2] = {a.box_inner, a.box_outer};
    const cuuint32_t estr[2] = {1, 1};
    if (g_encode(out, (CUtensorMapDataType)a.dtype, 2, const_cast<void*>(a.ptr), dims, strides,
                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, (CUtensorMapSwizzle)a.swizzle,
                 (CUtensorMapL2promotion)a.promotion,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(g_map_mu);
    slot.map = *out;
    slot.args = a;
    slot.used = true;
    return true;
}

MapArgs map_args(const void* ptr, int dtype, uint64_t inner, uint64_t outer, uint64_t stride_bytes,
                 uint32_t box_inner, uint32_t box_outer, int swizzle, int promotion) {
    MapArgs a;
    std::memset(&a, 0, sizeof(a));  // padding too: the cache compares bytes
    a.ptr = ptr;
    a.inner = inner;
    a.outer = outer;
    a.stride_bytes = stride_bytes;
    a.box_inner = box_inner;
    a.box_outer = box_outer;
    a.dtype = dtype;
    a.swizzle = swizzle;
    a.promotion = promotion;
    return a;
}

// 2-D map over a 16-bit matrix stored as `outer` rows of `inner` contiguous
// elements, `ld` elements apart; box {box_inner, box_outer}, 128-byte swizzle,
// zero fill outside the matrix.
bool encode_2d(CUtensorMap* map, bool bf16, const void* ptr, uint64_t inner, uint64_t outer,
               uint64_t ld, uint32_t box_inner, uint32_t box_outer) {
    return encode_cached(map, map_args(ptr,
                                       bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                                       inner, outer, ld * 2, box_inner, box_outer,
                                       CU_TENSOR_MAP_SWIZZLE_128B,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B));
}

}  // namespace

bool encode_tma_f32_2d(void* map, const float* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
                       uint32_t box_inner, uint32_t box_outer) {
    return encode_cached(static_cast<CUtensorMap*>(map),
                         map_args(ptr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, inner, outer, ld * 4,
                                  box_inner, box_outer, CU_TENSOR_MAP_SWIZZLE_NONE,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B));
}

int launch_gemm_tc(const Problem& pr, const DeviceInfo& dev, const TcLaunch& o,
                   cudaStream_t stream) {
    if (!get_encoder()) return kCuda;
    const bool want_mc = o.cta_group != 1 && o.multicast;
    const TcShape shape =
        plan_tc_shape(pr.M, pr.N, o.cta_group, o.tile_n, want_mc, dev.sm_count);
    const int CG = shape.cta_group;
    const bool mc = CG == 2 && want_mc;
    const bool bf16 = pr.dtype == 2 || pr.dtype == 4;
    const int tile_m = ROWS_A * CG;

    TcParams tp;
    std::memset(&tp, 0, sizeof(tp));
    // A: K-major -> dims {K, M}, box {64, 128}; M-major -> dims {M, K}, box {64, 64}.
    // B K-major (dims {K, N}): a CTA's share of a tile (tile_n / CG rows) per
    // box, and half that for half-width units; B N-major (dims {N, K}):
    // 64-column boxes, as many as the CTA's share of the unit's width.
    const uint32_t b_share = (uint32_t)(shape.tile_n / CG);
    bool ok = pr.a_kmajor
        ? encode_2d(&tp.tmap_a, bf16, pr.A, pr.K, pr.M, pr.lda, BK, ROWS_A)
        : encode_2d(&tp.tmap_a, bf16, pr.A, pr.M, pr.K, pr.lda, 64, BK);
    ok = ok && (pr.b_kmajor
        ? encode_2d(&tp.tmap_b, bf16, pr.B, pr.K, pr.N, pr.ldb, BK, mc ? 64 : b_share) &&
              (mc || b_share < 128 ||
               encode_2d(&tp.tmap_b_half, bf16, pr.B, pr.K, pr.N, pr.ldb, BK, b_share / 2))
        : encode_2d(&tp.tmap_b, bf16, pr.B, pr.N, pr.K, pr.ldb, 64, BK));
    if (!ok) return kCuda;

    const int out_bytes = pr.dtype <= 2 ? 4 : 2;
    // C through TMA when its base and rows are 16-byte aligned: box 32 x 32,
    // the staging tile's swizzle (128-byte rows for fp32, 64-byte for 16-bit).
    tp.c_tma = 0;
    tp.epi = pr.epi;  // an active epilogue reads/stores C itself (no TMA store)
    if ((reinterpret_cast<uintptr_t>(pr.C) & 15u) == 0 && ((pr.ldc * out_bytes) & 15) == 0 &&
        o.c_tma && !pr.epi.active) {
        const int dt = out_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                       : (bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
        if (encode_cached(&tp.tmap_c,
                          map_args(pr.C, dt, (uint64_t)pr.N, (uint64_t)pr.M,
                                   (uint64_t)(pr.ldc * out_bytes), 32, 32,
                                   out_bytes == 4 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                  : CU_TENSOR_MAP_SWIZZLE_64B,
                                   CU_TENSOR_MAP_L2_PROMOTION_NONE)))
            tp.c_tma = 1;
    }
    tp.C = pr.C;
    tp.ldc = pr.ldc;
    tp.M = (int)pr.M;
    tp.N = (int)pr.N;
    tp.K = (int)pr.K;
    tp.tile_n = shape.tile_n;
    tp.tiles_m = (int)((pr.M + tile_m - 1) / tile_m);
    tp.tiles_n = (int)((pr.N + shape.tile_n - 1) / shape.tile_n);
    tp.split_mode = o.split_mode;  // the split itself is planned at launch (resident clusters)
    // Every launch is a programmatic dependent of what precedes it on the
    // stream: the kernel waits (griddepcontrol.wait) before its first access
    // to global memory, so an earlier kernel's writes are visible, while its
    // launch and prologue overlap that kernel's tail when the earlier kernel
    // signals its dependents (the repack and this kernel do so at their start).
    tp.pdl = 1;
    tp.num_kb = (int)((pr.K + BK - 1) / BK);
    tp.c_vec = ((reinterpret_cast<uintptr_t>(pr.C) & 15u) == 0 &&
                ((pr.ldc * out_bytes) & 15) == 0) ? 1 : 0;
    tp.err = dev.err_word;
    tp.check = dev.check_word;
    tp.gen = next_generation();
    tp.wait_limit_ns = o.wait_limit_ns;
    tp.fault_inject = o.fault_inject;
    tp.clc = o.clc && !mc ? 1 : 0;  // the multicast variant keeps the static schedule
#ifdef LIBGEMM_TC_TRACE
    tp.trace = g_trace;
#endif
    // units (at most twice the tiles) x CTAs must fit the grid's int range
    if ((int64_t)tp.tiles_m * tp.tiles_n * 2 * CG > 0x7fffffffLL) return kUnsupported;

    const bool a_mn = !pr.a_kmajor, b_mn = !pr.b_kmajor;
    int rc = kInvalidArg;
    switch (pr.dtype) {
        case 1: rc = launch_gemm_tc_f16_f32(tp, CG, mc, a_mn, b_mn, dev, stream); break;
        case 2: rc = launch_gemm_tc_bf16_f32(tp, CG, mc, a_mn, b_mn, dev, stream); break;
        case 3: rc = launch_gemm_tc_f16_f16(tp, CG, mc, a_mn, b_mn, dev, stream); break;
        case 4: rc = launch_gemm_tc_bf16_bf16(tp, CG, mc, a_mn, b_mn, dev, stream); break;
        default: break;
    }
    if (rc == kOk && dispatch_log_on()) {
        // launch_variant has planned the split (tp.split_from) by now
        const int rows_u = mc ? (tp.tiles_m + 1) / 2 : tp.tiles_m;
        const int tiles = rows_u * tp.tiles_n;
        dispatch_log("tcgen05 %dx%dx%d: %s, %d x %d tiles (%d x %d), %d work units (tiles from "
                     "%d run as two half-width units), %s schedule, A %s, B %s, C by %s%s%s",
                     tp.M, tp.N, tp.K, CG == 2 ? "CTA pairs" : "one CTA per tile", tile_m,
                     tp.tile_n, tp.tiles_m, tp.tiles_n, tp.split_from + 2 * (tiles - tp.split_from),
                     tp.split_from, tp.clc ? "cluster-launch-control" : "persistent static",
                     a_mn ? "MN-major" : "K-major", b_mn ? "MN-major" : "K-major",
                     tp.c_tma ? "TMA stores" : "st.global", mc ? ", B multicast over two pairs" : "",
                     o.after_repack ? ", waits on the repack (programmatic launch)" : "");
    }
    return rc;
}

}  // namespace libgemm

#ifdef LIBGEMM_TC_TRACE
// Debug build only: device buffer of 64 timestamps per CTA for the next
// launches of the tensor-core kernel (NULL: no tracing).
extern "C" void libgemm_tc_trace_buffer(void* dev_ptr) {
    libgemm::g_trace = static_cast<unsigned long long*>(dev_ptr);
}
#endif
