// internal.h -- interface between the C-ABI layer (gemm_api.cu) and the
// kernel translation units. Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace libgemm {

// Fused epilogue D = act(alpha * acc + beta * C_old + bias) (gemm_ex); passed
// by value to the kernels.
struct EpiParams {
    int active;        // 0: plain store of the accumulator
    float alpha, beta;
    const void* bias;  // C's element type; may be null
    int bias_rows;     // 1: bias indexed by the row of the stored (normalised) C
    int act;           // 0 none, 1 ReLU, 2 GELU
};

// A problem after layout normalisation: C is always row-major (N-major) with
// leading dimension ldc; A is M x K and B is N x K, each K- or MN-major.
struct Problem {
    int64_t M, N, K;
    const void* A;
    int64_t lda;
    bool a_kmajor;
    const void* B;
    int64_t ldb;
    bool b_kmajor;
    void* C;
    int64_t ldc;
    int dtype;  // gemm_dtype
    EpiParams epi;
};

// The per-device error word: 0 while no bounded wait has run out since the
// last gemm_check_device_error(), else the largest launch generation whose
// wait ran out. Every launch with bounded waits gets a generation of its own
// (next_generation(), never 0); its threads give up early only when the word
// holds that generation, so a timeout left over from an earlier launch does
// not stop later ones.
using ErrWord = unsigned long long;

struct DeviceInfo {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    ErrWord* err_word;  // device address of this device's error word
    unsigned long long* check_word;  // device address of its device-check word
};

// Device-side checks of the debug build (-DLIBGEMM_DEVICE_CHECKS): tile
// coordinates, TMA coordinates and store addresses are checked in the
// kernels; a failed check records (code << 56 | detail) in the device's check
// word (the first failure wins) and the checked access is skipped. Without
// the flag the checks compile to nothing. gemm_device_checks() reads and
// clears the word.
enum DeviceCheckCode : unsigned {
    kCheckTcUnit = 1,      // tcgen05 work unit outside the tile grid (detail: unit)
    kCheckTcTmaX = 2,      // a TMA copy's innermost coordinate not 16-byte aligned
    kCheckTcStore = 3,     // an epilogue store outside C (detail: row << 24 | column)
    kCheckSgTile = 4,      // FFMA tile or K-slice outside the problem (detail: CTA)
    kCheckSgStore = 5,     // an FFMA store outside C (detail: row << 24 | column)
};

// A fresh launch generation (process-wide counter, starts at 1).
ErrWord next_generation();

#ifdef __CUDACC__
// Debug build: records a failed check (see DeviceCheckCode); returns `ok`.
__device__ __forceinline__ bool device_check(unsigned long long* word, bool ok, unsigned code,
                                             unsigned long long detail) {
#ifdef LIBGEMM_DEVICE_CHECKS
    if (!ok && word)
        atomicCAS(word, 0ull, ((unsigned long long)code << 56) | (detail & ((1ull << 56) - 1)));
    return ok;
#else
    (void)word; (void)code; (void)detail;
    return true;
#endif
}

// True when a wait of the launch with generation `gen` has run out.
__device__ __forceinline__ bool gen_failed(const ErrWord* err, ErrWord gen) {
    return *reinterpret_cast<const volatile ErrWord*>(err) == gen;
}
// Records that a wait of the launch `gen` ran out.
__device__ __forceinline__ void gen_record_timeout(ErrWord* err, ErrWord gen) {
    atomicMax(err, gen);
}
#endif

// Launchers return 0 or a gemm_status. They enqueue exactly the kernels they
// report through note_launch().

// Device scratch of one call, enqueued on `stream`: get() returns the
// buffer (its first call sizes it), release() ends the call's use of it.
// Buffers up to 64 MB come from a per-(device, stream) cache that keeps them
// across calls (see scratch_cache_acquire in gemm_api.cu); larger ones, and
// any the cache cannot give, are stream-ordered pool allocations freed on
// release.
struct Scratch {
    cudaMemPool_t pool;
    cudaStream_t stream;
    int device;
    void* ptr = nullptr;
    int slot = -1;  // >= 0: the cache entry lent to this call
    void* get(size_t bytes);
    void release();
};
// config: the FFMA tile configuration, 1..9 (GEMM_OPT_SIMT_CONFIG in gemm.h).
// split_mode: 0 automatic (K-split the tiles after the last full round of
// tiles over the SMs when a per-SM model predicts >= 10% saved; plan_split in
// sgemm_ffma.cu), 1 never, 2 always split the last wave (tests).
// wait_limit_ns / fault_inject: the bounded mbarrier waits of configuration 9
// (TMA-fed) and its test hook (1 = the first CTA never loads its second
// k-tile, so its waits run out and report a timeout in the error word).
int launch_sgemm_f32(const Problem& p, const DeviceInfo& dev, int config, int split_mode,
                     Scratch* scratch, uint64_t wait_limit_ns, int fault_inject,
                     cudaStream_t stream);
// A 2-D TMA tensor map (a 64-byte-aligned CUtensorMap at `map`) over an fp32
// matrix of `outer` rows of `inner` contiguous elements, `ld` elements
// apart; box {box_inner, box_outer}, no swizzle, zero fill outside the
// matrix. False when the driver's encoder is missing or rejects the map.
bool encode_tma_f32_2d(void* map, const float* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
                       uint32_t box_inner, uint32_t box_outer);
// dst[c * ldd + r] = src[r * lds + c] (fp32), rows x cols.
int launch_transpose_f32(const float* src, int64_t lds, float* dst, int64_t ldd, int64_t rows,
                         int64_t cols, const DeviceInfo& dev, cudaStream_t stream);
// How one tensor-core launch runs (every field resolved except where 0 means
// automatic; the shape rules are plan_tc_shape / plan_tc_split in policy.h).
struct TcLaunch {
    int cta_group;   // 0 automatic, 1 a CTA per tile, 2 a CTA pair per tile
    int tile_n;      // 0 automatic, or 64, 128, 256 columns per tile
    int split_mode;  // last-round split into half-width units: 0 auto, 1 never, 2 always
    int c_tma;       // 1: TMA stores of C where its rows are 16-byte aligned; 0: st.global
    int multicast;   // 1: clusters of two CTA pairs sharing B through TMA multicast
    int clc;         // 1: one cluster per unit, cluster launch control takes over
                     // unstarted ones; 0: persistent static schedule
    uint64_t wait_limit_ns;
    int fault_inject;  // test hook (GEMM_OPT_TC_FAULT_INJECT)
    int after_repack;  // 1: the previous launch on the stream is this call's repack
                       // kernel: launch as its programmatic dependent
};
int launch_gemm_tc(const Problem& p, const DeviceInfo& dev, const TcLaunch& o,
                   cudaStream_t stream);

void note_launch(uint64_t n = 1);

// Dispatch log (debug aid): when the environment variable GEMM_LOG is set to
// a non-empty value other than "0" when the library first checks it, every
// call writes one line per decision it takes (kernel, tile shape, split,
// repack, transpose) to stderr, prefixed "libgemm: ". Off by default.
bool dispatch_log_on();
void dispatch_log(const char* fmt, ...)
#if defined(__GNUC__)
    __attribute__((format(printf, 1, 2)))
#endif
    ;

// Host-side argument checks and layout normalisation of gemm() (no CUDA calls),
// and the current device's error-word address (cudaGetSymbolAddress only).
int check_args(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_major,
               const void* B, int64_t ldb, int b_major, void* C, int64_t ldc, int c_major,
               int dtype);
Problem normalised(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_major,
                   const void* B, int64_t ldb, int b_major, void* C, int64_t ldc, int c_major,
                   int dtype);
int error_word_address(ErrWord** out);
// Device address of the current device's device-check word (debug build).
int check_word_address(unsigned long long** out);
// kOk when every non-null pointer of ptrs[0..n) is device memory of device
// `device` (cudaPointerGetAttributes: type device, same ordinal), else
// kInvalidArg. Host, managed and peer-device pointers are rejected before any
// launch, so no kernel -- in particular no cluster-multicast TMA load -- ever
// addresses another GPU's memory.
int check_device_pointers(const void* const* ptrs, int n, int device);
// The tensor-core launch options gemm() resolves for a problem: an option the
// caller set wins, then a gemm_tune() entry for the problem, then the default.
TcLaunch resolve_tc_options(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                            int a_major, const void* B, int64_t ldb, int b_major, const void* C,
                            int64_t ldc, int c_major, int dtype);

// Row softmax over thread-block clusters (softmax_cluster.cu); rows longer
// than softmax_max_cols() are not supported.
int64_t softmax_max_cols();
int launch_softmax_rows(int64_t M, int64_t N, const float* x, int64_t ldx, float* y, int64_t ldy,
                        const DeviceInfo& dev, uint64_t wait_limit_ns, int fault_inject,
                        cudaStream_t stream);

// C = act(beta * C + bias) in place (the K == 0 case of gemm_ex), rows x cols
// of the normalised row-major C.
int launch_epilogue_only(const Problem& p, const DeviceInfo& dev, cudaStream_t stream);

// Status codes shared with the public header (kept numerically identical).
enum : int {
    kOk = 0,
    kInvalidArg = -1,
    kUnsupported = -2,
    kCuda = -3,
    kTimeout = -4,
};


}  // namespace libgemm
