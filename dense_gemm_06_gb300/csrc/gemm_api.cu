// gemm_api.cu -- the C ABI of libgemm (include/gemm.h): argument checks,
// layout normalisation, kernel selection, scratch memory and error reporting.
//
// Argument model after the CuTe DSL Ampere SGEMM example's run() (a_major
// "k"|"m", b_major "k"|"n", c_major "n"|"m", leading dimension = stride of the
// non-contiguous mode) and the validation of the Gluon Multi-CTA tutorial's
// matmul_multicta wrapper (shape and dtype checks before any launch), but
// reporting status codes instead of raising, and accepting any element-aligned
// layout.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstdint>
#include <cstring>
#include <map>
#include <numeric>
#include <mutex>

#include "../../include/gemm.h"
#include "epilogue.cuh"
#include "internal.h"
#include "policy.h"
#include "repack16.cuh"

namespace libgemm {

namespace {

constexpr int kMaxDevices = 64;

// Per-device error word written by kernels that give up on a wait (the
// largest generation of a launch whose wait ran out; see internal.h).
__device__ ErrWord g_err_word;
__device__ unsigned long long g_check_word;  // first failed device-side check (debug build)
std::atomic<ErrWord> g_generation{1};

std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_wait_limit_ns{1000000000ull};
std::atomic<int> g_cta_group{0};
std::atomic<int> g_fault_inject{0};
std::atomic<int> g_softmax_fault_inject{0};
std::atomic<int> g_simt_config{0};
std::atomic<int> g_simt_transpose{0};
std::atomic<int> g_simt_split{0};
std::atomic<int> g_simt_fault_inject{0};
std::atomic<int> g_tc_scheduler{0};
std::atomic<int> g_tc_store{0};
std::atomic<int> g_tc_multicast{0};
std::atomic<int> g_tc_tile_n{0};
std::atomic<int> g_tc_split{0};

// The kernel configuration one call runs with. Every field is resolved
// (no "automatic" values): an option set to a non-zero value wins, then a
// gemm_tune() entry for the problem, then the built-in choice.
struct RunConfig {
    int simt_config;     // 1..9
    int simt_transpose;  // 0 automatic size rule, 1 never, 2 always
    int cta_group;       // 1 or 2
    int multicast;       // 1 off, 2 on
    int tc_store;        // 0 TMA where possible, 1 st.global
    int simt_split;      // 0 automatic K-split of the last wave, 1 never, 2 always
    int tc_scheduler;    // 1 static persistent, 2 cluster launch control
    int tc_tile_n;       // 0 automatic, 64, 128, 256
    int tc_split;        // 0 automatic, 1 never, 2 always
};

// Problems gemm_tune() has measured: shape, types, layouts and whether each
// operand's base/pitch is 16-byte aligned (which changes the kernels run).
struct TuneKey {
    int64_t M, N, K;
    int dtype, a_major, b_major, c_major, align;
    bool operator<(const TuneKey& o) const {
        if (M != o.M) return M < o.M;
        if (N != o.N) return N < o.N;
        if (K != o.K) return K < o.K;
        if (dtype != o.dtype) return dtype < o.dtype;
        if (a_major != o.a_major) return a_major < o.a_major;
        if (b_major != o.b_major) return b_major < o.b_major;
        if (c_major != o.c_major) return c_major < o.c_major;
        return align < o.align;
    }
};
std::mutex g_tune_mu;
std::map<TuneKey, gemm_tuning> g_tune_table;

struct DeviceState {
    std::once_flag once;
    int status = kOk;
    DeviceInfo info{};
    cudaMemPool_t pool = nullptr;
    cudaStream_t h2d = nullptr, d2h = nullptr;  // gemm_host's copy streams
};
DeviceState g_dev[kMaxDevices];

int in_bytes(int dtype) { return dtype == GEMM_F32 ? 4 : 2; }
int out_bytes(int dtype) { return dtype <= GEMM_BF16_F32 ? 4 : 2; }

// Resolve the current device once: capability check, error word, scratch pool.
int current_device(DeviceInfo** out, cudaMemPool_t* pool) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return kUnsupported;
    }
    if (dev >= kMaxDevices) return kUnsupported;
    DeviceState& st = g_dev[dev];
    std::call_once(st.once, [&st, dev] {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            cudaGetLastError();
            st.status = kUnsupported;
            return;
        }
        if (prop.major != 10 || prop.minor != 3) {  // built for sm_103a only
            st.status = kUnsupported;
            return;
        }
        void* err = nullptr;
        if (cudaGetSymbolAddress(&err, g_err_word) != cudaSuccess) {
            cudaGetLastError();
            st.status = kCuda;
            return;
        }
        cudaMemPoolProps pp;
        std::memset(&pp, 0, sizeof(pp));
        pp.allocType = cudaMemAllocationTypePinned;
        pp.location.type = cudaMemLocationTypeDevice;
        pp.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &pp) != cudaSuccess) {
            cudaGetLastError();
            st.status = kCuda;
            return;
        }
        uint64_t keep = ~0ull;  // keep freed scratch cached until released
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        st.pool = pool;
        st.info.device = dev;
        st.info.sm_count = prop.multiProcessorCount;
        st.info.cc_major = prop.major;
        st.info.cc_minor = prop.minor;
        st.info.err_word = static_cast<ErrWord*>(err);
        if (check_word_address(&st.info.check_word) != kOk) {
            st.status = kCuda;
            return;
        }
        if (cudaStreamCreateWithFlags(&st.h2d, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&st.d2h, cudaStreamNonBlocking) != cudaSuccess) {
            cudaGetLastError();
            st.status = kCuda;
            return;
        }
        st.status = kOk;
    });
    if (st.status != kOk) return st.status;
    *out = &st.info;
    if (pool) *pool = st.pool;
    return kOk;
}

// gemm_host's copy streams of the current device (after current_device()).
void copy_streams(const DeviceInfo& dev, cudaStream_t* h2d, cudaStream_t* d2h) {
    *h2d = g_dev[dev.device].h2d;
    *d2h = g_dev[dev.device].d2h;
}

bool mul_fits(int64_t a, int64_t b, int64_t limit) { return a == 0 || b <= limit / a; }

// Elements spanned by `outer` rows of `inner` elements, `ld` apart.
bool span_ok(int64_t outer, int64_t inner, int64_t ld, int esize) {
    if (outer == 0 || inner == 0) return true;
    const int64_t lim = INT64_MAX / esize;
    if (!mul_fits(outer - 1, ld, lim)) return false;
    return (outer - 1) * ld <= lim - inner;
}

int64_t span_elems(int64_t outer, int64_t inner, int64_t ld) {
    return (outer == 0 || inner == 0) ? 0 : (outer - 1) * ld + inner;
}

// Host-side validation shared by gemm() and gemm_host(). No CUDA calls.
int validate(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_major,
             const void* B, int64_t ldb, int b_major, void* C, int64_t ldc, int c_major,
             int dtype) {
    if (dtype < GEMM_F32 || dtype > GEMM_BF16_BF16) return kInvalidArg;
    if ((a_major != 0 && a_major != 1) || (b_major != 0 && b_major != 1) ||
        (c_major != 0 && c_major != 1))
        return kInvalidArg;
    if (M < 0 || N < 0 || K < 0) return kInvalidArg;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return kInvalidArg;
    if (M == 0 || N == 0) return kOk;
    const int ie = in_bytes(dtype), oe = out_bytes(dtype);
    // C: N-major (row-major) -> rows M of N; M-major -> rows N of M.
    const int64_t c_inner = c_major == GEMM_MAJOR_MN ? N : M;
    const int64_t c_outer = c_major == GEMM_MAJOR_MN ? M : N;
    if (!C || ldc < c_inner || ldc < 1) return kInvalidArg;
    if (reinterpret_cast<uintptr_t>(C) % oe) return kInvalidArg;
    if (!span_ok(c_outer, c_inner, ldc, oe)) return kInvalidArg;
    if (K == 0) return kOk;
    const int64_t a_inner = a_major == GEMM_MAJOR_K ? K : M;
    const int64_t a_outer = a_major == GEMM_MAJOR_K ? M : K;
    const int64_t b_inner = b_major == GEMM_MAJOR_K ? K : N;
    const int64_t b_outer = b_major == GEMM_MAJOR_K ? N : K;
    if (!A || !B) return kInvalidArg;
    if (lda < a_inner || ldb < b_inner) return kInvalidArg;
    if (reinterpret_cast<uintptr_t>(A) % ie || reinterpret_cast<uintptr_t>(B) % ie)
        return kInvalidArg;
    if (!span_ok(a_outer, a_inner, lda, ie) || !span_ok(b_outer, b_inner, ldb, ie))
        return kInvalidArg;
    return kOk;
}

// ------------------------------------------------------------- helpers --

__global__ void zero_rows_kernel(uint8_t* C, int64_t rows, int64_t row_bytes,
                                 int64_t pitch_bytes) {
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x)  // a block per row
        for (int64_t c = threadIdx.x; c < row_bytes; c += blockDim.x) C[r * pitch_bytes + c] = 0;
}

// Blocks for a row-per-block kernel over `rows` rows: at most 8 per SM.
int grid_rows(int64_t rows, const DeviceInfo& dev) {
    const int64_t cap = (int64_t)dev.sm_count * 8;
    return (int)(rows < 1 ? 1 : (rows > cap ? cap : rows));
}


int zero_fill(void* C, int64_t rows, int64_t cols, int64_t ld, int esize, const DeviceInfo& dev,
              cudaStream_t s) {
    const int64_t rb = cols * esize;
    zero_rows_kernel<<<grid_rows(rows, dev), 256, 0, s>>>(static_cast<uint8_t*>(C), rows, rb,
                                                           ld * esize);
    if (cudaGetLastError() != cudaSuccess) return kCuda;
    note_launch();
    return kOk;
}

bool tma_ok(const void* p, int64_t ld, int esize) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && ((ld * esize) & 15) == 0;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Normalised problem on the device: column-major C becomes row-major C^T by
// exchanging the roles of A and B (C^T[n][m] = sum_k B(n,k) A(m,k)).
Problem normalise(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_major,
                  const void* B, int64_t ldb, int b_major, void* C, int64_t ldc, int c_major,
                  int dtype) {
    Problem p;
    if (c_major == GEMM_MAJOR_MN) {
        p = {M, N, K, A, lda, a_major == GEMM_MAJOR_K, B, ldb, b_major == GEMM_MAJOR_K, C, ldc,
             dtype, EpiParams{}};
    } else {
        p = {N, M, K, B, ldb, b_major == GEMM_MAJOR_K, A, lda, a_major == GEMM_MAJOR_K, C, ldc,
             dtype, EpiParams{}};
    }
    return p;
}

// ------------------------------------------------------------ scratch cache --
// Scratch buffers kept across calls, one per (device, stream): the operand
// repack of the tensor-core path and the split-K / stream-K workspace of the
// FFMA path reuse the previous call's buffer on the same stream instead of a
// stream-ordered pool allocation and free per call (those two operations cost
// about 1.6 us of stream time per call on top of their host time). Reuse on
// the same stream is ordered by the stream itself. A call holds its entry
// busy, so a concurrent call on the same stream from another host thread
// takes the pool path. An entry of another stream is evicted only after the
// evicting stream waits for the event recorded at that entry's last release,
// so a buffer still in use is never freed; streams are told apart by their
// process-unique id, not by the reusable handle. Calls captured into a CUDA
// graph bypass the cache.
constexpr size_t kCachedScratchMax = 64ull << 20;
constexpr int kCachedScratchEntries = 8;
struct CachedScratch {
    int device = -1;
    unsigned long long stream_id = 0;
    void* ptr = nullptr;
    size_t bytes = 0;
    cudaEvent_t last_use = nullptr;  // recorded on the entry's stream at each release
    bool recorded = false;           // last_use covers every use so far (else never evicted)
    bool busy = false;
    uint64_t tick = 0;               // last release, for least-recently-used eviction
};
std::mutex g_scratch_mu;
CachedScratch g_scratch[kCachedScratchEntries];
uint64_t g_scratch_tick = 0;

// An entry of at least `bytes` for work on `s` (marked busy), or -1.
int scratch_cache_acquire(int device, cudaStream_t s, size_t bytes, cudaMemPool_t pool) {
    if (bytes > kCachedScratchMax) return -1;
    // A stream being captured into a CUDA graph takes the pool path: the
    // graph then owns its allocation, where a cached buffer would be baked
    // into the graph and raced by later calls on the stream.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (cap != cudaStreamCaptureStatusNone) return -1;
    unsigned long long id = 0;
    if (cudaStreamGetId(s, &id) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    int slot = -1;
    for (int i = 0; i < kCachedScratchEntries; ++i)
        if (g_scratch[i].ptr && g_scratch[i].device == device && g_scratch[i].stream_id == id) {
            slot = i;
            break;
        }
    if (slot >= 0 && g_scratch[slot].busy) return -1;
    if (slot < 0) {  // an empty entry, else this device's least recently used idle one
        for (int i = 0; i < kCachedScratchEntries && slot < 0; ++i)
            if (!g_scratch[i].ptr && !g_scratch[i].busy) slot = i;
        for (int i = 0; i < kCachedScratchEntries && slot < 0; ++i) {
            const CachedScratch& e = g_scratch[i];
            if (e.busy || !e.recorded || e.device != device) continue;
            int lru = i;
            for (int k = i + 1; k < kCachedScratchEntries; ++k)
                if (!g_scratch[k].busy && g_scratch[k].recorded &&
                    g_scratch[k].device == device && g_scratch[k].tick < g_scratch[lru].tick)
                    lru = k;
            slot = lru;
        }
        if (slot < 0) return -1;
        CachedScratch& e = g_scratch[slot];
        if (e.ptr) {  // evict: free after the entry's last use on its own stream
            if (cudaStreamWaitEvent(s, e.last_use, 0) != cudaSuccess ||
                cudaFreeAsync(e.ptr, s) != cudaSuccess) {
                cudaGetLastError();
                return -1;
            }
            e.ptr = nullptr;
            e.bytes = 0;
        }
        if (e.last_use && e.device != device) {
            cudaEventDestroy(e.last_use);
            e.last_use = nullptr;
        }
        if (!e.last_use &&
            cudaEventCreateWithFlags(&e.last_use, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            e.last_use = nullptr;
            return -1;
        }
        e.device = device;
        e.stream_id = id;
        e.recorded = false;
    }
    CachedScratch& e = g_scratch[slot];
    if (e.bytes < bytes) {  // grow: earlier uses were on this stream, so ordered
        if (e.ptr && cudaFreeAsync(e.ptr, s) != cudaSuccess) cudaGetLastError();
        e.ptr = nullptr;
        e.bytes = 0;
        if (cudaMallocFromPoolAsync(&e.ptr, bytes, pool, s) != cudaSuccess) {
            cudaGetLastError();
            e.ptr = nullptr;
            return -1;
        }
        e.bytes = bytes;
    }
    e.busy = true;
    return slot;
}

// Frees every idle cached buffer (after the caller has synchronised the
// devices; entries in use by a call are kept).
void scratch_cache_clear() {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    for (CachedScratch& e : g_scratch) {
        if (e.busy || e.device < 0) continue;
        if (cudaSetDevice(e.device) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (e.ptr) cudaFree(e.ptr);
        if (e.last_use) cudaEventDestroy(e.last_use);
        e = CachedScratch{};
    }
    cudaSetDevice(cur);
    cudaGetLastError();
}

void scratch_cache_release(int slot, cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    CachedScratch& e = g_scratch[slot];
    if (cudaEventRecord(e.last_use, s) == cudaSuccess) {
        e.recorded = true;
    } else {
        cudaGetLastError();
        e.recorded = false;  // its stream's later uses stay ordered; only eviction is barred
    }
    e.busy = false;
    e.tick = ++g_scratch_tick;
}

int run_sgemm(Problem p, const DeviceInfo& dev, cudaMemPool_t pool, const RunConfig& cfg,
              cudaStream_t s) {
    void* scratch[2] = {nullptr, nullptr};
    int rc = kOk;
    const void** ops[2] = {&p.A, &p.B};
    int64_t* lds[2] = {&p.lda, &p.ldb};
    bool* kmaj[2] = {&p.a_kmajor, &p.b_kmajor};
    const int64_t rows[2] = {p.M, p.N};
    const int64_t other[2] = {p.N, p.M};
    for (int i = 0; i < 2 && rc == kOk; ++i) {
        if (!*kmaj[i] || !want_transpose(other[i], p.M, p.N, p.K, cfg.simt_transpose)) continue;
        const int64_t ld2 = round_up(rows[i], 4);  // 16-byte rows for vector copies
        if (cudaMallocFromPoolAsync(&scratch[i], (size_t)(p.K * ld2 * 4), pool, s) !=
            cudaSuccess) {
            cudaGetLastError();
            rc = kCuda;
            break;
        }
        rc = launch_transpose_f32(static_cast<const float*>(*ops[i]), *lds[i],
                                  static_cast<float*>(scratch[i]), ld2, rows[i], p.K, dev, s);
        dispatch_log("transpose of K-major fp32 %s (%lld x %lld) to MN-major", i ? "B" : "A",
                     (long long)rows[i], (long long)p.K);
        *ops[i] = scratch[i];
        *lds[i] = ld2;
        *kmaj[i] = false;
    }
    Scratch tail{pool, s, dev.device};
    if (rc == kOk)
        rc = launch_sgemm_f32(p, dev, cfg.simt_config, cfg.simt_split, &tail,
                              g_wait_limit_ns.load(), g_simt_fault_inject.load(), s);
    tail.release();
    for (int i = 0; i < 2; ++i)
        if (scratch[i]) cudaFreeAsync(scratch[i], s);
    return rc;
}

TcLaunch tc_launch(const RunConfig& c);

int run_device(Problem p, const DeviceInfo& dev, cudaMemPool_t pool, const RunConfig& cfg,
               cudaStream_t s) {
    if (p.K == 0) return zero_fill(p.C, p.M, p.N, p.ldc, out_bytes(p.dtype), dev, s);
    if (p.dtype == GEMM_F32) return run_sgemm(p, dev, pool, cfg, s);

    // Tensor-core path: TMA needs 16-byte aligned bases and row pitches.
    // Misaligned operands are repacked into one scratch buffer (each
    // operand's part 256-byte aligned), in one launch.
    Scratch scratch{pool, s, dev.device};
    int rc = kOk;
    const void** ops[2] = {&p.A, &p.B};
    int64_t* lds[2] = {&p.lda, &p.ldb};
    const bool kmaj[2] = {p.a_kmajor, p.b_kmajor};
    const int64_t rows[2] = {p.M, p.N};
    Repack16 job[2] = {};  // outer == 0: nothing to repack
    int64_t off[2] = {0, 0}, bytes = 0;
    for (int i = 0; i < 2; ++i) {
        if (tma_ok(*ops[i], *lds[i], 2)) continue;
        const int64_t inner = kmaj[i] ? p.K : rows[i];
        const int64_t outer = kmaj[i] ? rows[i] : p.K;
        const int64_t ld2 = round_up(inner, 8);
        job[i] = {static_cast<const uint16_t*>(*ops[i]), nullptr, *lds[i], ld2, outer, inner};
        off[i] = bytes;
        bytes += round_up(outer * ld2 * 2, 256);
    }
    if (bytes > 0) {
        if (!scratch.get((size_t)bytes)) return kCuda;
        for (int i = 0; i < 2; ++i) {
            if (job[i].outer == 0) continue;
            job[i].dst = reinterpret_cast<uint16_t*>(static_cast<char*>(scratch.ptr) + off[i]);
            *ops[i] = job[i].dst;
            *lds[i] = job[i].ldd;
        }
        repack16_kernel<<<repack16_blocks(job[0].outer + job[1].outer, dev.sm_count), 256, 0,
                          s>>>(job[0], job[1]);
        if (cudaGetLastError() != cudaSuccess) rc = kCuda;
        else note_launch();
        dispatch_log("repack of misaligned 16-bit operands: A %s, B %s (%lld bytes of scratch)",
                     job[0].outer ? "yes" : "no", job[1].outer ? "yes" : "no", (long long)bytes);
    }
    if (rc == kOk) {
        TcLaunch o = tc_launch(cfg);
        o.after_repack = bytes > 0 ? 1 : 0;
        rc = launch_gemm_tc(p, dev, o, s);
    }
    scratch.release();
    return rc;
}

bool aligned16_ld(const void* p, int64_t ld, int esize) {
    return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && ((ld * esize) & 15) == 0;
}

TuneKey make_key(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_major,
                 const void* B, int64_t ldb, int b_major, const void* C, int64_t ldc,
                 int c_major, int dtype) {
    const int ie = in_bytes(dtype), oe = out_bytes(dtype);
    const int align = (aligned16_ld(A, lda, ie) ? 1 : 0) | (aligned16_ld(B, ldb, ie) ? 2 : 0) |
                      (aligned16_ld(C, ldc, oe) ? 4 : 0);
    return TuneKey{M, N, K, dtype, a_major, b_major, c_major, align};
}

RunConfig resolve(const TuneKey& key) {
    RunConfig c{g_simt_config.load(), g_simt_transpose.load(), g_cta_group.load(),
                g_tc_multicast.load(), g_tc_store.load(), g_simt_split.load(),
                g_tc_scheduler.load(), g_tc_tile_n.load(), g_tc_split.load()};
    gemm_tuning t{};
    bool tuned = false;
    {
        std::lock_guard<std::mutex> lock(g_tune_mu);
        auto it = g_tune_table.find(key);
        if (it != g_tune_table.end()) {
            t = it->second;
            tuned = true;
        }
    }
    if (c.simt_config == 0) c.simt_config = tuned && t.simt_config ? t.simt_config : 9;
    if (c.simt_transpose == 0 && tuned) c.simt_transpose = t.simt_transpose;
    // CTA group and tile width stay automatic (0) unless asked for or tuned:
    // the launch picks them from the shape (plan_tc_shape)
    if (c.cta_group == 0 && tuned) c.cta_group = t.tc_cta_group;
    c.multicast = c.multicast == 2 ? 2 : 1;  // only on request, never from a tuned entry
    if (c.tc_store == 0 && tuned) c.tc_store = t.tc_store;
    if (c.tc_scheduler == 0) c.tc_scheduler = tuned && t.tc_scheduler ? t.tc_scheduler : 1;
    return c;
}

TcLaunch tc_launch(const RunConfig& c) {
    return TcLaunch{c.cta_group,         c.tc_tile_n,          c.tc_split,
                    c.tc_store != 1,     c.multicast == 2,     c.tc_scheduler == 2,
                    g_wait_limit_ns.load(), g_fault_inject.load(), 0};
}

}  // namespace

void* Scratch::get(size_t bytes) {
    if (ptr) return ptr;
    slot = scratch_cache_acquire(device, stream, bytes, pool);
    if (slot >= 0) {
        ptr = g_scratch[slot].ptr;
        return ptr;
    }
    if (cudaMallocFromPoolAsync(&ptr, bytes, pool, stream) != cudaSuccess) {
        cudaGetLastError();
        ptr = nullptr;
    }
    return ptr;
}

void Scratch::release() {
    if (slot >= 0) scratch_cache_release(slot, stream);
    else if (ptr) cudaFreeAsync(ptr, stream);
    ptr = nullptr;
    slot = -1;
}

void note_launch(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

bool dispatch_log_on() {
    static const bool on = [] {
        const char* v = std::getenv("GEMM_LOG");
        return v && v[0] && std::strcmp(v, "0") != 0;
    }();
    return on;
}

void dispatch_log(const char* fmt, ...) {
    if (!dispatch_log_on()) return;
    char line[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(line, sizeof(line), fmt, ap);
    va_end(ap);
    std::fprintf(stderr, "libgemm: %s\n", line);
}

namespace {

// C = act(beta * C + bias) for K == 0 (the product term is zero).
template <typename OutT>
__global__ void epilogue_only_kernel(OutT* C, int64_t ldc, int rows, int cols, EpiParams e) {
    for (int r = blockIdx.x; r < rows; r += gridDim.x)  // a block per row
        for (int c = threadIdx.x; c < cols; c += blockDim.x) {
            OutT* d = C + (int64_t)r * ldc + c;
            const float old = e.beta != 0.f ? to_f32(*d) : 0.f;
            *d = from_f32<OutT>(epilogue_value<OutT>(e, 0.f, old, r, c));
        }
}

}  // namespace

int launch_epilogue_only(const Problem& p, const DeviceInfo& dev, cudaStream_t s) {
    const int grid = grid_rows(p.M, dev);
    if (out_bytes(p.dtype) == 4)
        epilogue_only_kernel<float><<<grid, 256, 0, s>>>(static_cast<float*>(p.C), p.ldc,
                                                          (int)p.M, (int)p.N, p.epi);
    else if (p.dtype == GEMM_BF16_BF16)
        epilogue_only_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<__nv_bfloat16*>(p.C), p.ldc, (int)p.M, (int)p.N, p.epi);
    else
        epilogue_only_kernel<__half><<<grid, 256, 0, s>>>(static_cast<__half*>(p.C), p.ldc,
                                                           (int)p.M, (int)p.N, p.epi);
    if (cudaGetLastError() != cudaSuccess) return kCuda;
    note_launch();
    return kOk;
}

int check_args(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_major,
               const void* B, int64_t ldb, int b_major, void* C, int64_t ldc, int c_major,
               int dtype) {
    return validate(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype);
}

Problem normalised(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_major,
                   const void* B, int64_t ldb, int b_major, void* C, int64_t ldc, int c_major,
                   int dtype) {
    return normalise(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype);
}

int error_word_address(ErrWord** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) {
        cudaGetLastError();
        return kCuda;
    }
    *out = static_cast<ErrWord*>(p);
    return kOk;
}

int check_word_address(unsigned long long** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_check_word) != cudaSuccess) {
        cudaGetLastError();
        return kCuda;
    }
    *out = static_cast<unsigned long long*>(p);
    return kOk;
}

ErrWord next_generation() { return g_generation.fetch_add(1, std::memory_order_relaxed); }

TcLaunch resolve_tc_options(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                            int a_major, const void* B, int64_t ldb, int b_major, const void* C,
                            int64_t ldc, int c_major, int dtype) {
    return tc_launch(
        resolve(make_key(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype)));
}

int check_device_pointers(const void* const* ptrs, int n, int device) {
    for (int i = 0; i < n; ++i) {
        if (!ptrs[i]) continue;
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, ptrs[i]) != cudaSuccess) {
            cudaGetLastError();
            return kInvalidArg;
        }
        if (at.type != cudaMemoryTypeDevice || at.device != device) return kInvalidArg;
    }
    return kOk;
}

}  // namespace libgemm

using namespace libgemm;

extern "C" {

int gemm(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_major, const void* B,
         int64_t ldb, int b_major, void* C, int64_t ldc, int c_major, int dtype, void* stream) {
    try {
        int rc = validate(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype);
        if (rc != kOk) return rc;
        if (M == 0 || N == 0) return kOk;
        DeviceInfo* dev = nullptr;
        cudaMemPool_t pool = nullptr;
        rc = current_device(&dev, &pool);
        if (rc != kOk) return rc;
        const void* ptrs[3] = {K > 0 ? A : nullptr, K > 0 ? B : nullptr, C};
        rc = check_device_pointers(ptrs, 3, dev->device);
        if (rc != kOk) return rc;
        const Problem p =
            normalise(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype);
        const RunConfig cfg = resolve(
            make_key(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype));
        return run_device(p, *dev, pool, cfg, static_cast<cudaStream_t>(stream));
    } catch (...) {
        return kCuda;
    }
}

int gemm_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_major,
            const void* B, int64_t ldb, int b_major, void* C, int64_t ldc, int c_major, int dtype,
            const gemm_epilogue* epi, void* stream) {
    try {
        if (!epi)
            return gemm(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype, stream);
        int rc = validate(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype);
        if (rc != kOk) return rc;
        if (epi->activation < GEMM_ACT_NONE || epi->activation > GEMM_ACT_GELU) return kInvalidArg;
        if (epi->bias && reinterpret_cast<uintptr_t>(epi->bias) % out_bytes(dtype))
            return kInvalidArg;
        if (M == 0 || N == 0) return kOk;
        const bool plain = epi->alpha == 1.f && epi->beta == 0.f && !epi->bias &&
                           epi->activation == GEMM_ACT_NONE;
        if (plain)
            return gemm(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype, stream);
        DeviceInfo* dev = nullptr;
        cudaMemPool_t pool = nullptr;
        rc = current_device(&dev, &pool);
        if (rc != kOk) return rc;
        const void* ptrs[4] = {K > 0 ? A : nullptr, K > 0 ? B : nullptr, C, epi->bias};
        rc = check_device_pointers(ptrs, 4, dev->device);
        if (rc != kOk) return rc;
        Problem p = normalise(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype);
        // a column-major C is stored transposed: its columns are our rows
        p.epi = EpiParams{1, epi->alpha, epi->beta, epi->bias, c_major == GEMM_MAJOR_K ? 1 : 0,
                          epi->activation};
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        if (K == 0) return launch_epilogue_only(p, *dev, s);
        const RunConfig cfg = resolve(
            make_key(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype));
        return run_device(p, *dev, pool, cfg, s);
    } catch (...) {
        return kCuda;
    }
}

int gemm_host(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_major,
              const void* B, int64_t ldb, int b_major, void* C, int64_t ldc, int c_major,
              int dtype, void* stream) {
    try {
        int rc = validate(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype);
        if (rc != kOk) return rc;
        if (M == 0 || N == 0) return kOk;
        DeviceInfo* dev = nullptr;
        cudaMemPool_t pool = nullptr;
        rc = current_device(&dev, &pool);
        if (rc != kOk) return rc;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        cudaStream_t h2d = nullptr, d2h = nullptr;
        copy_streams(*dev, &h2d, &d2h);
        const int ie = in_bytes(dtype), oe = out_bytes(dtype);

        // Device copies with 16-byte aligned row pitches.
        const int64_t a_inner = a_major == GEMM_MAJOR_K ? K : M, a_outer = a_major == GEMM_MAJOR_K ? M : K;
        const int64_t b_inner = b_major == GEMM_MAJOR_K ? K : N, b_outer = b_major == GEMM_MAJOR_K ? N : K;
        const int64_t c_inner = c_major == GEMM_MAJOR_MN ? N : M, c_outer = c_major == GEMM_MAJOR_MN ? M : N;
        const int64_t lda_d = round_up(a_inner > 0 ? a_inner : 1, 16 / ie);
        const int64_t ldb_d = round_up(b_inner > 0 ? b_inner : 1, 16 / ie);
        const int64_t ldc_d = round_up(c_inner, 16 / oe);
        const size_t a_bytes = (size_t)(a_outer * lda_d * ie), b_bytes = (size_t)(b_outer * ldb_d * ie);
        const size_t c_bytes = (size_t)(c_outer * ldc_d * oe);

        // One flat copy when both sides are packed rows, else a pitched copy.
        auto copy = [](void* dst, size_t dpitch, const void* src, size_t spitch, size_t width,
                       size_t height, cudaMemcpyKind kind, cudaStream_t st) {
            if (dpitch == width && spitch == width)
                return cudaMemcpyAsync(dst, src, width * height, kind, st);
            return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, kind, st);
        };
        void *dA = nullptr, *dB = nullptr, *dC = nullptr;
        if (cudaMallocFromPoolAsync(&dC, c_bytes, pool, s) != cudaSuccess ||
            (K > 0 && (cudaMallocFromPoolAsync(&dA, a_bytes, pool, s) != cudaSuccess ||
                       cudaMallocFromPoolAsync(&dB, b_bytes, pool, s) != cudaSuccess))) {
            cudaGetLastError();
            if (dA) cudaFreeAsync(dA, s);
            if (dB) cudaFreeAsync(dB, s);
            if (dC) cudaFreeAsync(dC, s);
            return kCuda;
        }
        // The same normalisation (C column-major: the transposed problem) of
        // the host and the device views; panels run over its rows.
        const Problem ph = normalise(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major,
                                     dtype);
        const Problem pd = normalise(M, N, K, dA, lda_d, a_major, dB, ldb_d, b_major, dC, ldc_d,
                                     c_major, dtype);
        const RunConfig cfg = resolve(make_key(M, N, K, dA, lda_d, a_major, dB, ldb_d, b_major,
                                               dC, ldc_d, c_major, dtype));
        // host_panel_rows gives at most about 8 panels; more than kMaxPanels
        // would only come from a model error, and then the call runs whole.
        constexpr int kMaxPanels = 64;
        // FFMA configurations 5 and 6 are sized for one CTA per SM, the others two
        const int ctas_per_sm = cfg.simt_config == 5 || cfg.simt_config == 6 ? 1 : 2;
        int64_t rows = host_panel_rows(pd.M, pd.N, pd.K, dtype == GEMM_F32, ctas_per_sm,
                                       cfg.cta_group ? cfg.cta_group : 2, cfg.multicast,
                                       dev->sm_count);
        if ((pd.M + rows - 1) / rows > kMaxPanels) rows = pd.M;
        const int np = (int)((pd.M + rows - 1) / rows);

        // Events: allocation done (s), each input piece in (B and the first
        // A panel in up to 4 pieces, the other A panels), each C panel
        // computed, both copy streams done.
        constexpr int kMaxEvents = 2 * kMaxPanels + 8;
        cudaEvent_t ev[kMaxEvents] = {};
        int nev = 0;
        auto event = [&]() -> cudaEvent_t {
            cudaEvent_t e = nullptr;
            if (nev < kMaxEvents &&
                cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess) {
                ev[nev++] = e;
                return e;
            }
            cudaGetLastError();
            return nullptr;
        };
        auto ok = [&](cudaError_t e) {
            if (e != cudaSuccess && rc == kOk) rc = kCuda;
            return rc == kOk;
        };
        // A goes in panel by panel (either major) when there are several.
        const bool a_panels = np > 1;
        const int64_t prow = rows;
        // With an fp32 C the first panel is pipelined over K as well: B and
        // that panel's A arrive in kp pieces of K and the panel runs as kp
        // GEMMs accumulating into C (host_k_pieces / host_k_bound, policy.h).
        const int kp = host_k_pieces(np, (int)oe, K);
        auto kbound = [&](int j) { return host_k_bound(K, kp, j); };
        dispatch_log("gemm_host %lldx%lldx%lld: %d row panel(s) of %lld rows, the first in %d "
                     "piece(s) of K",
                     (long long)pd.M, (long long)pd.N, (long long)K, np, (long long)rows, kp);
        Problem pb = pd;  // B replaced by its MN-major copy, if made
        void* bt = nullptr;
        cudaEvent_t e_alloc = event();
        if (!e_alloc) rc = kCuda;
        if (rc == kOk) ok(cudaEventRecord(e_alloc, s));
        if (rc == kOk) ok(cudaStreamWaitEvent(h2d, e_alloc, 0));
        // A K-major fp32 B that every panel would transpose for the FFMA
        // kernel is transposed once instead (piece by piece as it arrives).
        bool b_transpose = false;
        if (rc == kOk && np > 1 && K > 0 && dtype == GEMM_F32 && pd.b_kmajor) {
            if (want_transpose(prow, prow, pd.N, K, cfg.simt_transpose)) {
                const int64_t ld2 = round_up(pd.N, 4);
                if (cudaMallocFromPoolAsync(&bt, (size_t)(K * ld2 * 4), pool, s) != cudaSuccess) {
                    cudaGetLastError();
                    bt = nullptr;
                    rc = kCuda;
                } else {
                    pb.B = bt;
                    pb.ldb = ld2;
                    pb.b_kmajor = false;
                    b_transpose = true;
                }
            }
        }
        // Copies of B's k-range [k0, k1) and of rows m0 .. m1 of A's k-range.
        auto copy_b = [&](int64_t k0, int64_t k1) {
            const char* hB = static_cast<const char*>(ph.B);
            char* dBp = static_cast<char*>(const_cast<void*>(pd.B));
            if (pd.b_kmajor)  // columns k0 .. k1 of every row of B
                return ok(copy(dBp + k0 * ie, pd.ldb * ie, hB + k0 * ie, ph.ldb * ie,
                               (k1 - k0) * ie, pd.N, cudaMemcpyHostToDevice, h2d));
            return ok(copy(dBp + k0 * pd.ldb * ie, pd.ldb * ie, hB + k0 * ph.ldb * ie,
                           ph.ldb * ie, pd.N * ie, k1 - k0, cudaMemcpyHostToDevice, h2d));
        };
        auto copy_a = [&](int64_t m0, int64_t m1, int64_t k0, int64_t k1) {
            const char* hA = static_cast<const char*>(ph.A);
            char* dAp = static_cast<char*>(const_cast<void*>(pd.A));
            if (pd.a_kmajor)  // rows m0 .. m1, columns k0 .. k1
                return ok(copy(dAp + (m0 * pd.lda + k0) * ie, pd.lda * ie,
                               hA + (m0 * ph.lda + k0) * ie, ph.lda * ie, (k1 - k0) * ie, m1 - m0,
                               cudaMemcpyHostToDevice, h2d));
            return ok(copy(dAp + (k0 * pd.lda + m0) * ie, pd.lda * ie, hA + (k0 * ph.lda + m0) * ie,
                           ph.lda * ie, (m1 - m0) * ie, k1 - k0, cudaMemcpyHostToDevice, h2d));
        };
        for (int i = 0; i < np && rc == kOk; ++i) {
            const int64_t m0 = i * prow, m1 = std::min<int64_t>(pd.M, m0 + prow);
            Problem q = pb;
            q.M = m1 - m0;
            q.C = static_cast<char*>(pd.C) + m0 * pd.ldc * oe;
            if (K > 0) q.A = static_cast<const char*>(pd.A) + (pd.a_kmajor ? m0 * pd.lda : m0) * ie;
            // panel 0 in kp pieces of K (B piece by piece with it); later
            // panels whole, once their A rows are in (B is in by then)
            const int pieces = i == 0 ? kp : 1;
            for (int j = 0; j < pieces && rc == kOk; ++j) {
                const int64_t k0 = i == 0 ? kbound(j) : 0, k1 = i == 0 ? kbound(j + 1) : K;
                if (K > 0) {
                    cudaEvent_t e_in = event();
                    if (!e_in) { rc = kCuda; break; }
                    if (i == 0) copy_b(k0, k1);
                    if (rc == kOk && (a_panels || i == 0)) copy_a(m0, m1, k0, k1);
                    if (rc == kOk) ok(cudaEventRecord(e_in, h2d));
                    if (rc == kOk) ok(cudaStreamWaitEvent(s, e_in, 0));
                }
                if (rc == kOk && i == 0 && b_transpose)
                    rc = launch_transpose_f32(static_cast<const float*>(pd.B) + k0, pd.ldb,
                                              static_cast<float*>(bt) + k0 * pb.ldb, pb.ldb,
                                              pd.N, k1 - k0, *dev, s);
                Problem qk = q;
                if (pieces > 1) {
                    qk.K = k1 - k0;
                    qk.A = static_cast<const char*>(q.A) + (pb.a_kmajor ? k0 : k0 * pb.lda) * ie;
                    qk.B = static_cast<const char*>(q.B) + (pb.b_kmajor ? k0 : k0 * pb.ldb) * ie;
                    if (j > 0) qk.epi = EpiParams{1, 1.f, 1.f, nullptr, 0, GEMM_ACT_NONE};
                }
                if (rc == kOk) rc = run_device(qk, *dev, pool, cfg, s);
            }
            cudaEvent_t e_c = rc == kOk ? event() : nullptr;
            if (rc == kOk && !e_c) rc = kCuda;
            if (rc == kOk) ok(cudaEventRecord(e_c, s));
            if (rc == kOk) ok(cudaStreamWaitEvent(d2h, e_c, 0));
            if (rc == kOk)
                ok(copy(static_cast<char*>(ph.C) + m0 * ph.ldc * oe, ph.ldc * oe, q.C,
                        pd.ldc * oe, pd.N * oe, q.M, cudaMemcpyDeviceToHost, d2h));
        }
        // Whatever was enqueued on the copy streams finishes before the
        // caller's stream goes on (and before the scratch is freed).
        cudaEvent_t e_in = event(), e_out = event();
        if (e_in && cudaEventRecord(e_in, h2d) == cudaSuccess) cudaStreamWaitEvent(s, e_in, 0);
        else rc = rc == kOk ? kCuda : rc;
        if (e_out && cudaEventRecord(e_out, d2h) == cudaSuccess) cudaStreamWaitEvent(s, e_out, 0);
        else rc = rc == kOk ? kCuda : rc;
        cudaGetLastError();
        if (bt) cudaFreeAsync(bt, s);
        if (dA) cudaFreeAsync(dA, s);
        if (dB) cudaFreeAsync(dB, s);
        cudaFreeAsync(dC, s);
        for (int i = 0; i < nev; ++i) cudaEventDestroy(ev[i]);
        return rc;
    } catch (...) {
        return kCuda;
    }
}

int gemm_tune(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, int a_major,
              const void* B, int64_t ldb, int b_major, void* C, int64_t ldc, int c_major,
              int dtype, int iterations, void* stream, gemm_tuning* out) {
    try {
        gemm_tuning best{};
        if (out) *out = best;
        int rc = validate(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype);
        if (rc != kOk) return rc;
        if (M == 0 || N == 0 || K == 0) return kOk;
        DeviceInfo* dev = nullptr;
        cudaMemPool_t pool = nullptr;
        rc = current_device(&dev, &pool);
        if (rc != kOk) return rc;
        const void* ptrs[3] = {A, B, C};
        rc = check_device_pointers(ptrs, 3, dev->device);
        if (rc != kOk) return rc;
        if (iterations <= 0) iterations = 5;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        const Problem p =
            normalise(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype);

        // candidate configurations for this problem
        RunConfig cands[32];
        int n = 0;
        if (dtype == GEMM_F32) {
            const bool any_kmajor = p.a_kmajor || p.b_kmajor;
            for (int c = 1; c <= 9; ++c)
                for (int t = 1; t <= (any_kmajor ? 2 : 1); ++t) cands[n++] = {c, t, 2, 1, 0};
        } else {
            const bool c_aligned = aligned16_ld(C, ldc, out_bytes(dtype));
            // (CTA group, multicast, scheduler). The operand-multicast variant
            // is never a candidate: it runs only when the caller asks for it
            // (GEMM_OPT_TC_MULTICAST = 2).
            const int modes[4][3] = {{1, 1, 1}, {1, 1, 2}, {2, 1, 1}, {2, 1, 2}};
            for (const auto& m : modes)
                for (int st = c_aligned ? 0 : 1; st <= 1; ++st)
                    cands[n++] = {1, 0, m[0], m[1], st, 0, m[2]};
        }

        cudaEvent_t e0 = nullptr, e1 = nullptr;
        if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
            cudaGetLastError();
            if (e0) cudaEventDestroy(e0);
            return kCuda;
        }
        float best_ms = -1.f;
        RunConfig best_cfg = cands[0];
        for (int i = 0; i < n && rc == kOk; ++i) {
            rc = run_device(p, *dev, pool, cands[i], s);  // warm-up
            if (rc == kOk && cudaEventRecord(e0, s) != cudaSuccess) rc = kCuda;
            for (int it = 0; it < iterations && rc == kOk; ++it)
                rc = run_device(p, *dev, pool, cands[i], s);
            float ms = 0.f;
            if (rc == kOk && (cudaEventRecord(e1, s) != cudaSuccess ||
                              cudaEventSynchronize(e1) != cudaSuccess ||
                              cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess))
                rc = kCuda;
            if (rc != kOk) break;
            ms /= (float)iterations;
            if (best_ms < 0.f || ms < best_ms) {
                best_ms = ms;
                best_cfg = cands[i];
            }
        }
        cudaEventDestroy(e0);
        cudaEventDestroy(e1);
        if (rc != kOk) {
            cudaGetLastError();
            return rc;
        }
        best = gemm_tuning{best_cfg.simt_config, best_cfg.simt_transpose, best_cfg.cta_group,
                           best_cfg.multicast, best_cfg.tc_store, best_ms, n,
                           best_cfg.tc_scheduler};
        {
            std::lock_guard<std::mutex> lock(g_tune_mu);
            g_tune_table[make_key(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major,
                                  dtype)] = best;
        }
        if (out) *out = best;
        return kOk;
    } catch (...) {
        return kCuda;
    }
}

void gemm_tune_reset(void) {
    std::lock_guard<std::mutex> lock(g_tune_mu);
    g_tune_table.clear();
}

int softmax_rows(int64_t M, int64_t N, const float* x, int64_t ldx, float* y, int64_t ldy,
                 void* stream) {
    try {
        if (M < 0 || N < 0 || M > INT32_MAX || N > INT32_MAX) return kInvalidArg;
        if (M == 0 || N == 0) return kOk;
        if (!x || !y || ldx < N || ldy < N) return kInvalidArg;
        if (reinterpret_cast<uintptr_t>(x) % 4 || reinterpret_cast<uintptr_t>(y) % 4)
            return kInvalidArg;
        if (!span_ok(M, N, ldx, 4) || !span_ok(M, N, ldy, 4)) return kInvalidArg;
        if (N > softmax_max_cols()) return kUnsupported;
        DeviceInfo* dev = nullptr;
        int rc = current_device(&dev, nullptr);
        if (rc != kOk) return rc;
        const void* ptrs[2] = {x, y};
        rc = check_device_pointers(ptrs, 2, dev->device);
        if (rc != kOk) return rc;
        return launch_softmax_rows(M, N, x, ldx, y, ldy, *dev, g_wait_limit_ns.load(),
                                   g_softmax_fault_inject.load(),
                                   static_cast<cudaStream_t>(stream));
    } catch (...) {
        return kCuda;
    }
}

const char* gemm_strerror(int status) {
    switch (status) {
        case GEMM_OK: return "success";
        case GEMM_ERR_INVALID_ARG:
            return "invalid argument (size, pointer, leading dimension, enum or alignment)";
        case GEMM_ERR_UNSUPPORTED: return "no usable device, or the device is not sm_103";
        case GEMM_ERR_CUDA: return "a CUDA runtime call failed";
        case GEMM_ERR_TIMEOUT:
            return "a kernel gave up waiting on a pipeline barrier (time limit exceeded)";
        default: return "unknown status";
    }
}

int gemm_check_device_error(void* stream) {
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev, nullptr);
    if (rc != kOk) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return kCuda;
    }
    ErrWord word = 0;
    if (cudaMemcpy(&word, dev->err_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return kCuda;
    }
    if (word == 0) return kOk;
    const ErrWord zero = 0;
    if (cudaMemcpy(dev->err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return kCuda;
    }
    return kTimeout;
}

int gemm_device_checks(void* stream, uint64_t* first) {
    if (!first) return kInvalidArg;
    *first = 0;
#ifndef LIBGEMM_DEVICE_CHECKS
    (void)stream;
    return kUnsupported;
#else
    DeviceInfo* dev = nullptr;
    int rc = current_device(&dev, nullptr);
    if (rc != kOk) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return kCuda;
    }
    unsigned long long word = 0;
    if (cudaMemcpy(&word, dev->check_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return kCuda;
    }
    if (word != 0) {
        const unsigned long long zero = 0;
        if (cudaMemcpy(dev->check_word, &zero, sizeof(zero), cudaMemcpyHostToDevice) !=
            cudaSuccess) {
            cudaGetLastError();
            return kCuda;
        }
    }
    *first = word;
    return kOk;
#endif
}

void gemm_release_workspace(void) {
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    for (int d = 0; d < kMaxDevices; ++d) {
        if (!g_dev[d].pool) continue;
        if (cudaSetDevice(d) != cudaSuccess) { cudaGetLastError(); continue; }
        cudaDeviceSynchronize();
    }
    cudaSetDevice(cur);
    scratch_cache_clear();  // the per-stream buffers go back to the pools
    for (int d = 0; d < kMaxDevices; ++d) {
        if (!g_dev[d].pool) continue;
        if (cudaSetDevice(d) != cudaSuccess) { cudaGetLastError(); continue; }
        cudaMemPoolTrimTo(g_dev[d].pool, 0);
    }
    cudaSetDevice(cur);
    cudaGetLastError();
}

uint64_t gemm_launch_count(void) { return g_launches.load(); }

int gemm_set_option(int option, int64_t value) {
    switch (option) {
        case GEMM_OPT_WAIT_LIMIT_NS:
            if (value < 0) return GEMM_ERR_INVALID_ARG;
            g_wait_limit_ns.store(value == 0 ? 1000000000ull : (uint64_t)value);
            return GEMM_OK;
        case GEMM_OPT_TC_CTA_GROUP:
            if (value != 0 && value != 1 && value != 2) return GEMM_ERR_INVALID_ARG;
            g_cta_group.store((int)value);
            return GEMM_OK;
        case GEMM_OPT_TC_FAULT_INJECT:
            if (value != 0 && value != 1) return GEMM_ERR_INVALID_ARG;
            g_fault_inject.store((int)value);
            return GEMM_OK;
        case GEMM_OPT_SIMT_CONFIG:
            if (value < 0 || value > 9) return GEMM_ERR_INVALID_ARG;
            g_simt_config.store((int)value);
            return GEMM_OK;
        case GEMM_OPT_SIMT_TRANSPOSE:
            if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
            g_simt_transpose.store((int)value);
            return GEMM_OK;
        case GEMM_OPT_TC_STORE:
            if (value != 0 && value != 1) return GEMM_ERR_INVALID_ARG;
            g_tc_store.store((int)value);
            return GEMM_OK;
        case GEMM_OPT_TC_MULTICAST:
            if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
            g_tc_multicast.store((int)value);
            return GEMM_OK;
        case GEMM_OPT_SOFTMAX_FAULT_INJECT:
            if (value != 0 && value != 1) return GEMM_ERR_INVALID_ARG;
            g_softmax_fault_inject.store((int)value);
            return GEMM_OK;
        case GEMM_OPT_SIMT_SPLIT_TAIL:
            if (value < 0 || value > 3) return GEMM_ERR_INVALID_ARG;
            g_simt_split.store((int)value);
            return GEMM_OK;
        case GEMM_OPT_TC_SCHEDULER:
            if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
            g_tc_scheduler.store((int)value);
            return GEMM_OK;
        case GEMM_OPT_SIMT_FAULT_INJECT:
            if (value != 0 && value != 1) return GEMM_ERR_INVALID_ARG;
            g_simt_fault_inject.store((int)value);
            return GEMM_OK;
        case GEMM_OPT_TC_TILE_N:
            if (value != 0 && value != 64 && value != 128 && value != 256)
                return GEMM_ERR_INVALID_ARG;
            g_tc_tile_n.store((int)value);
            return GEMM_OK;
        case GEMM_OPT_TC_SPLIT_TAIL:
            if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
            g_tc_split.store((int)value);
            return GEMM_OK;
        default: return GEMM_ERR_INVALID_ARG;
    }
}

int64_t gemm_get_option(int option) {
    switch (option) {
        case GEMM_OPT_WAIT_LIMIT_NS: return (int64_t)g_wait_limit_ns.load();
        case GEMM_OPT_TC_CTA_GROUP: return g_cta_group.load();
        case GEMM_OPT_TC_FAULT_INJECT: return g_fault_inject.load();
        case GEMM_OPT_SIMT_CONFIG: return g_simt_config.load();
        case GEMM_OPT_SIMT_TRANSPOSE: return g_simt_transpose.load();
        case GEMM_OPT_TC_STORE: return g_tc_store.load();
        case GEMM_OPT_TC_MULTICAST: return g_tc_multicast.load();
        case GEMM_OPT_SOFTMAX_FAULT_INJECT: return g_softmax_fault_inject.load();
        case GEMM_OPT_SIMT_SPLIT_TAIL: return g_simt_split.load();
        case GEMM_OPT_TC_SCHEDULER: return g_tc_scheduler.load();
        case GEMM_OPT_SIMT_FAULT_INJECT: return g_simt_fault_inject.load();
        case GEMM_OPT_TC_TILE_N: return g_tc_tile_n.load();
        case GEMM_OPT_TC_SPLIT_TAIL: return g_tc_split.load();
        default: return -1;
    }
}

}  // extern "C"
