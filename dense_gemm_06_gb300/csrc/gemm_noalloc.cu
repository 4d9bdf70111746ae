// gemm_noalloc.cu -- gemm_noalloc(): the 16-bit tensor-core GEMM for callers
// that must not allocate device memory.
//
// gemm() takes scratch for repacking A or B (rows whose byte pitch or base is
// not a multiple of 16, which TMA cannot read) from a stream-ordered pool, and
// the pool may have to grow. Some callers cannot allow that: a serving loop
// that has reserved all device memory up front for its own allocator, or a
// latency-critical path where a device allocation (and the synchronisation
// cudaMalloc may imply) is not acceptable after start-up. For them this entry
// point repacks into a fixed array that lives in the library's own device
// image instead, and never calls cudaMalloc, cudaFree or any other
// allocating routine.
//
// The array (kFixedScratchBytes = 32 MiB) is a file-scope __device__ variable,
// so every GPU that loads the library holds it until the process exits. In
// host code its name is only a host-side stand-in, never a device address:
// the address is looked up once per device with cudaGetSymbolAddress (with
// that device current) and passed to the kernels.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/gemm.h"
#include "internal.h"
#include "repack16.cuh"

namespace libgemm {
namespace {

constexpr int64_t kFixedScratchBytes = 32ll << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

struct FixedDevice {
    std::once_flag once;
    int status = kOk;
    DeviceInfo info{};
    unsigned char* scratch = nullptr;  // device address of g_fixed_scratch
};
FixedDevice g_fixed[kMaxDevices];

// One-time set-up for the current device (run by its first gemm_noalloc call).
int fixed_device(FixedDevice** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return kUnsupported;
    }
    FixedDevice& st = g_fixed[dev];
    std::call_once(st.once, [&st, dev] {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            st.status = kUnsupported;
            return;
        }
        if (major != 10 || minor != 3) {
            st.status = kUnsupported;
            return;
        }
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fixed_scratch) != cudaSuccess) {
            cudaGetLastError();
            st.status = kCuda;
            return;
        }
        ErrWord* err = nullptr;
        if (error_word_address(&err) != kOk) {
            st.status = kCuda;
            return;
        }
        st.scratch = static_cast<unsigned char*>(p);
        st.info.device = dev;
        st.info.sm_count = sms;
        st.info.cc_major = major;
        st.info.cc_minor = minor;
        st.info.err_word = err;
        if (check_word_address(&st.info.check_word) != kOk) {
            st.status = kCuda;
            return;
        }
        st.status = kOk;
    });
    if (st.status != kOk) return st.status;
    *out = &st;
    return kOk;
}

// C = 0 for K == 0: `rows` rows of `row_bytes` bytes, `pitch` bytes apart.
__global__ void zero_fixed_kernel(unsigned char* C, int64_t rows, int64_t row_bytes,
                                  int64_t pitch) {
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x)  // a block per row
        for (int64_t c = threadIdx.x; c < row_bytes; c += blockDim.x) C[r * pitch + c] = 0;
}

bool rows_tma_ready(const void* p, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && ((ld * 2) & 15) == 0;
}

}  // namespace
}  // namespace libgemm

using namespace libgemm;

extern "C" int gemm_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                            int a_major, const void* B, int64_t ldb, int b_major, void* C,
                            int64_t ldc, int c_major, int dtype, void* stream) {
    try {
        if (dtype == GEMM_F32) return kUnsupported;  // 16-bit inputs only
        int rc = check_args(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major, dtype);
        if (rc != kOk) return rc;
        if (M == 0 || N == 0) return kOk;
        Problem p = normalised(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc, c_major,
                               dtype);
        FixedDevice* fd = nullptr;
        rc = fixed_device(&fd);
        if (rc != kOk) return rc;
        const void* ptrs[3] = {K > 0 ? A : nullptr, K > 0 ? B : nullptr, C};
        rc = check_device_pointers(ptrs, 3, fd->info.device);
        if (rc != kOk) return rc;
        if (K == 0) {  // C = 0, as gemm() does
            const int64_t esize = dtype <= GEMM_BF16_F32 ? 4 : 2;
            int64_t blocks = p.M;  // a block per row of C
            const int64_t cap = (int64_t)fd->info.sm_count * 8;
            if (blocks > cap) blocks = cap;
            zero_fixed_kernel<<<(int)(blocks < 1 ? 1 : blocks), 256, 0,
                                static_cast<cudaStream_t>(stream)>>>(
                static_cast<unsigned char*>(p.C), p.M, p.N * esize, p.ldc * esize);
            if (cudaGetLastError() != cudaSuccess) return kCuda;
            note_launch();
            return kOk;
        }

        // Plan the repacked copies inside the fixed array before launching
        // anything, and reject problems that do not fit.
        const void** ops[2] = {&p.A, &p.B};
        int64_t* lds[2] = {&p.lda, &p.ldb};
        const bool kmaj[2] = {p.a_kmajor, p.b_kmajor};
        const int64_t rows[2] = {p.M, p.N};
        int64_t off[2] = {-1, -1}, ld2[2] = {0, 0}, inner[2] = {0, 0}, outer[2] = {0, 0};
        int64_t used = 0;
        for (int i = 0; i < 2; ++i) {
            if (rows_tma_ready(*ops[i], *lds[i])) continue;
            inner[i] = kmaj[i] ? p.K : rows[i];
            outer[i] = kmaj[i] ? rows[i] : p.K;
            ld2[i] = (inner[i] + 7) / 8 * 8;
            const int64_t bytes = (outer[i] * ld2[i] * 2 + 255) / 256 * 256;
            if (bytes > kFixedScratchBytes - used) return kInvalidArg;  // over the limit
            off[i] = used;
            used += bytes;
        }

        cudaStream_t s = static_cast<cudaStream_t>(stream);
        Repack16 job[2] = {};  // outer == 0: nothing to repack
        for (int i = 0; i < 2; ++i) {
            if (off[i] < 0) continue;
            uint16_t* dst = reinterpret_cast<uint16_t*>(fd->scratch + off[i]);
            job[i] = {static_cast<const uint16_t*>(*ops[i]), dst, *lds[i], ld2[i], outer[i],
                      inner[i]};
            *ops[i] = dst;
            *lds[i] = ld2[i];
        }
        const int64_t rows_all = job[0].outer + job[1].outer;
        if (rows_all > 0) {  // both operands in one launch, a warp per row
            repack16_kernel<<<repack16_blocks(rows_all, fd->info.sm_count), 256, 0, s>>>(job[0],
                                                                                       job[1]);
            if (cudaGetLastError() != cudaSuccess) return kCuda;
            note_launch();
        }
        // The same kernel options gemm() would resolve for this problem
        // (caller's options, then a gemm_tune() entry, then the default).
        TcLaunch o = resolve_tc_options(M, N, K, A, lda, a_major, B, ldb, b_major, C, ldc,
                                        c_major, dtype);
        o.after_repack = rows_all > 0 ? 1 : 0;
        return launch_gemm_tc(p, fd->info, o, s);
    } catch (...) {
        return kCuda;
    }
}
