// sgemm_cfg9.cu -- FFMA tile configuration 9: configuration 7's 128 x 128
// tile with shared memory filled by TMA (the kernel is in sgemm_tma.cuh)
// when both operands are MN-major with 16-byte aligned bases and row
// pitches; other operand variants, and pitches the driver's tensor-map
// encoder rejects, run configuration 7's cp.async kernel.
#include "sgemm_sk.cuh"
#include "sgemm_tma.cuh"

namespace libgemm {
namespace {

using Cfg7 = SgCfg<16, 4, true, 2, 16>;  // the cp.async fallback

// Launches the TMA-fed kernel for maps `ta` (A) and `tb` (B).
template <class TC>
int launch_tma(SgemmParams sp, const CUtensorMap& ta, const CUtensorMap& tb,
               const DeviceInfo& dev, int split_mode, Scratch* scratch, uint64_t wait_limit_ns,
               int fault_inject, cudaStream_t stream) {
    using Cfg = typename TC::Cfg;
    auto kern = sgemm_ffma_tma_kernel<TC>;
    auto kern_sk = sgemm_ffma_tma_sk_kernel<TC>;
    static std::atomic<uint64_t> configured{0}, configured_sk{0};
    static std::atomic<int> per_sm[64];
    const int device = dev.device;
    if (!configure_once(kern, configured, device, TC::SMEM) ||
        !configure_once(kern_sk, configured_sk, device, TC::SMEM))
        return kCuda;
    int occ = per_sm[device & 63].load();
    if (occ == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Cfg::THREADS, TC::SMEM) !=
            cudaSuccess) {
            cudaGetLastError();
            occ = -1;
        }
        per_sm[device & 63].store(occ);
    }
    const int nkt = (sp.K + TC::BK - 1) / TC::BK;
    SkArgs sk{0, nullptr};
    plan_split(sp, occ > 0 ? occ * dev.sm_count : 0, dev.sm_count, nkt, split_mode, &sk.ctas);
    const int64_t tail = (int64_t)sp.tiles_m * sp.tiles_n - sp.dp_tiles;
    if (tail > 0) {
        // K-slices: a partial tile per slice; stream-K: one per stream-K CTA
        // and the CTAs' flags
        const size_t parts = sk.ctas > 0 ? (size_t)sk.ctas : (size_t)tail * sp.splits;
        const size_t flags = sk.ctas > 0 ? (size_t)sk.ctas * 8 : 0;
        sp.ws = scratch
            ? static_cast<float*>(scratch->get(parts * BM * BN * sizeof(float) + flags))
            : nullptr;
        sk.flags = sp.ws && flags
            ? reinterpret_cast<unsigned long long*>(sp.ws + parts * BM * BN)
            : nullptr;
        if (!sp.ws) {  // no scratch: compute every tile whole
            sp.dp_tiles = sp.tiles_m * sp.tiles_n;
            sp.splits = 1;
            sk.ctas = 0;
        }
    }
    const TmaArgs x{dev.err_word, next_generation(), (unsigned long long)wait_limit_ns,
                    fault_inject};
    const int64_t fix = (int64_t)sp.tiles_m * sp.tiles_n - sp.dp_tiles;
    const int64_t units = sk.ctas > 0 ? sp.dp_tiles + sk.ctas : sp.dp_tiles + fix * sp.splits;
    if (sk.ctas > 0)
        kern_sk<<<dim3((unsigned)units), dim3(Cfg::THREADS), TC::SMEM, stream>>>(sp, ta, tb, x,
                                                                                 sk);
    else
        kern<<<dim3((unsigned)units), dim3(Cfg::THREADS), TC::SMEM, stream>>>(sp, ta, tb, x);
    if (cudaGetLastError() != cudaSuccess) return kCuda;
    note_launch();
    if (sk.ctas > 0)
        dispatch_log("FFMA SGEMM (TMA) %dx%dx%d: %d x %d tiles of 128 x 128, %d whole, "
                     "%d stream-K CTAs over the rest",
                     sp.M, sp.N, sp.K, sp.tiles_m, sp.tiles_n, sp.dp_tiles, sk.ctas);
    else
        dispatch_log("FFMA SGEMM (TMA) %dx%dx%d: %d x %d tiles of 128 x 128, %d whole, "
                     "the rest in %d K-slices of %d k-tiles",
                     sp.M, sp.N, sp.K, sp.tiles_m, sp.tiles_n, sp.dp_tiles, sp.splits,
                     sp.kt_slice);
    if (fix > 0 && sk.ctas == 0) {  // stream-K CTAs add up partials themselves
        sgemm_split_fixup_kernel<Cfg::TN>
            <<<dim3((unsigned)fix), dim3(Cfg::THREADS), 0, stream>>>(sp);
        if (cudaGetLastError() != cudaSuccess) return kCuda;
        note_launch();
    }
    return kOk;
}

}  // namespace

int launch_sgemm_cfg9(const SgemmParams& sp, int av, int bv, const DeviceInfo& dev,
                      int split_mode, Scratch* scratch, uint64_t wait_limit_ns, int fault_inject,
                      cudaStream_t s) {
    using TC = TmaCfg<SgCfg<16, 6, true, 2, 16>, 2>;
    if (av == 4 && bv == 4) {
        // A: M x K MN-major = K rows of M contiguous floats; box 128 (M) x 16 (K); B likewise.
        alignas(64) CUtensorMap ta, tb;
        if (encode_tma_f32_2d(&ta, sp.A, (uint64_t)sp.M, (uint64_t)sp.K, (uint64_t)sp.lda, BM,
                              TC::BK) &&
            encode_tma_f32_2d(&tb, sp.B, (uint64_t)sp.N, (uint64_t)sp.K, (uint64_t)sp.ldb, BN,
                              TC::BK))
            return launch_tma<TC>(sp, ta, tb, dev, split_mode, scratch, wait_limit_ns,
                                  fault_inject, s);
        // a map the encoder rejects (e.g. a row pitch of 2^40 bytes or more): cp.async
    }
    return launch_layout<Cfg7>(sp, av, bv, dev.device, dev.sm_count, split_mode, scratch, s);
}

}  // namespace libgemm
