// gemm_tc_bf16_f32.cu -- the tcgen05 GEMM for bf16 operands and a f32 C, every
// CTA mode and operand major; the kernel templates are in gemm_tc.cuh.
#include "gemm_tc.cuh"

namespace libgemm {

int launch_gemm_tc_bf16_f32(TcParams& tp, int cg, bool mc, bool a_mn, bool b_mn,
                       const DeviceInfo& dev, cudaStream_t s) {
    if (cg == 1) return dispatch_majors<1, false, true, float>(tp, a_mn, b_mn, dev, s);
    if (mc) return dispatch_majors<2, true, true, float>(tp, a_mn, b_mn, dev, s);
    return dispatch_majors<2, false, true, float>(tp, a_mn, b_mn, dev, s);
}

}  // namespace libgemm
