// sgemm_cfg1.cu -- FFMA tile configuration 1 (SgCfg<16, 4, true, 2>), all operand
// variants; the kernel templates are in sgemm_ffma.cuh.
#include "sgemm_ffma.cuh"

namespace libgemm {

int launch_sgemm_cfg1(const SgemmParams& sp, int av, int bv, int device, int sm_count,
                      int split_mode, Scratch* scratch, cudaStream_t s) {
    return launch_layout<SgCfg<16, 4, true, 2>>(sp, av, bv, device, sm_count, split_mode, scratch, s);
}

}  // namespace libgemm
