// sgemm_cfg8.cu -- FFMA tile configuration 8 (SgCfg<32, 3, true, 2, 16>), all operand
// variants; the kernel templates are in sgemm_ffma.cuh.
#include "sgemm_ffma.cuh"

namespace libgemm {

int launch_sgemm_cfg8(const SgemmParams& sp, int av, int bv, int device, int sm_count,
                      int split_mode, Scratch* scratch, cudaStream_t s) {
    return launch_layout<SgCfg<32, 3, true, 2, 16>>(sp, av, bv, device, sm_count, split_mode, scratch, s);
}

}  // namespace libgemm
