// Tensor-core MLA decode for sm_103a (tcgen05 + TMEM + TMA): placeholder
// until the kernel lands; every shape goes to the CUDA-core kernel.
#include "common.cuh"
#include "internal.h"

namespace mla {

bool tc_supported(int dtype, int H, int T_q, int d_c, int d_r) {
  (void)dtype; (void)H; (void)T_q; (void)d_c; (void)d_r;
  return false;
}

int tc_workers(int num_sms) { return num_sms / 2; }

cudaError_t launch_decode_tc(const DecodeArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace mla
