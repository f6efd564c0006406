// mla_tc.cu -- tensor-core (tcgen05) partial MLA decode.  (Kernel pending.)
#include "mla_internal.h"

namespace mla {
int launch_tc(const DecodeArgs&) {
  return fail(MLA_ERR_UNSUPPORTED, "tensor-core kernel not built yet");
}
}  // namespace mla

extern "C" int mla_pair_slots(void) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mla::cuda_fail(e, "cudaGetDevice");
  int n = mla_num_sms(dev);
  return n < 0 ? n : n / 2;
}
