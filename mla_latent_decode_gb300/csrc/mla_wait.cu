// mla_wait.cu -- test entry point of the bounded pipeline waits.
//
// Every wait of the decode kernels goes through ptx::mbar_wait, which gives up
// after a time limit of %globaltimer or when the CTA's abort flag is raised,
// so a broken pipeline ends with MLA_STATUS_WAIT_TIMEOUT instead of a hung
// GPU.  This kernel runs that same wait on a barrier phase that nothing
// completes (or that another warp completes or aborts late), so a test can
// watch it give up and return.  It holds no tensor memory and starts no TMA,
// bulk copy or MMA, so the CTA always ends cleanly.
#include "mla_internal.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

using namespace ptx;

__global__ void __launch_bounds__(64, 1)
    mla_wait_probe_kernel(int mode, uint64_t delay_ns, int* status,
                          unsigned long long* elapsed_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // the waiter: phase 0 of a one-arrival barrier
    const uint64_t t0 = globaltimer();
    const bool ok = mbar_wait(smem_u32(&bar), 0, &abort_flag);
    *elapsed_ns = globaltimer() - t0;
    if (!ok) atomicOr(status, MLA_STATUS_WAIT_TIMEOUT);
  } else if (threadIdx.x == 32 && mode != 0) {
    // the other warp: after delay_ns (a loop bounded by that delay), raise
    // the abort flag (mode 1) or complete the phase (mode 2)
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < delay_ns) __nanosleep(1000);
    if (mode == 1)
      *reinterpret_cast<volatile int*>(&abort_flag) = 1;
    else
      mbar_arrive(smem_u32(&bar));
  }
  __syncthreads();
}

}  // namespace
}  // namespace mla

extern "C" int mla_debug_wait(int mode, int delay_us, int* status,
                              uint64_t* elapsed_ns, mla_stream_t stream) {
  using namespace mla;
  if (mode < 0 || mode > 2)
    return fail(MLA_ERR_INVALID_ARG, "mode %d: expected 0, 1 or 2", mode);
  if (delay_us < 0 || delay_us > 1000000)
    return fail(MLA_ERR_INVALID_ARG, "delay_us %d outside [0, 1000000]",
                delay_us);
  if (!status || !elapsed_ns)
    return fail(MLA_ERR_INVALID_ARG, "status and elapsed_ns are required");
  if (!aligned(status, 4) || !aligned(elapsed_ns, 8))
    return fail(MLA_ERR_MISALIGNED, "status or elapsed_ns misaligned");
  mla_wait_probe_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(
      mode, (uint64_t)delay_us * 1000u, status,
      reinterpret_cast<unsigned long long*>(elapsed_ns));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch mla_wait_probe_kernel");
  return MLA_OK;
}
