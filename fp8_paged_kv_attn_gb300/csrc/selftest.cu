// Self-test of the split attention kernels' failure path (kvq_selftest_wait,
// which = 0; the weight ring's twin, which = 1, sits beside its wait in
// wq_gemm.cu).  No fault and no hang: every wait here is the bounded wait the
// kernels use, and the barrier it waits on is one that nothing arrives at.
#include "kvq_internal.h"
#include "decode_common.cuh"

namespace kvq {

// One CTA starts a real 64-byte bulk copy on one mbarrier, then every thread
// waits with ctl_wait on a second barrier that nothing arrives at.  The wait
// gives up after its bound, raises KVQ_ERRBIT_TIMEOUT once and sets the fail
// flag; thread 0 then drains the copy it started (the bounded mbar_wait on
// the first barrier) and stores the copied word in *landed.
__global__ void attn_wait_selftest_kernel(const uint32_t *src, uint32_t *err_word,
                                          uint32_t *landed) {
  __shared__ __align__(128) uint32_t buf[16];
  __shared__ Ctrl ctl;
  if (threadIdx.x == 0) ctrl_init(ctl, 2, 1);
  __syncthreads();
  grid_dependency_wait();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&ctl.full[0], sizeof(buf));
    bulk_g2s(buf, src, sizeof(buf), &ctl.full[0]);
  }
  const bool ok = ctl_wait(ctl, &ctl.full[1], 0, err_word);  // nothing arrives on full[1]
  if (threadIdx.x == 0) {
    const bool drained = mbar_wait(&ctl.full[0], 0);
    *landed = (!ok && drained) ? buf[0] : 0u;
  }
}

kvq_status selftest_attn_wait(const uint32_t *src, uint32_t *err_word, uint32_t *landed,
                              cudaStream_t stream) {
  const cudaError_t e =
      launch_dependent(attn_wait_selftest_kernel, dim3(1), dim3(64), 0, stream, src, err_word,
                       landed);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
