// ep_selftest_bounded_waits: a self-test of the bounded device waits that
// the library's kernels rely on so that no wait can hang the GPU.  Block 0
// waits on an mbarrier that nothing arrives on (the form of every stage wait
// in the dispatch and combine kernels); block 1 enters a grid barrier that
// block 0 never reaches (the form of the expanded layout's barrier).  Both
// waits must give up after the wait limit, set EP_ERRBIT_TIMEOUT and let the
// kernel return, so that the context stays usable for the next call.
#include <cstdint>

#include "ep_device.cuh"

namespace ep {
namespace {

// The grid barrier's words.  Zero at module load; the block whose wait gives
// up zeroes them again, so every call starts from zero.
__device__ GridBarrierWords g_selftest_barrier;

__global__ void __launch_bounds__(kWarpSize)
    selftest_wait_kernel(uint32_t *error_word, int32_t *gave_up, uint64_t *elapsed_ns) {
  __shared__ uint64_t bar;
  __shared__ int s_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const uint64_t t0 = global_timer_ns();
  bool ok;
  if (blockIdx.x == 0) {
    ok = mbar_wait_bounded(&bar, 0u);  // the phase never completes: no arrival
  } else {
    ok = grid_barrier(&g_selftest_barrier, &s_flag);  // block 0 never arrives
    if (!ok && threadIdx.x == 0) atomicExch(&g_selftest_barrier.arrive, 0u);
  }
  const uint64_t t1 = global_timer_ns();
  if (threadIdx.x == 0) {
    gave_up[blockIdx.x] = ok ? 0 : 1;
    elapsed_ns[blockIdx.x] = t1 - t0;
    if (!ok) atomicOr(error_word, EP_ERRBIT_TIMEOUT);
  }
}

}  // namespace
}  // namespace ep

extern "C" ep_status_t ep_selftest_bounded_waits(uint32_t *error_word, int32_t *gave_up, uint64_t *elapsed_ns,
                                                 ep_stream_t stream) {
  using namespace ep;
  static const char *fn = "ep_selftest_bounded_waits";
  clear_error();
  ep_status_t s = check_ptr(fn, "error_word", error_word, 4, true);
  if (s == EP_OK) s = check_ptr(fn, "gave_up", gave_up, 4, true);
  if (s == EP_OK) s = check_ptr(fn, "elapsed_ns", elapsed_ns, 8, true);
  if (s != EP_OK) return s;
  if (current_device_info() == nullptr) return EP_ERR_CUDA;
  // A plain launch (no programmatic dependent launch): the kernel starts once
  // the work ahead of it on the stream has finished.
  selftest_wait_kernel<<<2, kWarpSize, 0, reinterpret_cast<cudaStream_t>(stream)>>>(error_word, gave_up,
                                                                                     elapsed_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch selftest_wait_kernel");
  return EP_OK;
}
