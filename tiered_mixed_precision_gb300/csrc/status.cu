// Device-side status: reading the status words that kernels write when a bounded wait gives
// up, and a self-test of that mechanism. The library's kernels never trap and never spin
// without a limit: a wait on an mbarrier that does not complete within its limit records a
// nonzero code in status[0] and the kernel returns; the results of that call are then
// invalid, and fade_check_status reports it.
#include "fade_internal.cuh"

namespace fade {
namespace {

// Two warps share one mbarrier: warp 1 (the producer) arrives on it only when `arrive` is
// nonzero; lane 0 of warp 0 (the consumer) waits with the bounded wait the attention kernel
// uses, with a limit of `limit` cycles, and records code 1 on a timeout.
__global__ void __launch_bounds__(64) bounded_wait_selftest_kernel(int32_t* status, int arrive,
                                                                   long long limit) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 32 && arrive) mbar_arrive(b);
  if (threadIdx.x == 0) mbar_wait_limit(b, 0, status, 1, limit);
}

}  // namespace
}  // namespace fade

using namespace fade;

extern "C" fade_status_t fade_check_status(const fade_layer_t* L, void* stream) {
  clear_error();
  if (!L || !L->status) return set_error(FADE_ERR_INVALID_ARGUMENT, "layer or status is NULL");
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess)
    return set_error(FADE_ERR_CUDA, "fade_check_status: %s", cudaGetErrorString(e));
  int32_t w[FADE_STATUS_WORDS];
  e = cudaMemcpy(w, L->status, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess)
    return set_error(FADE_ERR_CUDA, "fade_check_status: %s", cudaGetErrorString(e));
  if (w[0] >= kDevCheckBase)
    return set_error(FADE_ERR_DEVICE_CHECK,
                     "a device-side check failed (code %d: 16 demote slot, 17 append slot, "
                     "18 compaction row, 19 attention tile); results since the last reset are "
                     "invalid", w[0]);
  if (w[0] != 0)
    return set_error(FADE_ERR_TIMEOUT,
                     "a kernel gave up a bounded wait (code %d: 1 consumer stage, 2 producer "
                     "slot, 3 producer drain); results since the last reset are invalid",
                     w[0]);
  return FADE_OK;
}

extern "C" fade_status_t fade_selftest_bounded_wait(int32_t* status, int32_t producer_arrives,
                                                    int64_t limit_cycles, void* stream) {
  clear_error();
  FADE_RANGE("fade_selftest_bounded_wait");
  if (!status || (reinterpret_cast<uintptr_t>(status) & 3))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "status is NULL or not 4-byte aligned");
  if (limit_cycles < 1 || limit_cycles > kWaitCycles)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "limit_cycles outside [1, %lld]", kWaitCycles);
  bounded_wait_selftest_kernel<<<1, 64, 0, as_stream(stream)>>>(status, producer_arrives != 0,
                                                               (long long)limit_cycles);
  return launch_status("fade_selftest_bounded_wait");
}
