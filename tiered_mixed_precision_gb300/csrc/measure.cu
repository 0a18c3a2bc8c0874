// Measurement helper: the rate of separately rounded fp32 operations on this device, the
// denominator of the re-positioning kernel's ALU roofline. The kernel runs independent chains
// of packed fp32 multiplies (mul.rn.f32x2: two fp32 operations per lane per instruction, the
// form the re-positioning arithmetic takes) on registers only, so its time divided into the
// operations it performs is the device's peak for that instruction form.
#include "fade_internal.cuh"

namespace fade {
namespace {

constexpr int kRateChains = 8;      // independent chains per thread
constexpr int kRateThreads = 256;

__global__ void __launch_bounds__(kRateThreads) fp32_rate_kernel(int iters, float one,
                                                                 float* sink) {
  f2x x[kRateChains];
  const f2x c = f2_pack(one, one);
#pragma unroll
  for (int k = 0; k < kRateChains; ++k)
    x[k] = f2_pack(1.0f + 1e-3f * (threadIdx.x + k), 0.5f + 1e-3f * k);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < kRateChains; ++k)
      asm volatile("mul.rn.f32x2 %0, %0, %1;" : "+l"(x[k]) : "l"(c));
  }
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kRateChains; ++k) {
    float lo, hi;
    f2_unpack(x[k], lo, hi);
    s += lo + hi;
  }
  if (s == 12345.f) sink[threadIdx.x] = s;  // never true: keeps the chains alive
}

}  // namespace
}  // namespace fade

using namespace fade;

extern "C" fade_status_t fade_measure_fp32_rate(int32_t blocks, int32_t iters, float* sink,
                                                double* ops_out, void* stream) {
  clear_error();
  FADE_RANGE("fade_measure_fp32_rate");
  if (blocks < 1 || iters < 1 || !sink)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "blocks and iters must be positive, sink set");
  fp32_rate_kernel<<<blocks, kRateThreads, 0, as_stream(stream)>>>(iters, 1.0f, sink);
  if (ops_out)
    *ops_out = (double)blocks * kRateThreads * (double)iters * kRateChains * 2.0;
  return launch_status("fade_measure_fp32_rate");
}
