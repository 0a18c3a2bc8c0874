// Symmetric absmax quantisation with little-endian bit-packing, and its inverse.
// Source: page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术", §量化与Bit-Packing (INT4/INT2
// symmetric quantisation with bit-packing); one fp16 scale per 32-channel group.
#include "fade_internal.cuh"

namespace fade {
namespace {

// One warp per vector; lane = channel within the current 32-channel group.
template <int BITS>
__global__ void __launch_bounds__(256) quantize_pack_kernel(const uint16_t* __restrict__ x,
                                                            long long n_vec, int dim,
                                                            uint8_t* __restrict__ codes,
                                                            uint16_t* __restrict__ scales) {
  const long long v = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (v >= n_vec) return;
  const int lane = threadIdx.x & 31;
  constexpr int qmax = (1 << (BITS - 1)) - 1;
  const int groups = dim / kGroup;
  const uint16_t* xr = x + v * dim;
  uint8_t* cr = codes + v * (long long)(dim * BITS / 8);
  uint16_t* sr = scales + v * groups;
  for (int g = 0; g < groups; ++g) {
    uint16_t sb;
    int q;
    quant_group_lane(h2f(xr[g * kGroup + lane]), qmax, sb, q);
    pack_group_store<BITS>(q, cr + g * (kGroup * BITS / 8));
    if (lane == 0) sr[g] = sb;
  }
}

template <int BITS>
__global__ void dequantize_kernel(const uint8_t* __restrict__ codes,
                                  const uint16_t* __restrict__ scales, long long n_vec, int dim,
                                  float* __restrict__ out) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_vec * dim) return;
  const long long v = i / dim;
  const int c = (int)(i % dim);
  const int q = unpack_code<BITS>(codes + v * (long long)(dim * BITS / 8), c);
  out[i] = (float)q * h2f(scales[v * (dim / kGroup) + c / kGroup]);
}

fade_status_t check_codec_args(const void* a, const void* b, const void* c, long long n_vec,
                               int dim, int bits) {
  if (!a || !b || !c) return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL buffer");
  if (n_vec < 0) return set_error(FADE_ERR_INVALID_ARGUMENT, "n_vec < 0");
  if (dim <= 0 || dim % kGroup)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "dim %d is not a positive multiple of 32", dim);
  if (bits != 2 && bits != 4) return set_error(FADE_ERR_UNSUPPORTED, "bits %d not in {2,4}", bits);
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
       reinterpret_cast<uintptr_t>(c)) & 3)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "buffers must be 4-byte aligned");
  return FADE_OK;
}

}  // namespace
}  // namespace fade

using namespace fade;

extern "C" fade_status_t fade_quantize_pack(const uint16_t* x, int64_t n_vec, int32_t dim,
                                            int32_t bits, uint8_t* codes, uint16_t* scales,
                                            void* stream) {
  clear_error();
  FADE_RANGE("fade_quantize_pack");
  fade_status_t st = check_codec_args(x, codes, scales, n_vec, dim, bits);
  if (st) return st;
  if (n_vec == 0) return FADE_OK;
  const int blocks = ceil_div(n_vec, 8);
  if (bits == 4)
    quantize_pack_kernel<4><<<blocks, 256, 0, as_stream(stream)>>>(x, n_vec, dim, codes, scales);
  else
    quantize_pack_kernel<2><<<blocks, 256, 0, as_stream(stream)>>>(x, n_vec, dim, codes, scales);
  return launch_status("fade_quantize_pack");
}

extern "C" fade_status_t fade_dequantize(const uint8_t* codes, const uint16_t* scales,
                                         int64_t n_vec, int32_t dim, int32_t bits, float* out,
                                         void* stream) {
  clear_error();
  FADE_RANGE("fade_dequantize");
  fade_status_t st = check_codec_args(codes, scales, out, n_vec, dim, bits);
  if (st) return st;
  if (n_vec == 0) return FADE_OK;
  const long long n = (long long)n_vec * dim;
  const int blocks = ceil_div(n, 256);
  if (bits == 4)
    dequantize_kernel<4><<<blocks, 256, 0, as_stream(stream)>>>(codes, scales, n_vec, dim, out);
  else
    dequantize_kernel<2><<<blocks, 256, 0, as_stream(stream)>>>(codes, scales, n_vec, dim, out);
  return launch_status("fade_dequantize");
}
