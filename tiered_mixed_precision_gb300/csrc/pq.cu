// Product quantisation of V: encoding, decoding and codebook training (Lloyd's k-means).
// Source: page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术" — §高级功能 / §产品量化 (a
// codebook trained from calibration vectors with 256 centroids replaces INT2 at about 2 bits
// per element; vectors are encoded to uint8 codes and decoded back). Each code covers one
// 4-channel sub-vector; sub-space s has its own 256 centroids.
#include "fade_internal.cuh"

namespace fade {
namespace {

constexpr int kPqThreads = 256;

// grid (ceil(n / 256), dim / 4): the block stages sub-space s's 256 centroids (2 KB) and
// codes that sub-vector of 256 rows. With `sums` set, the block also adds each row's
// sub-vector to its centroid's member sum (integers of 2^-24, exact) and count.
__global__ void __launch_bounds__(kPqThreads)
    pq_assign_kernel(const uint16_t* __restrict__ codebook, const uint16_t* __restrict__ x,
                     long long n, int dim, uint8_t* __restrict__ codes,
                     unsigned long long* __restrict__ sums, int* __restrict__ counts) {
  __shared__ uint2 cb[kPqCentroids];
  const int s = blockIdx.y, S = dim / kPqSub;
  cb[threadIdx.x] =
      reinterpret_cast<const uint2*>(codebook)[(size_t)s * kPqCentroids + threadIdx.x];
  __syncthreads();
  const long long r = (long long)blockIdx.x * kPqThreads + threadIdx.x;
  if (r >= n) return;
  const uint2 raw = *reinterpret_cast<const uint2*>(x + r * dim + kPqSub * s);
  const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
  const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
  const float xv[4] = {x01.x, x01.y, x23.x, x23.y};
  const int c = pq_nearest(xv, cb);
  if (codes) codes[r * S + s] = (uint8_t)c;
  if (sums) {
    const size_t e = (size_t)s * kPqCentroids + c;
#pragma unroll
    for (int j = 0; j < kPqSub; ++j) {
      // an fp16 value times 2^24 is an integer below 2^40: exact in fp32 and in int64
      const long long v = (long long)(xv[j] * 16777216.0f);
      atomicAdd(sums + e * kPqSub + j, (unsigned long long)v);  // two's complement sum
    }
    atomicAdd(counts + e, 1);
  }
}

// One thread per (sub-space, centroid): the mean of the members, rounded once to fp16.
__global__ void pq_update_kernel(uint16_t* __restrict__ codebook,
                                 const unsigned long long* __restrict__ sums,
                                 const int* __restrict__ counts, int n_entries) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n_entries) return;
  const int cnt = counts[e];
  if (cnt == 0) return;  // no members: the centroid keeps its value
#pragma unroll
  for (int j = 0; j < kPqSub; ++j) {
    // |sum| < 2^53, so the conversion is exact; scaling by 2^-24 is exact; one division
    const double total = (double)(long long)sums[(size_t)e * kPqSub + j] * (1.0 / 16777216.0);
    codebook[(size_t)e * kPqSub + j] = __half_as_ushort(__double2half(total / (double)cnt));
  }
}

// One thread per (sub-space, centroid): centroid c starts at calibration row idx[c].
__global__ void pq_init_kernel(const uint16_t* __restrict__ calib, const int* __restrict__ idx,
                               int dim, uint16_t* __restrict__ codebook) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  const int S = dim / kPqSub;
  if (e >= S * kPqCentroids) return;
  const int s = e / kPqCentroids, c = e % kPqCentroids;
  reinterpret_cast<uint2*>(codebook)[e] =
      *reinterpret_cast<const uint2*>(calib + (size_t)idx[c] * dim + kPqSub * s);
}

// One thread per (row, sub-space).
__global__ void pq_decode_kernel(const uint16_t* __restrict__ codebook,
                                 const uint8_t* __restrict__ codes, long long n, int dim,
                                 uint16_t* __restrict__ out) {
  const int S = dim / kPqSub;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n * S) return;
  const int s = (int)(i % S);
  reinterpret_cast<uint2*>(out)[i] =
      reinterpret_cast<const uint2*>(codebook)[(size_t)s * kPqCentroids + codes[i]];
}

fade_status_t check_dim(int32_t dim, int64_t n_vec) {
  if (dim < kPqSub || dim > 1024 || dim % kPqSub)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "PQ dim %d: a multiple of 4 in [4, 1024]", dim);
  if (n_vec < 0) return set_error(FADE_ERR_INVALID_ARGUMENT, "n_vec < 0");
  // keeps both grids below 2^28 blocks of 256 threads
  if (n_vec > (1LL << 36) || n_vec * (dim / kPqSub) > (1LL << 36))
    return set_error(FADE_ERR_UNSUPPORTED, "n_vec x dim/4 above 2^36");
  return FADE_OK;
}

bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7) == 0; }

}  // namespace
}  // namespace fade

using namespace fade;

extern "C" fade_status_t fade_pq_encode(const uint16_t* codebook, const uint16_t* x,
                                        int64_t n_vec, int32_t dim, uint8_t* codes,
                                        void* stream) {
  clear_error();
  FADE_RANGE("fade_pq_encode");
  fade_status_t st = check_dim(dim, n_vec);
  if (st) return st;
  if (n_vec == 0) return FADE_OK;
  if (!codebook || !x || !codes)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "fade_pq_encode: NULL pointer");
  if (!aligned8(codebook) || !aligned8(x))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "fade_pq_encode: codebook and x need 8-byte "
                                                "alignment");
  const dim3 grid((unsigned)((n_vec + kPqThreads - 1) / kPqThreads), dim / kPqSub);
  pq_assign_kernel<<<grid, kPqThreads, 0, as_stream(stream)>>>(codebook, x, n_vec, dim, codes,
                                                               nullptr, nullptr);
  return launch_status("fade_pq_encode");
}

extern "C" fade_status_t fade_pq_decode(const uint16_t* codebook, const uint8_t* codes,
                                        int64_t n_vec, int32_t dim, uint16_t* out,
                                        void* stream) {
  clear_error();
  FADE_RANGE("fade_pq_decode");
  fade_status_t st = check_dim(dim, n_vec);
  if (st) return st;
  if (n_vec == 0) return FADE_OK;
  if (!codebook || !codes || !out)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "fade_pq_decode: NULL pointer");
  if (!aligned8(codebook) || !aligned8(out))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "fade_pq_decode: codebook and out need 8-byte "
                                                "alignment");
  const long long total = n_vec * (dim / kPqSub);
  pq_decode_kernel<<<(unsigned)((total + 255) / 256), 256, 0, as_stream(stream)>>>(
      codebook, codes, n_vec, dim, out);
  return launch_status("fade_pq_decode");
}

extern "C" fade_status_t fade_pq_train(const uint16_t* calib, int64_t n_vec, int32_t dim,
                                       const int32_t* h_init_idx, int32_t iters,
                                       uint16_t* codebook, void* ws, size_t ws_bytes,
                                       void* stream) {
  clear_error();
  FADE_RANGE("fade_pq_train");
  fade_status_t st = check_dim(dim, n_vec);
  if (st) return st;
  if (n_vec < 1 || n_vec > FADE_PQ_MAX_CALIB)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "calibration rows %lld outside [1, %d]",
                     (long long)n_vec, FADE_PQ_MAX_CALIB);
  if (iters < 0) return set_error(FADE_ERR_INVALID_ARGUMENT, "iters < 0");
  if (!calib || !h_init_idx || !codebook || !ws)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "fade_pq_train: NULL pointer");
  if (!aligned8(calib) || !aligned8(codebook) || (reinterpret_cast<uintptr_t>(ws) & 15))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "fade_pq_train: misaligned buffer");
  if (ws_bytes < FADE_PQ_TRAIN_WS_BYTES(dim))
    return set_error(FADE_ERR_CAPACITY, "fade_pq_train workspace %zu bytes, %zu needed",
                     ws_bytes, FADE_PQ_TRAIN_WS_BYTES(dim));
  for (int c = 0; c < kPqCentroids; ++c)
    if (h_init_idx[c] < 0 || h_init_idx[c] >= n_vec)
      return set_error(FADE_ERR_INVALID_ARGUMENT, "init index %d = %d outside [0, %lld)", c,
                       h_init_idx[c], (long long)n_vec);
  const int S = dim / kPqSub, entries = S * kPqCentroids;
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto* sums = reinterpret_cast<unsigned long long*>(base);  // [S][256][4]
  const size_t sums_bytes = (size_t)entries * kPqSub * 8;
  auto* counts = reinterpret_cast<int*>(base + sums_bytes);  // [S][256]
  const size_t counts_bytes = (size_t)entries * 4;
  auto* idx = reinterpret_cast<int*>(base + sums_bytes + counts_bytes);  // [256]
  cudaStream_t s = as_stream(stream);
  if (cudaMemcpyAsync(idx, h_init_idx, kPqCentroids * sizeof(int32_t), cudaMemcpyHostToDevice,
                      s) != cudaSuccess)
    return launch_status("fade_pq_train: copy of the init indices");
  pq_init_kernel<<<ceil_div(entries, 256), 256, 0, s>>>(calib, idx, dim, codebook);
  const dim3 grid((unsigned)((n_vec + kPqThreads - 1) / kPqThreads), S);
  for (int it = 0; it < iters; ++it) {
    if (cudaMemsetAsync(base, 0, sums_bytes + counts_bytes, s) != cudaSuccess)
      return launch_status("fade_pq_train: clearing the member sums");
    pq_assign_kernel<<<grid, kPqThreads, 0, s>>>(codebook, calib, n_vec, dim, nullptr, sums,
                                                 counts);
    pq_update_kernel<<<ceil_div(entries, 256), 256, 0, s>>>(codebook, sums, counts, entries);
  }
  return launch_status("fade_pq_train");
}
