// Prefill attention mass: the H2O importance of every prompt token before decoding starts.
// Sources: page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术", §四种驱逐策略详解 1 (H2O needs the
// attention captured at prefill); page "探秘Transformer系列之（25）--- KV Cache优化之处理长文本序列",
// §1.3.1 H2O (a token's importance is the column sum of the attention matrix).
//
// mass[b][hk][j] = sum over the query heads h of KV head hk and over the causal queries i >= j
// of softmax_j(q_{h,i} . k_j / sqrt(d)). Two kernels, both in fp32 with one fixed operation
// order, so the result is the same bit for bit on every run:
//   1. row statistics: one CTA per (64-query tile, query head, row) streams the causal keys
//      and keeps each query row's running (max, sum of exp) in the workspace;
//   2. column sums: one CTA per (64-key tile, KV head, row) walks the group's query heads in
//      order and, for each, the query tiles from the key tile's own onwards in order; it
//      recomputes each score exactly as kernel 1 did (same loop, same fused multiply-adds),
//      normalises it with the row's statistics and adds it to its column's register sum.
// No atomics: every mass entry is written once, by the thread owning its column.
#include <math.h>

#include "fade_internal.cuh"

namespace fade {
namespace {

constexpr int kQ = 64;        // query rows per tile
constexpr int kK = 64;        // keys per tile
constexpr int kThr = 256;

// Scores of one (query tile, key tile) pair into sm: s = (q . k) * scale for causal pairs
// j <= i of valid rows, -inf elsewhere. Both kernels call this with the same operands, so
// they see identical scores.
template <int D>
__device__ __forceinline__ void score_tile(const float (*qs)[D + 1], const float (*ks)[D + 1],
                                           float (*sm)[kK + 1], int q0, int nq, int k0,
                                           float scale) {
  for (int e = threadIdx.x; e < kQ * kK; e += kThr) {
    const int r = e / kK, cidx = e % kK;
    const int i = q0 + r, j = k0 + cidx;
    float s = -INFINITY;
    if (r < nq && j <= i) {
      float acc = 0.f;
#pragma unroll 8
      for (int c = 0; c < D; ++c) acc = fmaf(qs[r][c], ks[cidx][c], acc);
      s = acc * scale;
    }
    sm[r][cidx] = s;
  }
}

template <int D>
__device__ __forceinline__ void load_rows(float (*dst)[D + 1], const uint16_t* src, int first,
                                          int n_valid) {
  for (int i = threadIdx.x; i < 64 * D; i += kThr) {
    const int r = i / D, c = i % D;
    dst[r][c] = r < n_valid ? h2f(src[(size_t)(first + r) * D + c]) : 0.f;
  }
}

// Kernel 1: stats[b][hq][i] = (max_j s_ij, sum_j exp(s_ij - max)) over the causal keys j <= i.
// Dynamic shared memory of both kernels: q rows, k rows, scores (fp32, rows padded by one).
template <int D>
constexpr size_t smem_bytes() {
  return (size_t)(kQ * (D + 1) + kK * (D + 1) + kQ * (kK + 1)) * sizeof(float);
}

template <int D>
__global__ void __launch_bounds__(kThr) prefill_rowstats_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ k, float2* __restrict__ stats,
    int Hq, int H, int maxP, RowLens lens, float scale) {
  extern __shared__ float dyn[];
  float(*qs)[D + 1] = reinterpret_cast<float(*)[D + 1]>(dyn);
  float(*ks)[D + 1] = reinterpret_cast<float(*)[D + 1]>(dyn + kQ * (D + 1));
  float(*sm)[kK + 1] = reinterpret_cast<float(*)[kK + 1]>(dyn + (kQ + kK) * (D + 1));
  __shared__ float rmax[kQ], rsum[kQ];
  const int b = blockIdx.z, hq = blockIdx.y, q0 = blockIdx.x * kQ;
  const int P = lens.v[b];
  if (q0 >= P) return;
  const int G = Hq / H, hk = hq / G;
  const int nq = min(kQ, P - q0);
  load_rows<D>(qs, q + ((size_t)(b * Hq + hq) * maxP) * D, q0, nq);
  if (threadIdx.x < kQ) {
    rmax[threadIdx.x] = -INFINITY;
    rsum[threadIdx.x] = 0.f;
  }
  const uint16_t* kb = k + ((size_t)(b * H + hk) * maxP) * D;
  const int n_kt = (q0 + nq - 1) / kK + 1;  // causal: keys 0..i for row i
  for (int kt = 0; kt < n_kt; ++kt) {
    const int k0 = kt * kK;
    __syncthreads();
    load_rows<D>(ks, kb, k0, min(kK, P - k0));
    __syncthreads();
    score_tile<D>(qs, ks, sm, q0, nq, k0, scale);
    __syncthreads();
    if (threadIdx.x < kQ) {  // running row statistics, keys in index order
      const int r = threadIdx.x;
      float mx = rmax[r];
      for (int c = 0; c < kK; ++c) mx = fmaxf(mx, sm[r][c]);
      float sum = (rmax[r] == -INFINITY) ? 0.f : rsum[r] * expf(rmax[r] - mx);
      if (mx != -INFINITY)
        for (int c = 0; c < kK; ++c)
          if (sm[r][c] != -INFINITY) sum += expf(sm[r][c] - mx);
      rmax[r] = mx;
      rsum[r] = sum;
    }
  }
  __syncthreads();
  if (threadIdx.x < nq)
    stats[(size_t)(b * Hq + hq) * maxP + q0 + threadIdx.x] =
        make_float2(rmax[threadIdx.x], rsum[threadIdx.x]);
}

// Kernel 2: mass of the keys of one tile, summed over the group's query heads (in order) and
// the query rows i >= j (query tiles in order, rows in order within a tile).
template <int D>
__global__ void __launch_bounds__(kThr) prefill_colsum_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
    const float2* __restrict__ stats, float* __restrict__ mass, int Hq, int H, int maxP,
    RowLens lens, float scale) {
  extern __shared__ float dyn[];
  float(*qs)[D + 1] = reinterpret_cast<float(*)[D + 1]>(dyn);
  float(*ks)[D + 1] = reinterpret_cast<float(*)[D + 1]>(dyn + kQ * (D + 1));
  float(*sm)[kK + 1] = reinterpret_cast<float(*)[kK + 1]>(dyn + (kQ + kK) * (D + 1));
  __shared__ float2 st[kQ];
  const int b = blockIdx.z, hk = blockIdx.y, k0 = blockIdx.x * kK;
  const int P = lens.v[b];
  float* out = mass + (size_t)(b * H + hk) * maxP;
  if (k0 >= P) {  // past the row's prompt: zeros
    for (int j = k0 + threadIdx.x; j < min(k0 + kK, maxP); j += kThr) out[j] = 0.f;
    return;
  }
  const int G = Hq / H;
  load_rows<D>(ks, k + ((size_t)(b * H + hk) * maxP) * D, k0, min(kK, P - k0));
  float col = 0.f;  // thread c < kK owns column k0 + c
  const int n_qt = (P + kQ - 1) / kQ;
  for (int g = 0; g < G; ++g) {
    const int hq = hk * G + g;
    const uint16_t* qb = q + ((size_t)(b * Hq + hq) * maxP) * D;
    for (int qt = k0 / kQ; qt < n_qt; ++qt) {
      const int q0 = qt * kQ, nq = min(kQ, P - q0);
      __syncthreads();
      load_rows<D>(qs, qb, q0, nq);
      if (threadIdx.x < kQ)
        st[threadIdx.x] = threadIdx.x < nq ? stats[(size_t)(b * Hq + hq) * maxP + q0 + threadIdx.x]
                                           : make_float2(-INFINITY, 1.f);
      __syncthreads();
      score_tile<D>(qs, ks, sm, q0, nq, k0, scale);
      __syncthreads();
      if (threadIdx.x < kK) {
        const int c = threadIdx.x;
        for (int r = 0; r < nq; ++r)
          if (sm[r][c] != -INFINITY) col += expf(sm[r][c] - st[r].x) / st[r].y;
      }
    }
  }
  if (threadIdx.x < kK && k0 + threadIdx.x < maxP)
    out[k0 + threadIdx.x] = (k0 + threadIdx.x < P) ? col : 0.f;
}

template <int D>
fade_status_t launch_mass(const fade_config_t* c, const uint16_t* q_rot, const uint16_t* k_rot,
                          int32_t max_prompt, RowLens lens, float* mass, float2* stats,
                          cudaStream_t s) {
  constexpr size_t smem = smem_bytes<D>();
  // above the 48 KB default: opt in (per function, on the current device; cheap, so on
  // every call rather than once per process)
  cudaError_t opt = cudaFuncSetAttribute(prefill_rowstats_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (opt == cudaSuccess)
    opt = cudaFuncSetAttribute(prefill_colsum_kernel<D>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (opt != cudaSuccess)
    return set_error(FADE_ERR_CUDA, "fade_prefill_mass: shared-memory opt-in failed: %s",
                     cudaGetErrorString(opt));
  const float scale = 1.0f / sqrtf((float)c->head_dim);
  const dim3 g1(ceil_div(max_prompt, kQ), c->num_q_heads, c->batch);
  const dim3 g2(ceil_div(max_prompt, kK), c->num_kv_heads, c->batch);
  prefill_rowstats_kernel<D><<<g1, kThr, smem, s>>>(q_rot, k_rot, stats, c->num_q_heads,
                                                    c->num_kv_heads, max_prompt, lens, scale);
  fade_status_t st = launch_status("fade_prefill_mass rows");
  if (st) return st;
  prefill_colsum_kernel<D><<<g2, kThr, smem, s>>>(q_rot, k_rot, stats, mass, c->num_q_heads,
                                                  c->num_kv_heads, max_prompt, lens, scale);
  return launch_status("fade_prefill_mass columns");
}

}  // namespace
}  // namespace fade

using namespace fade;

extern "C" fade_status_t fade_prefill_mass(const fade_config_t* c, const uint16_t* q_rot,
                                           const uint16_t* k_rot, int32_t max_prompt,
                                           const int32_t* h_prompt_len, float* mass, void* ws,
                                           size_t ws_bytes, void* stream) {
  clear_error();
  FADE_RANGE("fade_prefill_mass");
  fade_status_t st = validate_config(c);
  if (st) return st;
  if (!q_rot || !k_rot || !h_prompt_len || !mass)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL q, k, lengths or mass");
  if (max_prompt < 1) return set_error(FADE_ERR_INVALID_ARGUMENT, "max_prompt < 1");
  const size_t need = (size_t)c->batch * c->num_q_heads * (size_t)max_prompt * sizeof(float2);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 7))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "workspace is NULL or not 8-byte aligned");
  if (ws_bytes < need)
    return set_error(FADE_ERR_CAPACITY, "prefill-mass workspace of %zu bytes < %zu needed",
                     ws_bytes, need);
  RowLens lens{};
  for (int b = 0; b < c->batch; ++b) {
    if (h_prompt_len[b] < 0 || h_prompt_len[b] > max_prompt)
      return set_error(FADE_ERR_INVALID_ARGUMENT, "row %d prompt length %d outside [0, %d]", b,
                       h_prompt_len[b], max_prompt);
    lens.v[b] = h_prompt_len[b];
  }
  cudaStream_t s = as_stream(stream);
  float2* stats = reinterpret_cast<float2*>(ws);
  if (c->head_dim == 64)
    return launch_mass<64>(c, q_rot, k_rot, max_prompt, lens, mass, stats, s);
  return launch_mass<128>(c, q_rot, k_rot, max_prompt, lens, mass, stats, s);
}
