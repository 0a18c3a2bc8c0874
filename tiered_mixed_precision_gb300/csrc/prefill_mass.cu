// Prefill attention mass: the H2O importance of every prompt token before decoding starts.
// Sources: page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术", §四种驱逐策略详解 1 (H2O needs the
// attention captured at prefill); page "探秘Transformer系列之（25）--- KV Cache优化之处理长文本序列",
// §1.3.1 H2O (a token's importance is the column sum of the attention matrix).
//
// mass[b][hk][j] = sum over the query heads h of KV head hk and over the causal queries i >= j
// of softmax_j(q_{h,i} . k_j / sqrt(d)). Two passes per 64-query tile: the row statistics
// (max, sum) over all causal keys, then the normalised probabilities summed by column and
// added to the mass with one atomic per (tile, column). fp32 arithmetic; the atomic order is
// not fixed, so results may differ between runs in the last bits.
#include <math.h>

#include "fade_internal.cuh"

namespace fade {
namespace {

constexpr int kQ = 64;        // query rows per CTA
constexpr int kK = 64;        // keys per tile
constexpr int kThr = 256;

template <int D>
__global__ void __launch_bounds__(kThr) prefill_mass_kernel(const uint16_t* __restrict__ q,
                                                            const uint16_t* __restrict__ k,
                                                            float* __restrict__ mass, int Hq,
                                                            int H, int maxP, RowLens lens,
                                                            float scale) {
  __shared__ float qs[kQ][D + 1];
  __shared__ float ks[kK][D + 1];
  __shared__ float sm[kQ][kK + 1];
  __shared__ float rmax[kQ], rsum[kQ];
  const int b = blockIdx.z, hq = blockIdx.y, q0 = blockIdx.x * kQ;
  const int P = lens.v[b];
  if (q0 >= P) return;
  const int G = Hq / H, hk = hq / G;
  const int nq = min(kQ, P - q0);
  const uint16_t* qb = q + ((size_t)(b * Hq + hq) * maxP) * D;
  const uint16_t* kb = k + ((size_t)(b * H + hk) * maxP) * D;
  for (int i = threadIdx.x; i < kQ * D; i += kThr) {
    const int r = i / D, c = i % D;
    qs[r][c] = r < nq ? h2f(qb[(size_t)(q0 + r) * D + c]) : 0.f;
  }
  if (threadIdx.x < kQ) {
    rmax[threadIdx.x] = -INFINITY;
    rsum[threadIdx.x] = 0.f;
  }
  const int last_key = q0 + nq - 1;            // causal: keys 0..i for row i
  const int n_kt = last_key / kK + 1;
  for (int pass = 0; pass < 2; ++pass) {
    for (int kt = 0; kt < n_kt; ++kt) {
      const int k0 = kt * kK;
      __syncthreads();
      for (int i = threadIdx.x; i < kK * D; i += kThr) {
        const int r = i / D, c = i % D;
        ks[r][c] = (k0 + r < P) ? h2f(kb[(size_t)(k0 + r) * D + c]) : 0.f;
      }
      __syncthreads();
      // scores: 16 (row, key) entries per thread
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
      __syncthreads();
      if (pass == 0) {
        if (threadIdx.x < kQ) {  // online row statistics
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
      } else if (threadIdx.x < kK) {  // column sums of the normalised probabilities
        const int cidx = threadIdx.x, j = k0 + cidx;
        if (j < P) {
          float col = 0.f;
          for (int r = 0; r < nq; ++r)
            if (sm[r][cidx] != -INFINITY) col += expf(sm[r][cidx] - rmax[r]) / rsum[r];
          if (col != 0.f) atomicAdd(&mass[(size_t)(b * H + hk) * maxP + j], col);
        }
      }
    }
  }
}

__global__ void zero_kernel(float* p, long long n) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0.f;
}

}  // namespace
}  // namespace fade

using namespace fade;

extern "C" fade_status_t fade_prefill_mass(const fade_config_t* c, const uint16_t* q_rot,
                                           const uint16_t* k_rot, int32_t max_prompt,
                                           const int32_t* h_prompt_len, float* mass,
                                           void* stream) {
  clear_error();
  fade_status_t st = validate_config(c);
  if (st) return st;
  if (!q_rot || !k_rot || !h_prompt_len || !mass)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL q, k, lengths or mass");
  if (max_prompt < 1) return set_error(FADE_ERR_INVALID_ARGUMENT, "max_prompt < 1");
  RowLens lens{};
  int maxlen = 0;
  for (int b = 0; b < c->batch; ++b) {
    if (h_prompt_len[b] < 0 || h_prompt_len[b] > max_prompt)
      return set_error(FADE_ERR_INVALID_ARGUMENT, "row %d prompt length %d outside [0, %d]", b,
                       h_prompt_len[b], max_prompt);
    lens.v[b] = h_prompt_len[b];
    if (lens.v[b] > maxlen) maxlen = lens.v[b];
  }
  cudaStream_t s = as_stream(stream);
  const long long n = (long long)c->batch * c->num_kv_heads * max_prompt;
  zero_kernel<<<ceil_div(n, 256), 256, 0, s>>>(mass, n);
  if ((st = launch_status("fade_prefill_mass zero"))) return st;
  if (maxlen == 0) return FADE_OK;
  const dim3 grid(ceil_div(maxlen, kQ), c->num_q_heads, c->batch);
  const float scale = 1.0f / sqrtf((float)c->head_dim);
  if (c->head_dim == 64)
    prefill_mass_kernel<64><<<grid, kThr, 0, s>>>(q_rot, k_rot, mass, c->num_q_heads,
                                                  c->num_kv_heads, max_prompt, lens, scale);
  else
    prefill_mass_kernel<128><<<grid, kThr, 0, s>>>(q_rot, k_rot, mass, c->num_q_heads,
                                                   c->num_kv_heads, max_prompt, lens, scale);
  return launch_status("fade_prefill_mass");
}
