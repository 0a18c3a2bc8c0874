// RoPE table and rotation of q/k to cache positions.
// Sources: page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术", §RoPE重计算 (float32 RoPE math,
// cast through the model dtype) and §RoPE方案兼容性 (standard RoPE; llama3, linear, ntk, dynamic
// and yarn scaling, as their published definitions: position interpolation, NTK-aware base
// scaling, with the factor from the sequence length for dynamic, and YaRN's ramp over rotations
// per original context); page
// "探秘Transformer系列之（25）--- KV Cache优化之处理长文本序列", §1.2.2 StreamingLLM (positions are
// indices inside the cache).
#include <math.h>

#include "fade_internal.cuh"

namespace fade {
namespace {

struct InvFreq {
  float v[64];  // d/2 <= 64
};

// inv_freq_i in fp64 per the scheme (fade_rope_kind_t), rounded once to fp32, for the r/2
// pairs of the rotated width r (proportional RoPE: every formula reads the head dimension as
// r). Host code: compiled without floating-point contraction so every step rounds as written.
InvFreq host_inv_freq(const fade_config_t* c, int max_pos) {
  InvFreq f{};
  const int rd = rotary_width(c);
  const int half = rd / 2;
  const fade_rope_t& r = c->rope;
  // NTK-aware scaling raises the base so that the lowest frequency is divided by the factor;
  // dynamic NTK takes that factor from the sequence length (the table's length)
  double ntk = 0.0;
  if (r.kind == FADE_ROPE_NTK) ntk = r.factor;
  if (r.kind == FADE_ROPE_DYNAMIC && max_pos > r.original_max_position)
    ntk = r.factor * (double)max_pos / (double)r.original_max_position - (r.factor - 1.0);
  const double base = ntk > 0.0 ? r.base * pow(ntk, (double)rd / (rd - 2)) : r.base;
  for (int i = 0; i < half; ++i) {
    double x = pow(base, -(2.0 * i) / rd);
    if (r.kind == FADE_ROPE_LINEAR) x = x / r.factor;
    if (r.kind == FADE_ROPE_LLAMA3 || r.kind == FADE_ROPE_YARN) {
      const double lam = 2.0 * M_PI / x;
      const double L = (double)r.original_max_position;
      const double low_wl = L / r.low_freq_factor;
      const double high_wl = L / r.high_freq_factor;
      if (lam < high_wl) {
        // unchanged
      } else if (lam > low_wl) {
        x = x / r.factor;
      } else {
        const double t = (L / lam - r.low_freq_factor) / (r.high_freq_factor - r.low_freq_factor);
        x = (1.0 - t) * x / r.factor + t * x;
      }
    }
    f.v[i] = (float)x;
  }
  return f;
}

// Pairs k < npairs (= r/2) of every position; rows of `half` (= d/2) pairs.
__global__ void rope_table_kernel(InvFreq inv, int half, int npairs, int max_pos,
                                  float* __restrict__ table) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)max_pos * npairs) return;
  const int pos = (int)(i / npairs);
  const int k = (int)(i % npairs);
  const float ang = __fmul_rn((float)pos, inv.v[k]);
  const double a = (double)ang;
  const size_t base = (size_t)pos * 2 * half + (k >> 1) * 4 + (k & 1);
  table[base] = (float)cos(a);
  table[base + 2] = (float)sin(a);
}

// One thread per (vector, slot k < d/2): slot k < rh = r/2 rotates the pair (k, k + rh);
// a slot k >= rh copies the two pass-through channels r + 2 (k - rh) and the next one.
__global__ void rope_apply_kernel(const float* __restrict__ table, int max_pos, int half, int rh,
                                  const uint16_t* __restrict__ x, uint16_t* __restrict__ y,
                                  long long n_slots, int group_len,
                                  const int32_t* __restrict__ pos_start, int pos_step) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_slots) return;
  const long long vec = i / half;
  const int k = (int)(i % half);
  const long long base = vec * (2LL * half);
  if (k >= rh) {
    const int c = 2 * rh + 2 * (k - rh);
    y[base + c] = x[base + c];
    y[base + c + 1] = x[base + c + 1];
    return;
  }
  const long long g = vec / group_len;
  const int j = (int)(vec % group_len);
  int pos = (pos_start ? pos_start[g] : 0) + j * pos_step;
  pos = min(max(pos, 0), max_pos - 1);  // out-of-range positions are clamped (memory safety)
  const float x1 = h2f(x[base + k]), x2 = h2f(x[base + k + rh]);
  float y1, y2;
  rotate_pair(x1, x2, rope_cos(table, half, pos, k), rope_sin(table, half, pos, k), y1, y2);
  y[base + k] = f2h(y1);
  y[base + k + rh] = f2h(y2);
}

}  // namespace
}  // namespace fade

using namespace fade;

extern "C" fade_status_t fade_rope_table_init(const fade_config_t* cfg, float* table,
                                              int32_t max_pos, void* stream) {
  clear_error();
  FADE_RANGE("fade_rope_table_init");
  fade_status_t st = validate_config(cfg);
  if (st) return st;
  if (cfg->rope.kind == FADE_ROPE_NONE)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "no RoPE table for FADE_ROPE_NONE");
  if (!table || max_pos < 1)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL table or max_pos < 1");
  if (reinterpret_cast<uintptr_t>(table) & 15)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "table must be 16-byte aligned");
  const int half = cfg->head_dim / 2, npairs = rotary_width(cfg) / 2;
  const long long n = (long long)max_pos * npairs;
  rope_table_kernel<<<ceil_div(n, 256), 256, 0, as_stream(stream)>>>(
      host_inv_freq(cfg, max_pos), half, npairs, max_pos, table);
  return launch_status("fade_rope_table_init");
}

extern "C" fade_status_t fade_rope_apply(const fade_config_t* cfg, const float* table,
                                         int32_t max_pos, const uint16_t* x, uint16_t* y,
                                         int64_t n_groups, int32_t group_len,
                                         const int32_t* pos_start, int32_t pos_step,
                                         void* stream) {
  clear_error();
  FADE_RANGE("fade_rope_apply");
  fade_status_t st = validate_config(cfg);
  if (st) return st;
  if (!x || !y) return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL x or y");
  if (n_groups < 0 || group_len < 0)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "negative n_groups or group_len");
  const long long n_vec = (long long)n_groups * group_len;
  if (cfg->rope.kind == FADE_ROPE_NONE) {
    if (x != y && n_vec)
      if (cudaMemcpyAsync(y, x, n_vec * cfg->head_dim * 2, cudaMemcpyDeviceToDevice,
                          as_stream(stream)) != cudaSuccess)
        return launch_status("fade_rope_apply copy");
    return FADE_OK;
  }
  if (!table || max_pos < 1) return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL RoPE table");
  if (!pos_start && group_len > 0 && (long long)(group_len - 1) * pos_step >= max_pos)
    return set_error(FADE_ERR_CAPACITY, "positions up to %lld exceed the table (%d)",
                     (long long)(group_len - 1) * pos_step, max_pos);
  if (pos_step < 0) return set_error(FADE_ERR_INVALID_ARGUMENT, "pos_step < 0");
  if (n_vec == 0) return FADE_OK;
  const int half = cfg->head_dim / 2;
  const long long n_slots = n_vec * half;
  rope_apply_kernel<<<ceil_div(n_slots, 256), 256, 0, as_stream(stream)>>>(
      table, max_pos, half, rotary_width(cfg) / 2, x, y, n_slots, group_len, pos_start,
      pos_step);
  return launch_status("fade_rope_apply");
}
