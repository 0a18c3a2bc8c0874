// Decode attention over the tiered cache: the entry point (schedule, workspace), the combine of
// the tensor-core kernel's partials (attention_mma.cuh), and H2O / EMA score accumulation.
// Sources: page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术" — §项目结构与代码质量 (kernels/:
// fused INT4 dequant + SDPA), §四种驱逐策略详解 1 (H2O: keep the highest accumulated attention)
// and 2 (EMA of attention during decode); page "探秘Transformer系列之（25）--- KV Cache优化之处理
// 长文本序列" — §1.2 (softmax attention as a weighted average of V), §1.3.1 H2O (a token's
// score is its accumulated attention, the column sum of the attention matrix).
#include <math.h>

#include "fade_internal.cuh"

namespace fade {
namespace {

constexpr int kF = FADE_META_FIELDS;

// What the combine reads: the partials of every (row, query head) and each unit's count.
struct AttnArgs {
  float* part_ml;                       // [B][Hq][nsplit][2]
  float* part_acc;                      // [B][Hq][nsplit][D]
  const int32_t* seg_count;             // [B][H]: partials of each unit
  int Hq, H, nsplit;
};

// The tensor-core kernel's partials (split 0 + one per stream-K segment of the unit).
// One CTA per unit (row, KV head), one warp per query head, D/32 channels per lane. No
// shared memory and no barrier: every lane reads the unit's partial count and the head's
// (m, l) of every partial (the same addresses across the warp) and merges the partials in
// chunks of kChunk with a running maximum: per chunk M' = max(M, m_s), the running sums are
// scaled by e^(M - M') and each partial adds l_s e^(m_s - M') and acc_s e^(m_s - M');
// out = acc / L. A chunk's loads depend only on nsplit (every slot below it is in bounds), so
// they are issued before the count is known and masked by it afterwards. With at most kChunk
// partials this is one pass with no rescaling.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_sk_kernel(AttnArgs a,
                                                              uint16_t* __restrict__ out,
                                                              float* __restrict__ ml) {
  constexpr int CPL = D / 32;       // channels per lane
  constexpr int kChunk = 8;
  const int unit = blockIdx.x;
  const int b = unit / a.H, hk = unit % a.H;
  const int G = a.Hq / a.H;
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t bh = (size_t)b * a.Hq + hk * G + h;
  const float* pa = a.part_acc + bh * a.nsplit * D + CPL * lane;
  const float* pm = a.part_ml + bh * a.nsplit * 2;
  // launched as a programmatic dependent of the attention kernel: this CTA may start while
  // the attention grid's last CTAs still run; wait here until that grid has completed and its
  // partials are visible (a no-op when launched without the dependency)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the score update that may follow is a programmatic dependent in turn
  asm volatile("griddepcontrol.launch_dependents;");
  const int ns = max(1, min(a.nsplit, a.seg_count[unit]));
  float M = -INFINITY, L = 0.f, o[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) o[c] = 0.f;
  int s0 = 0;
  do {
    float acc[kChunk][CPL], mv[kChunk], lv[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int s = s0 + i;
      const bool in = s < a.nsplit;
      mv[i] = in ? pm[2 * s] : -INFINITY;
      lv[i] = in ? pm[2 * s + 1] : 0.f;
      if constexpr (CPL == 4) {
        const float4 v = in ? *reinterpret_cast<const float4*>(pa + (size_t)s * D)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        acc[i][0] = v.x; acc[i][1] = v.y; acc[i][2] = v.z; acc[i][3] = v.w;
      } else {
        const float2 v = in ? *reinterpret_cast<const float2*>(pa + (size_t)s * D)
                            : make_float2(0.f, 0.f);
        acc[i][0] = v.x; acc[i][1] = v.y;
      }
    }
    float Mc = M;
#pragma unroll
    for (int i = 0; i < kChunk; ++i)
      if (s0 + i < ns) Mc = fmaxf(Mc, mv[i]);
    if (s0 > 0) {  // rescale what the earlier chunks summed (M finite: a partial has m > -inf)
      const float r = (M == -INFINITY) ? 0.f : __expf(M - Mc);
      L *= r;
#pragma unroll
      for (int c = 0; c < CPL; ++c) o[c] *= r;
    }
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      if (s0 + i < ns) {
        const float w = (mv[i] == -INFINITY) ? 0.f : __expf(mv[i] - Mc);
        L = fmaf(lv[i], w, L);
#pragma unroll
        for (int c = 0; c < CPL; ++c) o[c] = fmaf(acc[i][c], w, o[c]);
      }
    }
    M = Mc;
    s0 += kChunk;
  } while (s0 < ns);
  if (lane == 0) {
    ml[2 * bh] = M;
    ml[2 * bh + 1] = L;
  }
  uint16_t r[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) r[c] = f2h(o[c] / L);
  if constexpr (CPL == 4)
    *reinterpret_cast<uint2*>(out + bh * D + CPL * lane) =
        make_uint2(r[0] | ((uint32_t)r[1] << 16), r[2] | ((uint32_t)r[3] << 16));
  else
    *reinterpret_cast<uint32_t*>(out + bh * D + CPL * lane) = r[0] | ((uint32_t)r[1] << 16);
}

struct AccArgs {
  const float* logits;
  const float* ml;
  float *sink_sc, *mid_sc[2], *rec_sc;
  const int32_t* meta;
  int Hq, H, S, W, C, NS, policy;
  float decay;
};

// One thread per storage slot of a unit: score update from the G heads' probabilities. Every
// load is issued before any of them is used: the G logits of the slot and the heads' (M, L)
// do not depend on the unit's counts, and neither does the score's address except for a
// middle slot, whose score is read from both ping-pong buffers and the live one kept (for
// slots the unit does not hold the values are read and dropped). One round trip to memory
// per thread, then the update.
__global__ void __launch_bounds__(256) h2o_accumulate_kernel(AccArgs a) {
  // launched as a programmatic dependent of the attention call's combine: wait here until that
  // grid has completed and its (M, L) are visible (a no-op when launched without the dependency)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next layer's RoPE + append launch may be a programmatic dependent in turn
  asm volatile("griddepcontrol.launch_dependents;");
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= a.NS) return;
  const int hk = blockIdx.y, b = blockIdx.z, unit = b * a.H + hk;
  const int G = a.Hq / a.H;
  float lg[8], mh[8], lh[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h < G) {
      const size_t bh = (size_t)b * a.Hq + hk * G + h;
      lg[h] = a.logits[bh * a.NS + j];
      mh[h] = a.ml[2 * bh];
      lh[h] = a.ml[2 * bh + 1];
    }
  }
  const int32_t* mp = a.meta + unit * kF;
  const int4 m = make_int4(mp[FADE_META_N_SINK], mp[FADE_META_N_MID], mp[FADE_META_N_RECENT],
                           mp[FADE_META_HEAD]);
  const int cur = mp[FADE_META_CUR];
  float* sc;
  float old0, old1 = 0.f;
  int region;  // 0 sink, 1 middle, 2 ring
  int idx;
  if (j < a.S) {
    region = 0;
    idx = j;
    sc = a.sink_sc + (size_t)unit * a.S + j;
    old0 = *sc;
  } else if (j < a.S + a.C) {
    region = 1;
    idx = j - a.S;
    const size_t o = (size_t)unit * a.C + idx;
    old0 = a.mid_sc[0][o];
    old1 = a.mid_sc[1][o];
    sc = nullptr;
  } else {
    region = 2;
    idx = j - a.S - a.C;
    sc = a.rec_sc + (size_t)unit * a.W + idx;
    old0 = *sc;
  }
  bool held;
  float old;
  if (region == 0) {
    held = idx < m.x;
    old = old0;
  } else if (region == 1) {
    held = idx < m.y;
    sc = (cur ? a.mid_sc[1] : a.mid_sc[0]) + (size_t)unit * a.C + idx;
    old = cur ? old1 : old0;
  } else {
    const int age = (idx - m.w + a.W) % a.W;
    held = age < m.z;
    old = old0;
  }
  if (!held) return;
  float psum = 0.f;
#pragma unroll
  for (int h = 0; h < 8; ++h)
    if (h < G) psum += __expf(lg[h] - mh[h]) / lh[h];
  if (a.policy == FADE_EVICT_H2O)
    *sc = old + psum;
  else
    *sc = a.decay * old + (1.f - a.decay) * psum;
}

// The same update for four consecutive slots per thread (when the sink count and the slot
// count are multiples of 4, so that a group of four never straddles two tiers and every
// vector access is 16-byte aligned): the G heads' (M, L) are loaded once per four slots, the
// logits and the scores (both middle buffers) as float4. Per slot the arithmetic is the scalar
// kernel's, term for term.
template <int G>
__global__ void __launch_bounds__(256) h2o_accumulate4_kernel(AccArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // as in h2o_accumulate_kernel
  asm volatile("griddepcontrol.launch_dependents;");
  const int j0 = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (j0 >= a.NS) return;
  const int hk = blockIdx.y, b = blockIdx.z, unit = b * a.H + hk;
  float4 lg[G];
  float mh[G], lh[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const size_t bh = (size_t)b * a.Hq + hk * G + h;
    lg[h] = *reinterpret_cast<const float4*>(a.logits + bh * a.NS + j0);
    mh[h] = a.ml[2 * bh];
    lh[h] = a.ml[2 * bh + 1];
  }
  const int32_t* mp = a.meta + unit * kF;
  const int n_sink = mp[FADE_META_N_SINK], n_mid = mp[FADE_META_N_MID];
  const int n_rec = mp[FADE_META_N_RECENT], head = mp[FADE_META_HEAD], cur = mp[FADE_META_CUR];
  float* sc;
  float4 o0, o1 = make_float4(0.f, 0.f, 0.f, 0.f);
  int region, idx;
  if (j0 < a.S) {
    region = 0;
    idx = j0;
    sc = a.sink_sc + (size_t)unit * a.S + j0;
    o0 = *reinterpret_cast<const float4*>(sc);
  } else if (j0 < a.S + a.C) {
    region = 1;
    idx = j0 - a.S;
    const size_t off = (size_t)unit * a.C + idx;
    o0 = *reinterpret_cast<const float4*>(a.mid_sc[0] + off);
    o1 = *reinterpret_cast<const float4*>(a.mid_sc[1] + off);
    sc = (cur ? a.mid_sc[1] : a.mid_sc[0]) + off;
  } else {
    region = 2;
    idx = j0 - a.S - a.C;
    sc = a.rec_sc + (size_t)unit * a.W + idx;
    o0 = *reinterpret_cast<const float4*>(sc);
  }
  const float4 ov = (region == 1 && cur) ? o1 : o0;
  const float old[4] = {ov.x, ov.y, ov.z, ov.w};
  float nv[4];
  bool held[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (region == 0) {
      held[e] = idx + e < n_sink;
    } else if (region == 1) {
      held[e] = idx + e < n_mid;
    } else {
      int age = idx + e - head;
      if (age < 0) age += a.W;
      held[e] = age < n_rec;
    }
    float psum = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float l = e == 0 ? lg[h].x : e == 1 ? lg[h].y : e == 2 ? lg[h].z : lg[h].w;
      psum += __expf(l - mh[h]) / lh[h];
    }
    nv[e] = a.policy == FADE_EVICT_H2O ? old[e] + psum
                                       : a.decay * old[e] + (1.f - a.decay) * psum;
  }
  if (held[0] && held[1] && held[2] && held[3]) {
    *reinterpret_cast<float4*>(sc) = make_float4(nv[0], nv[1], nv[2], nv[3]);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (held[e]) sc[e] = nv[e];
  }
}

}  // namespace
}  // namespace fade

using namespace fade;

extern "C" fade_status_t fade_decode_attention(const fade_config_t* c, const fade_layer_t* L,
                                               const uint16_t* q_rot, uint16_t* out,
                                               float* logits_ws, float* ml_ws, void* ws,
                                               size_t ws_bytes, void* stream) {
  clear_error();
  FADE_RANGE("fade_decode_attention");
  fade_status_t st = validate_config(c);
  if (!st) st = validate_layer(c, L);
  if (st) return st;
  if (!q_rot || !out || !ml_ws || !ws)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL q, out, ml_ws or ws");
  int max_mid = 0, max_fp16 = 0;
  for (int b = 0; b < c->batch; ++b) {
    if (L->h_n_mid[b] > max_mid) max_mid = L->h_n_mid[b];
    const int f = L->h_n_sink[b] + L->h_n_recent[b];
    if (f > max_fp16) max_fp16 = f;
  }
  if (max_mid == 0 && max_fp16 == 0)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "the cache is empty");
  const int units = c->batch * c->num_kv_heads;
  if (!mid_mma_supported(c))
    return set_error(FADE_ERR_UNSUPPORTED, "no tensor-core attention for these code widths");
  StreamK sk{};  // the stream-K schedule of the middle tiles (from the host mirror)
  build_stream_k(c, L, mid_mma_ctas(c), &sk);
  AttnArgs a;
  a.Hq = c->num_q_heads;
  a.H = c->num_kv_heads;
  a.nsplit = 1 + sk.smax;
  const size_t part = (size_t)c->batch * c->num_q_heads * a.nsplit * (c->head_dim + 2) * 4;
  const size_t need = part + (size_t)units * 4;
  if (ws_bytes < need)
    return set_error(FADE_ERR_CAPACITY, "attention workspace %zu bytes, %zu needed", ws_bytes,
                     need);
  a.part_ml = reinterpret_cast<float*>(ws);
  a.part_acc = a.part_ml + (size_t)c->batch * c->num_q_heads * a.nsplit * 2;
  int32_t* seg_count = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + part);
  a.seg_count = seg_count;
  cudaStream_t s = as_stream(stream);
  // one launch: FP16 tiers (split 0) and the packed middle tier (tensor cores)
  if ((st = launch_mid_mma(c, L, q_rot, logits_ws, a.part_ml, a.part_acc, seg_count, sk,
                           a.nsplit, s)))
    return st;
  // the combine launches as a programmatic dependent of the attention kernel (its CTAs are
  // scheduled while the attention grid drains and wait on the device for its completion)
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(units);
  lc.blockDim = dim3(32 * (a.Hq / a.H));
  lc.dynamicSmemBytes = 0;
  lc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  const cudaError_t e =
      c->head_dim == 64 ? cudaLaunchKernelEx(&lc, attn_combine_sk_kernel<64>, a, out, ml_ws)
                        : cudaLaunchKernelEx(&lc, attn_combine_sk_kernel<128>, a, out, ml_ws);
  if (e != cudaSuccess)
    return set_error(FADE_ERR_CUDA, "fade_decode_attention combine: %s", cudaGetErrorString(e));
  return launch_status("fade_decode_attention combine");
}

extern "C" fade_status_t fade_h2o_accumulate(const fade_config_t* c, fade_layer_t* L,
                                             const float* logits_ws, const float* ml_ws,
                                             void* stream) {
  clear_error();
  FADE_RANGE("fade_h2o_accumulate");
  fade_status_t st = validate_config(c);
  if (!st) st = validate_layer(c, L);
  if (st) return st;
  if (c->policy != FADE_EVICT_H2O && c->policy != FADE_EVICT_EMA) return FADE_OK;
  if (!logits_ws || !ml_ws) return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL logits or ml");
  AccArgs a;
  a.logits = logits_ws;
  a.ml = ml_ws;
  a.sink_sc = L->sink_scores;
  a.mid_sc[0] = L->mid_scores[0];
  a.mid_sc[1] = L->mid_scores[1];
  a.rec_sc = L->recent_scores;
  a.meta = L->meta;
  a.Hq = c->num_q_heads;
  a.H = c->num_kv_heads;
  a.S = c->n_sink;
  a.W = c->recent_window;
  a.C = mid_stride(c);
  a.NS = a.S + a.C + a.W;
  a.policy = c->policy;
  a.decay = c->ema_decay;
  const int G = c->num_q_heads / c->num_kv_heads;
  // a programmatic dependent of the kernel before it on the stream (the attention call's
  // combine, in a decode step): its CTAs are scheduled while that grid drains and wait on the
  // device for its completion
  cudaLaunchConfig_t lc{};
  lc.blockDim = dim3(256);
  lc.dynamicSmemBytes = 0;
  lc.stream = as_stream(stream);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  cudaError_t e;
  if (a.S % 4 == 0 && a.NS % 4 == 0 && al16(a.logits) && al16(a.sink_sc) && al16(a.mid_sc[0]) &&
      al16(a.mid_sc[1]) && al16(a.rec_sc)) {
    lc.gridDim = dim3(ceil_div(a.NS / 4, 256), c->num_kv_heads, c->batch);
    switch (G) {
      case 1: e = cudaLaunchKernelEx(&lc, h2o_accumulate4_kernel<1>, a); break;
      case 2: e = cudaLaunchKernelEx(&lc, h2o_accumulate4_kernel<2>, a); break;
      case 4: e = cudaLaunchKernelEx(&lc, h2o_accumulate4_kernel<4>, a); break;
      default: e = cudaLaunchKernelEx(&lc, h2o_accumulate4_kernel<8>, a); break;
    }
  } else {
    lc.gridDim = dim3(ceil_div(a.NS, 256), c->num_kv_heads, c->batch);
    e = cudaLaunchKernelEx(&lc, h2o_accumulate_kernel, a);
  }
  if (e != cudaSuccess)
    return set_error(FADE_ERR_CUDA, "fade_h2o_accumulate: %s", cudaGetErrorString(e));
  return launch_status("fade_h2o_accumulate");
}
