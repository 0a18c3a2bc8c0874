// Host-side part of the C ABI: error state, validation, buffer layout, position and byte
// accounting. No device code here.
#include <stdarg.h>
#include <stdio.h>

#include "fade_internal.cuh"

#if FADE_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace fade {

static thread_local char g_err[512] = "";

fade_status_t set_error(fade_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_err[0] = '\0'; }

fade_status_t launch_status(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return set_error(FADE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
                     cudaGetErrorString(e));
  return FADE_OK;
}

fade_status_t validate_config(const fade_config_t* c) {
  if (!c) return set_error(FADE_ERR_INVALID_ARGUMENT, "config is NULL");
  if (c->batch < 1 || c->batch > FADE_MAX_BATCH)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "batch %d outside [1, %d]", c->batch,
                     FADE_MAX_BATCH);
  if (c->num_kv_heads < 1 || c->num_q_heads < 1 || c->num_q_heads % c->num_kv_heads)
    return set_error(FADE_ERR_INVALID_ARGUMENT,
                     "num_q_heads %d must be a positive multiple of num_kv_heads %d",
                     c->num_q_heads, c->num_kv_heads);
  const int g = c->num_q_heads / c->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return set_error(FADE_ERR_UNSUPPORTED, "query heads per KV head %d not in {1,2,4,8}", g);
  if (c->head_dim != 64 && c->head_dim != 128)
    return set_error(FADE_ERR_UNSUPPORTED, "head_dim %d not in {64, 128}", c->head_dim);
  if (c->n_sink < 0 || c->recent_window < 1)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "n_sink %d < 0 or recent_window %d < 1",
                     c->n_sink, c->recent_window);
  if ((c->middle_k_bits != 2 && c->middle_k_bits != 4) ||
      (c->middle_v_bits != 2 && c->middle_v_bits != 4))
    return set_error(FADE_ERR_UNSUPPORTED, "middle bits (K %d, V %d) not in {2, 4}",
                     c->middle_k_bits, c->middle_v_bits);
  if (c->policy < FADE_EVICT_NONE || c->policy > FADE_EVICT_POSITION)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "unknown eviction policy %d", c->policy);
  if (c->v_codec != FADE_V_INT && c->v_codec != FADE_V_PQ)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "unknown v_codec %d", c->v_codec);
  if (c->v_codec == FADE_V_PQ && c->middle_v_bits != 2)
    return set_error(FADE_ERR_INVALID_ARGUMENT,
                     "PQ-coded V uses the INT2 row layout: middle_v_bits must be 2");
  if (c->shared_rows != 0 && c->shared_rows != 1)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "shared_rows must be 0 or 1");
  if (!(c->ema_decay >= 0.f && c->ema_decay < 1.f))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "ema_decay must lie in [0, 1)");
  if (c->mid_capacity < 1)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "mid_capacity %d < 1", c->mid_capacity);
  if ((long long)c->batch * c->num_kv_heads * (((long long)c->mid_capacity + 63) / 64 * 64) >
      0x7fffffffLL)
    return set_error(FADE_ERR_UNSUPPORTED,
                     "batch x num_kv_heads x mid_capacity exceeds 2^31 middle slots");
  const bool evicts = c->policy != FADE_EVICT_NONE && c->int4_budget >= 0;
  if (evicts && c->mid_capacity < c->int4_budget + 1)
    return set_error(FADE_ERR_CAPACITY,
                     "mid_capacity %d must hold int4_budget + 1 = %d tokens (demotion "
                     "precedes eviction)",
                     c->mid_capacity, c->int4_budget + 1);
  const fade_rope_t& r = c->rope;
  if (r.kind < FADE_ROPE_NONE || r.kind > FADE_ROPE_DYNAMIC)
    return set_error(FADE_ERR_UNSUPPORTED, "unknown rope kind %d", r.kind);
  if (r.kind != FADE_ROPE_NONE && !(r.base > 1.0))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "rope base must exceed 1");
  if ((r.kind == FADE_ROPE_LLAMA3 || r.kind == FADE_ROPE_YARN) &&
      !(r.factor > 0.0 && r.low_freq_factor > 0.0 && r.high_freq_factor > r.low_freq_factor &&
        r.original_max_position > 0))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "bad llama3 / yarn rope scaling parameters");
  if ((r.kind == FADE_ROPE_LINEAR || r.kind == FADE_ROPE_NTK) && !(r.factor > 0.0))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "rope scaling factor must be positive");
  if (r.kind == FADE_ROPE_DYNAMIC && !(r.factor >= 1.0 && r.original_max_position > 0))
    return set_error(FADE_ERR_INVALID_ARGUMENT,
                     "dynamic NTK needs factor >= 1 and original_max_position > 0");
  if (r.rotary_dim != 0 && (r.rotary_dim < 4 || r.rotary_dim > c->head_dim || r.rotary_dim % 4))
    return set_error(FADE_ERR_INVALID_ARGUMENT,
                     "rotary_dim %d must be 0 or a multiple of 4 in [4, head_dim]",
                     r.rotary_dim);
  return FADE_OK;
}

fade_status_t validate_layer(const fade_config_t* c, const fade_layer_t* L) {
  if (!L) return set_error(FADE_ERR_INVALID_ARGUMENT, "layer is NULL");
  if (c->n_sink > 0 && (!L->sink_k || !L->sink_v || !L->sink_scores))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "sink buffers are NULL");
  if (!L->recent_k || !L->recent_v || !L->recent_scores)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "recent buffers are NULL");
  for (int i = 0; i < 2; ++i)
    if (!L->mid_k_codes[i] || !L->mid_k_scales[i] || !L->mid_v_codes[i] ||
        !L->mid_v_scales[i] || !L->mid_scores[i])
      return set_error(FADE_ERR_INVALID_ARGUMENT, "middle buffer %d is NULL", i);
  if (!L->meta || !L->victims || !L->chunk_base || !L->status)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "meta, status or scratch buffers are NULL");
  if (!L->h_n_sink || !L->h_n_mid || !L->h_n_recent)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "host mirror arrays are NULL");
  if (c->v_codec == FADE_V_PQ &&
      (!L->pq_codebook || (reinterpret_cast<uintptr_t>(L->pq_codebook) & 15)))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "PQ-coded V needs a 16-byte aligned codebook");
  return FADE_OK;
}

}  // namespace fade

#if FADE_NVTX
fade::NvtxRange::NvtxRange(const char* name) { nvtxRangePushA(name); }
fade::NvtxRange::~NvtxRange() { nvtxRangePop(); }
#endif

using namespace fade;

// Smallest split of the middle tier in fade_decode_attention; bounds the partial slots.
static const int kMinSplitTokens = 128;

extern "C" fade_status_t fade_layout(const fade_config_t* c, int32_t max_prompt,
                                     fade_layout_t* o) {
  clear_error();
  fade_status_t st = validate_config(c);
  if (st) return st;
  if (!o) return set_error(FADE_ERR_INVALID_ARGUMENT, "layout output is NULL");
  if (max_prompt < 0) return set_error(FADE_ERR_INVALID_ARGUMENT, "max_prompt < 0");
  const size_t B = c->batch, H = c->num_kv_heads, Hq = c->num_q_heads, d = c->head_dim;
  const size_t S = c->n_sink, W = c->recent_window, C = mid_stride(c);
  const size_t units = B * H;
  o->sink_k = o->sink_v = units * S * d * 2;
  o->recent_k = o->recent_v = units * W * d * 2;
  o->mid_k_codes = units * C * d * c->middle_k_bits / 8;
  o->mid_v_codes = units * C * d * c->middle_v_bits / 8;
  o->mid_k_scales = o->mid_v_scales = units * C * (d / kGroup) * 2;
  o->sink_scores = units * S * 4;
  o->mid_scores = units * C * 4;
  o->recent_scores = units * W * 4;
  o->meta = units * FADE_META_FIELDS * 4;
  const long long span = (long long)(C > (size_t)max_prompt ? C : (size_t)max_prompt);
  o->victim_words = ceil_div(span, 32) + 1;
  o->chunk_slots = ceil_div(span, kChunk) + 1;
  o->victims = units * o->victim_words * 4;
  o->chunk_base = units * o->chunk_slots * 4;
  o->status = FADE_STATUS_WORDS * 4;
  o->logits_ws = B * Hq * (S + C + W) * 4;
  o->ml_ws = B * Hq * 2 * 4;
  o->max_splits = 1 + ceil_div((long long)C, kMinSplitTokens);
  o->attn_ws = B * Hq * (size_t)o->max_splits * (d + 2) * 4 + units * 4;
  o->max_prompt = max_prompt;
  o->mid_stride = (int32_t)C;
  o->prefill_mass_ws = B * Hq * (size_t)max_prompt * 8;
  return FADE_OK;
}

extern "C" int32_t fade_attention_tiled(const fade_config_t* c) {
  clear_error();
  if (validate_config(c)) return -1;
  return mid_mma_supported(c) ? 1 : 0;
}

extern "C" int32_t fade_next_position(const fade_config_t* c, const fade_layer_t* L,
                                      int32_t row) {
  clear_error();
  if (validate_config(c) || !L || !L->h_n_sink || !L->h_n_mid || !L->h_n_recent || row < 0 ||
      row >= c->batch) {
    set_error(FADE_ERR_INVALID_ARGUMENT, "fade_next_position: bad arguments");
    return -1;
  }
  const int held = L->h_n_sink[row] + L->h_n_mid[row] + L->h_n_recent[row];
  int mid = L->h_n_mid[row] + (L->h_n_recent[row] == c->recent_window ? 1 : 0);
  const bool evicts = c->policy != FADE_EVICT_NONE && c->int4_budget >= 0;
  const int ev = (evicts && mid > c->int4_budget) ? mid - c->int4_budget : 0;
  return held - ev;
}

extern "C" uint64_t fade_compressed_bytes(const fade_config_t* c, const fade_layer_t* L) {
  clear_error();
  if (validate_config(c) || !L || !L->h_n_sink || !L->h_n_mid || !L->h_n_recent) {
    set_error(FADE_ERR_INVALID_ARGUMENT, "fade_compressed_bytes: bad arguments");
    return 0;
  }
  const uint64_t d = c->head_dim;
  const uint64_t fp16_tok = 4 * d;
  // a PQ middle token's V is d/4 code bytes without scales (the codebook is counted apart)
  const uint64_t mid_tok = c->v_codec == FADE_V_PQ
                               ? d * c->middle_k_bits / 8 + 2 * (d / kGroup) + d / 4
                               : d * (c->middle_k_bits + c->middle_v_bits) / 8 +
                                     2 * 2 * (d / kGroup);
  uint64_t total = 0;
  for (int b = 0; b < c->batch; ++b)
    total += (uint64_t)c->num_kv_heads *
             ((uint64_t)(L->h_n_sink[b] + L->h_n_recent[b]) * fp16_tok +
              (uint64_t)L->h_n_mid[b] * mid_tok);
  return total;
}

extern "C" const char* fade_last_error(void) { return g_err; }

extern "C" fade_status_t fade_tier_counts(const fade_config_t* c, const fade_layer_t* L,
                                          int32_t* out) {
  clear_error();
  if (validate_config(c) || !L || !L->h_n_sink || !L->h_n_mid || !L->h_n_recent || !out)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "fade_tier_counts: bad arguments");
  for (int b = 0; b < c->batch; ++b) {
    out[3 * b + 0] = L->h_n_sink[b];
    out[3 * b + 1] = L->h_n_mid[b];
    out[3 * b + 2] = L->h_n_recent[b];
  }
  return FADE_OK;
}
