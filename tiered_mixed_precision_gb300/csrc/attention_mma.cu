// Decode attention on the tensor cores: the host side (schedule, dispatch) and the kernels for
// INT4 K codes; the kernel itself is in attention_mma.cuh, the INT2-K instantiations in
// attention_mma_k2.cu.
#include "attention_mma.cuh"

namespace fade {

bool mid_mma_supported(const fade_config_t* c) {
  // INT4 or INT2 K, with INT2 V (or PQ-coded V, whose codes fill the INT2 rows) or INT4 V
  return (c->middle_k_bits == 4 || c->middle_k_bits == 2) &&
         (c->middle_v_bits == 2 || (c->middle_v_bits == 4 && c->v_codec != FADE_V_PQ));
}

int mid_mma_ctas(const fade_config_t* c) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 1;
  const int G = c->num_q_heads / c->num_kv_heads;
  const int minb = c->v_codec == FADE_V_PQ ? 1                        // MmaShape::MINB
                   : (FADE_MMA_WIDE && G <= 4) ? FADE_MMA_CTAS_PER_SM : 1;
  return std::max(1, std::min(kMaxCtaSK, sms * minb));
}

void build_stream_k(const fade_config_t* c, const fade_layer_t* L, int ctas, StreamK* k) {
  k->P = ctas;
  k->B = c->batch;
  k->H = c->num_kv_heads;
  long long T = 0;
  for (int b = 0; b < c->batch; ++b) {
    k->row_start[b] = (int)T;
    T += (long long)k->H * ((L->h_n_mid[b] + kTileTok - 1) / kTileTok);
  }
  for (int b = c->batch; b <= FADE_MAX_BATCH; ++b) k->row_start[b] = (int)T;
  // an FP16-tier item (sinks + recent window) costs about kFp16Weight middle tiles
  constexpr long long kFp16Weight = FADE_F16_ITEM_WEIGHT;
  const long long F = (long long)c->batch * c->num_kv_heads, P = ctas;
  const long long Wtot = T + kFp16Weight * F;
  long long f16_before = 0, prev = 0;
  k->cta_start[0] = 0;
  for (long long cc = 1; cc <= P; ++cc) {
    const long long n16 = (cc - 1) < F ? (F - (cc - 1) + P - 1) / P : 0;
    f16_before += n16;
    long long v = cc * Wtot / P - kFp16Weight * f16_before;
    v = std::max(prev, std::min(T, v));
    k->cta_start[cc] = (int)v;
    prev = v;
  }
  k->cta_start[P] = (int)T;
  int smax = 0;
  for (int b = 0; b < c->batch; ++b)
    for (int h = 0; h < k->H; ++h) smax = std::max(smax, sk_segments(*k, b, h));
  k->smax = smax;
}

fade_status_t launch_mid_mma(const fade_config_t* c, const fade_layer_t* L, const uint16_t* q,
                             float* logits, float* part_ml, float* part_acc, int32_t* seg_count,
                             const StreamK& sk, int nsplit, cudaStream_t st) {
  MmaArgs a;
  a.q = q;
  a.sink_k = L->sink_k;
  a.sink_v = L->sink_v;
  a.rec_k = L->recent_k;
  a.rec_v = L->recent_v;
  a.W = c->recent_window;
  for (int i = 0; i < 2; ++i) {
    a.ks[i] = L->mid_k_scales[i];
    a.vs[i] = L->mid_v_scales[i];
  }
  a.meta = L->meta;
  a.logits = logits;
  a.part_ml = part_ml;
  a.part_acc = part_acc;
  a.seg_count = seg_count;
  a.status = L->status;
  a.B = c->batch;
  a.Hq = c->num_q_heads;
  a.H = c->num_kv_heads;
  a.S = c->n_sink;
  a.C = mid_stride(c);
  a.NS = c->n_sink + a.C + c->recent_window;
  a.chunk = kTileTok;
  a.nsplit = nsplit;
  a.inv_sqrt_d = 1.0f / sqrtf((float)c->head_dim);
  a.pq_cb = L->pq_codebook;
  const int G = c->num_q_heads / c->num_kv_heads;
  const bool pq = c->v_codec == FADE_V_PQ;
  if (c->middle_k_bits == 2) return launch_mid_mma_k2(c, L, a, sk, st);
  const bool v4 = c->middle_v_bits == 4;
#define FADE_CASE(D_, G_)                                                     \
  if (c->head_dim == D_ && G == G_)                                           \
    return pq ? launch_mma<D_, G_, true, 2, 4>(c, L, a, sk, st)               \
              : v4 ? launch_mma<D_, G_, false, 4, 4>(c, L, a, sk, st)         \
                   : launch_mma<D_, G_, false, 2, 4>(c, L, a, sk, st);
  FADE_CASE(64, 1) FADE_CASE(64, 2) FADE_CASE(64, 4) FADE_CASE(64, 8)
  FADE_CASE(128, 1) FADE_CASE(128, 2) FADE_CASE(128, 4) FADE_CASE(128, 8)
#undef FADE_CASE
  return set_error(FADE_ERR_UNSUPPORTED, "no tensor-core attention for this shape");
}

}  // namespace fade
