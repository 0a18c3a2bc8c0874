// Decode attention on the tensor cores for INT2 K codes (with INT2, INT4 or PQ-coded V): the
// instantiations of the kernel in attention_mma.cuh, in their own translation unit so that the
// two halves compile in parallel.
#include "attention_mma.cuh"

namespace fade {

fade_status_t launch_mid_mma_k2(const fade_config_t* c, const fade_layer_t* L, MmaArgs a,
                                const StreamK& sk, cudaStream_t st) {
  const int G = c->num_q_heads / c->num_kv_heads;
  const bool pq = c->v_codec == FADE_V_PQ, v4 = c->middle_v_bits == 4;
#define FADE_CASE(D_, G_)                                                     \
  if (c->head_dim == D_ && G == G_)                                           \
    return pq ? launch_mma<D_, G_, true, 2, 2>(c, L, a, sk, st)               \
              : v4 ? launch_mma<D_, G_, false, 4, 2>(c, L, a, sk, st)         \
                   : launch_mma<D_, G_, false, 2, 2>(c, L, a, sk, st);
  FADE_CASE(64, 1) FADE_CASE(64, 2) FADE_CASE(64, 4) FADE_CASE(64, 8)
  FADE_CASE(128, 1) FADE_CASE(128, 2) FADE_CASE(128, 4) FADE_CASE(128, 8)
#undef FADE_CASE
  return set_error(FADE_ERR_UNSUPPORTED, "no tensor-core attention for this shape");
}

}  // namespace fade
