// Tier maintenance of the FADE cache: reset, prefill, demote, append, evict + re-position.
// Sources: page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术" — §核心机制 (three tiers),
// §第一层 (FP16 sinks and recent window), §第二层/§第三层 (INT4 middle tier, INT2 V),
// §驱逐策略 (eviction at INT4_BUDGET with un-RoPE/re-RoPE to contiguous positions),
// §四种驱逐策略详解 (H2O, EMA, position), §RoPE重计算 (fp32 RoPE math, cast via fp16);
// page "探秘Transformer系列之（25）--- KV Cache优化之处理长文本序列" — §1.2.2 StreamingLLM
// (sinks + rolling window, positions inside the cache), §1.3.1 H2O (evict the lowest
// accumulated attention).
#include "fade_internal.cuh"

namespace fade {
namespace {

constexpr int kSelThreads = kChunk;  // one selection CTA covers one chunk per pass
constexpr int kF = FADE_META_FIELDS;

// Unsigned key whose order is the float order (-0 and +0 equal).
__device__ __forceinline__ uint32_t ord_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive prefix count of `f` over the CTA (all threads must call); `total` = count.
__device__ __forceinline__ int block_excl_count(bool f, int* sh /*[33]*/, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const uint32_t b = __ballot_sync(0xffffffffu, f);
  const int in_warp = __popc(b & ((1u << lane) - 1u));
  if (lane == 0) sh[warp] = __popc(b);
  __syncthreads();
  if (warp == 0) {
    const int v = lane < nw ? sh[lane] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    sh[lane] = incl - v;
    if (lane == 31) sh[32] = incl;
  }
  __syncthreads();
  const int r = sh[warp] + in_warp;
  total = sh[32];
  __syncthreads();
  return r;
}

// Selects the k smallest (key, index) among n candidates with one CTA of kSelThreads
// threads: an exact 4-pass radix select finds the k-th smallest key T, then one pass in index
// order marks keys < T and the first (k - #below) keys equal to T. keys == nullptr means all
// keys are equal (the oldest k go first). Writes bitmap words [0, ceil(n/32)) and
// chunk_base[c] = victims among candidates [0, c*kChunk), c = 0..ceil(n/kChunk).
__device__ void block_select(const float* __restrict__ keys, int n, int k,
                             uint32_t* __restrict__ bitmap, int32_t* __restrict__ chunk_base) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_rem;
  __shared__ int sh[33];
  const int tid = threadIdx.x;
  uint32_t T = ord_key(0.f);
  int remaining = k;
  if (keys && k > 0) {
    uint32_t prefix = 0, mask = 0;
    int rem = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < n; i += blockDim.x) {
        const uint32_t u = ord_key(keys[i]);
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        int cum = 0;
        for (int dgt = 0; dgt < 256; ++dgt) {
          const int h = (int)hist[dgt];
          if (cum + h >= rem) {
            s_prefix = prefix | (uint32_t(dgt) << shift);
            s_rem = rem - cum;
            break;
          }
          cum += h;
        }
      }
      __syncthreads();
      prefix = s_prefix;
      rem = s_rem;
      mask |= 255u << shift;
      __syncthreads();
    }
    T = prefix;
    remaining = rem;
  }
  int carry = 0, eq_carry = 0;
  for (int base = 0; base < n; base += kSelThreads) {
    const int i = base + tid;
    const bool valid = i < n;
    const uint32_t u = valid ? (keys ? ord_key(keys[i]) : T) : 0u;
    const bool eq = valid && k > 0 && u == T;
    int eq_tot;
    const int eq_rank = block_excl_count(eq, sh, eq_tot) + eq_carry;
    const bool flag = valid && k > 0 && (u < T || (eq && eq_rank < remaining));
    const uint32_t word = __ballot_sync(0xffffffffu, flag);
    if ((tid & 31) == 0 && i < n) bitmap[i >> 5] = word;
    if (tid == 0) chunk_base[base / kChunk] = carry;
    int f_tot;
    block_excl_count(flag, sh, f_tot);
    carry += f_tot;
    eq_carry += eq_tot;
  }
  if (tid == 0) chunk_base[(n + kChunk - 1) / kChunk] = carry;
}

// Victims before candidate `ci`, from the chunk prefix plus the bitmap words of its chunk
// (warp-cooperative; all lanes get the result).
__device__ __forceinline__ int victims_before(const uint32_t* __restrict__ bitmap,
                                              const int32_t* __restrict__ chunk_base, int ci) {
  const int lane = threadIdx.x & 31;
  const int w = ci >> 5;
  const int w0 = (ci / kChunk) * (kChunk / 32);
  int cnt = (w0 + lane < w) ? __popc(bitmap[w0 + lane]) : 0;
#pragma unroll
  for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  return chunk_base[ci / kChunk] + cnt + __popc(bitmap[w] & ((1u << (ci & 31)) - 1u));
}

// ----------------------------------------------------------------- shared layer view
struct LayerArgs {
  uint16_t *sink_k, *sink_v, *rec_k, *rec_v;
  uint8_t *mk[2], *mv[2];
  uint16_t *mks[2], *mvs[2];
  float *sink_sc, *mid_sc[2], *rec_sc;
  int32_t* meta;
  uint32_t* victims;
  int32_t* chunk_base;
  int victim_words, chunk_slots;
  int H, S, W, C, budget, policy;
  bool evicts;
  bool positional;  // position policy: the victims are the oldest middle slots (no selection)
  const float* table;   // nullptr: RoPE kind NONE (re-positioning is the identity)
  int half;
};

LayerArgs make_args(const fade_config_t* c, const fade_layer_t* L, const float* table) {
  LayerArgs a;
  a.sink_k = L->sink_k;
  a.sink_v = L->sink_v;
  a.rec_k = L->recent_k;
  a.rec_v = L->recent_v;
  for (int i = 0; i < 2; ++i) {
    a.mk[i] = L->mid_k_codes[i];
    a.mv[i] = L->mid_v_codes[i];
    a.mks[i] = L->mid_k_scales[i];
    a.mvs[i] = L->mid_v_scales[i];
    a.mid_sc[i] = L->mid_scores[i];
  }
  a.sink_sc = L->sink_scores;
  a.rec_sc = L->recent_scores;
  a.meta = L->meta;
  a.victims = L->victims;
  a.chunk_base = L->chunk_base;
  a.victim_words = L->victim_words;
  a.chunk_slots = L->chunk_slots;
  a.H = c->num_kv_heads;
  a.S = c->n_sink;
  a.W = c->recent_window;
  a.C = mid_stride(c);
  a.budget = c->int4_budget;
  a.policy = c->policy;
  a.evicts = c->policy != FADE_EVICT_NONE && c->int4_budget >= 0;
  a.positional = c->policy == FADE_EVICT_POSITION;
  a.table = (c->rope.kind == FADE_ROPE_NONE) ? nullptr : table;
  a.half = c->head_dim / 2;
  return a;
}

// Load a middle key row (dequantised, exact in fp32) as warp pairs.
template <int D, int KB>
__device__ __forceinline__ WarpKey<D> load_mid_key(const uint8_t* codes, const uint16_t* scales) {
  const int lane = threadIdx.x & 31;
  WarpKey<D> k;
#pragma unroll
  for (int gp = 0; gp < D / 64; ++gp) {
    const int c1 = 32 * gp + lane, c2 = c1 + D / 2;
    k.lo[gp] = (float)unpack_code<KB>(codes, c1) * h2f(scales[c1 / kGroup]);
    k.hi[gp] = (float)unpack_code<KB>(codes, c2) * h2f(scales[c2 / kGroup]);
  }
  return k;
}

template <int D>
__device__ __forceinline__ WarpKey<D> load_fp16_key(const uint16_t* row) {
  const int lane = threadIdx.x & 31;
  WarpKey<D> k;
#pragma unroll
  for (int gp = 0; gp < D / 64; ++gp) {
    k.lo[gp] = h2f(row[32 * gp + lane]);
    k.hi[gp] = h2f(row[32 * gp + lane + D / 2]);
  }
  return k;
}

template <int D>
__device__ __forceinline__ void reposition_key(const LayerArgs& a, WarpKey<D>& k, int pold,
                                               int pnew) {
  if (!a.table || pold == pnew) return;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int gp = 0; gp < D / 64; ++gp) {
    float y1, y2;
    reposition_pair(a.table, a.half, 32 * gp + lane, pold, pnew, k.lo[gp], k.hi[gp], y1, y2);
    k.lo[gp] = y1;
    k.hi[gp] = y2;
  }
}

template <int D>
__device__ __forceinline__ void store_fp16_key(const WarpKey<D>& k, uint16_t* row) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int gp = 0; gp < D / 64; ++gp) {
    row[32 * gp + lane] = f2h(k.lo[gp]);
    row[32 * gp + lane + D / 2] = f2h(k.hi[gp]);
  }
}

// Quantise an fp16 row (V, or an unmoved K) with one warp.
template <int D, int BITS>
__device__ __forceinline__ void warp_quantize_row(const uint16_t* x, uint8_t* codes,
                                                  uint16_t* scales) {
  const int lane = threadIdx.x & 31;
  constexpr int qmax = (1 << (BITS - 1)) - 1;
#pragma unroll
  for (int g = 0; g < D / kGroup; ++g) {
    uint16_t sb;
    int q;
    quant_group_lane(h2f(x[g * kGroup + lane]), qmax, sb, q);
    pack_group_store<BITS>(q, codes + g * (kGroup * BITS / 8));
    if (lane == 0) scales[g] = sb;
  }
}

template <int BYTES>
__device__ __forceinline__ void copy_row(const void* src, void* dst) {
  if constexpr (BYTES % 16 == 0) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < BYTES / 16; ++i) d[i] = s[i];
  } else if constexpr (BYTES % 8 == 0) {
    const uint2* s = reinterpret_cast<const uint2*>(src);
    uint2* d = reinterpret_cast<uint2*>(dst);
#pragma unroll
    for (int i = 0; i < BYTES / 8; ++i) d[i] = s[i];
  } else {
    const uint32_t* s = reinterpret_cast<const uint32_t*>(src);
    uint32_t* d = reinterpret_cast<uint32_t*>(dst);
#pragma unroll
    for (int i = 0; i < BYTES / 4; ++i) d[i] = s[i];
  }
}

// ----------------------------------------------------------------- reset / demote / append
__global__ void reset_kernel(int32_t* meta, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) meta[i] = 0;
}

// One warp per unit: if the ring is full, quantise its oldest token into middle slot N_MID.
template <int D, int KB, int VB>
__global__ void __launch_bounds__(32) demote_kernel(LayerArgs a) {
  const int unit = blockIdx.y * a.H + blockIdx.x;
  int32_t* m = a.meta + unit * kF;
  const int n_rec = m[FADE_META_N_RECENT];
  if (n_rec != a.W) return;
  const int n_mid = m[FADE_META_N_MID], cur = m[FADE_META_CUR], head = m[FADE_META_HEAD];
  if (n_mid >= a.C || head < 0 || head >= a.W) return;  // host checks capacity; never overrun
  const size_t rrow = ((size_t)unit * a.W + head) * D;
  const size_t mrow = (size_t)unit * a.C + n_mid;
  warp_quantize_row<D, KB>(a.rec_k + rrow, (cur ? a.mk[1] : a.mk[0]) + mrow * (D * KB / 8),
                           (cur ? a.mks[1] : a.mks[0]) + mrow * (D / kGroup));
  warp_quantize_row<D, VB>(a.rec_v + rrow, (cur ? a.mv[1] : a.mv[0]) + mrow * (D * VB / 8),
                           (cur ? a.mvs[1] : a.mvs[0]) + mrow * (D / kGroup));
  __syncwarp();
  if (threadIdx.x == 0) {
    (cur ? a.mid_sc[1] : a.mid_sc[0])[mrow] = a.rec_sc[(size_t)unit * a.W + head];
    m[FADE_META_N_MID] = n_mid + 1;
    m[FADE_META_N_RECENT] = n_rec - 1;
    m[FADE_META_HEAD] = (head + 1) % a.W;
  }
}

// One warp per unit: the new token becomes a sink or the newest ring entry (score 0).
template <int D>
__global__ void __launch_bounds__(32) append_kernel(LayerArgs a, const uint16_t* __restrict__ k,
                                                    const uint16_t* __restrict__ v) {
  const int unit = blockIdx.y * a.H + blockIdx.x;
  int32_t* m = a.meta + unit * kF;
  const int n_sink = m[FADE_META_N_SINK], n_rec = m[FADE_META_N_RECENT];
  uint16_t *dk, *dv;
  float* dsc;
  const bool to_sink = n_sink < a.S;
  if (!to_sink && n_rec >= a.W) return;  // host checks capacity; never overwrite the ring
  if (to_sink) {
    const size_t row = (size_t)unit * a.S + n_sink;
    dk = a.sink_k + row * D;
    dv = a.sink_v + row * D;
    dsc = a.sink_sc + row;
  } else {
    const int slot = (m[FADE_META_HEAD] + n_rec) % a.W;
    const size_t row = (size_t)unit * a.W + slot;
    dk = a.rec_k + row * D;
    dv = a.rec_v + row * D;
    dsc = a.rec_sc + row;
  }
  const uint16_t* sk = k + (size_t)unit * D;
  const uint16_t* sv = v + (size_t)unit * D;
  for (int c = threadIdx.x; c < D; c += 32) {
    dk[c] = sk[c];
    dv[c] = sv[c];
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    *dsc = 0.f;
    if (to_sink)
      m[FADE_META_N_SINK] = n_sink + 1;
    else
      m[FADE_META_N_RECENT] = n_rec + 1;
  }
}

// ----------------------------------------------------------------- eviction (decode)
// One CTA per unit: choose N_MID - budget victims among the live middle tier.
__global__ void __launch_bounds__(kSelThreads) evict_select_kernel(LayerArgs a) {
  const int unit = blockIdx.y * a.H + blockIdx.x;
  int32_t* m = a.meta + unit * kF;
  const int n_mid = m[FADE_META_N_MID], cur = m[FADE_META_CUR];
  const int k = (a.evicts && n_mid > a.budget) ? n_mid - a.budget : 0;
  __syncthreads();
  if (threadIdx.x == 0) m[FADE_META_N_EV] = k;
  if (k == 0) return;
  const float* keys = (a.policy == FADE_EVICT_POSITION)
                          ? nullptr
                          : (cur ? a.mid_sc[1] : a.mid_sc[0]) + (size_t)unit * a.C;
  block_select(keys, n_mid, k, a.victims + (size_t)unit * a.victim_words,
               a.chunk_base + (size_t)unit * a.chunk_slots);
}

// Compact survivors of the live middle buffer into the other one, re-positioning keys whose
// index drops; the last x-block re-positions the recent ring in place.
// grid = (ceil(max_mid / compact_tok<D>()) + 1, H, B), 256 threads. Middle tokens: D/32 threads
// per token; thread (gp, hf) owns rotation pairs 32gp + 16hf .. +15, i.e. half of group gp
// (channels 32gp + 16hf + j) and the matching half of its partner group gp + D/64 (channels
// D/2 + 32gp + 16hf + j). A moved key is dequantised, un-RoPE'd / re-RoPE'd and re-quantised;
// each group's absmax is completed with the neighbouring thread (lane ^ 1).
template <int D>
__host__ __device__ constexpr int compact_tok() { return 256 / (D / 32); }

// Resident CTAs per SM asked of the register allocator for the compaction kernel.
#ifndef FADE_COMPACT_MIN_CTAS
#define FADE_COMPACT_MIN_CTAS 3
#endif

template <int D, int KB, int VB>
__global__ void __launch_bounds__(256, FADE_COMPACT_MIN_CTAS) evict_compact_kernel(LayerArgs a) {
  constexpr int TPT = D / 32;            // threads per token
  constexpr int TOK = compact_tok<D>();  // tokens per CTA
  constexpr int HB = 16 * KB / 8;        // bytes of half a group's K codes
  constexpr int VROW = D * VB / 8, SROW = D / kGroup, KROW = D * KB / 8;
  const int unit = blockIdx.z * a.H + blockIdx.y;
  const int32_t* m = a.meta + unit * kF;
  const int n_mid = m[FADE_META_N_MID], cur = m[FADE_META_CUR];
  // the position policy evicts the oldest slots: no selection pass, no victim bitmap
  const int n_ev = a.positional ? max(0, n_mid - a.budget) : m[FADE_META_N_EV];
  if (n_ev == 0) return;
  const int n_sink = m[FADE_META_N_SINK], n_rec = m[FADE_META_N_RECENT];
  const int head = m[FADE_META_HEAD];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nblk = gridDim.x - 1;

  if ((int)blockIdx.x == nblk) {
    // recent ring: every token's index drops by n_ev; rewrite keys in place
    for (int t = warp; t < n_rec; t += 8) {
      const int slot = (head + t) % a.W;
      uint16_t* row = a.rec_k + ((size_t)unit * a.W + slot) * D;
      WarpKey<D> k = load_fp16_key<D>(row);
      const int pold = n_sink + n_mid + t;
      reposition_key<D>(a, k, pold, pold - n_ev);
      store_fp16_key<D>(k, row);
    }
    return;
  }

  const int lo = blockIdx.x * TOK;
  if (lo >= n_mid) return;  // uniform per CTA
  const int hi = min(lo + TOK, n_mid);
  const uint32_t* bm = a.victims + (size_t)unit * a.victim_words;
  __shared__ int wpre[TOK / 32 + 1];
  __shared__ int s_base;
  if (warp == 0 && !a.positional) {
    // victims before `lo`: chunk prefix plus the words of lo's chunk that precede it
    const int w_lo = lo >> 5, w0 = (lo / kChunk) * (kChunk / 32);
    int c = (w0 + lane < w_lo) ? __popc(bm[w0 + lane]) : 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    const int nw = (hi - lo + 31) / 32;
    const int wc = lane < nw ? __popc(bm[w_lo + lane]) : 0;
    int incl = wc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int tt = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += tt;
    }
    if (lane <= TOK / 32) wpre[lane] = incl - wc;
    if (lane == 0) s_base = a.chunk_base[(size_t)unit * a.chunk_slots + lo / kChunk] + c;
  }
  __syncthreads();
  const int i = lo + threadIdx.x / TPT, t_ = threadIdx.x % TPT;
  const int gp = t_ >> 1, hf = t_ & 1;
  // The lanes of one token are adjacent (TPT divides 32) and share every flag below, so the
  // warp-wide ballot and the absmax exchange see whole tokens; nothing exits before them.
  const bool in_range = i < hi;
  bool keep = in_range;
  int nv = 0;
  if (in_range) {
    if (a.positional) {
      keep = i >= n_ev;
      nv = i - n_ev;
    } else {
      const uint32_t word = bm[i >> 5];
      keep = !((word >> (i & 31)) & 1u);
      nv = i - (s_base + wpre[(i - lo) >> 5] + __popc(word & ((1u << (i & 31)) - 1u)));
    }
  }
  const bool moved = keep && nv != i && a.table != nullptr;

  const uint8_t* mk_s = cur ? a.mk[1] : a.mk[0];
  uint8_t* mk_d = cur ? a.mk[0] : a.mk[1];
  const uint8_t* mv_s = cur ? a.mv[1] : a.mv[0];
  uint8_t* mv_d = cur ? a.mv[0] : a.mv[1];
  const uint16_t* mks_s = cur ? a.mks[1] : a.mks[0];
  uint16_t* mks_d = cur ? a.mks[0] : a.mks[1];
  const uint16_t* mvs_s = cur ? a.mvs[1] : a.mvs[0];
  uint16_t* mvs_d = cur ? a.mvs[0] : a.mvs[1];
  const float* sc_s = cur ? a.mid_sc[1] : a.mid_sc[0];
  float* sc_d = cur ? a.mid_sc[0] : a.mid_sc[1];
  const size_t si = (size_t)unit * a.C + i, di = (size_t)unit * a.C + nv;
  const int g1 = gp, g2 = gp + D / 64;
  const uint8_t* krow_s = mk_s + si * KROW;
  uint8_t* krow_d = mk_d + di * KROW;

  if (keep) {
    // V codes (this thread's share of the row), the V scales and the score
    constexpr int VSH = VROW / TPT;
    copy_row<VSH>(mv_s + si * VROW + t_ * VSH, mv_d + di * VROW + t_ * VSH);
    if (hf == 0) {
      mvs_d[di * SROW + g1] = mvs_s[si * SROW + g1];
      mvs_d[di * SROW + g2] = mvs_s[si * SROW + g2];
    }
    if (t_ == 0) sc_d[di] = sc_s[si];
    if (!moved) {
      copy_row<HB>(krow_s + g1 * 2 * HB + hf * HB, krow_d + g1 * 2 * HB + hf * HB);
      copy_row<HB>(krow_s + g2 * 2 * HB + hf * HB, krow_d + g2 * 2 * HB + hf * HB);
      if (hf == 0) {
        mks_d[di * SROW + g1] = mks_s[si * SROW + g1];
        mks_d[di * SROW + g2] = mks_s[si * SROW + g2];
      }
    }
  }
  if (__ballot_sync(0xffffffffu, moved) == 0u) return;  // warp-uniform
  f2x X1[8], X2[8];
  float a1m = 0.f, a2m = 0.f;
  if (moved) {
    const float s1 = h2f(mks_s[si * SROW + g1]), s2 = h2f(mks_s[si * SROW + g2]);
    uint32_t w1[HB / 4], w2[HB / 4];
#pragma unroll
    for (int w = 0; w < HB / 4; ++w) {
      w1[w] = reinterpret_cast<const uint32_t*>(krow_s + g1 * 2 * HB + hf * HB)[w];
      w2[w] = reinterpret_cast<const uint32_t*>(krow_s + g2 * 2 * HB + hf * HB)[w];
    }
    if constexpr (KB == 4) {
      dequant16_int4(w1, s1, X1);
      dequant16_int4(w2, s2, X2);
    } else {
      constexpr int per = 32 / KB;
      constexpr uint32_t msk = (1u << KB) - 1u, flip = 1u << (KB - 1);
      const float off = 8388608.f + (float)flip;   // 2^23 + 2^(bits-1)
      const f2x OFF = f2_pack(off, off), S1 = f2_pack(s1, s1), S2 = f2_pack(s2, s2);
      // dequantise (exact): the offset-binary code sits in the mantissa of 2^23
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int j0 = 2 * k, j1 = 2 * k + 1;
        const uint32_t c10 = ((w1[j0 / per] >> (KB * (j0 % per))) & msk) ^ flip;
        const uint32_t c11 = ((w1[j1 / per] >> (KB * (j1 % per))) & msk) ^ flip;
        const uint32_t c20 = ((w2[j0 / per] >> (KB * (j0 % per))) & msk) ^ flip;
        const uint32_t c21 = ((w2[j1 / per] >> (KB * (j1 % per))) & msk) ^ flip;
        X1[k] = f2_mul(f2_sub(f2_pack(__uint_as_float(0x4B000000u | c10),
                                      __uint_as_float(0x4B000000u | c11)), OFF), S1);
        X2[k] = f2_mul(f2_sub(f2_pack(__uint_as_float(0x4B000000u | c20),
                                      __uint_as_float(0x4B000000u | c21)), OFF), S2);
      }
    }
    // un-RoPE at the old index, re-RoPE at the new one, every product and sum rounded
    // separately: products as packed fp32x2 multiplies (two rotation pairs at once), sums as
    // scalar IEEE adds. (A packed sum fed by a packed product may be fused into one rounding
    // by the assembler; packed products read by scalar sums were bit-identical to the scalar
    // form on 16.7M probe values.) Then the cast to fp16.
    const float4* to = reinterpret_cast<const float4*>(a.table) +
                       (size_t)(n_sink + i) * (a.half / 2) + 16 * gp + 8 * hf;
    const float4* tn = reinterpret_cast<const float4*>(a.table) +
                       (size_t)(n_sink + nv) * (a.half / 2) + 16 * gp + 8 * hf;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 co = __ldg(to + k), cn = __ldg(tn + k);  // (cos, cos, sin, sin) of 2 pairs
      rotate2(X1[k], X2[k], f2_pack(co.x, co.y), f2_pack(-co.z, -co.w));
      rotate2(X1[k], X2[k], f2_pack(cn.x, cn.y), f2_pack(cn.z, cn.w));
      X1[k] = f2_round_f16(X1[k]);
      X2[k] = f2_round_f16(X2[k]);
      float p1[2], p2[2];
      f2_unpack(X1[k], p1[0], p1[1]);
      f2_unpack(X2[k], p2[0], p2[1]);
      a1m = fmaxf(a1m, fmaxf(fabsf(p1[0]), fabsf(p1[1])));
      a2m = fmaxf(a2m, fmaxf(fabsf(p2[0]), fabsf(p2[1])));
    }
  }
  // absmax of each group over the token's two half-threads (adjacent lanes)
  a1m = fmaxf(a1m, __shfl_xor_sync(0xffffffffu, a1m, 1));
  a2m = fmaxf(a2m, __shfl_xor_sync(0xffffffffu, a2m, 1));
  if (!moved) return;
  constexpr int qmax = (1 << (KB - 1)) - 1;
  float s1 = __half2float(__float2half_rn(__fdiv_rn(a1m, (float)qmax)));
  float s2 = __half2float(__float2half_rn(__fdiv_rn(a2m, (float)qmax)));
  if (a1m > 0.f && s1 == 0.f) s1 = kSubnormalMin;
  if (a2m > 0.f && s2 == 0.f) s2 = kSubnormalMin;
  uint32_t o1[HB / 4], o2[HB / 4];
#pragma unroll
  for (int w = 0; w < HB / 4; ++w) o1[w] = o2[w] = 0u;
  if (s1 > 0.f) codes_half_group<KB>(X1, s1, o1);
  if (s2 > 0.f) codes_half_group<KB>(X2, s2, o2);
#pragma unroll
  for (int w = 0; w < HB / 4; ++w) {
    reinterpret_cast<uint32_t*>(krow_d + g1 * 2 * HB + hf * HB)[w] = o1[w];
    reinterpret_cast<uint32_t*>(krow_d + g2 * 2 * HB + hf * HB)[w] = o2[w];
  }
  if (hf == 0) {
    mks_d[di * SROW + g1] = __half_as_ushort(__float2half_rn(s1));
    mks_d[di * SROW + g2] = __half_as_ushort(__float2half_rn(s2));
  }
}

__global__ void evict_commit_kernel(int32_t* meta, int units, bool positional, int budget) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  int32_t* m = meta + u * kF;
  const int n_ev = positional ? max(0, m[FADE_META_N_MID] - budget) : m[FADE_META_N_EV];
  if (n_ev > 0) {
    m[FADE_META_N_MID] -= n_ev;
    m[FADE_META_CUR] ^= 1;
    m[FADE_META_N_EV] = 0;
  }
}

// ----------------------------------------------------------------- prefill
struct PrefillArgs {
  const uint16_t* k;    // [B][H][maxP][D], RoPE'd at 0..P-1
  const uint16_t* v;
  const float* mass;    // [B][H][maxP] or nullptr
  int maxP;
};

struct PrefillSplit {
  int n_s, n_r, n_m0, k;
};

__device__ __forceinline__ PrefillSplit prefill_split(const LayerArgs& a, int P) {
  PrefillSplit s;
  s.n_s = min(a.S, P);
  s.n_r = min(a.W, P - s.n_s);
  s.n_m0 = P - s.n_s - s.n_r;
  s.k = (a.evicts && s.n_m0 > a.budget) ? s.n_m0 - a.budget : 0;
  return s;
}

__global__ void __launch_bounds__(kSelThreads) prefill_select_kernel(LayerArgs a, PrefillArgs p,
                                                                     RowLens lens) {
  const int unit = blockIdx.y * a.H + blockIdx.x;
  const PrefillSplit s = prefill_split(a, lens.v[blockIdx.y]);
  if (s.k == 0) return;
  const float* keys = (a.policy == FADE_EVICT_H2O) ? p.mass + (size_t)unit * p.maxP + s.n_s
                                                   : nullptr;  // EMA: all 0; position: index
  block_select(keys, s.n_m0, s.k, a.victims + (size_t)unit * a.victim_words,
               a.chunk_base + (size_t)unit * a.chunk_slots);
}

// grid = (ceil(maxP / kChunk), H, B), 8 warps; one warp per prompt token.
template <int D, int KB, int VB>
__global__ void __launch_bounds__(256) prefill_place_kernel(LayerArgs a, PrefillArgs p,
                                                            RowLens lens) {
  const int b = blockIdx.z, unit = b * a.H + blockIdx.y;
  const int P = lens.v[b];
  const PrefillSplit s = prefill_split(a, P);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lo = blockIdx.x * kChunk, hi = min(lo + kChunk, P);
  const uint32_t* bm = a.victims + (size_t)unit * a.victim_words;
  const int32_t* cb = a.chunk_base + (size_t)unit * a.chunk_slots;
  const int m_keep = s.n_m0 - s.k;
  constexpr int KROW = D * KB / 8, VROW = D * VB / 8, SROW = D / kGroup;
  for (int i = lo + warp; i < hi; i += 8) {
    int nv;
    int tier;  // 0 sink, 1 middle, 2 recent
    if (i < s.n_s) {
      nv = i;
      tier = 0;
    } else if (i < s.n_s + s.n_m0) {
      const int ci = i - s.n_s;
      if (s.k > 0) {
        if ((bm[ci >> 5] >> (ci & 31)) & 1u) continue;  // evicted
        nv = i - victims_before(bm, cb, ci);
      } else {
        nv = i;
      }
      tier = 1;
    } else {
      nv = i - s.k;
      tier = 2;
    }
    const size_t src = ((size_t)unit * p.maxP + i) * D;
    WarpKey<D> key = load_fp16_key<D>(p.k + src);
    reposition_key<D>(a, key, i, nv);
    const float score = (a.policy == FADE_EVICT_H2O && p.mass) ? p.mass[(size_t)unit * p.maxP + i]
                                                               : 0.f;
    if (tier == 1) {
      const size_t row = (size_t)unit * a.C + (nv - s.n_s);
      warp_store_quantized<D, KB>(key, a.mk[0] + row * KROW, a.mks[0] + row * SROW);
      warp_quantize_row<D, VB>(p.v + src, a.mv[0] + row * VROW, a.mvs[0] + row * SROW);
      if (lane == 0) a.mid_sc[0][row] = score;
    } else {
      size_t row;
      uint16_t *dk, *dv;
      float* dsc;
      if (tier == 0) {
        row = (size_t)unit * a.S + nv;
        dk = a.sink_k;
        dv = a.sink_v;
        dsc = a.sink_sc;
      } else {
        row = (size_t)unit * a.W + (nv - s.n_s - m_keep);  // ring head is slot 0
        dk = a.rec_k;
        dv = a.rec_v;
        dsc = a.rec_sc;
      }
      store_fp16_key<D>(key, dk + row * D);
      for (int c = lane; c < D; c += 32) dv[row * D + c] = p.v[src + c];
      if (lane == 0) dsc[row] = score;
    }
  }
}

__global__ void prefill_commit_kernel(LayerArgs a, RowLens lens, int units) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= units) return;
  const PrefillSplit s = prefill_split(a, lens.v[u / a.H]);
  int32_t* m = a.meta + u * kF;
  m[FADE_META_N_SINK] = s.n_s;
  m[FADE_META_N_MID] = s.n_m0 - s.k;
  m[FADE_META_N_RECENT] = s.n_r;
  m[FADE_META_HEAD] = 0;
  m[FADE_META_CUR] = 0;
  m[FADE_META_N_EV] = 0;
  m[FADE_META_P0] = 0;
  m[FADE_META_P1] = 0;
}

// ----------------------------------------------------------------- dispatch
template <template <int, int, int> class F, typename... Args>
fade_status_t dispatch_dkv(const fade_config_t* c, Args&&... args) {
  const int d = c->head_dim, kb = c->middle_k_bits, vb = c->middle_v_bits;
#define FADE_CASE(D_, KB_, VB_) \
  if (d == D_ && kb == KB_ && vb == VB_) return F<D_, KB_, VB_>::run(args...);
  FADE_CASE(64, 4, 2) FADE_CASE(64, 4, 4) FADE_CASE(64, 2, 2) FADE_CASE(64, 2, 4)
  FADE_CASE(128, 4, 2) FADE_CASE(128, 4, 4) FADE_CASE(128, 2, 2) FADE_CASE(128, 2, 4)
#undef FADE_CASE
  return set_error(FADE_ERR_UNSUPPORTED, "unsupported (head_dim, k_bits, v_bits)");
}

template <int D, int KB, int VB>
struct DemoteLaunch {
  static fade_status_t run(const LayerArgs& a, int B, cudaStream_t st) {
    demote_kernel<D, KB, VB><<<dim3(a.H, B), 32, 0, st>>>(a);
    return launch_status("fade_cache_demote");
  }
};

template <int D, int KB, int VB>
struct CompactLaunch {
  static fade_status_t run(const LayerArgs& a, int B, int chunks, cudaStream_t st) {
    evict_compact_kernel<D, KB, VB><<<dim3(chunks + 1, a.H, B), 256, 0, st>>>(a);  // chunks of compact_tok<D>() tokens
    return launch_status("fade_evict_rerope compact");
  }
};

template <int D, int KB, int VB>
struct PlaceLaunch {
  static fade_status_t run(const LayerArgs& a, const PrefillArgs& p, const RowLens& lens, int B,
                           cudaStream_t st) {
    prefill_place_kernel<D, KB, VB>
        <<<dim3(ceil_div(p.maxP, kChunk), a.H, B), 256, 0, st>>>(a, p, lens);
    return launch_status("fade_cache_prefill place");
  }
};

fade_status_t check_table(const fade_config_t* c, const float* table, int max_pos, int need) {
  if (c->rope.kind == FADE_ROPE_NONE) return FADE_OK;
  if (!table) return set_error(FADE_ERR_INVALID_ARGUMENT, "RoPE table is NULL");
  if (max_pos < need)
    return set_error(FADE_ERR_CAPACITY, "RoPE table holds %d positions, %d needed", max_pos,
                     need);
  return FADE_OK;
}

}  // namespace
}  // namespace fade

using namespace fade;

extern "C" fade_status_t fade_cache_reset(const fade_config_t* c, fade_layer_t* L, void* stream) {
  clear_error();
  fade_status_t st = validate_config(c);
  if (!st) st = validate_layer(c, L);
  if (st) return st;
  const int n = c->batch * c->num_kv_heads * FADE_META_FIELDS;
  reset_kernel<<<ceil_div(n, 256), 256, 0, as_stream(stream)>>>(L->meta, n);
  if ((st = launch_status("fade_cache_reset"))) return st;
  reset_kernel<<<1, 32, 0, as_stream(stream)>>>(L->status, FADE_STATUS_WORDS);
  for (int b = 0; b < c->batch; ++b) L->h_n_sink[b] = L->h_n_mid[b] = L->h_n_recent[b] = 0;
  return launch_status("fade_cache_reset");
}

extern "C" fade_status_t fade_cache_prefill(const fade_config_t* c, fade_layer_t* L,
                                            const uint16_t* k_rot, const uint16_t* v,
                                            int32_t max_prompt, const int32_t* h_prompt_len,
                                            const float* mass, const float* table,
                                            int32_t max_pos, void* stream) {
  clear_error();
  fade_status_t st = validate_config(c);
  if (!st) st = validate_layer(c, L);
  if (st) return st;
  if (!k_rot || !v || !h_prompt_len)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL prompt or lengths");
  if (max_prompt < 1) return set_error(FADE_ERR_INVALID_ARGUMENT, "max_prompt < 1");
  if (c->policy == FADE_EVICT_H2O && c->int4_budget >= 0 && !mass)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "H2O prefill needs the prefill mass");
  if ((long long)L->victim_words < (max_prompt + 31) / 32 + 1 ||
      (long long)L->chunk_slots < (max_prompt + kChunk - 1) / kChunk + 1)
    return set_error(FADE_ERR_CAPACITY, "scratch buffers are sized for a shorter prompt");
  if ((st = check_table(c, table, max_pos, max_prompt))) return st;
  RowLens lens{};
  const bool evicts = c->policy != FADE_EVICT_NONE && c->int4_budget >= 0;
  for (int b = 0; b < c->batch; ++b) {
    if (L->h_n_sink[b] || L->h_n_mid[b] || L->h_n_recent[b])
      return set_error(FADE_ERR_INVALID_ARGUMENT, "prefill needs an empty cache (reset first)");
    const int P = h_prompt_len[b];
    if (P < 0 || P > max_prompt)
      return set_error(FADE_ERR_INVALID_ARGUMENT, "row %d prompt length %d outside [0, %d]", b,
                       P, max_prompt);
    lens.v[b] = P;
    const int n_s = P < c->n_sink ? P : c->n_sink;
    const int n_r = (P - n_s) < c->recent_window ? (P - n_s) : c->recent_window;
    int n_m = P - n_s - n_r;
    if (evicts && n_m > c->int4_budget) n_m = c->int4_budget;
    if (n_m > c->mid_capacity)
      return set_error(FADE_ERR_CAPACITY, "row %d needs %d middle slots, capacity %d", b, n_m,
                       c->mid_capacity);
  }
  const LayerArgs a = make_args(c, L, table);
  const PrefillArgs p{k_rot, v, mass, max_prompt};
  cudaStream_t s = as_stream(stream);
  prefill_select_kernel<<<dim3(c->num_kv_heads, c->batch), kSelThreads, 0, s>>>(a, p, lens);
  if ((st = launch_status("fade_cache_prefill select"))) return st;
  if ((st = dispatch_dkv<PlaceLaunch>(c, a, p, lens, c->batch, s))) return st;
  const int units = c->batch * c->num_kv_heads;
  prefill_commit_kernel<<<ceil_div(units, 128), 128, 0, s>>>(a, lens, units);
  if ((st = launch_status("fade_cache_prefill commit"))) return st;
  for (int b = 0; b < c->batch; ++b) {
    const int P = lens.v[b];
    const int n_s = P < c->n_sink ? P : c->n_sink;
    const int n_r = (P - n_s) < c->recent_window ? (P - n_s) : c->recent_window;
    int n_m = P - n_s - n_r;
    if (evicts && n_m > c->int4_budget) n_m = c->int4_budget;
    L->h_n_sink[b] = n_s;
    L->h_n_mid[b] = n_m;
    L->h_n_recent[b] = n_r;
  }
  return FADE_OK;
}

extern "C" fade_status_t fade_cache_demote(const fade_config_t* c, fade_layer_t* L,
                                           void* stream) {
  clear_error();
  fade_status_t st = validate_config(c);
  if (!st) st = validate_layer(c, L);
  if (st) return st;
  bool any = false;
  for (int b = 0; b < c->batch; ++b)
    if (L->h_n_recent[b] == c->recent_window) {
      if (L->h_n_mid[b] + 1 > c->mid_capacity)
        return set_error(FADE_ERR_CAPACITY, "row %d: middle tier full (%d slots)", b,
                         c->mid_capacity);
      any = true;
    }
  if (!any) return FADE_OK;
  const LayerArgs a = make_args(c, L, nullptr);
  if ((st = dispatch_dkv<DemoteLaunch>(c, a, c->batch, as_stream(stream)))) return st;
  for (int b = 0; b < c->batch; ++b)
    if (L->h_n_recent[b] == c->recent_window) {
      L->h_n_mid[b] += 1;
      L->h_n_recent[b] -= 1;
    }
  return FADE_OK;
}

extern "C" fade_status_t fade_cache_append(const fade_config_t* c, fade_layer_t* L,
                                           const uint16_t* k_rot, const uint16_t* v,
                                           void* stream) {
  clear_error();
  fade_status_t st = validate_config(c);
  if (!st) st = validate_layer(c, L);
  if (st) return st;
  if (!k_rot || !v) return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL k or v");
  for (int b = 0; b < c->batch; ++b)
    if (L->h_n_sink[b] >= c->n_sink && L->h_n_recent[b] >= c->recent_window)
      return set_error(FADE_ERR_CAPACITY, "row %d: recent window full (demote first)", b);
  const LayerArgs a = make_args(c, L, nullptr);
  const dim3 grid(c->num_kv_heads, c->batch);
  if (c->head_dim == 64)
    append_kernel<64><<<grid, 32, 0, as_stream(stream)>>>(a, k_rot, v);
  else
    append_kernel<128><<<grid, 32, 0, as_stream(stream)>>>(a, k_rot, v);
  if ((st = launch_status("fade_cache_append"))) return st;
  for (int b = 0; b < c->batch; ++b) {
    if (L->h_n_sink[b] < c->n_sink)
      L->h_n_sink[b] += 1;
    else
      L->h_n_recent[b] += 1;
  }
  return FADE_OK;
}

extern "C" fade_status_t fade_evict_rerope(const fade_config_t* c, fade_layer_t* L,
                                           const float* table, int32_t max_pos, void* stream) {
  clear_error();
  fade_status_t st = validate_config(c);
  if (!st) st = validate_layer(c, L);
  if (st) return st;
  const bool evicts = c->policy != FADE_EVICT_NONE && c->int4_budget >= 0;
  if (!evicts) return FADE_OK;
  int max_mid = 0;
  bool any = false;
  for (int b = 0; b < c->batch; ++b) {
    if (L->h_n_mid[b] > max_mid) max_mid = L->h_n_mid[b];
    if (L->h_n_mid[b] > c->int4_budget) any = true;
  }
  if (!any) return FADE_OK;
  if ((long long)L->victim_words < (c->mid_capacity + 31) / 32 + 1 ||
      (long long)L->chunk_slots < (c->mid_capacity + kChunk - 1) / kChunk + 1)
    return set_error(FADE_ERR_CAPACITY, "scratch buffers are smaller than the middle tier");
  if ((st = check_table(c, table, max_pos, c->n_sink + c->mid_capacity + c->recent_window)))
    return st;
  const LayerArgs a = make_args(c, L, table);
  cudaStream_t s = as_stream(stream);
  if (!a.positional) {  // the position policy needs no selection pass
    evict_select_kernel<<<dim3(c->num_kv_heads, c->batch), kSelThreads, 0, s>>>(a);
    if ((st = launch_status("fade_evict_rerope select"))) return st;
  }
  const int ctok = c->head_dim == 128 ? compact_tok<128>() : compact_tok<64>();
  if ((st = dispatch_dkv<CompactLaunch>(c, a, c->batch, ceil_div(max_mid, ctok), s))) return st;
  const int units = c->batch * c->num_kv_heads;
  evict_commit_kernel<<<ceil_div(units, 128), 128, 0, s>>>(L->meta, units, a.positional,
                                                            c->int4_budget);
  if ((st = launch_status("fade_evict_rerope commit"))) return st;
  for (int b = 0; b < c->batch; ++b)
    if (L->h_n_mid[b] > c->int4_budget) L->h_n_mid[b] = c->int4_budget;
  return FADE_OK;
}
