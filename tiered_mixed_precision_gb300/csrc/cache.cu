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
// Resident CTAs per SM the compaction kernel is compiled for (its register budget).
#ifndef FADE_COMPACT_MINB
#define FADE_COMPACT_MINB 2
#endif
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

// Selection keys: one unit's scores, or (rows sharing their tier decisions) the sum over the
// batch rows of the same candidate's scores, added in ascending row order in fp32. `p` null:
// every key equal (the oldest go first).
struct KeysOne {
  const float* p;
  __device__ float operator()(int i) const { return p[i]; }
};
struct KeysRows {
  const float* p;   // row 0's scores of the unit
  size_t stride;    // floats from one row's unit to the next row's
  int rows;
  __device__ float operator()(int i) const {
    float s = p[i];
    for (int r = 1; r < rows; ++r) s += p[(size_t)r * stride + i];
    return s;
  }
};

// Selects the k smallest (key, index) among n candidates with one CTA of kSelThreads
// threads: an exact 4-pass radix select finds the k-th smallest key T, then one pass in index
// order marks keys < T and the first (k - #below) keys equal to T. keys == nullptr means all
// keys are equal (the oldest k go first). Writes bitmap words [0, ceil(n/32)) and
// chunk_base[c] = victims among candidates [0, c*kChunk), c = 0..ceil(n/kChunk).
template <class Keys>
__device__ void block_select(Keys keys, int n, int k, uint32_t* __restrict__ bitmap,
                             int32_t* __restrict__ chunk_base) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_rem;
  __shared__ int sh[33];
  const int tid = threadIdx.x;
  uint32_t T = ord_key(0.f);
  int remaining = k;
  if (keys.p && k > 0) {
    uint32_t prefix = 0, mask = 0;
    int rem = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < n; i += blockDim.x) {
        const uint32_t u = ord_key(keys(i));
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
    const uint32_t u = valid ? (keys.p ? ord_key(keys(i)) : T) : 0u;
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

// block_select for k = 1 (one victim: the steady state of a decode step) in one pass: the
// smallest (key, index) pair, i.e. the lowest index among the smallest keys, by a block-wide
// minimum over 64-bit (ordered key, index) words; then the bitmap and the chunk prefixes.
template <class Keys>
__device__ void block_select_one(Keys keys, int n, uint32_t* __restrict__ bitmap,
                                 int32_t* __restrict__ chunk_base) {
  __shared__ unsigned long long s_best[kSelThreads / 32];
  __shared__ int s_victim;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long best = ~0ull;
  if (keys.p) {
    for (int i = tid; i < n; i += kSelThreads) {
      const unsigned long long c = ((unsigned long long)ord_key(keys(i)) << 32) | (uint32_t)i;
      best = c < best ? c : best;
    }
  } else if (tid == 0) {
    best = 0ull;  // all keys equal: the oldest
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(0xffffffffu, best, o);
    best = t < best ? t : best;
  }
  if (lane == 0) s_best[warp] = best;
  __syncthreads();
  if (warp == 0) {
    best = lane < kSelThreads / 32 ? s_best[lane] : ~0ull;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const unsigned long long t = __shfl_xor_sync(0xffffffffu, best, o);
      best = t < best ? t : best;
    }
    if (lane == 0) s_victim = (int)(uint32_t)(best & 0xffffffffull);
  }
  __syncthreads();
  const int vic = s_victim;
  for (int w = tid; w < (n + 31) / 32; w += kSelThreads)
    bitmap[w] = (w == (vic >> 5)) ? (1u << (vic & 31)) : 0u;
  const int nc = (n + kChunk - 1) / kChunk;
  for (int c = tid; c <= nc; c += kSelThreads) chunk_base[c] = (vic < c * kChunk) ? 1 : 0;
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
  bool shared;      // the rows share their tier decisions (row-summed selection keys)
  int B;            // batch rows
  const float* table;   // nullptr: RoPE kind NONE (re-positioning is the identity)
  int half;
  bool pq;                    // middle-tier V is product-quantised (codes in the INT2 rows)
  const uint16_t* pq_cb;      // the layer's PQ codebook, fp16 [d/4][256][4]
  float one, neg_one;         // 1 and -1, opaque to the compiler (see PlusMinus)
  int rd;                     // rotated width (head_dim unless proportional RoPE)
  int32_t* status;            // the layer's device status words (device-side checks)
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
  a.shared = c->shared_rows != 0;
  a.B = c->batch;
  a.table = (c->rope.kind == FADE_ROPE_NONE) ? nullptr : table;
  a.half = c->head_dim / 2;
  a.pq = c->v_codec == FADE_V_PQ;
  a.pq_cb = L->pq_codebook;
  a.one = 1.0f;
  a.neg_one = -1.0f;
  a.rd = rotary_width(c);
  a.status = L->status;
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

// One warp: the oldest ring token (slot `head`) of a unit quantise-packed into middle slot
// n_mid of buffer `cur` (K at KB bits; V at VB bits, or PQ-encoded), its score moved with it.
// The unit's counts are the caller's to update.
// The two halves of a demotion, each for one warp: K codes and scales plus the score, and V.
template <int D, int KB>
__device__ __forceinline__ void warp_demote_k(const LayerArgs& a, int unit, int n_mid, int cur,
                                              int head) {
  const size_t rrow = ((size_t)unit * a.W + head) * D;
  const size_t mrow = (size_t)unit * a.C + n_mid;
  warp_quantize_row<D, KB>(a.rec_k + rrow, (cur ? a.mk[1] : a.mk[0]) + mrow * (D * KB / 8),
                           (cur ? a.mks[1] : a.mks[0]) + mrow * (D / kGroup));
  if ((threadIdx.x & 31) == 0)
    (cur ? a.mid_sc[1] : a.mid_sc[0])[mrow] = a.rec_sc[(size_t)unit * a.W + head];
}
template <int D, int VB>
__device__ __forceinline__ void warp_demote_v(const LayerArgs& a, int unit, int n_mid, int cur,
                                              int head) {
  const size_t rrow = ((size_t)unit * a.W + head) * D;
  const size_t mrow = (size_t)unit * a.C + n_mid;
  if (a.pq)
    warp_pq_encode_row<D>(a.rec_v + rrow, a.pq_cb, (cur ? a.mv[1] : a.mv[0]) + mrow * (D / 4),
                          (cur ? a.mvs[1] : a.mvs[0]) + mrow * (D / kGroup));
  else
    warp_quantize_row<D, VB>(a.rec_v + rrow, (cur ? a.mv[1] : a.mv[0]) + mrow * (D * VB / 8),
                             (cur ? a.mvs[1] : a.mvs[0]) + mrow * (D / kGroup));
}

// Two warps per unit: if the ring is full, quantise its oldest token into middle slot N_MID
// (warp 0 its K and score, warp 1 its V, side by side).
template <int D, int KB, int VB>
__global__ void __launch_bounds__(64) demote_kernel(LayerArgs a) {
  const int unit = blockIdx.y * a.H + blockIdx.x;
  int32_t* m = a.meta + unit * kF;
  const int n_rec = m[FADE_META_N_RECENT];
  if (n_rec != a.W) return;  // uniform per CTA
  const int n_mid = m[FADE_META_N_MID], cur = m[FADE_META_CUR], head = m[FADE_META_HEAD];
  if (n_mid >= a.C || head < 0 || head >= a.W) {  // the host checks capacity; never overrun
    if (threadIdx.x == 0) record_status(a.status, kCheckDemoteSlot);
    return;
  }
  if (threadIdx.x < 32)
    warp_demote_k<D, KB>(a, unit, n_mid, cur, head);
  else
    warp_demote_v<D, VB>(a, unit, n_mid, cur, head);
  __syncthreads();  // both warps have read the counts and the ring slot
  if (threadIdx.x == 0) {
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
  if (!to_sink && n_rec >= a.W) {  // the host checks capacity; never overwrite the ring
    if (threadIdx.x == 0) record_status(a.status, kCheckAppendSlot);
    return;
  }
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

// One CTA per unit (row b, KV head h): a decode step's RoPE and append in one launch. The
// unit's G query heads and its new key are rotated at the row's position exactly as
// rope_apply_kernel rotates them (slot k < rh rotates the pair (k, k + rh) with the table's
// cos and sin, the remaining slots copy their two pass-through channels; no table: a copy),
// the queries into q_rot and the key straight into the slot append_kernel gives it (a sink
// while fewer than n_sink are held, else the newest ring entry), with its value and score 0.
// DEMOTE: first, if the ring is full, warps 0 and 1 demote its oldest token exactly as
// demote_kernel does (while the other warps rotate queries); the new token then takes the freed
// slot.
#ifndef FADE_ROPE_APPEND_THREADS
#define FADE_ROPE_APPEND_THREADS 256
#endif
static_assert(FADE_ROPE_APPEND_THREADS >= 128 && FADE_ROPE_APPEND_THREADS % 32 == 0,
              "two demoting warps; one thread per channel of the new token (D <= 128)");
template <int D, int KB, int VB, bool DEMOTE>
__global__ void __launch_bounds__(FADE_ROPE_APPEND_THREADS)
    rope_append_kernel(LayerArgs a, const float* __restrict__ table, int max_pos, int rh,
                       const uint16_t* __restrict__ q_raw, const uint16_t* __restrict__ k_raw,
                       const uint16_t* __restrict__ v, const int32_t* __restrict__ pos,
                       uint16_t* __restrict__ q_rot, int Hq) {
  // the attention kernel that follows may be a programmatic dependent: let it be scheduled now
  asm volatile("griddepcontrol.launch_dependents;");
  constexpr int half = D / 2;
  const int h = blockIdx.x, b = blockIdx.y, unit = b * a.H + h;
  const int G = Hq / a.H;
  const int p = table ? min(max(pos[b], 0), max_pos - 1) : 0;
  int32_t* m = a.meta + unit * kF;
  const int n_sink = m[FADE_META_N_SINK], n_rec0 = m[FADE_META_N_RECENT];
  const int head0 = m[FADE_META_HEAD];
  int n_rec = n_rec0, head = head0;
  const bool demote = DEMOTE && n_rec0 == a.W;  // uniform per CTA
  if (demote) {
    const int n_mid = m[FADE_META_N_MID], cur = m[FADE_META_CUR];
    if (n_mid >= a.C || head0 < 0 || head0 >= a.W) {  // the host checks capacity
      if (threadIdx.x == 0) record_status(a.status, kCheckDemoteSlot);
      asm volatile("griddepcontrol.wait;" ::: "memory");  // see the end of the kernel
      return;
    }
    if (threadIdx.x < 32)
      warp_demote_k<D, KB>(a, unit, n_mid, cur, head0);
    else if (threadIdx.x < 64)
      warp_demote_v<D, VB>(a, unit, n_mid, cur, head0);
    n_rec = n_rec0 - 1;
    head = (head0 + 1) % a.W;
  }
  // slot k of vector x (D channels): its two output channels c0, c1 and their values
  auto rot = [&](const uint16_t* x, int k, int& c0, int& c1, uint16_t& y0, uint16_t& y1) {
    if (!table) {
      c0 = k;
      c1 = k + half;
      y0 = x[c0];
      y1 = x[c1];
    } else if (k >= rh) {
      c0 = 2 * rh + 2 * (k - rh);
      c1 = c0 + 1;
      y0 = x[c0];
      y1 = x[c1];
    } else {
      float f1, f2;
      rotate_pair(h2f(x[k]), h2f(x[k + rh]), rope_cos(table, half, p, k),
                  rope_sin(table, half, p, k), f1, f2);
      c0 = k;
      c1 = k + rh;
      y0 = f2h(f1);
      y1 = f2h(f2);
    }
  };
  for (int i = threadIdx.x; i < G * half; i += blockDim.x) {
    const size_t base = ((size_t)b * Hq + (size_t)h * G + i / half) * D;
    int c0, c1;
    uint16_t y0, y1;
    rot(q_raw + base, i % half, c0, c1, y0, y1);
    q_rot[base + c0] = y0;
    q_rot[base + c1] = y1;
  }
  // the new token's key slot (thread k < D/2) rotated and its value channel (thread c < D) read
  // now; both are stored once the demotion has read the slot they may overwrite
  int kc0 = 0, kc1 = 0;
  uint16_t ky0 = 0, ky1 = 0, vy = 0;
  if (threadIdx.x < half) rot(k_raw + (size_t)unit * D, threadIdx.x, kc0, kc1, ky0, ky1);
  if (threadIdx.x < D) vy = v[(size_t)unit * D + threadIdx.x];
  if (demote) __syncthreads();  // the demoted slot is read before the new token overwrites it
  const bool to_sink = n_sink < a.S;
  if (!to_sink && n_rec >= a.W) {  // the host checks capacity; never overwrite the ring
    if (threadIdx.x == 0) record_status(a.status, kCheckAppendSlot);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // see the end of the kernel
    return;
  }
  size_t row;
  uint16_t *dk, *dv;
  float* dsc;
  if (to_sink) {
    row = (size_t)unit * a.S + n_sink;
    dk = a.sink_k + row * D;
    dv = a.sink_v + row * D;
    dsc = a.sink_sc + row;
  } else {
    row = (size_t)unit * a.W + (head + n_rec) % a.W;
    dk = a.rec_k + row * D;
    dv = a.rec_v + row * D;
    dsc = a.rec_sc + row;
  }
  if (threadIdx.x < half) {
    dk[kc0] = ky0;
    dk[kc1] = ky1;
  }
  if (threadIdx.x < D) dv[threadIdx.x] = vy;
  __syncthreads();  // every thread has read the counts
  if (threadIdx.x == 0) {
    *dsc = 0.f;
    if (demote) {
      m[FADE_META_N_MID] += 1;
      m[FADE_META_HEAD] = head;
    }
    if (to_sink)
      m[FADE_META_N_SINK] = n_sink + 1;
    else
      m[FADE_META_N_RECENT] = n_rec + 1;
  }
  // launched as a programmatic dependent of the previous layer's last kernel (the score update
  // or the combine), which this kernel's work does not touch: finish only once that grid has
  // completed, so that whatever follows this kernel finds it done (the attention call reuses the
  // workspaces it reads)
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ----------------------------------------------------------------- eviction (decode)
// One CTA per unit: choose N_MID - budget victims among the live middle tier.
// Copies unit `from`'s victim bitmap (n candidates) and chunk prefixes to unit `to`.
__device__ void copy_selection(const LayerArgs& a, int from, int to, int n) {
  const uint32_t* bs = a.victims + (size_t)from * a.victim_words;
  uint32_t* bd = a.victims + (size_t)to * a.victim_words;
  for (int w = threadIdx.x; w < (n + 31) / 32; w += blockDim.x) bd[w] = bs[w];
  const int32_t* cs = a.chunk_base + (size_t)from * a.chunk_slots;
  int32_t* cd = a.chunk_base + (size_t)to * a.chunk_slots;
  for (int c = threadIdx.x; c <= (n + kChunk - 1) / kChunk; c += blockDim.x) cd[c] = cs[c];
}

// grid = (H, B) with one CTA per unit; rows sharing their decisions: grid = (H, 1), the CTA
// selects by the row-summed scores of head h and gives every row the same victims (the rows
// hold equal counts and evolve alike, so their live buffers agree).
__global__ void __launch_bounds__(kSelThreads) evict_select_kernel(LayerArgs a) {
  const int unit = blockIdx.y * a.H + blockIdx.x;
  int32_t* m = a.meta + unit * kF;
  const int n_mid = m[FADE_META_N_MID], cur = m[FADE_META_CUR];
  const int k = (a.evicts && n_mid > a.budget) ? n_mid - a.budget : 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    m[FADE_META_N_EV] = k;
    if (a.shared)
      for (int r = 1; r < a.B; ++r) a.meta[(r * a.H + blockIdx.x) * kF + FADE_META_N_EV] = k;
  }
  if (k == 0) return;
  const float* sc = (a.policy == FADE_EVICT_POSITION)
                        ? nullptr
                        : (cur ? a.mid_sc[1] : a.mid_sc[0]) + (size_t)unit * a.C;
  uint32_t* bm = a.victims + (size_t)unit * a.victim_words;
  int32_t* cb = a.chunk_base + (size_t)unit * a.chunk_slots;
  if (a.shared) {
    const KeysRows keys{sc, (size_t)a.H * a.C, a.B};
    if (k == 1)
      block_select_one(keys, n_mid, bm, cb);
    else
      block_select(keys, n_mid, k, bm, cb);
    __syncthreads();
    for (int r = 1; r < a.B; ++r) copy_selection(a, unit, r * a.H + blockIdx.x, n_mid);
  } else {
    const KeysOne keys{sc};
    if (k == 1)
      block_select_one(keys, n_mid, bm, cb);
    else
      block_select(keys, n_mid, k, bm, cb);
  }
}

// 8 consecutive fp16 values (16-byte aligned) as 4 packed fp32 pairs, and back (RN to fp16).
__device__ __forceinline__ void load_f16x8(const uint16_t* p, f2x (&X)[4]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
    X[k] = f2_pack(f.x, f.y);
  }
}
__device__ __forceinline__ void store_f16x8(const f2x (&X)[4], uint16_t* p) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float lo, hi;
    f2_unpack(X[k], lo, hi);
    const __half2 h = __floats2half2_rn(lo, hi);
    w[k] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Recent-ring re-positioning: geometry. D/32 threads per ring token; thread t_ owns the rotation
// pairs 16 t_ .. 16 t_ + 15.
template <int D>
struct RecentCfg {
  static constexpr int TPT = D / 32;        // threads per ring token
  static constexpr int TOK = 256 / TPT;     // ring tokens per pass of the CTA
  static constexpr int ROWF4 = D / 4;       // float4 per RoPE row: d/2 pairs x (cos, sin)
  static constexpr int NROWS = TOK + 32;    // staged RoPE rows
  static constexpr int TPW = 32 / TPT;      // tokens per warp
  static constexpr int TABF4 = NROWS * (ROWF4 + 1);  // staged rows padded by one float4
};

// Float4 slot of (row, j) in the staged table: rows padded by one float4, so the eight
// threads of a quarter warp (eight consecutive tokens with the same t_, reading the same j of
// eight consecutive rows) hit eight different bank quads.
template <int D>
__device__ __forceinline__ int tab_slot(int row, int j) {
  return row * (D / 4 + 1) + j;
}

// Middle-tier compaction: geometry. D/64 threads per middle token; thread t_ of a token owns
// the rotation pairs 32 t_ .. 32 t_ + 31, i.e. the whole quantisation groups t_ (channels
// 32 t_ + j) and t_ + D/64 (their partners D/2 + 32 t_ + j), so a group's absmax, scale and
// codes stay in one thread.
template <int D>
struct MidCfg {
  static constexpr int TPT = D / 64;        // threads per middle token
  static constexpr int TOK = 256 / TPT;     // middle indices per CTA
  static constexpr int TPW = 32 / TPT;      // tokens per warp
  static constexpr int ROWF4 = D / 4;       // float4 per RoPE row: d/2 pairs x (cos, sin)
  static constexpr int NROWS = TOK + 16;    // staged RoPE rows (blocks with n_ev <= 16)
  static constexpr int TABF4 = NROWS * (ROWF4 + 1);  // staged rows padded by one float4
  static constexpr int PRE = TOK / 32 + 2;  // per-head ints: victim prefix words + base
  // with the block's TOK/32 bitmap words after them (selection policies, staged bitmap)
  static constexpr int PRE_SEL = PRE + TOK / 32;
};
// Shared memory of the compaction kernel: the staged RoPE rows, then per head the counts and
// the victim prefixes of the block.
template <int D>
size_t compact_smem(int H) {
  return (size_t)MidCfg<D>::TABF4 * 16 + (size_t)H * (MidCfg<D>::PRE_SEL + 5) * 4;
}

template <int D>
__host__ __device__ constexpr int compact_tok() { return MidCfg<D>::TOK; }

// Packed (1, 1) and (-1, -1) whose values the compiler cannot see (they come from kernel
// arguments). A sum or difference of two separately rounded products is taken as
// fma(p, +-1, q): that rounds p +- q once, exactly like the scalar IEEE sum, and the product
// that made p cannot be fused into it.
struct PlusMinus {
  f2x one, neg;
};

// Rotation of two pairs at once with every product and every sum rounded on its own:
// X1 = (x_a, x_b) of the first half, X2 = their partners, C and S the pairs' cos and sin.
__device__ __forceinline__ void rot2_inv_pm(f2x& X1, f2x& X2, f2x C, f2x S, const PlusMinus& u) {
  const f2x p = f2_mul(X1, C), q = f2_mul(X2, S), r = f2_mul(X2, C), t = f2_mul(X1, S);
  X1 = f2_fma(p, u.one, q);  // x1 c + x2 s
  X2 = f2_fma(t, u.neg, r);  // x2 c - x1 s
}
__device__ __forceinline__ void rot2_fwd_pm(f2x& X1, f2x& X2, f2x C, f2x S, const PlusMinus& u) {
  const f2x p = f2_mul(X1, C), q = f2_mul(X2, S), r = f2_mul(X2, C), t = f2_mul(X1, S);
  X1 = f2_fma(q, u.neg, p);  // x1 c - x2 s
  X2 = f2_fma(r, u.one, t);  // x2 c + x1 s
}

// Exact dequantisation of one INT4 group (4 little-endian words, channel j at bits 4j), pair k
// = channels (2k, 2k+1) as one packed pair. The offset-binary nibble u = q + 8 of an even
// channel (low nibble of its byte) goes to mantissa bits 8..11 of 2^15, giving 2^15 + u; an
// odd channel's (high nibble) to bits 12..15, giving 2^15 + 16u. One fused multiply-add then
// yields q s exactly: (2^15 + u) s - (2^15 + 8) s and (2^15 + 16u) (s/16) - (2^11 + 8) s. Its
// exact result q s is representable, and so are the constants: (2^15 + 8) s = 8 s (2^12 + 1)
// and (2^11 + 8) s = 8 s (2^8 + 1) need at most 11 + 13 significant bits, and s/16 is a
// power-of-two scaling (no underflow for any fp16 s).
struct Int4Group {
  uint32_t ev[4], od[4];  // bytes: offset-binary even nibbles (low), odd nibbles (high)
  f2x S, C;               // (s, s/16), (-(2^15 + 8) s, -(2^11 + 8) s)
};
__device__ __forceinline__ Int4Group int4_group(const uint32_t (&w)[4], float s) {
  Int4Group g;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    g.ev[i] = (w[i] & 0x0F0F0F0Fu) ^ 0x08080808u;
    g.od[i] = (w[i] & 0xF0F0F0F0u) ^ 0x80808080u;
  }
  g.S = f2_pack(s, s * 0.0625f);
  g.C = f2_pack(s * -32776.f, s * -2056.f);
  return g;
}
template <int K>
__device__ __forceinline__ f2x int4_pair(const Int4Group& g) {
  constexpr uint32_t sel = 0x7504u | ((uint32_t)(K & 3) << 4);  // byte 1 <- byte K%4
  const float lo = __uint_as_float(prmt(g.ev[K >> 2], 0x47000000u, sel));
  const float hi = __uint_as_float(prmt(g.od[K >> 2], 0x47000000u, sel));
  return f2_fma(f2_pack(lo, hi), g.S, g.C);
}

// Codes of 16 fp16 values (8 half2 words) for a scale s >= 2^-14 (normal), packed little-endian
// from bit 0 of out[0] (INT4: two words, INT2: one): exact round_half_even(x / s). The candidate
// rint(x * r) (r = an approximate 1/s; the product is exact inside the fused multiply-add that
// adds 1.5 * 2^23) is within 8e-7 of x / s, while x / s is either exactly a half-integer or at
// least 2^-13 from one (fp16 operands), so only exact ties can be mis-rounded; the exact
// residual x - q s, equal to s/2 in magnitude exactly at a tie, confirms all 16 codes or sends
// the half group to the exact scalar path (ties to even).
template <int BITS>
__device__ __forceinline__ void codes_half_group_fast(const uint32_t (&H)[8], float s,
                                                      uint32_t* out) {
  constexpr uint32_t mask = (1u << BITS) - 1u;
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  const f2x R = f2_pack(r, r), M = f2_pack(12582912.f, 12582912.f), NS = f2_pack(-s, -s);
  uint32_t qb[16];
  float emax = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&H[k]));
    const f2x X = f2_pack(f.x, f.y);
    const f2x QM = f2_fma(X, R, M);
    const f2x E = f2_fma(f2_sub(QM, M), NS, X);
    float e0, e1, qm0, qm1;
    f2_unpack(E, e0, e1);
    f2_unpack(QM, qm0, qm1);
    qb[2 * k] = __float_as_uint(qm0);
    qb[2 * k + 1] = __float_as_uint(qm1);
    emax = fmaxf(emax, fmaxf(fabsf(e0), fabsf(e1)));
  }
  if (emax < 0.5f * s) {
    if constexpr (BITS == 4) {
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const uint32_t a = prmt(prmt(qb[8 * v], qb[8 * v + 2], 0x0040u),
                                prmt(qb[8 * v + 4], qb[8 * v + 6], 0x0040u), 0x5410u);
        const uint32_t b = prmt(prmt(qb[8 * v + 1], qb[8 * v + 3], 0x0040u),
                                prmt(qb[8 * v + 5], qb[8 * v + 7], 0x0040u), 0x5410u);
        out[v] = (a & 0x0F0F0F0Fu) | ((b << 4) & 0xF0F0F0F0u);
      }
    } else {
      uint32_t o = 0u;
#pragma unroll
      for (int j = 0; j < 16; ++j) o |= (qb[j] & mask) << (BITS * j);
      out[0] = o;
    }
    return;
  }
  const uint2 ex = codes_half_group_exact<BITS>(make_uint4(H[0], H[1], H[2], H[3]),
                                                make_uint4(H[4], H[5], H[6], H[7]), s);
  out[0] = ex.x;
  if constexpr (BITS == 4) out[1] = ex.y;
}

// Quantise one group of 32 fp16 values (16 half2 words) whose fp32 absmax (before the fp16
// cast) is a32: scale s = fp16(fp16(a32) / qmax) (the fp16 absmax equals the fp16 rounding of
// the fp32 one: rounding is monotone and odd), 2^-24 if it underflows; codes into `o`.
// Returns the scale's fp16 bits.
template <int KB>
__device__ __forceinline__ uint16_t quantize_group16(const uint32_t (&H)[16], float a32,
                                                     uint32_t (&o)[KB]) {
  constexpr int qmax = (1 << (KB - 1)) - 1;
  const float ah = __half2float(__float2half_rn(a32));
  float s = __half2float(__float2half_rn(div_by_qmax<qmax>(ah)));
  if (ah > 0.f && s == 0.f) s = kSubnormalMin;
#pragma unroll
  for (int w = 0; w < KB; ++w) o[w] = 0u;
  if (s >= 6.103515625e-05f) {
    codes_half_group_fast<KB>(*reinterpret_cast<const uint32_t(*)[8]>(&H[0]), s, o);
    codes_half_group_fast<KB>(*reinterpret_cast<const uint32_t(*)[8]>(&H[8]), s, o + KB / 2);
  } else if (s > 0.f) {  // subnormal scale: the clamp can bind; the exact path
    const uint2 lo = codes_half_group_exact<KB>(make_uint4(H[0], H[1], H[2], H[3]),
                                                make_uint4(H[4], H[5], H[6], H[7]), s);
    const uint2 hi = codes_half_group_exact<KB>(make_uint4(H[8], H[9], H[10], H[11]),
                                                make_uint4(H[12], H[13], H[14], H[15]), s);
    if constexpr (KB == 4) {
      o[0] = lo.x; o[1] = lo.y; o[2] = hi.x; o[3] = hi.y;
    } else {
      o[0] = lo.x; o[1] = hi.x;
    }
  }
  return __half_as_ushort(__float2half_rn(s));
}

// One thread's two key groups of a moved middle token: codes k1 (group g1) and k2 (group g2,
// the rotation partners of g1), scales s1, s2. Dequantise (exact), un-RoPE with the old
// position's row `to`, re-RoPE with the new one's `tn` (16 float4 each: pairs 2k, 2k+1 in
// float4 k), every product and sum rounded on its own, cast to fp16 and requantise. Writes the
// new codes and returns the two scales' fp16 bits in sb1, sb2.
// RoPE rows of the table: staged in shared memory (a 32-bit shared address, read with
// ld.shared) or in global memory.
struct SharedRow {
  uint32_t addr;
  __device__ __forceinline__ float4 operator[](int k) const {
    float4 v;
    // not volatile: the rows are written before the CTA barrier that precedes every read
    // (the address depends on values read after it), so the load may be scheduled freely
    asm("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "r"(addr + 16u * (uint32_t)k));
    return v;
  }
};
struct GlobalRow {
  const float4* p;
  __device__ __forceinline__ float4 operator[](int k) const { return __ldg(p + k); }
};

template <int KB, class Row>
__device__ __forceinline__ void requant_moved(const uint32_t (&k1)[KB], const uint32_t (&k2)[KB],
                                              float s1, float s2, const Row to, const Row tn,
                                              const PlusMinus& pm, uint32_t (&o1)[KB],
                                              uint32_t (&o2)[KB], uint16_t& sb1,
                                              uint16_t& sb2) {
  uint32_t H1[16], H2[16];
  float a1 = 0.f, a2 = 0.f;
  if constexpr (KB == 4) {
    const Int4Group G1 = int4_group(k1, s1), G2 = int4_group(k2, s2);
#define FADE_REQ_PAIR(K)                                                                  \
  {                                                                                       \
    f2x X1 = int4_pair<K>(G1), X2 = int4_pair<K>(G2);                                     \
    const float4 co = to[K], cn = tn[K];                                                  \
    rot2_inv_pm(X1, X2, f2_pack(co.x, co.y), f2_pack(co.z, co.w), pm);                    \
    rot2_fwd_pm(X1, X2, f2_pack(cn.x, cn.y), f2_pack(cn.z, cn.w), pm);                    \
    float y10, y11, y20, y21;                                                             \
    f2_unpack(X1, y10, y11);                                                              \
    f2_unpack(X2, y20, y21);                                                              \
    a1 = fmaxf(a1, fmaxf(fabsf(y10), fabsf(y11)));                                       \
    a2 = fmaxf(a2, fmaxf(fabsf(y20), fabsf(y21)));                                        \
    const __half2 r1 = __floats2half2_rn(y10, y11), r2 = __floats2half2_rn(y20, y21);     \
    H1[K] = *reinterpret_cast<const uint32_t*>(&r1);                                      \
    H2[K] = *reinterpret_cast<const uint32_t*>(&r2);                                      \
  }
    FADE_REQ_PAIR(0) FADE_REQ_PAIR(1) FADE_REQ_PAIR(2) FADE_REQ_PAIR(3)
    FADE_REQ_PAIR(4) FADE_REQ_PAIR(5) FADE_REQ_PAIR(6) FADE_REQ_PAIR(7)
    FADE_REQ_PAIR(8) FADE_REQ_PAIR(9) FADE_REQ_PAIR(10) FADE_REQ_PAIR(11)
    FADE_REQ_PAIR(12) FADE_REQ_PAIR(13) FADE_REQ_PAIR(14) FADE_REQ_PAIR(15)
#undef FADE_REQ_PAIR
  } else {
    const f2x S1 = f2_pack(s1, s1), S2 = f2_pack(s2, s2);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      f2x X1 = dequant_pair_bits<KB>(k1, k, S1), X2 = dequant_pair_bits<KB>(k2, k, S2);
      const float4 co = to[k], cn = tn[k];
      rot2_inv_pm(X1, X2, f2_pack(co.x, co.y), f2_pack(co.z, co.w), pm);
      rot2_fwd_pm(X1, X2, f2_pack(cn.x, cn.y), f2_pack(cn.z, cn.w), pm);
      float y10, y11, y20, y21;
      f2_unpack(X1, y10, y11);
      f2_unpack(X2, y20, y21);
      a1 = fmaxf(a1, fmaxf(fabsf(y10), fabsf(y11)));
      a2 = fmaxf(a2, fmaxf(fabsf(y20), fabsf(y21)));
      const __half2 r1 = __floats2half2_rn(y10, y11), r2 = __floats2half2_rn(y20, y21);
      H1[k] = *reinterpret_cast<const uint32_t*>(&r1);
      H2[k] = *reinterpret_cast<const uint32_t*>(&r2);
    }
  }
  sb1 = quantize_group16<KB>(H1, a1, o1);
  sb2 = quantize_group16<KB>(H2, a2, o2);
}

// One head's data of one middle token for one thread, loaded ahead of its use: the K codes
// of the thread's two groups, the token's K scale row, the thread's share of the V codes, its
// share of the V scale row and the score.
template <int D, int KB, int VB>
struct MidToken {
  static constexpr int KW = KB;                        // words of one group's codes
  static constexpr int SW = D / kGroup / 2;            // words of the scale row (1 or 2)
  static constexpr int VW = D * VB / 8 / MidCfg<D>::TPT / 4;  // words of V (4 or 8)
  uint32_t k1[KW], k2[KW];
  uint32_t ks[SW];
  uint32_t v[VW];
  uint32_t vs;     // the thread's 4 bytes of the V scale row
  float sc;
};

template <int W>
__device__ __forceinline__ void ldg_words(const void* p, uint32_t (&w)[W]) {
  static_assert(W == 1 || W == 2 || W % 4 == 0, "1, 2 or a multiple of 4 words");
  if constexpr (W == 1) {
    w[0] = __ldg(reinterpret_cast<const uint32_t*>(p));
  } else if constexpr (W == 2) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = u.x;
    w[1] = u.y;
  } else {
#pragma unroll
    for (int i = 0; i < W / 4; ++i) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(p) + i);
      w[4 * i] = u.x;
      w[4 * i + 1] = u.y;
      w[4 * i + 2] = u.z;
      w[4 * i + 3] = u.w;
    }
  }
}
template <int W>
__device__ __forceinline__ void stg_words(void* p, const uint32_t (&w)[W]) {
  if constexpr (W == 1) {
    *reinterpret_cast<uint32_t*>(p) = w[0];
  } else if constexpr (W == 2) {
    *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  } else {
#pragma unroll
    for (int i = 0; i < W / 4; ++i)
      reinterpret_cast<uint4*>(p)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}

// Compact survivors of the live middle buffer into the other one, re-positioning keys whose
// index drops (the recent rings follow in evict_recent_commit_kernel).
// grid = (B, ceil(max_mid / TOK)), 256 threads (a row's blocks in reverse order); one CTA
// takes one block of TOK middle indices of one batch row and loops over the row's KV heads.
// A middle token is handled by D/64 adjacent threads (MidCfg); thread t_ of a token owns its
// quantisation groups g1 = t_ and g2 = t_ + D/64, whose channels are each other's rotation
// partners. A moved key is dequantised, un-RoPE'd at its old position and re-RoPE'd at its new
// one, rounded to fp16 and re-quantised, all in the owning thread. The RoPE rows the block
// needs (its old positions and the new ones, at most 16 below) are staged once per CTA in
// shared memory and serve every head; each head's codes, scales and score are loaded into
// registers one head ahead.
// SEL: a selection policy (victims from the bitmap of evict_select_kernel) whose block's bitmap
// words are staged in shared memory with their prefix counts; false: the code for every policy,
// with the victims' prefix read from the bitmap per token (the position policy's instantiation).
template <int D, int KB, int VB, bool SEL>
__global__ void __launch_bounds__(256, FADE_COMPACT_MINB) evict_compact_kernel(LayerArgs a) {
  using CC = MidCfg<D>;
  using TD = MidToken<D, KB, VB>;
  constexpr int PRE = SEL ? CC::PRE_SEL : CC::PRE;
  constexpr int TOK = CC::TOK, TPW = CC::TPW;
  constexpr int GB = 32 * KB / 8;              // bytes of one group's codes
  constexpr int VROW = D * VB / 8, SROW = D / kGroup, KROW = D * KB / 8;
  constexpr int VSH = VROW / CC::TPT;          // bytes of V per thread
  extern __shared__ float4 tab[];              // [NROWS][ROWF4 + 1], then hinfo, hpre
  int* hinfo = reinterpret_cast<int*>(tab + CC::TABF4);  // [H][4]: n_mid n_ev n_sink cur
  int* hpre = hinfo + a.H * 4;                           // [H][PRE]
  // [H]: the head's block lies below both the agreement index of the two middle buffers and
  // the first victim: its codes and scales are already in place, only its scores are copied
  int* hlight = hpre + a.H * PRE;
  __shared__ int s_rlo, s_rhi, s_any;
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // blocks in reverse index order, rows fastest: under a selection policy a block's work
  // grows with its index (every key after a unit's victim is re-positioned, the ones before
  // it are copied), so the heaviest blocks of every row are scheduled first
  const int lo = (gridDim.y - 1 - blockIdx.y) * TOK;
  if (threadIdx.x == 0) {
    s_rlo = 0x7fffffff;
    s_rhi = -1;
    s_any = 0;
  }
  __syncthreads();
  // per-head bookkeeping (warp w takes heads w, w+8, ...): counts, the victims before each
  // 32-token word of the block, and the block's range of RoPE rows
  for (int h = warp; h < a.H; h += 8) {
    const int unit = b * a.H + h;
    const int32_t* m = a.meta + unit * kF;
    const int n_mid = m[FADE_META_N_MID];
    const int n_ev = a.positional ? max(0, n_mid - a.budget) : m[FADE_META_N_EV];
    const int n_sink = m[FADE_META_N_SINK];
    if (lane == 0) {
      const int cur = m[FADE_META_CUR];
      hinfo[4 * h + 0] = n_mid;
      hinfo[4 * h + 1] = n_ev;
      hinfo[4 * h + 2] = n_sink;
      hinfo[4 * h + 3] = cur;
    }
    if (n_ev == 0 || lo >= n_mid) continue;
    const int hi = min(lo + TOK, n_mid);
    if (!a.positional) {
      const uint32_t* bm = a.victims + (size_t)unit * a.victim_words;
      // victims before `lo`: chunk prefix plus the words of lo's chunk that precede it
      const int w_lo = lo >> 5, w0 = (lo / kChunk) * (kChunk / 32);
      int c = (w0 + lane < w_lo) ? __popc(bm[w0 + lane]) : 0;
#pragma unroll
      for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      const int nw = (hi - lo + 31) / 32;
      int wc;
      if constexpr (SEL) {
        const uint32_t wv = lane < nw ? bm[w_lo + lane] : 0u;
        wc = __popc(wv);
        if (lane < TOK / 32) hpre[h * PRE + TOK / 32 + 2 + lane] = (int)wv;
      } else {
        wc = lane < nw ? __popc(bm[w_lo + lane]) : 0;
      }
      int incl = wc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int tt = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += tt;
      }
      if (lane <= TOK / 32) hpre[h * PRE + lane] = incl - wc;
      const int before_lo = a.chunk_base[(size_t)unit * a.chunk_slots + lo / kChunk] + c;
      if (lane == 0) hpre[h * PRE + TOK / 32 + 1] = before_lo;
      if constexpr (SEL) {
        const int in_block = __shfl_sync(0xffffffffu, incl, TOK / 32 - 1);
        const bool light = hi <= m[FADE_META_SYNC] && before_lo + in_block == 0;
        if (lane == 0) hlight[h] = light ? 1 : 0;
        if (light) {
          if (lane == 0) s_any = 1;
          continue;
        }
      }
    }
    if (lane == 0) {
      s_any = 1;
      atomicMin(&s_rlo, n_sink + max(0, lo - n_ev));  // lowest new position of the block
      atomicMax(&s_rhi, n_sink + hi);                  // one past the highest old position
    }
  }
  __syncthreads();
  const int rlo = s_rlo, rhi = s_rhi;
  if (!s_any) return;  // no head has work in this block (uniform per CTA)
  const bool staged = a.table != nullptr && rhi >= 0 && rhi - rlo <= CC::NROWS;
  if (staged) {
    const float4* src = reinterpret_cast<const float4*>(a.table) + (size_t)rlo * CC::ROWF4;
    for (int e = threadIdx.x; e < (rhi - rlo) * CC::ROWF4; e += 256) {
      const int r = e / CC::ROWF4, j = e % CC::ROWF4;
      tab[tab_slot<D>(r, j)] = __ldg(src + e);
    }
  }
  __syncthreads();

  const PlusMinus pm{f2_pack(a.one, a.one), f2_pack(a.neg_one, a.neg_one)};
  // lanes: token-minor (TPW consecutive tokens per t_), so a quarter warp reads one float4 of
  // eight consecutive RoPE rows (the padding puts them in eight different bank quads)
  const int it = warp * TPW + lane % TPW, t_ = lane / TPW;
  const int i = lo + it;
  const int g1 = t_, g2 = t_ + D / 64;
  const int4* hinfo4 = reinterpret_cast<const int4*>(hinfo);
  const uint32_t row0 = (uint32_t)(b * a.H) * (uint32_t)a.C;  // slot 0 of the row's first unit
  auto has_work = [&](int hh) {
    const int4 m = hinfo4[hh];
    return m.y != 0 && lo < m.x;
  };
  // a head's data for this thread (zeros past the unit's middle tier)
  auto load = [&](int hh, TD& d) {
    const int4 m = hinfo4[hh];
    if (i < m.x) {
      const uint32_t r = row0 + (uint32_t)hh * (uint32_t)a.C + (uint32_t)i;
      if (SEL && hlight[hh]) {  // the score only
        d.sc = __ldg((m.w ? a.mid_sc[1] : a.mid_sc[0]) + r);
        return;
      }
      const uint8_t* kr = (m.w ? a.mk[1] : a.mk[0]) + (size_t)r * KROW;
      ldg_words(kr + g1 * GB, d.k1);
      ldg_words(kr + g2 * GB, d.k2);
      ldg_words((m.w ? a.mks[1] : a.mks[0]) + (size_t)r * SROW, d.ks);
      ldg_words((m.w ? a.mv[1] : a.mv[0]) + (size_t)r * VROW + t_ * VSH, d.v);
      d.vs = __ldg(reinterpret_cast<const uint32_t*>((m.w ? a.mvs[1] : a.mvs[0]) +
                                                     (size_t)r * SROW) + t_);
      d.sc = __ldg((m.w ? a.mid_sc[1] : a.mid_sc[0]) + r);
    }
  };
  int h = 0;
  while (h < a.H && !has_work(h)) ++h;
  TD cur;
  if (h < a.H) load(h, cur);
  while (h < a.H) {  // uniform per CTA
    int hn = h + 1;
    while (hn < a.H && !has_work(hn)) ++hn;
    TD nxt;
    if (hn < a.H) load(hn, nxt);
    const int4 m = hinfo4[h];
    const int n_mid = m.x, n_ev = m.y, n_sink = m.z;
    const bool cbuf = m.w != 0;
    if (SEL && hlight[h]) {  // uniform per CTA: no victim before the block, codes in place
      if (i < n_mid && t_ == 0)
        (cbuf ? a.mid_sc[0] : a.mid_sc[1])[row0 + (uint32_t)h * (uint32_t)a.C + (uint32_t)i] =
            cur.sc;
      cur = nxt;
      h = hn;
      continue;
    }
    // The TPT lanes of one token lie in one warp and share every flag below, so the warp-wide
    // ballot sees whole tokens; nothing exits before it.
    const bool in_range = i < n_mid;
    bool keep = in_range;
    int nv = 0;
    if (in_range) {
      if (a.positional) {
        keep = i >= n_ev;
        nv = i - n_ev;
      } else {
        uint32_t word;
        if constexpr (SEL) {  // the block's bitmap word from shared memory (lo % 32 == 0)
          word = (uint32_t)hpre[h * PRE + TOK / 32 + 2 + ((i - lo) >> 5)];
        } else {
          const uint32_t* bm = a.victims + (size_t)(b * a.H + h) * a.victim_words;
          word = bm[i >> 5];
        }
        keep = !((word >> (i & 31)) & 1u);
        nv = i - (hpre[h * PRE + TOK / 32 + 1] + hpre[h * PRE + ((i - lo) >> 5)] +
                  __popc(word & ((1u << (i & 31)) - 1u)));
      }
    }
    if (FADE_DEBUG && keep && (nv < 0 || nv >= a.C)) {  // a destination outside the unit
      record_status(a.status, kCheckCompactRow);
      keep = false;
    }
    const bool moved = keep && nv != i && a.table != nullptr;
    const uint32_t dr = row0 + (uint32_t)h * (uint32_t)a.C + (uint32_t)nv;  // destination row
    uint8_t* krow_d = (cbuf ? a.mk[0] : a.mk[1]) + (size_t)dr * KROW;
    uint16_t* ks_d = (cbuf ? a.mks[0] : a.mks[1]) + (size_t)dr * SROW;
    const uint16_t* ksrc = reinterpret_cast<const uint16_t*>(cur.ks);
    if (keep && !moved) {  // survivor at its own index (or no RoPE): K as it is
      stg_words(krow_d + g1 * GB, cur.k1);
      stg_words(krow_d + g2 * GB, cur.k2);
      ks_d[g1] = ksrc[g1];
      ks_d[g2] = ksrc[g2];
    }
    if (__ballot_sync(0xffffffffu, moved) != 0u && moved) {
      uint32_t o1[KB], o2[KB];
      uint16_t sb1, sb2;
      // this thread's 16 float4 (pairs 32 t_ .. 32 t_ + 31) of the old and the new RoPE row
      if (staged)
        requant_moved<KB>(cur.k1, cur.k2, h2f(ksrc[g1]), h2f(ksrc[g2]),
                          SharedRow{smem_u32(tab + tab_slot<D>(n_sink + i - rlo, 16 * t_))},
                          SharedRow{smem_u32(tab + tab_slot<D>(n_sink + nv - rlo, 16 * t_))}, pm,
                          o1, o2, sb1, sb2);
      else
        requant_moved<KB>(
            cur.k1, cur.k2, h2f(ksrc[g1]), h2f(ksrc[g2]),
            GlobalRow{reinterpret_cast<const float4*>(a.table) + (size_t)(n_sink + i) * CC::ROWF4 +
                      16 * t_},
            GlobalRow{reinterpret_cast<const float4*>(a.table) + (size_t)(n_sink + nv) * CC::ROWF4 +
                      16 * t_},
            pm, o1, o2, sb1, sb2);
      stg_words(krow_d + g1 * GB, o1);
      stg_words(krow_d + g2 * GB, o2);
      ks_d[g1] = sb1;
      ks_d[g2] = sb2;
    }
    if (keep) {  // V codes (this thread's share), its V scales and the score move unchanged
      stg_words((cbuf ? a.mv[0] : a.mv[1]) + (size_t)dr * VROW + t_ * VSH, cur.v);
      reinterpret_cast<uint32_t*>((cbuf ? a.mvs[0] : a.mvs[1]) + (size_t)dr * SROW)[t_] = cur.vs;
      if (t_ == 0) (cbuf ? a.mid_sc[0] : a.mid_sc[1])[dr] = cur.sc;
    }
    cur = nxt;
    h = hn;
  }
}

// Recent rings after compaction: every ring token's index drops by its unit's n_ev, so its key
// is re-positioned in place; then the unit's counts are committed (middle count, live buffer).
// grid = (H, B), 256 threads: one CTA per unit. Thread (token t, t_) owns the same rotation
// pairs as in the middle tier; the RoPE rows of the ring's old and new positions are staged.
template <int D>
__global__ void __launch_bounds__(256) evict_recent_commit_kernel(LayerArgs a) {
  using CC = RecentCfg<D>;
  constexpr int TOK = CC::TOK;
  extern __shared__ float4 tab[];
  int* hinfo = reinterpret_cast<int*>(tab + CC::TABF4);  // [H][4]
  __shared__ int s_rlo, s_rhi;
  const int b = blockIdx.y, hb = blockIdx.x;  // one unit per CTA: (row b, KV head hb)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // the unit's recent ring: every token's index drops by the unit's n_ev; keys rewritten in
  // place. Thread (token t, t_) owns the same rotation pairs as in the middle tier; the RoPE
  // rows of the ring's old and new positions are staged first.
  if (threadIdx.x == 0) {
    s_rlo = 0x7fffffff;
    s_rhi = -1;
  }
  __syncthreads();
  for (int h = hb + warp; h < hb + 1; h += 8) {
    const int32_t* m = a.meta + (b * a.H + h) * kF;
    const int n_mid = m[FADE_META_N_MID];
    const int n_ev = a.positional ? max(0, n_mid - a.budget) : m[FADE_META_N_EV];
    const int n_rec = m[FADE_META_N_RECENT];
    if (lane == 0) {
      hinfo[4 * h + 0] = n_mid;
      hinfo[4 * h + 1] = n_ev;
      hinfo[4 * h + 2] = m[FADE_META_N_SINK];
      hinfo[4 * h + 3] = n_rec | (m[FADE_META_HEAD] << 16);
      if (n_ev > 0 && n_rec > 0) {
        const int p0 = m[FADE_META_N_SINK] + n_mid;  // old position of ring token 0
        atomicMin(&s_rlo, p0 - n_ev);
        atomicMax(&s_rhi, p0 + n_rec);
      }
    }
  }
  __syncthreads();
  const int rlo = s_rlo, rhi = s_rhi;
  const bool rotate = rhi >= 0 && a.table != nullptr;  // uniform per CTA
  const bool staged = rotate && rhi - rlo <= CC::NROWS;
  if (staged) {
    const float4* src = reinterpret_cast<const float4*>(a.table) + (size_t)rlo * CC::ROWF4;
    for (int e = threadIdx.x; e < (rhi - rlo) * CC::ROWF4; e += 256) {
      const int r = e / CC::ROWF4, j = e % CC::ROWF4;
      tab[tab_slot<D>(r, j)] = __ldg(src + e);
    }
  }
  __syncthreads();
  const int tt = warp * CC::TPW + lane % CC::TPW, t_ = lane / CC::TPW;
  const int gp = t_ >> 1, hf = t_ & 1;
  for (int h = hb; h < hb + 1 && rotate; ++h) {
    const int n_mid = hinfo[4 * h + 0], n_ev = hinfo[4 * h + 1];
    const int n_rec = hinfo[4 * h + 3] & 0xFFFF, head = hinfo[4 * h + 3] >> 16;
    if (n_ev == 0) continue;
    const int unit = b * a.H + h;
    for (int t = tt; t < n_rec; t += TOK) {
      const int slot = (head + t) % a.W;
      uint16_t* row = a.rec_k + ((size_t)unit * a.W + slot) * D;
      const int pold = hinfo[4 * h + 2] + n_mid + t, pnew = pold - n_ev;
      const float4* to = reinterpret_cast<const float4*>(a.table) + (size_t)pold * (a.half / 2) +
                         8 * t_;
      const float4* tn = reinterpret_cast<const float4*>(a.table) + (size_t)pnew * (a.half / 2) +
                         8 * t_;
#pragma unroll
      for (int q = 0; q < 2; ++q) {  // 8 channels of the first half and their partners
        uint16_t* p1 = row + 32 * gp + 16 * hf + 8 * q;
        uint16_t* p2 = p1 + D / 2;
        f2x X1[4], X2[4];
        load_f16x8(p1, X1);
        load_f16x8(p2, X2);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = 8 * t_ + 4 * q + k;
          float4 co, cn;
          if (staged) {
            co = tab[tab_slot<D>(pold - rlo, j)];
            cn = tab[tab_slot<D>(pnew - rlo, j)];
          } else {
            co = __ldg(to + 4 * q + k);
            cn = __ldg(tn + 4 * q + k);
          }
          rotate2_inv(X1[k], X2[k], f2_pack(co.x, co.y), f2_pack(co.z, co.w));
          rotate2(X1[k], X2[k], f2_pack(cn.x, cn.y), f2_pack(cn.z, cn.w));
        }
        store_f16x8(X1, p1);
        store_f16x8(X2, p2);
      }
    }
  }
  // the first victim of the unit: both middle buffers now hold the same codes and scales
  // below it (the compaction copied them or found them equal), which the next compaction
  // uses to skip them. Position eviction drops the oldest tokens: 0.
  __shared__ int s_first;
  if (threadIdx.x == 0) s_first = 0x7fffffff;
  __syncthreads();  // every thread is done with the counts read above
  if (!a.positional && hinfo[4 * hb + 1] > 0) {
    const uint32_t* bm = a.victims + (size_t)(b * a.H + hb) * a.victim_words;
    for (int w = threadIdx.x; w < (hinfo[4 * hb + 0] + 31) / 32; w += 256) {
      const uint32_t x = bm[w];
      if (x) atomicMin(&s_first, 32 * w + __ffs(x) - 1);
    }
  }
  __syncthreads();
  for (int h = hb + threadIdx.x; h < hb + 1; h += 256) {
    int32_t* m = a.meta + (b * a.H + h) * kF;
    const int n_ev = a.positional ? max(0, m[FADE_META_N_MID] - a.budget) : m[FADE_META_N_EV];
    if (n_ev > 0) {
      m[FADE_META_N_MID] -= n_ev;
      m[FADE_META_CUR] ^= 1;
      m[FADE_META_N_EV] = 0;
      m[FADE_META_SYNC] = (a.positional || s_first == 0x7fffffff) ? 0 : s_first;
    }
  }
}


// ----------------------------------------------------------------- proportional RoPE
// With a rotated width rd < D (proportional RoPE) the rotation pairs (i, i + rd/2) no longer
// line up with the thread-per-group layout of the kernels above, so keys are re-positioned by
// a warp through a row of fp32 values in shared memory (one row per warp). Every product and
// sum is rounded on its own, exactly as in the full-width path; channels rd..D-1 only go
// through the same fp16 cast and requantisation.

// Re-position the fp32 key `row` [D] (shared memory, one warp): pairs i < rd/2.
template <int D>
__device__ __forceinline__ void warp_reposition_row(float* row, const LayerArgs& a, int pold,
                                                    int pnew) {
  const int lane = threadIdx.x & 31, rh = a.rd / 2;
  __syncwarp();
  if (a.table && pold != pnew)
    for (int i = lane; i < rh; i += 32) {
      float y1, y2;
      reposition_pair(a.table, a.half, i, pold, pnew, row[i], row[i + rh], y1, y2);
      row[i] = y1;
      row[i + rh] = y2;
    }
  __syncwarp();
}

template <int D>
__device__ __forceinline__ void warp_key_to_row(const WarpKey<D>& k, float* row) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int gp = 0; gp < D / 64; ++gp) {
    row[32 * gp + lane] = k.lo[gp];
    row[32 * gp + lane + D / 2] = k.hi[gp];
  }
}
template <int D>
__device__ __forceinline__ WarpKey<D> row_to_warp_key(const float* row) {
  const int lane = threadIdx.x & 31;
  WarpKey<D> k;
#pragma unroll
  for (int gp = 0; gp < D / 64; ++gp) {
    k.lo[gp] = row[32 * gp + lane];
    k.hi[gp] = row[32 * gp + lane + D / 2];
  }
  return k;
}

// Re-position a warp-held key (WarpKey layout) with any rotated width: the full-width pairing
// in registers, otherwise through the warp's shared row.
template <int D>
__device__ __forceinline__ void reposition_key_any(const LayerArgs& a, WarpKey<D>& k, int pold,
                                                   int pnew, float* row) {
  if (a.rd == D) {
    reposition_key<D>(a, k, pold, pnew);
    return;
  }
  if (!a.table || pold == pnew) return;
  warp_key_to_row<D>(k, row);
  warp_reposition_row<D>(row, a, pold, pnew);
  k = row_to_warp_key<D>(row);
  __syncwarp();
}

// Compaction with proportional RoPE: one warp per middle index of one unit.
// grid = (ceil(max_mid / 8), H, B), 256 threads.
template <int D, int KB, int VB>
__global__ void __launch_bounds__(256) evict_compact_rows_kernel(LayerArgs a) {
  __shared__ float rows[8][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h = blockIdx.y, unit = b * a.H + h;
  const int i = blockIdx.x * 8 + warp;
  const int32_t* m = a.meta + unit * kF;
  const int n_mid = m[FADE_META_N_MID], n_sink = m[FADE_META_N_SINK];
  const int n_ev = a.positional ? max(0, n_mid - a.budget) : m[FADE_META_N_EV];
  const bool cur = m[FADE_META_CUR] != 0;
  if (n_ev == 0 || i >= n_mid) return;  // warp-uniform
  int nv;
  if (a.positional) {
    if (i < n_ev) return;
    nv = i - n_ev;
  } else {
    const uint32_t* bm = a.victims + (size_t)unit * a.victim_words;
    const int32_t* cb = a.chunk_base + (size_t)unit * a.chunk_slots;
    if ((bm[i >> 5] >> (i & 31)) & 1u) return;
    nv = i - victims_before(bm, cb, i);
  }
  constexpr int KROW = D * KB / 8, VROW = D * VB / 8, SROW = D / kGroup;
  const size_t r = (size_t)unit * a.C + i, dr = (size_t)unit * a.C + nv;
  const uint8_t* ks = (cur ? a.mk[1] : a.mk[0]) + r * KROW;
  const uint16_t* kss = (cur ? a.mks[1] : a.mks[0]) + r * SROW;
  uint8_t* kd = (cur ? a.mk[0] : a.mk[1]) + dr * KROW;
  uint16_t* ksd = (cur ? a.mks[0] : a.mks[1]) + dr * SROW;
  if (nv == i || !a.table) {
    for (int c = lane; c < KROW; c += 32) kd[c] = ks[c];
    if (lane < SROW) ksd[lane] = kss[lane];
  } else {
    WarpKey<D> key = load_mid_key<D, KB>(ks, kss);
    reposition_key_any<D>(a, key, n_sink + i, n_sink + nv, rows[warp]);
    warp_store_quantized<D, KB>(key, kd, ksd);
  }
  const uint8_t* vs = (cur ? a.mv[1] : a.mv[0]) + r * VROW;
  uint8_t* vd = (cur ? a.mv[0] : a.mv[1]) + dr * VROW;
  for (int c = lane; c < VROW; c += 32) vd[c] = vs[c];
  if (lane < SROW) (cur ? a.mvs[0] : a.mvs[1])[dr * SROW + lane] = (cur ? a.mvs[1] : a.mvs[0])[r * SROW + lane];
  if (lane == 0) (cur ? a.mid_sc[0] : a.mid_sc[1])[dr] = (cur ? a.mid_sc[1] : a.mid_sc[0])[r];
}

// Recent rings after the compaction above, with proportional RoPE: every ring key's index
// drops by the unit's n_ev (re-positioned in place, one warp per ring token); then the unit's
// counts are committed. grid = (H, B), 256 threads.
template <int D>
__global__ void __launch_bounds__(256) evict_recent_commit_rows_kernel(LayerArgs a) {
  __shared__ float rows[8][D];
  const int warp = threadIdx.x >> 5;
  const int b = blockIdx.y, h = blockIdx.x, unit = b * a.H + h;
  int32_t* m = a.meta + unit * kF;
  const int n_mid = m[FADE_META_N_MID], n_sink = m[FADE_META_N_SINK];
  const int n_rec = m[FADE_META_N_RECENT], head = m[FADE_META_HEAD];
  const int n_ev = a.positional ? max(0, n_mid - a.budget) : m[FADE_META_N_EV];
  if (n_ev > 0 && a.table) {
    for (int t = warp; t < n_rec; t += 8) {
      uint16_t* row = a.rec_k + ((size_t)unit * a.W + (head + t) % a.W) * D;
      WarpKey<D> key = load_fp16_key<D>(row);
      const int pold = n_sink + n_mid + t;
      reposition_key_any<D>(a, key, pold, pold - n_ev, rows[warp]);
      store_fp16_key<D>(key, row);
    }
  }
  __syncthreads();  // every warp has read the counts
  if (threadIdx.x == 0 && n_ev > 0) {
    m[FADE_META_N_MID] = n_mid - n_ev;
    m[FADE_META_CUR] ^= 1;
    m[FADE_META_N_EV] = 0;
    m[FADE_META_SYNC] = 0;  // (this path's compaction reads no agreement index)
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

// grid = (H, B); rows sharing their decisions (equal prompt lengths): grid = (H, 1), the
// row-summed prefill mass decides and every row gets the same victims.
__global__ void __launch_bounds__(kSelThreads) prefill_select_kernel(LayerArgs a, PrefillArgs p,
                                                                     RowLens lens) {
  const int unit = blockIdx.y * a.H + blockIdx.x;
  const PrefillSplit s = prefill_split(a, lens.v[blockIdx.y]);
  if (s.k == 0) return;
  const float* mass = (a.policy == FADE_EVICT_H2O) ? p.mass + (size_t)unit * p.maxP + s.n_s
                                                   : nullptr;  // EMA: all 0; position: index
  uint32_t* bm = a.victims + (size_t)unit * a.victim_words;
  int32_t* cb = a.chunk_base + (size_t)unit * a.chunk_slots;
  if (a.shared) {
    block_select(KeysRows{mass, (size_t)a.H * p.maxP, a.B}, s.n_m0, s.k, bm, cb);
    __syncthreads();
    for (int r = 1; r < a.B; ++r) copy_selection(a, unit, r * a.H + blockIdx.x, s.n_m0);
  } else {
    block_select(KeysOne{mass}, s.n_m0, s.k, bm, cb);
  }
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
  __shared__ float rows[8][D];  // proportional RoPE: each warp's key during re-positioning
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
    reposition_key_any<D>(a, key, i, nv, rows[warp]);
    const float score = (a.policy == FADE_EVICT_H2O && p.mass) ? p.mass[(size_t)unit * p.maxP + i]
                                                               : 0.f;
    if (tier == 1) {
      const size_t row = (size_t)unit * a.C + (nv - s.n_s);
      warp_store_quantized<D, KB>(key, a.mk[0] + row * KROW, a.mks[0] + row * SROW);
      if (a.pq)
        warp_pq_encode_row<D>(p.v + src, a.pq_cb, a.mv[0] + row * VROW, a.mvs[0] + row * SROW);
      else
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
  m[FADE_META_SYNC] = 0;
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
    demote_kernel<D, KB, VB><<<dim3(a.H, B), 64, 0, st>>>(a);
    return launch_status("fade_cache_demote");
  }
};

template <int D, int KB, int VB>
struct CompactLaunch {
  static fade_status_t run(const LayerArgs& a, int B, int max_mid, cudaStream_t st) {
    if (a.rd < D) {  // proportional RoPE: one warp per middle index
      evict_compact_rows_kernel<D, KB, VB><<<dim3(ceil_div(max_mid, 8), a.H, B), 256, 0, st>>>(a);
      return launch_status("fade_evict_rerope compact (proportional RoPE)");
    }
    // chunks of compact_tok<D>() middle indices per batch row
    const int chunks = ceil_div(max_mid, compact_tok<D>());
    const size_t smem = compact_smem<D>(a.H);
    auto kern = a.positional ? evict_compact_kernel<D, KB, VB, false>
                             : evict_compact_kernel<D, KB, VB, true>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
      return launch_status("fade_evict_rerope compact shared-memory opt-in");
    kern<<<dim3(B, chunks), 256, smem, st>>>(a);
    return launch_status("fade_evict_rerope compact");
  }
};

template <int D>
fade_status_t launch_recent_commit(const LayerArgs& a, int B, cudaStream_t st) {
  if (a.rd < D) {
    evict_recent_commit_rows_kernel<D><<<dim3(a.H, B), 256, 0, st>>>(a);
    return launch_status("fade_evict_rerope recent + commit (proportional RoPE)");
  }
  using CC = RecentCfg<D>;
  const size_t smem = (size_t)CC::TABF4 * 16 + (size_t)a.H * 4 * 4;
  auto kern = evict_recent_commit_kernel<D>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return launch_status("fade_evict_rerope recent shared-memory opt-in");
  kern<<<dim3(a.H, B), 256, smem, st>>>(a);
  return launch_status("fade_evict_rerope recent + commit");
}

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
  FADE_RANGE("fade_cache_reset");
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
  FADE_RANGE("fade_cache_prefill");
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
  if (c->shared_rows)
    for (int b = 1; b < c->batch; ++b)
      if (lens.v[b] != lens.v[0])
        return set_error(FADE_ERR_INVALID_ARGUMENT,
                         "rows sharing their tier decisions need equal prompt lengths "
                         "(row %d: %d, row 0: %d)", b, lens.v[b], lens.v[0]);
  const LayerArgs a = make_args(c, L, table);
  const PrefillArgs p{k_rot, v, mass, max_prompt};
  cudaStream_t s = as_stream(stream);
  prefill_select_kernel<<<dim3(c->num_kv_heads, c->shared_rows ? 1 : c->batch), kSelThreads, 0,
                          s>>>(a, p, lens);
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
  FADE_RANGE("fade_cache_demote");
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
  FADE_RANGE("fade_cache_append");
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

template <int D, int KB, int VB>
struct RopeAppendLaunch {
  static fade_status_t run(const LayerArgs& a, bool demote, const float* t, int max_pos, int rh,
                           const uint16_t* q_raw, const uint16_t* k_raw, const uint16_t* v,
                           const int32_t* pos, uint16_t* q_rot, int Hq, int B, cudaStream_t s) {
    // a programmatic dependent of the kernel before it on the stream (see the kernel's end)
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(a.H, B);
    lc.blockDim = dim3(FADE_ROPE_APPEND_THREADS);
    lc.dynamicSmemBytes = 0;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    const cudaError_t e =
        demote ? cudaLaunchKernelEx(&lc, rope_append_kernel<D, KB, VB, true>, a, t, max_pos, rh,
                                    q_raw, k_raw, v, pos, q_rot, Hq)
               : cudaLaunchKernelEx(&lc, rope_append_kernel<D, 4, 2, false>, a, t, max_pos, rh,
                                    q_raw, k_raw, v, pos, q_rot, Hq);
    if (e != cudaSuccess)
      return set_error(FADE_ERR_CUDA, "fade_rope_append: %s", cudaGetErrorString(e));
    return launch_status("fade_rope_append");
  }
};

extern "C" fade_status_t fade_rope_append(const fade_config_t* c, fade_layer_t* L,
                                          const float* table, int32_t max_pos,
                                          const uint16_t* q_raw, const uint16_t* k_raw,
                                          const uint16_t* v, const int32_t* pos,
                                          uint16_t* q_rot, int32_t demote, void* stream) {
  clear_error();
  FADE_RANGE("fade_rope_append");
  fade_status_t st = validate_config(c);
  if (!st) st = validate_layer(c, L);
  if (st) return st;
  if (!q_raw || !k_raw || !v || !pos || !q_rot)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL q_raw, k_raw, v, pos or q_rot");
  const bool rope = c->rope.kind != FADE_ROPE_NONE;
  if (rope && (!table || max_pos < 1))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "NULL RoPE table");
  for (int b = 0; b < c->batch; ++b) {
    const bool full = L->h_n_recent[b] == c->recent_window;
    if (demote && full && L->h_n_mid[b] + 1 > c->mid_capacity)
      return set_error(FADE_ERR_CAPACITY, "row %d: middle tier full (%d slots)", b,
                       c->mid_capacity);
    if (!demote && L->h_n_sink[b] >= c->n_sink && full)
      return set_error(FADE_ERR_CAPACITY, "row %d: recent window full (demote first)", b);
  }
  const LayerArgs a = make_args(c, L, nullptr);
  if ((st = dispatch_dkv<RopeAppendLaunch>(c, a, demote != 0, rope ? table : nullptr, max_pos,
                                           rotary_width(c) / 2, q_raw, k_raw, v, pos, q_rot,
                                           c->num_q_heads, c->batch, as_stream(stream))))
    return st;
  for (int b = 0; b < c->batch; ++b) {
    if (demote && L->h_n_recent[b] == c->recent_window) {
      L->h_n_mid[b] += 1;
      L->h_n_recent[b] -= 1;
    }
    if (L->h_n_sink[b] < c->n_sink)
      L->h_n_sink[b] += 1;
    else
      L->h_n_recent[b] += 1;
  }
  return FADE_OK;
}

namespace {
// One step's count changes of one layer's mirror: pass 0 checks every row, pass 1 stores.
fade_status_t advance_host_pass(const fade_config_t* c, fade_layer_t* L, int pass) {
  const bool evicts = c->policy != FADE_EVICT_NONE && c->int4_budget >= 0;
  for (int b = 0; b < c->batch; ++b) {
    int s = L->h_n_sink[b], m = L->h_n_mid[b], r = L->h_n_recent[b];
    if (r == c->recent_window) {  // demote
      if (m + 1 > c->mid_capacity)
        return set_error(FADE_ERR_CAPACITY, "row %d: middle tier full (%d slots)", b,
                         c->mid_capacity);
      m += 1;
      r -= 1;
    }
    if (evicts && m > c->int4_budget) m = c->int4_budget;  // evict
    if (s >= c->n_sink && r >= c->recent_window)             // append
      return set_error(FADE_ERR_CAPACITY, "row %d: recent window full (demote first)", b);
    if (s < c->n_sink)
      s += 1;
    else
      r += 1;
    if (pass == 1) {
      L->h_n_sink[b] = s;
      L->h_n_mid[b] = m;
      L->h_n_recent[b] = r;
    }
  }
  return FADE_OK;
}
}  // namespace

extern "C" fade_status_t fade_cache_advance_host(const fade_config_t* c, fade_layer_t* L) {
  clear_error();
  fade_status_t st = validate_config(c);
  if (st) return st;
  if (!L || !L->h_n_sink || !L->h_n_mid || !L->h_n_recent)
    return set_error(FADE_ERR_INVALID_ARGUMENT, "host mirror arrays are NULL");
  // every row's counts after the step, checked before any of them is stored
  if ((st = advance_host_pass(c, L, 0))) return st;
  return advance_host_pass(c, L, 1);
}

extern "C" fade_status_t fade_cache_advance_host_layers(const fade_config_t* c,
                                                        fade_layer_t* const* layers,
                                                        int32_t n_layers) {
  clear_error();
  fade_status_t st = validate_config(c);
  if (st) return st;
  if (n_layers < 0 || (n_layers > 0 && !layers))
    return set_error(FADE_ERR_INVALID_ARGUMENT, "bad layer array");
  for (int i = 0; i < n_layers; ++i) {
    const fade_layer_t* L = layers[i];
    if (!L || !L->h_n_sink || !L->h_n_mid || !L->h_n_recent)
      return set_error(FADE_ERR_INVALID_ARGUMENT, "layer %d: host mirror arrays are NULL", i);
  }
  // every layer's rows checked before any count is stored
  for (int pass = 0; pass < 2; ++pass)
    for (int i = 0; i < n_layers; ++i)
      if ((st = advance_host_pass(c, layers[i], pass))) return st;
  return FADE_OK;
}

extern "C" fade_status_t fade_evict_rerope(const fade_config_t* c, fade_layer_t* L,
                                           const float* table, int32_t max_pos, void* stream) {
  clear_error();
  FADE_RANGE("fade_evict_rerope");
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
  if (c->shared_rows)
    for (int b = 1; b < c->batch; ++b)
      if (L->h_n_sink[b] != L->h_n_sink[0] || L->h_n_mid[b] != L->h_n_mid[0] ||
          L->h_n_recent[b] != L->h_n_recent[0])
        return set_error(FADE_ERR_INVALID_ARGUMENT,
                         "rows sharing their tier decisions need equal tier counts (row %d)", b);
  if ((long long)L->victim_words < (c->mid_capacity + 31) / 32 + 1 ||
      (long long)L->chunk_slots < (c->mid_capacity + kChunk - 1) / kChunk + 1)
    return set_error(FADE_ERR_CAPACITY, "scratch buffers are smaller than the middle tier");
  if ((st = check_table(c, table, max_pos, c->n_sink + c->mid_capacity + c->recent_window)))
    return st;
  const LayerArgs a = make_args(c, L, table);
  cudaStream_t s = as_stream(stream);
  if (!a.positional) {  // the position policy needs no selection pass
    evict_select_kernel<<<dim3(c->num_kv_heads, c->shared_rows ? 1 : c->batch), kSelThreads, 0,
                          s>>>(a);
    if ((st = launch_status("fade_evict_rerope select"))) return st;
  }
  if ((st = dispatch_dkv<CompactLaunch>(c, a, c->batch, max_mid, s))) return st;
  st = c->head_dim == 128 ? launch_recent_commit<128>(a, c->batch, s)
                          : launch_recent_commit<64>(a, c->batch, s);
  if (st) return st;
  for (int b = 0; b < c->batch; ++b)
    if (L->h_n_mid[b] > c->int4_budget) L->h_n_mid[b] = c->int4_budget;
  return FADE_OK;
}
