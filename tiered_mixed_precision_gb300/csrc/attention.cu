// Decode attention over the tiered cache (split-KV), the split combine, and H2O / EMA score
// accumulation.
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
constexpr int kThreads = 128;  // one token per thread in the score phase
constexpr int kTile = 128;     // tokens per shared-memory tile
constexpr int kPad = 16;       // bytes of padding per staged row (bank spread)

struct AttnArgs {
  const uint16_t* q;                    // [B][Hq][D]
  const uint16_t *sink_k, *sink_v, *rec_k, *rec_v;
  const uint8_t *mk[2], *mv[2];
  const uint16_t *mks[2], *mvs[2];
  const int32_t* meta;
  float* logits;                        // nullable, [B][Hq][NS]
  float* part_ml;                       // [B][Hq][nsplit][2]
  float* part_acc;                      // [B][Hq][nsplit][D]
  const int32_t* seg_count;             // [B][H]: partials of each unit (stream-K combine)
  int Hq, H, S, W, C, NS, chunk, nsplit;
  float scale;                          // 1/sqrt(D)
  const uint16_t* pq_cb;                // PQ-coded V: the layer's codebook [D/4][256][4]
};

template <int D, int KB, int VB, int G, bool PQ>
struct Smem {
  static constexpr int KROW = D * KB / 8, VROW = D * VB / 8, SROW = D / kGroup;
  static constexpr int KROWP = KROW + kPad, VROWP = VROW + kPad;
  static constexpr int FROWP = D * 2 + kPad;  // fp16 row, padded
  static constexpr int MID_BYTES = kTile * (KROWP + VROWP + 2 * SROW * 2);
  static constexpr int CB_BYTES = PQ ? kPqCentroids * D * 2 : 0;  // PQ codebook (middle splits)
  static constexpr int F16_BYTES = kTile * 2 * FROWP;
  static constexpr int MIDCB_BYTES = MID_BYTES + CB_BYTES;
  static constexpr int TILE_BYTES = MIDCB_BYTES > F16_BYTES ? MIDCB_BYTES : F16_BYTES;
  static constexpr int NSUB = kThreads / (D / 4);  // token subsets in the value phase
  static constexpr int Q_OFF = 0;                              // float [D][G]
  static constexpr int P_OFF = Q_OFF + D * G * 4;               // float [G][kTile]
  static constexpr int R_OFF = P_OFF + G * kTile * 4;           // float [4][G] + [G]*3
  static constexpr int T_OFF = R_OFF + (4 * G + 4 * G) * 4;     // tile buffers
  static constexpr int CB_OFF = T_OFF + MID_BYTES;              // codebook after the mid tile
  static constexpr int A_OFF = T_OFF;                           // acc reduction (reuses tile)
  static constexpr int TOTAL = T_OFF + (TILE_BYTES > NSUB * G * D * 4 ? TILE_BYTES : NSUB * G * D * 4);
};

// Copy `n` rows of `bytes` (a multiple of 16) from global rows given by `src_row(t)` into
// padded shared rows.
template <typename RowFn>
__device__ __forceinline__ void stage_rows(uint8_t* dst, int dst_stride, int bytes, int n,
                                           RowFn src_row) {
  const int per = bytes / 16;
  for (int i = threadIdx.x; i < n * per; i += kThreads) {
    const int t = i / per, c = i % per;
    *reinterpret_cast<uint4*>(dst + t * dst_stride + c * 16) =
        *reinterpret_cast<const uint4*>(src_row(t) + c * 16);
  }
}

template <int D, int KB, int VB, int G, bool PQ>
__global__ void __launch_bounds__(kThreads) attn_split_kernel(AttnArgs a) {
  using L = Smem<D, KB, VB, G, PQ>;
  extern __shared__ __align__(16) uint8_t smem[];
  float* qs = reinterpret_cast<float*>(smem + L::Q_OFF);    // [D][G]
  float* ps = reinterpret_cast<float*>(smem + L::P_OFF);    // [G][kTile]
  float* red = reinterpret_cast<float*>(smem + L::R_OFF);   // [4][G] then [4][G]
  uint8_t* tile = smem + L::T_OFF;

  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int unit = b * a.H + hk;
  const int32_t* m = a.meta + unit * kF;
  const int n_sink = m[FADE_META_N_SINK], n_mid = m[FADE_META_N_MID];
  const int n_rec = m[FADE_META_N_RECENT], head = m[FADE_META_HEAD], cur = m[FADE_META_CUR];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hq0 = hk * G;

  // token range of this split: split 0 = FP16 tiers, split s >= 1 = middle chunk s-1
  int n_tok;
  int lo = 0;
  if (split == 0) {
    n_tok = n_sink + n_rec;
  } else {
    lo = (split - 1) * a.chunk;
    n_tok = max(0, min(n_mid, lo + a.chunk) - lo);
  }
  const size_t pbase = ((size_t)(b * a.Hq + hq0)) * a.nsplit + split;  // (b, hq0, split)
  if (n_tok == 0) {
    for (int i = tid; i < G * D; i += kThreads) {
      const int h = i / D, c = i % D;
      a.part_acc[(pbase + (size_t)h * a.nsplit) * D + c] = 0.f;
    }
    if (tid < G) {
      a.part_ml[(pbase + (size_t)tid * a.nsplit) * 2 + 0] = -INFINITY;
      a.part_ml[(pbase + (size_t)tid * a.nsplit) * 2 + 1] = 0.f;
    }
    return;
  }

  for (int i = tid; i < G * D; i += kThreads) {
    const int h = i / D, c = i % D;
    qs[c * G + h] = h2f(a.q[((size_t)(b * a.Hq + hq0 + h)) * D + c]);
  }
  // PQ-coded V: the codebook sits in shared memory for the whole middle split (it stays
  // clear of the tile, which the loop below refills)
  const uint2* cbs = reinterpret_cast<const uint2*>(smem + L::CB_OFF);
  if constexpr (PQ) {
    if (split != 0)
      for (int i = tid; i < L::CB_BYTES / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + L::CB_OFF)[i] = reinterpret_cast<const uint4*>(a.pq_cb)[i];
  }

  constexpr int QUADS = D / 4, NSUB = L::NSUB;
  const int cq = tid % QUADS, ts = tid / QUADS;
  float acc[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[h][j] = 0.f;
  float m_run[G], l_run[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
  }

  const size_t urow_mid = (size_t)unit * a.C;
  for (int t0 = 0; t0 < n_tok; t0 += kTile) {
    const int nt = min(kTile, n_tok - t0);
    __syncthreads();  // previous tile fully consumed
    uint8_t *kt, *vt;
    uint16_t *kst = nullptr, *vst = nullptr;
    if (split == 0) {
      kt = tile;
      vt = tile + kTile * L::FROWP;
      auto krow = [&](int t) {
        const int u = t0 + t;
        const size_t r = u < n_sink ? ((size_t)unit * a.S + u) * D
                                    : ((size_t)unit * a.W + (head + u - n_sink) % a.W) * D;
        return reinterpret_cast<const uint8_t*>((u < n_sink ? a.sink_k : a.rec_k) + r);
      };
      auto vrow = [&](int t) {
        const int u = t0 + t;
        const size_t r = u < n_sink ? ((size_t)unit * a.S + u) * D
                                    : ((size_t)unit * a.W + (head + u - n_sink) % a.W) * D;
        return reinterpret_cast<const uint8_t*>((u < n_sink ? a.sink_v : a.rec_v) + r);
      };
      stage_rows(kt, L::FROWP, D * 2, nt, krow);
      stage_rows(vt, L::FROWP, D * 2, nt, vrow);
    } else {
      kt = tile;
      vt = tile + kTile * L::KROWP;
      kst = reinterpret_cast<uint16_t*>(vt + kTile * L::VROWP);
      vst = kst + kTile * L::SROW;
      const size_t r0 = urow_mid + lo + t0;
      const uint8_t* kg = (cur ? a.mk[1] : a.mk[0]) + r0 * L::KROW;
      const uint8_t* vg = (cur ? a.mv[1] : a.mv[0]) + r0 * L::VROW;
      stage_rows(kt, L::KROWP, L::KROW, nt, [&](int t) { return kg + (size_t)t * L::KROW; });
      stage_rows(vt, L::VROWP, L::VROW, nt, [&](int t) { return vg + (size_t)t * L::VROW; });
      const uint32_t* ksg =
          reinterpret_cast<const uint32_t*>((cur ? a.mks[1] : a.mks[0]) + r0 * L::SROW);
      const uint32_t* vsg =
          reinterpret_cast<const uint32_t*>((cur ? a.mvs[1] : a.mvs[0]) + r0 * L::SROW);
      const int words = nt * L::SROW / 2;
      for (int i = tid; i < words; i += kThreads) {
        reinterpret_cast<uint32_t*>(kst)[i] = ksg[i];
        if constexpr (!PQ) reinterpret_cast<uint32_t*>(vst)[i] = vsg[i];
      }
    }
    __syncthreads();

    // ---- scores: thread tid owns token tid of the tile
    float s[G];
#pragma unroll
    for (int h = 0; h < G; ++h) s[h] = -INFINITY;
    if (tid < nt) {
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = 0.f;
      if (split == 0) {
        const uint16_t* kr = reinterpret_cast<const uint16_t*>(kt + tid * L::FROWP);
        for (int c = 0; c < D; ++c) {
          const float kv = h2f(kr[c]);
#pragma unroll
          for (int h = 0; h < G; ++h) s[h] = fmaf(qs[c * G + h], kv, s[h]);
        }
      } else {
        const uint8_t* kr = kt + tid * L::KROWP;
        const uint16_t* sr = kst + tid * L::SROW;
#pragma unroll 1
        for (int g = 0; g < D / kGroup; ++g) {
          float part[G];
#pragma unroll
          for (int h = 0; h < G; ++h) part[h] = 0.f;
          const uint8_t* gr = kr + g * (kGroup * KB / 8);
#pragma unroll
          for (int w = 0; w < kGroup * KB / 32; ++w) {
            const uint32_t word = reinterpret_cast<const uint32_t*>(gr)[w];
#pragma unroll
            for (int e = 0; e < 32 / KB; ++e) {
              const uint32_t u = (word >> (KB * e)) & ((1u << KB) - 1u);
              const float code = (float)(int(u) - (int(u >> (KB - 1)) << KB));
              const int c = g * kGroup + w * (32 / KB) + e;
#pragma unroll
              for (int h = 0; h < G; ++h) part[h] = fmaf(qs[c * G + h], code, part[h]);
            }
          }
          const float sc = h2f(sr[g]);
#pragma unroll
          for (int h = 0; h < G; ++h) s[h] = fmaf(part[h], sc, s[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] *= a.scale;
      if (a.logits) {
        const int u = t0 + tid;
        int slot;
        if (split == 0)
          slot = u < n_sink ? u : a.S + a.C + (head + u - n_sink) % a.W;
        else
          slot = a.S + lo + u;
#pragma unroll
        for (int h = 0; h < G; ++h)
          a.logits[((size_t)(b * a.Hq + hq0 + h)) * a.NS + slot] = s[h];
      }
    }
    // ---- tile max per head
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float v = warp_max(s[h]);
      if (lane == 0) red[warp * G + h] = v;
    }
    __syncthreads();
    float alpha[G], mnew[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float tm = fmaxf(fmaxf(red[h], red[G + h]), fmaxf(red[2 * G + h], red[3 * G + h]));
      mnew[h] = fmaxf(m_run[h], tm);
      alpha[h] = __expf(m_run[h] - mnew[h]);  // m_run = -inf -> 0
    }
    float psum[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float p = (tid < nt) ? __expf(s[h] - mnew[h]) : 0.f;
      ps[h * kTile + tid] = p;
      psum[h] = warp_sum(p);
    }
    if (lane == 0)
#pragma unroll
      for (int h = 0; h < G; ++h) red[4 * G + warp * G + h] = psum[h];
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float ts_ = red[4 * G + h] + red[5 * G + h] + red[6 * G + h] + red[7 * G + h];
      l_run[h] = l_run[h] * alpha[h] + ts_;
      m_run[h] = mnew[h];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[h][j] *= alpha[h];
    }

    // ---- values: thread owns channels 4cq..4cq+3 for tokens ts, ts+NSUB, ...
    for (int t = ts; t < nt; t += NSUB) {
      float v4[4];
      if (split == 0) {
        const uint2 raw = *reinterpret_cast<const uint2*>(vt + t * L::FROWP + cq * 8);
        const __half2 h01 = *reinterpret_cast<const __half2*>(&raw.x);
        const __half2 h23 = *reinterpret_cast<const __half2*>(&raw.y);
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        v4[0] = f01.x;
        v4[1] = f01.y;
        v4[2] = f23.x;
        v4[3] = f23.y;
      } else if constexpr (PQ) {
        // channels 4cq..4cq+3 are sub-space cq: one code byte, one 8-byte centroid
        const uint32_t code = vt[t * L::VROWP + cq];
        const uint2 raw = cbs[cq * kPqCentroids + code];
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        v4[0] = f01.x;
        v4[1] = f01.y;
        v4[2] = f23.x;
        v4[3] = f23.y;
      } else {
        const float sc = h2f(vst[t * L::SROW + (4 * cq) / kGroup]);
        const uint8_t* vr = vt + t * L::VROWP;
        uint32_t bits;
        if (VB == 2)
          bits = vr[cq];
        else
          bits = *reinterpret_cast<const uint16_t*>(vr + 2 * cq);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t u = (bits >> (VB * j)) & ((1u << VB) - 1u);
          v4[j] = (float)(int(u) - (int(u >> (VB - 1)) << VB)) * sc;
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float p = ps[h * kTile + t];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[h][j] = fmaf(p, v4[j], acc[h][j]);
      }
    }
  }

  // ---- reduce value accumulators over token subsets, write the split's partial
  __syncthreads();
  float* ar = reinterpret_cast<float*>(smem + L::A_OFF);  // [NSUB][G][D]
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < 4; ++j) ar[(ts * G + h) * D + 4 * cq + j] = acc[h][j];
  __syncthreads();
  for (int i = tid; i < G * D; i += kThreads) {
    const int h = i / D, c = i % D;
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < NSUB; ++k) v += ar[(k * G + h) * D + c];
    a.part_acc[(pbase + (size_t)h * a.nsplit) * D + c] = v;
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
    if (tid == h) {
      a.part_ml[(pbase + (size_t)h * a.nsplit) * 2 + 0] = m_run[h];
      a.part_ml[(pbase + (size_t)h * a.nsplit) * 2 + 1] = l_run[h];
    }
}

// One CTA of D threads per (row, query head): merge the split partials of the CUDA-core
// kernel (split 0 + one per chunk of the middle tier).
template <int D>
__global__ void __launch_bounds__(D) attn_combine_kernel(AttnArgs a, uint16_t* __restrict__ out,
                                                         float* __restrict__ ml) {
  const int bh = blockIdx.x;
  const int b = bh / a.Hq, hq = bh % a.Hq;
  const int G = a.Hq / a.H;
  const int unit = b * a.H + hq / G;
  const int n_mid = a.meta[unit * kF + FADE_META_N_MID];
  const int ns = min(a.nsplit, 1 + (n_mid + a.chunk - 1) / a.chunk);
  const float* pm = a.part_ml + (size_t)bh * a.nsplit * 2;
  const float* pa = a.part_acc + (size_t)bh * a.nsplit * D;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, pm[2 * s]);
  float Lsum = 0.f, o = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float w = (pm[2 * s] == -INFINITY) ? 0.f : __expf(pm[2 * s] - M);
    Lsum = fmaf(pm[2 * s + 1], w, Lsum);
    o = fmaf(pa[(size_t)s * D + threadIdx.x], w, o);
  }
  out[(size_t)bh * D + threadIdx.x] = f2h(o / Lsum);
  if (threadIdx.x == 0) {
    ml[2 * bh] = M;
    ml[2 * bh + 1] = Lsum;
  }
}

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

template <int D, int KB, int VB, int G, bool PQ>
fade_status_t launch_split(const AttnArgs& a, int B, cudaStream_t st, int nx) {
  using L = Smem<D, KB, VB, G, PQ>;
  // opt in to more than 48 KB of dynamic shared memory (cheap; done on every launch so it
  // holds for whichever device is current)
  if (cudaFuncSetAttribute(attn_split_kernel<D, KB, VB, G, PQ>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL) != cudaSuccess)
    return launch_status("fade_decode_attention shared-memory opt-in");
  attn_split_kernel<D, KB, VB, G, PQ><<<dim3(nx, a.H, B), kThreads, L::TOTAL, st>>>(a);
  return launch_status("fade_decode_attention split");
}

template <int D, int KB, int VB, bool PQ = false>
fade_status_t launch_split_g(const AttnArgs& a, int G, int B, cudaStream_t st, int nx) {
  switch (G) {
    case 1: return launch_split<D, KB, VB, 1, PQ>(a, B, st, nx);
    case 2: return launch_split<D, KB, VB, 2, PQ>(a, B, st, nx);
    case 4: return launch_split<D, KB, VB, 4, PQ>(a, B, st, nx);
    case 8: return launch_split<D, KB, VB, 8, PQ>(a, B, st, nx);
  }
  return set_error(FADE_ERR_UNSUPPORTED, "query heads per KV head %d", G);
}

// Launches splits [0, nx) of the CUDA-core kernel.
fade_status_t launch_split_any(const fade_config_t* c, const AttnArgs& a, cudaStream_t st, int nx) {
  const int G = c->num_q_heads / c->num_kv_heads, B = c->batch;
  const int d = c->head_dim, kb = c->middle_k_bits, vb = c->middle_v_bits;
  if (c->v_codec == FADE_V_PQ) {  // PQ codes occupy the INT2 rows (validated)
    if (d == 64) return kb == 4 ? launch_split_g<64, 4, 2, true>(a, G, B, st, nx)
                                : launch_split_g<64, 2, 2, true>(a, G, B, st, nx);
    return kb == 4 ? launch_split_g<128, 4, 2, true>(a, G, B, st, nx)
                   : launch_split_g<128, 2, 2, true>(a, G, B, st, nx);
  }
#define FADE_CASE(D_, KB_, VB_) \
  if (d == D_ && kb == KB_ && vb == VB_) return launch_split_g<D_, KB_, VB_>(a, G, B, st, nx);
  FADE_CASE(64, 4, 2) FADE_CASE(64, 4, 4) FADE_CASE(64, 2, 2) FADE_CASE(64, 2, 4)
  FADE_CASE(128, 4, 2) FADE_CASE(128, 4, 4) FADE_CASE(128, 2, 2) FADE_CASE(128, 2, 4)
#undef FADE_CASE
  return set_error(FADE_ERR_UNSUPPORTED, "unsupported (head_dim, k_bits, v_bits)");
}

// Middle tokens per split: enough CTAs to fill the GPU several times over, splits of equal
// size, each a whole number of tiles.
int choose_chunk(int max_mid, int units, int tile, long long target_ctas) {
  if (max_mid <= 0) return tile;
  long long want = ((long long)max_mid * units + target_ctas - 1) / target_ctas;
  if (want < tile) want = tile;
  const long long n = (max_mid + want - 1) / want;
  long long ch = (max_mid + n - 1) / n;
  ch = ((ch + tile - 1) / tile) * tile;
  return (int)ch;
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
  AttnArgs a;
  a.q = q_rot;
  a.sink_k = L->sink_k;
  a.sink_v = L->sink_v;
  a.rec_k = L->recent_k;
  a.rec_v = L->recent_v;
  for (int i = 0; i < 2; ++i) {
    a.mk[i] = L->mid_k_codes[i];
    a.mv[i] = L->mid_v_codes[i];
    a.mks[i] = L->mid_k_scales[i];
    a.mvs[i] = L->mid_v_scales[i];
  }
  a.meta = L->meta;
  a.logits = logits_ws;
  a.Hq = c->num_q_heads;
  a.H = c->num_kv_heads;
  a.S = c->n_sink;
  a.W = c->recent_window;
  a.C = mid_stride(c);
  a.NS = a.S + a.C + a.W;
  const bool mma = mid_mma_supported(c);
  StreamK sk{};  // the tensor-core kernel's stream-K schedule (unused by the CUDA-core kernel)
  if (mma) {
    build_stream_k(c, L, mid_mma_ctas(c), &sk);
    a.chunk = kTileTokens;
    a.nsplit = 1 + sk.smax;
  } else {
    sk.P = 0;
    // splits sized by the middle capacity, not the current count: the launch is then the
    // same at every step while the cache grows (a captured step can be replayed), and splits
    // past a unit's tokens write empty partials. PQ: fewer, longer middle splits, so that
    // staging the codebook (256 x d fp16 from L2) stays small beside the split's own bytes
    a.chunk = choose_chunk(c->mid_capacity, units,
                           c->v_codec == FADE_V_PQ ? 16 * kTile : kTile,
                           (c->v_codec == FADE_V_PQ ? 4LL : 8LL) * 152);
    a.nsplit = 1 + (c->mid_capacity + a.chunk - 1) / a.chunk;
  }
  a.scale = 1.0f / sqrtf((float)c->head_dim);
  a.pq_cb = L->pq_codebook;
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
  if (mma) {
    // one launch: FP16 tiers (split 0) and the packed middle tier (tensor cores)
    if ((st = launch_mid_mma(c, L, q_rot, logits_ws, a.part_ml, a.part_acc, seg_count, sk,
                             a.nsplit, s)))
      return st;
  } else if ((st = launch_split_any(c, a, s, a.nsplit))) {
    return st;
  }
  const int bh = c->batch * c->num_q_heads;
  if (mma) {
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
        c->head_dim == 64
            ? cudaLaunchKernelEx(&lc, attn_combine_sk_kernel<64>, a, out, ml_ws)
            : cudaLaunchKernelEx(&lc, attn_combine_sk_kernel<128>, a, out, ml_ws);
    if (e != cudaSuccess)
      return set_error(FADE_ERR_CUDA, "fade_decode_attention combine: %s", cudaGetErrorString(e));
  } else if (c->head_dim == 64) {
    attn_combine_kernel<64><<<bh, 64, 0, s>>>(a, out, ml_ws);
  } else {
    attn_combine_kernel<128><<<bh, 128, 0, s>>>(a, out, ml_ws);
  }
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
  cudaStream_t cs = as_stream(stream);
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (a.S % 4 == 0 && a.NS % 4 == 0 && al16(a.logits) && al16(a.sink_sc) && al16(a.mid_sc[0]) &&
      al16(a.mid_sc[1]) && al16(a.rec_sc)) {
    const dim3 grid(ceil_div(a.NS / 4, 256), c->num_kv_heads, c->batch);
    switch (G) {
      case 1: h2o_accumulate4_kernel<1><<<grid, 256, 0, cs>>>(a); break;
      case 2: h2o_accumulate4_kernel<2><<<grid, 256, 0, cs>>>(a); break;
      case 4: h2o_accumulate4_kernel<4><<<grid, 256, 0, cs>>>(a); break;
      default: h2o_accumulate4_kernel<8><<<grid, 256, 0, cs>>>(a); break;
    }
  } else {
    h2o_accumulate_kernel<<<dim3(ceil_div(a.NS, 256), c->num_kv_heads, c->batch), 256, 0, cs>>>(a);
  }
  return launch_status("fade_h2o_accumulate");
}
