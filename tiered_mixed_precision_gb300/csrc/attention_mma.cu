// Decode attention over the packed middle tier on the tensor cores (INT4 K, INT2 V).
// Sources: page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术" — §项目结构与代码质量 (kernels/:
// fused INT4 dequant + SDPA), §第二层/§第三层 and §量化与Bit-Packing (INT4 K, INT2 V with one
// fp16 scale per 32 channels); page "探秘Transformer系列之（25）--- KV Cache优化之处理长文本序列"
// §1.2 (softmax-weighted average of V).
//
// One CTA = one (row, KV head) unit and one chunk of its middle tokens. A producer warp streams
// 256-token tiles into a shared-memory ring with TMA (2D tiled copies of the code rows with a
// bank-spreading swizzle, 1D bulk copies of the scale rows) under mbarrier completion; the
// consumer warps each take an equal share (64 or 32 tokens) of a tile:
//   QK^T: tokens are the MMA's M dimension, channels its K dimension. The packed codes become
//     exact fp16 integers in registers; each 64-channel half of the head dimension accumulates
//     in its own fragment whose 8 columns are (query head h, group parity), the query operand
//     being zero outside the column's group, so every 32-channel group's integer dot product
//     comes out separately and its K scale is applied in fp32 afterwards.
//   softmax: online, per warp, in the exp2 domain.
//   PV: channels are M, (query head, group parity) are N, tokens are K. V codes (exact fp16
//     integers) are the A operand, loaded transposed with ldmatrix.trans; the probabilities
//     times the V scale of the column's group are the B operand, transposed into place with
//     movmatrix. Columns whose group parity differs from the row's are discarded.
// mma.sync.m16n8k16 (fp16 in, fp32 accumulate) is used: at N = 8 query columns per KV head
// the contraction is far below the tile sizes of the 5th-generation tensor-core instructions.
#include <cuda.h>
#include <math.h>

#include <mutex>

#include "fade_internal.cuh"

namespace fade {
namespace {

constexpr int kF = FADE_META_FIELDS;
constexpr int kTileTok = 256;            // tokens per TMA tile
// Consumer warps per CTA (each takes kTileTok / kConsumers tokens of a tile), pipeline depth
// for head_dim 128, and the resident-CTA hint given to the register allocator.
#ifndef FADE_MMA_CONSUMERS
#define FADE_MMA_CONSUMERS 4
#endif
constexpr int kConsumers = FADE_MMA_CONSUMERS;
constexpr int kThreadsMma = 32 * (kConsumers + 1);
constexpr int kWarpTok = kTileTok / kConsumers;  // tokens per consumer warp per tile
constexpr int kMT = kWarpTok / 16;               // 16-token M-tiles per consumer warp
static_assert(kConsumers == 4 || kConsumers == 8, "4 or 8 consumer warps");
#ifndef FADE_MMA_STAGES_128
#define FADE_MMA_STAGES_128 3
#endif
#ifndef FADE_MMA_MIN_CTAS
#define FADE_MMA_MIN_CTAS 1
#endif
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz: a wait that never ends
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct MmaArgs {
  const uint16_t* q;                 // [B][Hq][D]
  const uint16_t *sink_k, *sink_v;   // [B][H][S][D]
  const uint16_t *rec_k, *rec_v;     // [B][H][W][D], ring
  const uint16_t* ks[2];             // K scales [B*H*C][D/32]
  const uint16_t* vs[2];             // V scales
  const int32_t* meta;
  float* logits;                     // nullable [B][Hq][NS]
  float* part_ml;                    // [B][Hq][nsplit][2]
  float* part_acc;                   // [B][Hq][nsplit][D]
  int32_t* status;
  int Hq, H, S, W, C, NS, chunk, nsplit;
  float inv_sqrt_d;
};

template <int D>
struct MmaCfg {
  static constexpr int KROW = D / 2;        // INT4 codes per token (bytes)
  static constexpr int VROW = D / 4;        // INT2 codes per token (bytes)
  static constexpr int SROW = D / kGroup;   // scales per token
  static constexpr int STAGE = kTileTok * (KROW + VROW + 2 * SROW * 2);
  static constexpr int NSTAGE = D == 128 ? FADE_MMA_STAGES_128 : 4;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = kTileTok * KROW;
  static constexpr int KS_OFF = V_OFF + kTileTok * VROW;
  static constexpr int VS_OFF = KS_OFF + kTileTok * SROW * 2;
  static constexpr int BAR_OFF = NSTAGE * STAGE;
  static constexpr int SMEM = BAR_OFF + 2 * NSTAGE * 8 + 1024;  // + alignment slack
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: gives up after kWaitCycles and records the failure in status[0].
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status,
                                          int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicCAS(status, 0, code);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// The N fp16 scales of one token row in shared memory (one 4- or 8-byte load) as fp32; zeros
// when `valid` is false.
template <int N>
__device__ __forceinline__ void load_scale_row(const uint16_t* p, bool valid, float (&f)[N]) {
  static_assert(N == 2 || N == 4, "2 or 4 groups per row");
  uint32_t w[N / 2];
  if constexpr (N == 4) {
    const uint2 u = valid ? *reinterpret_cast<const uint2*>(p) : make_uint2(0u, 0u);
    w[0] = u.x;
    w[1] = u.y;
  } else {
    w[0] = valid ? *reinterpret_cast<const uint32_t*>(p) : 0u;
  }
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    f[2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xFFFFu)));
    f[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
  }
}
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// INT4 codes -> exact fp16 integers. Word w holds 8 nibbles (nibble i = channel 8w'+i of its
// row). Pair kappa of a word is (nibble kappa', nibble kappa'+4) with kappa' = {0,1,2,3}: the
// nibble is placed in an fp16 mantissa above 1024 (offset-binary), then the offset is removed
// exactly.
template <int KAPPA>
__device__ __forceinline__ uint32_t k_pair(uint32_t w) {
  const uint32_t x = (KAPPA >= 2) ? (w >> 8) : w;
  if constexpr (KAPPA % 2 == 0) {
    const __half2 h = u32_as_h2((x & 0x000F000Fu) ^ 0x64086408u);       // 1024 + (n ^ 8)
    return h2_as_u32(__hsub2(h, __float2half2_rn(1032.f)));
  } else {
    const __half2 h = u32_as_h2((x & 0x00F000F0u) ^ 0x64806480u);       // 1024 + 16 (n ^ 8)
    return h2_as_u32(__hfma2(h, __float2half2_rn(0.0625f), __float2half2_rn(-72.f)));
  }
}

// INT2 codes -> exact fp16 integers: crumb c (bits 2c..2c+1 of each 16-bit half of x).
template <int C>
__device__ __forceinline__ uint32_t v_crumb(uint32_t x, uint32_t x10) {
  constexpr int cc = C <= 4 ? C : C - 5;
  const uint32_t src = C <= 4 ? x : x10;
  constexpr uint32_t mask = (0x3u << (2 * cc)) * 0x00010001u;
  constexpr uint32_t magic = (0x6400u | (2u << (2 * cc))) * 0x00010001u;
  const __half2 h = u32_as_h2((src & mask) ^ magic);                       // 1024 + (u^2)*4^cc
  constexpr float sc = 1.f / float(1 << (2 * cc));
  constexpr float off = -(1024.f / float(1 << (2 * cc)) + 2.f);
  return h2_as_u32(__hfma2(h, __float2half2_rn(sc), __float2half2_rn(off)));
}

template <int D, int G>
__global__ void __launch_bounds__(kThreadsMma, FADE_MMA_MIN_CTAS)
attn_mid_mma_kernel(const __grid_constant__ CUtensorMap tk0, const __grid_constant__ CUtensorMap tk1,
                    const __grid_constant__ CUtensorMap tv0, const __grid_constant__ CUtensorMap tv1,
                    MmaArgs a) {
  using Cfg = MmaCfg<D>;
  constexpr int NT = (2 * G + 7) / 8;    // 8-column n-tiles of (head, group parity)
  constexpr int NHALF = D / 64;          // 64-channel halves (accumulator sets)
  constexpr int NSTAGE = Cfg::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + Cfg::BAR_OFF;          // NSTAGE x 8 bytes
  const uint32_t bar_empty = bar_full + NSTAGE * 8;

  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int unit = b * a.H + hk;
  const int32_t* m = a.meta + unit * kF;
  const int n_mid = m[FADE_META_N_MID], cur = m[FADE_META_CUR];
  const int n_sink = m[FADE_META_N_SINK], n_rec = m[FADE_META_N_RECENT];
  const int head_slot = m[FADE_META_HEAD];
  const int lo = split > 0 ? (split - 1) * a.chunk : 0;
  const int hi = split > 0 ? min(n_mid, lo + a.chunk) : 0;
  const int n_tok = split > 0 ? max(0, hi - lo) : n_sink + n_rec;
  const int n_tiles = (n_tok + kTileTok - 1) / kTileTok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int hq0 = hk * G;
  const size_t pbase = ((size_t)(b * a.Hq + hq0)) * a.nsplit + split;

  if (n_tok == 0) {  // an empty split still publishes an empty partial
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
      const int h = i / D, c = i % D;
      a.part_acc[(pbase + (size_t)h * a.nsplit) * D + c] = 0.f;
    }
    if (threadIdx.x < G) {
      a.part_ml[(pbase + (size_t)threadIdx.x * a.nsplit) * 2] = -INFINITY;
      a.part_ml[(pbase + (size_t)threadIdx.x * a.nsplit) * 2 + 1] = 0.f;
    }
    return;
  }

  if (split > 0 && threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kConsumers);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const size_t row0 = (size_t)unit * a.C + lo;  // first global code row of this chunk
  bool failed = false;

  // per-warp online-softmax state (consumer warps): running max (exp2 domain), mass, and
  // the P.V accumulators
  float m2[NT], lsum[NT];
  float o[NHALF][4][NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    m2[j] = -INFINITY;
    lsum[j] = 0.f;
  }
#pragma unroll
  for (int s = 0; s < NHALF; ++s)
#pragma unroll
    for (int mm = 0; mm < 4; ++mm)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[s][mm][j][e] = 0.f;

  float* wm = reinterpret_cast<float*>(smem);                  // [kConsumers][8]
  float* wl = wm + kConsumers * 8;                             // [kConsumers][8]
  float* wo = wl + kConsumers * 8;                             // [kConsumers][G][D]

  if (split == 0) {
    // ------------------------------------------------------------ FP16 tiers (CUDA cores)
    // Warp w takes tokens w, w+4, ...; lane l holds channels l*CPL .. l*CPL+CPL-1.
    if (warp < kConsumers) {
      constexpr int CPL = D / 32;
      float qr[G][CPL], acc[G][CPL], mm_[G], ll[G];
      const uint16_t* qrow = a.q + (size_t)(b * a.Hq + hq0) * D;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        mm_[h] = -INFINITY;
        ll[h] = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          qr[h][c] = __half2float(__ushort_as_half(qrow[(size_t)h * D + lane * CPL + c]));
          acc[h][c] = 0.f;
        }
      }
      const float c2 = a.inv_sqrt_d * kLog2e;
      for (int u = warp; u < n_tok; u += kConsumers) {
        const bool is_sink = u < n_sink;
        const int slot = is_sink ? u : (head_slot + u - n_sink) % a.W;
        const size_t row = is_sink ? ((size_t)unit * a.S + u) * D : ((size_t)unit * a.W + slot) * D;
        const uint16_t* kr = (is_sink ? a.sink_k : a.rec_k) + row + lane * CPL;
        const uint16_t* vr = (is_sink ? a.sink_v : a.rec_v) + row + lane * CPL;
        float kv[CPL], vv[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          kv[c] = __half2float(__ushort_as_half(kr[c]));
          vv[c] = __half2float(__ushort_as_half(vr[c]));
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float d = 0.f;
#pragma unroll
          for (int c = 0; c < CPL; ++c) d = fmaf(qr[h][c], kv[c], d);
          d = warp_sum(d);
          if (a.logits && lane == 0)
            a.logits[(size_t)(b * a.Hq + hq0 + h) * a.NS + (is_sink ? u : a.S + a.C + slot)] =
                d * a.inv_sqrt_d;
          const float s2 = d * c2;
          const float mn = fmaxf(mm_[h], s2);
          const float al = exp2f(mm_[h] - mn);   // 0 when the old max is -inf
          const float p = exp2f(s2 - mn);
          ll[h] = ll[h] * al + p;
#pragma unroll
          for (int c = 0; c < CPL; ++c) acc[h][c] = fmaf(p, vv[c], acc[h][c] * al);
          mm_[h] = mn;
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (lane == 0) {
          wm[warp * 8 + h] = mm_[h];
          wl[warp * 8 + h] = ll[h];
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) wo[(warp * G + h) * D + lane * CPL + c] = acc[h][c];
      }
    }
    __syncthreads();
  } else if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const CUtensorMap* mk = cur ? &tk1 : &tk0;
      const CUtensorMap* mv = cur ? &tv1 : &tv0;
      const uint16_t* ksg = cur ? a.ks[1] : a.ks[0];
      const uint16_t* vsg = cur ? a.vs[1] : a.vs[0];
      int issued = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int s = it % NSTAGE;
        if (it >= NSTAGE &&
            !mbar_wait(bar_empty + 8 * s, ((it / NSTAGE) & 1) ^ 1, a.status, 2)) {
          failed = true;
          break;
        }
        const int nt = min(kTileTok, n_tok - it * kTileTok);
        // scale rows copied: rounded up so the copy is a multiple of 16 bytes (it stays inside
        // the unit: rows start at multiples of 4 and the slot stride is a multiple of 64)
        constexpr int kAlign = 16 / (Cfg::SROW * 2);
        const int ns = (nt + kAlign - 1) / kAlign * kAlign;
        const size_t r = row0 + (size_t)it * kTileTok;
        const uint32_t stage = sbase + s * Cfg::STAGE;
        const uint32_t bytes = kTileTok * (Cfg::KROW + Cfg::VROW) + 2u * ns * Cfg::SROW * 2;
        mbar_expect_tx(bar_full + 8 * s, bytes);
        tma_load_2d(stage + Cfg::K_OFF, mk, 0, (int)r, bar_full + 8 * s);
        tma_load_2d(stage + Cfg::V_OFF, mv, 0, (int)r, bar_full + 8 * s);
        bulk_load_1d(stage + Cfg::KS_OFF, ksg + r * Cfg::SROW, ns * Cfg::SROW * 2,
                     bar_full + 8 * s);
        bulk_load_1d(stage + Cfg::VS_OFF, vsg + r * Cfg::SROW, ns * Cfg::SROW * 2,
                     bar_full + 8 * s);
        ++issued;
      }
      // never leave the CTA with copies in flight: wait (bounded) for every issued tile
      for (int it = max(0, issued - NSTAGE); it < issued; ++it)
        mbar_wait(bar_full + 8 * (it % NSTAGE), (it / NSTAGE) & 1, a.status, 3);
    }
  } else {
    // ------------------------------------------------------------ consumers
    // query B operand: column n of n-tile j = (head 4j + n/2, parity n%2); thread (g, t)
    // holds column g, k-slots {2t, 2t+1} (group 2s of half s) and {2t+8, 2t+9} (group 2s+1)
    uint32_t qb[NHALF][4][NT][2];
    {
      const uint16_t* qrow = a.q + (size_t)(b * a.Hq + hq0) * D;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int h = 4 * j + g / 2, par = g & 1;
        const bool valid = h < G;
#pragma unroll
        for (int s = 0; s < NHALF; ++s)
#pragma unroll
          for (int kp = 0; kp < 4; ++kp) {
            const int c_lo = 64 * s + 8 * t + kp;        // group 2s
            const int c_hi = c_lo + 32;                  // group 2s+1
            uint16_t v0 = 0, v1 = 0, v2 = 0, v3 = 0;
            if (valid && par == 0) {
              v0 = qrow[(size_t)h * D + c_lo];
              v1 = qrow[(size_t)h * D + c_lo + 4];
            }
            if (valid && par == 1) {
              v2 = qrow[(size_t)h * D + c_hi];
              v3 = qrow[(size_t)h * D + c_hi + 4];
            }
            qb[s][kp][j][0] = uint32_t(v0) | (uint32_t(v1) << 16);
            qb[s][kp][j][1] = uint32_t(v2) | (uint32_t(v3) << 16);
          }
      }
    }
    const float c2 = a.inv_sqrt_d * kLog2e;

    for (int it = 0; it < n_tiles; ++it) {
      const int s_ = it % NSTAGE;
      if (!mbar_wait(bar_full + 8 * s_, (it / NSTAGE) & 1, a.status, 1)) {
        failed = true;
        break;
      }
      const int nt = min(kTileTok, n_tok - it * kTileTok);
      const int wr0 = warp * kWarpTok;
      const uint32_t stage = sbase + s_ * Cfg::STAGE;
      const uint8_t* st_ptr = smem + s_ * Cfg::STAGE;
      const uint16_t* kss = reinterpret_cast<const uint16_t*>(st_ptr + Cfg::KS_OFF);
      const uint16_t* vss = reinterpret_cast<const uint16_t*>(st_ptr + Cfg::VS_OFF);
      if (wr0 < nt) {
        float sc[kMT][NT][2];  // logits (exp2 domain) of tokens g, g+8 of each M-tile
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          const int r0 = wr0 + mt * 16;
          float ks_lo[D / kGroup], ks_hi[D / kGroup];
          load_scale_row<D / kGroup>(kss + (r0 + g) * Cfg::SROW, true, ks_lo);
          load_scale_row<D / kGroup>(kss + (r0 + g + 8) * Cfg::SROW, true, ks_hi);
          float acc_s[NT][2];
#pragma unroll
          for (int j = 0; j < NT; ++j) acc_s[j][0] = acc_s[j][1] = 0.f;
#pragma unroll
          for (int s = 0; s < NHALF; ++s) {
            // K rows r0..r0+15, 16-byte chunks 2s and 2s+1 (one 32-channel group each)
            const int lrow = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int chunk = 2 * s + (lane >> 4);
            int sw;
            if constexpr (D == 128)
              sw = (chunk ^ ((lrow >> 1) & 3));            // 64-byte swizzle
            else
              sw = (chunk ^ ((lrow >> 2) & 1));            // 32-byte swizzle
            uint32_t k0, k1, k2, k3;  // (rows g, chunk 2s) (g+8, 2s) (g, 2s+1) (g+8, 2s+1)
            ldsm_x4(stage + Cfg::K_OFF + lrow * Cfg::KROW + sw * 16, k0, k1, k2, k3);
            float cacc[NT][4];
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
              for (int e = 0; e < 4; ++e) cacc[j][e] = 0.f;
#define FADE_KSTEP(KP)                                                                    \
  {                                                                                       \
    const uint32_t a0 = k_pair<KP>(k0), a1 = k_pair<KP>(k1), a2 = k_pair<KP>(k2),         \
                   a3 = k_pair<KP>(k3);                                                   \
    _Pragma("unroll") for (int j = 0; j < NT; ++j)                                        \
        mma16816(cacc[j], a0, a1, a2, a3, qb[s][KP][j][0], qb[s][KP][j][1]);              \
  }
            FADE_KSTEP(0) FADE_KSTEP(1) FADE_KSTEP(2) FADE_KSTEP(3)
#undef FADE_KSTEP
            // column 2t = (head 4j+t, group 2s), column 2t+1 = (head 4j+t, group 2s+1)
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              acc_s[j][0] = fmaf(cacc[j][0], ks_lo[2 * s], acc_s[j][0]);
              acc_s[j][0] = fmaf(cacc[j][1], ks_lo[2 * s + 1], acc_s[j][0]);
              acc_s[j][1] = fmaf(cacc[j][2], ks_hi[2 * s], acc_s[j][1]);
              acc_s[j][1] = fmaf(cacc[j][3], ks_hi[2 * s + 1], acc_s[j][1]);
            }
          }
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const int h = 4 * j + t;
            const bool hv = h < G;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int tok = r0 + g + 8 * r;
              const bool tv = tok < nt;
              if (a.logits && hv && tv)
                a.logits[(size_t)(b * a.Hq + hq0 + h) * a.NS + a.S + lo + it * kTileTok + tok] =
                    acc_s[j][r] * a.inv_sqrt_d;
              sc[mt][j][r] = (hv && tv) ? acc_s[j][r] * c2 : -INFINITY;
            }
          }
        }
        // online softmax (per head column t of each n-tile; warp-uniform running max)
        float alpha[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          float mx = -INFINITY;
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt) mx = fmaxf(mx, fmaxf(sc[mt][j][0], sc[mt][j][1]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(m2[j], mx);
          alpha[j] = (mn == -INFINITY) ? 1.f : exp2f(m2[j] - mn);
          m2[j] = mn;
          float ps = 0.f;
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const float p = (sc[mt][j][r] == -INFINITY) ? 0.f : exp2f(sc[mt][j][r] - mn);
              sc[mt][j][r] = p;
              ps += p;
            }
          lsum[j] = lsum[j] * alpha[j] + ps;
        }
        // rescale the accumulators only when some column's running max moved (warp-uniform)
        bool moved = false;
#pragma unroll
        for (int j = 0; j < NT; ++j) moved |= alpha[j] != 1.f;
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
          for (int s = 0; s < NHALF; ++s)
#pragma unroll
            for (int mm = 0; mm < 4; ++mm)
#pragma unroll
              for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[s][mm][j][e] *= alpha[j];
        }

        // PV over the warp's M-tiles (16 tokens each = one MMA k-step)
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          const int r0 = wr0 + mt * 16;
          // past the tile's tokens the scale rows may never have been copied: use 0 so that a
          // zero probability cannot meet a non-finite leftover
          float vs_lo[D / kGroup], vs_hi[D / kGroup];
          load_scale_row<D / kGroup>(vss + (r0 + g) * Cfg::SROW, r0 + g < nt, vs_lo);
          load_scale_row<D / kGroup>(vss + (r0 + g + 8) * Cfg::SROW, r0 + g + 8 < nt, vs_hi);
          uint32_t X[2 * NHALF];  // (tokens 0-7 | 8-15) x (channel half)
          {
            const int lrow = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
            if constexpr (D == 128) {
              const int chunk = lane >> 4;
              const int sw = chunk ^ ((lrow >> 2) & 1);    // 32-byte swizzle
              ldsm_x4_t(stage + Cfg::V_OFF + lrow * Cfg::VROW + sw * 16, X[0], X[1], X[2], X[3]);
            } else {
              ldsm_x2_t(stage + Cfg::V_OFF + lrow * Cfg::VROW, X[0], X[1]);
            }
          }
#pragma unroll
          for (int s = 0; s < NHALF; ++s) {
            uint32_t pb[NT][2];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const float p0 = sc[mt][j][0], p1 = sc[mt][j][1];
              const uint32_t lo_ = h2_as_u32(__floats2half2_rn(p0 * vs_lo[2 * s], p0 * vs_lo[2 * s + 1]));
              const uint32_t hi_ = h2_as_u32(__floats2half2_rn(p1 * vs_hi[2 * s], p1 * vs_hi[2 * s + 1]));
              pb[j][0] = movm_t(lo_);
              pb[j][1] = movm_t(hi_);
            }
            const uint32_t xa = X[2 * s], xb = X[2 * s + 1];
            const uint32_t xa10 = xa >> 10, xb10 = xb >> 10;
#define FADE_PV(MM)                                                                         \
  {                                                                                         \
    const uint32_t a0 = v_crumb<2 * MM>(xa, xa10), a1 = v_crumb<2 * MM + 1>(xa, xa10);      \
    const uint32_t a2 = v_crumb<2 * MM>(xb, xb10), a3 = v_crumb<2 * MM + 1>(xb, xb10);      \
    _Pragma("unroll") for (int j = 0; j < NT; ++j)                                          \
        mma16816(o[s][MM][j], a0, a1, a2, a3, pb[j][0], pb[j][1]);                          \
  }
            FADE_PV(0) FADE_PV(1) FADE_PV(2) FADE_PV(3)
#undef FADE_PV
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s_);
    }

    // total probability mass of each head over the warp's tokens (lanes sharing t)
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      lsum[j] += __shfl_xor_sync(0xffffffffu, lsum[j], 4);
      lsum[j] += __shfl_xor_sync(0xffffffffu, lsum[j], 8);
      lsum[j] += __shfl_xor_sync(0xffffffffu, lsum[j], 16);
    }
  }
  // Past this barrier every tile is consumed and the producer has drained its copies, so
  // the stage memory can hold the per-warp results.
  if (split > 0) __syncthreads();
  if (split > 0 && warp < kConsumers) {
    const int gsel = g >= 4 ? 1 : 0;  // the column parity that matches row g's group
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int h = 4 * j + t;
      if (h < G) {
        if (g == 0) {
          wm[warp * 8 + h] = m2[j];
          wl[warp * 8 + h] = lsum[j];
        }
#pragma unroll
        for (int s = 0; s < NHALF; ++s)
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {
            const int c = 64 * s + 8 * g + 2 * mm;
            wo[(warp * G + h) * D + c] = gsel ? o[s][mm][j][1] : o[s][mm][j][0];
            wo[(warp * G + h) * D + c + 1] = gsel ? o[s][mm][j][3] : o[s][mm][j][2];
          }
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int h = i / D, c = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, wm[w * 8 + h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) {
      const float f = (wm[w * 8 + h] == -INFINITY) ? 0.f : exp2f(wm[w * 8 + h] - M);
      L = fmaf(wl[w * 8 + h], f, L);
      O = fmaf(wo[(w * G + h) * D + c], f, O);
    }
    a.part_acc[(pbase + (size_t)h * a.nsplit) * D + c] = O;
    if (c == 0) {
      a.part_ml[(pbase + (size_t)h * a.nsplit) * 2] = M * kLn2;  // natural-log units
      a.part_ml[(pbase + (size_t)h * a.nsplit) * 2 + 1] = L;
    }
  }
  (void)failed;
}

// ------------------------------------------------------------------ host side
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// 2D map over code rows: [rows][row_bytes] u8, boxes of kTileTok rows.
fade_status_t encode_rows(CUtensorMap* m, const void* base, unsigned long long rows,
                          int row_bytes) {
  EncodeFn fn = encode_fn();
  if (!fn) return set_error(FADE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)row_bytes, (cuuint32_t)kTileTok};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = row_bytes == 64   ? CU_TENSOR_MAP_SWIZZLE_64B
                                : row_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                  : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(FADE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return FADE_OK;
}

template <int D, int G>
fade_status_t launch_mma(const fade_config_t* c, const fade_layer_t* L, const MmaArgs& a,
                         int n_splits, cudaStream_t st) {
  using Cfg = MmaCfg<D>;
  const unsigned long long rows = (unsigned long long)c->batch * c->num_kv_heads * a.C;
  CUtensorMap tk[2], tv[2];
  fade_status_t s;
  for (int i = 0; i < 2; ++i) {
    if ((s = encode_rows(&tk[i], L->mid_k_codes[i], rows, Cfg::KROW))) return s;
    if ((s = encode_rows(&tv[i], L->mid_v_codes[i], rows, Cfg::VROW))) return s;
  }
  auto kern = attn_mid_mma_kernel<D, G>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) !=
      cudaSuccess)
    return launch_status("fade_decode_attention (middle tier) shared-memory opt-in");
  kern<<<dim3(n_splits, c->num_kv_heads, c->batch), kThreadsMma, Cfg::SMEM, st>>>(
      tk[0], tk[1], tv[0], tv[1], a);
  return launch_status("fade_decode_attention (middle tier)");
}

}  // namespace

bool mid_mma_supported(const fade_config_t* c) {
  return c->middle_k_bits == 4 && c->middle_v_bits == 2;
}

fade_status_t launch_mid_mma(const fade_config_t* c, const fade_layer_t* L, const uint16_t* q,
                             float* logits, float* part_ml, float* part_acc, int chunk,
                             int nsplit, cudaStream_t st) {
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
  a.status = L->status;
  a.Hq = c->num_q_heads;
  a.H = c->num_kv_heads;
  a.S = c->n_sink;
  a.C = mid_stride(c);
  a.NS = c->n_sink + a.C + c->recent_window;
  a.chunk = chunk;
  a.nsplit = nsplit;
  a.inv_sqrt_d = 1.0f / sqrtf((float)c->head_dim);
  const int G = c->num_q_heads / c->num_kv_heads;
#define FADE_CASE(D_, G_) \
  if (c->head_dim == D_ && G == G_) return launch_mma<D_, G_>(c, L, a, nsplit, st);
  FADE_CASE(64, 1) FADE_CASE(64, 2) FADE_CASE(64, 4) FADE_CASE(64, 8)
  FADE_CASE(128, 1) FADE_CASE(128, 2) FADE_CASE(128, 4) FADE_CASE(128, 8)
#undef FADE_CASE
  return set_error(FADE_ERR_UNSUPPORTED, "no tensor-core attention for this shape");
}

}  // namespace fade
