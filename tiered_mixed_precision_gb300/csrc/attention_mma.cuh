#pragma once
// Decode attention over the packed middle tier on the tensor cores (INT4 or INT2 K; INT2, INT4 or
// PQ-coded V).
// Sources: page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术" — §项目结构与代码质量 (kernels/:
// fused INT4 dequant + SDPA), §第二层/§第三层 and §量化与Bit-Packing (INT4 K, INT2 V with one
// fp16 scale per 32 channels); page "探秘Transformer系列之（25）--- KV Cache优化之处理长文本序列"
// §1.2 (softmax-weighted average of V).
//
// A persistent grid (a fixed number of CTAs per SM) under a stream-K schedule: every unit's
// middle tier is cut into 256-token tiles, and CTA c takes the FP16-tier items of units c,
// c + P, ... and then a contiguous run of tiles in global order (which may cross units; each
// run inside one unit is a segment with its own partial, merged by attn_combine_sk_kernel).
// A producer warp streams the items' tiles into a shared-memory ring with TMA (2D tiled copies
// of the code rows with a bank-spreading swizzle, 1D bulk copies of the scale rows) under
// mbarrier completion; the consumer warps each take an equal share (64 or 32 tokens) of a
// tile:
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

#include <algorithm>
#include <atomic>
#include <mutex>
#include <unordered_map>

#include "fade_internal.cuh"

namespace fade {

// Arguments of the tensor-core attention kernel (one layer).
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
  int32_t* seg_count;                // [B][H]: partials of each unit (split 0 + segments)
  int f16_sreg, f16_rreg;            // staged FP16 tiers: bytes of a sink / ring region (one
                                     // 64-channel half of the rows); f16_rreg 0: not staged
  int B, Hq, H, S, W, C, NS, chunk, nsplit;
  float inv_sqrt_d;
  const uint16_t* pq_cb;             // PQ-coded V: the layer's codebook [D/4][256][4]
};

// The kernel for INT2 K codes (instantiated in its own translation unit).
fade_status_t launch_mid_mma_k2(const fade_config_t* c, const fade_layer_t* L, MmaArgs a,
                                const StreamK& sk, cudaStream_t st);

// Everything below has internal linkage: attention_mma.cu (INT4 K) and attention_mma_k2.cu
// (INT2 K) each include this header and hold their own instantiations, and their own host-side
// tensor-map cache.
namespace {

constexpr int kF = FADE_META_FIELDS;
constexpr int kTileTok = FADE_ATTN_TILE_TOKENS;  // tokens per TMA tile
// Warp layout per (head_dim, query heads per KV head): consumer warps per CTA, each taking an
// equal share of a tile (32 or 64 tokens), one producer warp, and the resident-CTA hint given to
// the register allocator. Eight consumers: two CTAs per SM when the accumulators are small
// (G <= 4), one CTA for G = 8 (whose accumulators need the larger register budget); PQ-coded V
// at G = 8 keeps four (its codebook and V tiles fill the shared memory). FADE_MMA_WIDE=0 forces
// four consumers everywhere; FADE_MMA_STAGES_128 sets the pipeline
// depth for head_dim 128.
#ifndef FADE_MMA_WIDE
#define FADE_MMA_WIDE 1
#endif
#ifndef FADE_MMA_STAGES_128
#define FADE_MMA_STAGES_128 3
#endif
// Resident CTAs per SM of the eight-consumer shape (two: 96 registers a thread; one: more
// registers and a deeper ring per CTA).
#ifndef FADE_MMA_CTAS_PER_SM
#define FADE_MMA_CTAS_PER_SM 2
#endif
// Independent (code byte -> centroid -> store) chains a consumer lane keeps in flight when it
// decodes a PQ-coded V tile (all of them: the measured best).
#ifndef FADE_PQ_DECODE_UNROLL
#define FADE_PQ_DECODE_UNROLL 16
#endif
constexpr int kPqDecodeUnroll = FADE_PQ_DECODE_UNROLL;
// The FP16 tiers (sinks + recent ring) of an item on the tensor cores (1) or the CUDA cores (0;
// also the path when they do not fit a ring stage).
#ifndef FADE_F16_MMA
#define FADE_F16_MMA 1
#endif
constexpr bool kF16Mma = FADE_F16_MMA != 0;
// Weight of an FP16-tier item in the stream-K schedule, in middle tiles.
#ifndef FADE_F16_ITEM_WEIGHT
#define FADE_F16_ITEM_WEIGHT 3
#endif
template <int D, int G, bool PQ = false>
struct MmaShape {
  static constexpr int CONS = (FADE_MMA_WIDE && (G <= 4 || !PQ)) ? 8 : 4;
  static constexpr int THREADS = 32 * (CONS + 1);
  static constexpr int WARP_TOK = kTileTok / CONS;  // tokens per consumer warp per tile
  static constexpr int MT = WARP_TOK / 16;          // 16-token M-tiles per consumer warp
  // PQ-coded V keeps the codebook and per-warp V tiles in shared memory: one CTA per SM
  static constexpr int MINB = PQ ? 1 : ((CONS == 8 && G <= 4) ? FADE_MMA_CTAS_PER_SM : 1);
};
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;


// Stage layout of the ring for V codes of VB bits (2, or 4: the safe preset) and NST stages (0:
// the default for the head dimension); MROWS (consumer warps x query heads) rows of the merge;
// K codes of KB bits (4, or 2).
template <int D, int VB = 2, int NST = 0, int MROWS = 32, int KB = 4>
struct MmaCfg {
  static constexpr int KROW = D * KB / 8;   // INT4 / INT2 K codes per token (bytes)
  static constexpr int VROW = D * VB / 8;   // INT2 / INT4 V codes per token (bytes)
  static constexpr int SROW = D / kGroup;   // scales per token
  static constexpr int Q_BYTES = 8 * D * 2; // the item's query rows (up to 8 heads), fp16
  static constexpr int STAGE = kTileTok * (KROW + VROW + 2 * SROW * 2) + Q_BYTES;
  static constexpr int NSTAGE = NST ? NST : (D == 128 ? FADE_MMA_STAGES_128 : 4);
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = kTileTok * KROW;
  static constexpr int KS_OFF = V_OFF + kTileTok * VROW;
  static constexpr int VS_OFF = KS_OFF + kTileTok * SROW * 2;
  static constexpr int Q_OFF = VS_OFF + kTileTok * SROW * 2;
  // per-item merge of the consumer warps' partials: m, l [8][8], acc [8][8][D], weights [8][8]
  static constexpr int MERGE_OFF = NSTAGE * STAGE;
  // (acc rows padded by one float: the fragment-layout writes then hit 16 banks, not 4)
  static constexpr int WO_ROW = D + 1;
  static constexpr int MERGE_BYTES = (64 + 64 + MROWS * WO_ROW + 64) * 4;
  static constexpr int INFO_OFF = MERGE_OFF + MERGE_BYTES;  // per stage: kInfo ints
  static constexpr int BAR_OFF = INFO_OFF + NSTAGE * 8 * 4;
  static constexpr int SMEM = BAR_OFF + 2 * NSTAGE * 8 + 1024;  // + alignment slack
  static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned (TMA swizzle)");
};

// Ring depth of one shape: the default, except INT4 V at d = 128 (38 KB stages): two stages
// when two CTAs share an SM, four when one CTA holds it.
template <int D, int G, bool PQ, int VB>
__host__ __device__ constexpr int mma_stages() {
  return (VB == 4 && D == 128) ? (MmaShape<D, G, PQ>::MINB > 1 ? 2 : 4) : 0;
}
template <int D, int G, bool PQ, int VB, int KB>
using MmaCfgOf = MmaCfg<D, VB, mma_stages<D, G, PQ, VB>(), MmaShape<D, G, PQ>::CONS * G, KB>;

// Shared memory added for PQ-coded V, after the layout above: the layer's codebook stored
// centroid-major ([256][D/4] entries of 4 fp16 channels, so that the 32 lanes of a warp, one
// per sub-space, gather 32 different entries in two wavefronts whatever the codes) and one
// decoded 16-token V tile per consumer warp ([16][D] fp16, rows padded by 16 bytes so that the
// transposing matrix loads touch 32 distinct banks).
template <int D>
struct PqCfg {
  using C = MmaCfg<D>;
  static constexpr int SUBS = D / kPqSub;
  static constexpr int CB_OFF = (C::BAR_OFF + 2 * C::NSTAGE * 8 + 15) / 16 * 16;
  static constexpr int CB_BYTES = kPqCentroids * D * 2;
  static constexpr int VT_ROW = D * 2 + 16;
  static constexpr int VT_OFF = CB_OFF + CB_BYTES;
  static constexpr int VT_BYTES = 8 * 16 * VT_ROW;   // up to eight consumer warps
  static constexpr int SMEM = VT_OFF + VT_BYTES + 1024;  // + alignment slack
  static_assert(SMEM <= 227 * 1024, "PQ layout exceeds the shared memory of a CTA");
};

// Stage info written by the producer before it arms a stage: what the consumers find there.
enum StageInfo { kInfoUnit, kInfoSplit, kInfoNt, kInfoLast, kInfoTok0, kInfoSink, kInfoRec,
                 kInfoHead, kInfo };
// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
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
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
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

// 2^x by the hardware approximation (relative error ~2^-22; 2^-inf = +0; results below 2^-126
// flush to zero, which is far below anything that reaches an fp16 output).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Sums over the warp of N per-lane values, every lane receiving all N sums: a reduce-scatter
// (each step halves the values a lane carries and sends the other half across), a plain
// reduction of the last value, and a broadcast from the lanes that own each sum.
template <int N>
__device__ __forceinline__ void warp_allreduce(float (&v)[N], int lane) {
  if constexpr (N == 1) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
  } else {
    constexpr int LOG = N == 2 ? 1 : N == 4 ? 2 : 3;
    float w[N];
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = v[i];
#pragma unroll
    for (int st = 0; st < LOG; ++st) {
      const int half = N >> (st + 1), off = 16 >> st;
      const bool up = lane & off;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = up ? w[i] : w[i + half];
        const float keep = up ? w[i + half] : w[i];
        w[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
#pragma unroll
    for (int o = 16 >> LOG; o; o >>= 1) w[0] += __shfl_xor_sync(0xffffffffu, w[0], o);
#pragma unroll
    for (int h = 0; h < N; ++h) {
      int src = 0;
#pragma unroll
      for (int st = 0; st < LOG; ++st) src += ((h >> (LOG - 1 - st)) & 1) * (16 >> st);
      v[h] = __shfl_sync(0xffffffffu, w[0], src);
    }
  }
}

// CPL consecutive fp16 values (CPL = 2 or 4, 4- or 8-byte aligned) as fp32.
template <int CPL>
__device__ __forceinline__ void load_f16_lane(const uint16_t* p, float (&f)[CPL]) {
  if constexpr (CPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    f[0] = a.x;
    f[1] = a.y;
    f[2] = b.x;
    f[3] = b.y;
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u));
    f[0] = a.x;
    f[1] = a.y;
  }
}

// CPL consecutive fp16 values from shared memory (32-bit shared address) as fp32.
template <int CPL>
__device__ __forceinline__ void lds_f16_lane(uint32_t addr, float (&f)[CPL]);

// v[i] for a runtime index i < N, without indexing a register array dynamically.
template <int N>
__device__ __forceinline__ float pick(const float (&v)[N], int i) {
  float r = v[0];
#pragma unroll
  for (int k = 1; k < N; ++k) r = (i == k) ? v[k] : r;
  return r;
}

// Barrier among the NC consumer warps only (named barrier 1; the producer warp never joins).
template <int NC>
__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NC * 32) : "memory");
}

// (x & m) ^ c in one logic instruction.
__device__ __forceinline__ uint32_t and_xor(uint32_t x, uint32_t m, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(d) : "r"(x), "r"(m), "r"(c));
  return d;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts64(uint32_t addr, uint2 v) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}
template <int CPL>
__device__ __forceinline__ void lds_f16_lane(uint32_t addr, float (&f)[CPL]) {
  if constexpr (CPL == 4) {
    const uint2 u = lds64(addr);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    f[0] = a.x;
    f[1] = a.y;
    f[2] = b.x;
    f[3] = b.y;
  } else {
    const uint32_t u = lds32(addr);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u));
    f[0] = a.x;
    f[1] = a.y;
  }
}
__device__ __forceinline__ float h_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))); }
__device__ __forceinline__ float h_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// INT4 codes -> exact fp16 integers. Word w holds 8 nibbles (nibble i = channel 8w'+i of its
// row). Pair kappa of a word is (nibble kappa', nibble kappa'+4) with kappa' = {0,1,2,3}: the
// nibble is placed in an fp16 mantissa above 1024 (offset-binary), then the offset is removed
// exactly. x8 = w >> 8.
template <int KAPPA>
__device__ __forceinline__ uint32_t k_pair(uint32_t w, uint32_t x8) {
  const uint32_t x = (KAPPA >= 2) ? x8 : w;
  if constexpr (KAPPA % 2 == 0) {
    const __half2 h = u32_as_h2(and_xor(x, 0x000F000Fu, 0x64086408u));   // 1024 + (n ^ 8)
    return h2_as_u32(__hsub2(h, __float2half2_rn(1032.f)));
  } else {
    const __half2 h = u32_as_h2(and_xor(x, 0x00F000F0u, 0x64806480u));   // 1024 + 16 (n ^ 8)
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
  const __half2 h = u32_as_h2(and_xor(src, mask, magic));                  // 1024 + (u^2)*4^cc
  constexpr float sc = 1.f / float(1 << (2 * cc));
  constexpr float off = -(1024.f / float(1 << (2 * cc)) + 2.f);
  return h2_as_u32(__hfma2(h, __float2half2_rn(sc), __float2half2_rn(off)));
}

// Per-lane shared-memory byte offsets inside a stage, for M-tile 0 of the warp (M-tile mt adds
// mt * 16 rows). With the 64-/32-byte swizzles the XOR pattern depends only on the lane.
template <int D, int VB>
struct LaneOffsets {
  uint32_t k[D / 64];               // ldmatrix address of the K codes, per 64-channel half
  uint32_t v[VB == 4 ? D / 64 : 1]; // ldmatrix.trans address of the V codes (INT4: per half)
  uint32_t ks, vs;                  // K / V scale row of token g
};

// INT4 V rows have the K rows' width and swizzle, so they are addressed like the K rows (the
// 16-byte chunks 2s and 2s + 1, i.e. the quantisation groups of half s, of tokens 0-15).
template <int D, int G, bool PQ, int VB, int KB>
__device__ __forceinline__ LaneOffsets<D, VB> lane_offsets(int wr0, int lane) {
  using Cfg = MmaCfgOf<D, G, PQ, VB, KB>;
  LaneOffsets<D, VB> o;
  const int lr = (lane & 7) + ((lane >> 3) & 1) * 8, hi = lane >> 4, g = lane >> 2;
  // this lane's 16-byte chunk (2s + hi for 64-byte rows, hi otherwise) of row wr0 + lr, under the
  // swizzle the tensor map gives rows of that width (64 B: chunk ^ (row / 2) % 4; 32 B: chunk ^
  // (row / 4) % 2; 16 B: none)
  auto at = [&](int base, int row_bytes, int s) {
    const int r = wr0 + lr;
    if (row_bytes == 64) return base + r * 64 + (((2 * s + hi) ^ ((lr >> 1) & 3)) * 16);
    if (row_bytes == 32) return base + r * 32 + ((hi ^ ((lr >> 2) & 1)) * 16);
    return base + r * row_bytes;
  };
#pragma unroll
  for (int s = 0; s < (Cfg::KROW == 64 ? 2 : 1); ++s) o.k[s] = at(Cfg::K_OFF, Cfg::KROW, s);
#pragma unroll
  for (int s = 0; s < (Cfg::VROW == 64 ? 2 : 1); ++s) o.v[s] = at(Cfg::V_OFF, Cfg::VROW, s);
  o.ks = Cfg::KS_OFF + (wr0 + g) * Cfg::SROW * 2;
  o.vs = Cfg::VS_OFF + (wr0 + g) * Cfg::SROW * 2;
  return o;
}

// Scale words of one token row: D/32 fp16 scales as D/64 half2 words.
template <int D>
__device__ __forceinline__ void scale_words(uint32_t addr, uint32_t (&w)[D / 64]) {
  if constexpr (D == 128) {
    const uint2 v = lds64(addr);
    w[0] = v.x;
    w[1] = v.y;
  } else {
    w[0] = lds32(addr);
  }
}

// One consumer warp's share of one tile: QK^T on the tensor cores with the K scales applied per
// group in fp32, the online-softmax update, and PV. FULL: every token of the warp's share is
// valid (no masking). Invalid head columns (G < 4) carry logit 0 and are discarded later.
template <int D, int G, bool FULL, bool LOGITS, bool PQ, int VB, int KB>
__device__ __forceinline__ void consume_tile(
    const MmaArgs& a, uint32_t stage, const LaneOffsets<D, VB>& lo_, int nt, int wr0, int lane,
    const uint32_t (&qb)[D / 64][4][(2 * G + 7) / 8][2], float (&m2)[(2 * G + 7) / 8],
    float (&lsum)[(2 * G + 7) / 8], float (&o)[D / 64][4][(2 * G + 7) / 8][4], float c2,
    float* logit_row, uint32_t vt, uint32_t cbs) {
  using Cfg = MmaCfgOf<D, G, PQ, VB, KB>;
  constexpr int NT = (2 * G + 7) / 8;
  constexpr int NHALF = D / 64;
  const int g = lane >> 2, t = lane & 3;
  float sc[MmaShape<D, G, PQ>::MT][NT][2];  // logits (exp2 domain) of tokens g, g+8 of each M-tile
#pragma unroll
  for (int mt = 0; mt < MmaShape<D, G, PQ>::MT; ++mt) {
    const int r0 = wr0 + mt * 16;
    uint32_t kw_lo[NHALF], kw_hi[NHALF];
    scale_words<D>(stage + lo_.ks + mt * 16 * Cfg::SROW * 2, kw_lo);
    scale_words<D>(stage + lo_.ks + (mt * 16 + 8) * Cfg::SROW * 2, kw_hi);
    float acc_s[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc_s[j][0] = acc_s[j][1] = 0.f;
    // INT2 K: (rows g | g+8) x (16-byte chunk s = channels 64s .. 64s+63), one matrix load for
    // the whole row (two chunks at d = 128)
    uint32_t K2[2 * NHALF];
    if constexpr (KB == 2) {
      if constexpr (D == 128)
        ldsm_x4(stage + lo_.k[0] + mt * 16 * Cfg::KROW, K2[0], K2[1], K2[2], K2[3]);
      else
        ldsm_x2(stage + lo_.k[0] + mt * 16 * Cfg::KROW, K2[0], K2[1]);
    }
#pragma unroll
    for (int s = 0; s < NHALF; ++s) {
      float cacc[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) cacc[j][e] = 0.f;
      if constexpr (KB == 4) {
        uint32_t k0, k1, k2, k3;  // (rows g, chunk 2s) (g+8, 2s) (g, 2s+1) (g+8, 2s+1)
        ldsm_x4(stage + lo_.k[s] + mt * 16 * Cfg::KROW, k0, k1, k2, k3);
        const uint32_t k0s = k0 >> 8, k1s = k1 >> 8, k2s = k2 >> 8, k3s = k3 >> 8;
#define FADE_KSTEP(KP)                                                                        \
  {                                                                                           \
    const uint32_t a0 = k_pair<KP>(k0, k0s), a1 = k_pair<KP>(k1, k1s),                        \
                   a2 = k_pair<KP>(k2, k2s), a3 = k_pair<KP>(k3, k3s);                        \
    _Pragma("unroll") for (int j = 0; j < NT; ++j)                                            \
        mma16816(cacc[j], a0, a1, a2, a3, qb[s][KP][j][0], qb[s][KP][j][1]);                  \
  }
        FADE_KSTEP(0) FADE_KSTEP(1) FADE_KSTEP(2) FADE_KSTEP(3)
#undef FADE_KSTEP
      } else {
        // word t of each register: channels 16t .. 16t+7 (low half), 16t+8 .. 16t+15 (high
        // half) of the chunk; step st takes crumbs 2st (k-slots 2t, 2t+1 = channels 16t + 2st,
        // 16t + 8 + 2st) and 2st + 1 (k-slots 2t+8, 2t+9); lane t's channels lie in group
        // 2s + (t >= 2), and the query operand is zero outside the column's group
        const uint32_t X = K2[2 * s], Y = K2[2 * s + 1], X10 = X >> 10, Y10 = Y >> 10;
#define FADE_K2STEP(ST)                                                                       \
  {                                                                                           \
    const uint32_t a0 = v_crumb<2 * ST>(X, X10), a1 = v_crumb<2 * ST>(Y, Y10),                \
                   a2 = v_crumb<2 * ST + 1>(X, X10), a3 = v_crumb<2 * ST + 1>(Y, Y10);        \
    _Pragma("unroll") for (int j = 0; j < NT; ++j)                                            \
        mma16816(cacc[j], a0, a1, a2, a3, qb[s][ST][j][0], qb[s][ST][j][1]);                  \
  }
        FADE_K2STEP(0) FADE_K2STEP(1) FADE_K2STEP(2) FADE_K2STEP(3)
#undef FADE_K2STEP
      }
      // column 2t = (head 4j+t, group 2s), column 2t+1 = (head 4j+t, group 2s+1)
      const float kl0 = h_lo(kw_lo[s]), kl1 = h_hi(kw_lo[s]);
      const float kh0 = h_lo(kw_hi[s]), kh1 = h_hi(kw_hi[s]);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        acc_s[j][0] = fmaf(cacc[j][0], kl0, acc_s[j][0]);
        acc_s[j][0] = fmaf(cacc[j][1], kl1, acc_s[j][0]);
        acc_s[j][1] = fmaf(cacc[j][2], kh0, acc_s[j][1]);
        acc_s[j][1] = fmaf(cacc[j][3], kh1, acc_s[j][1]);
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int h = 4 * j + t;
      const bool hv = h < G;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int tok = r0 + g + 8 * r;
        const bool tv = FULL || tok < nt;
        if (LOGITS && hv && tv) logit_row[(size_t)h * a.NS + tok] = acc_s[j][r] * a.inv_sqrt_d;
        const float v = hv ? acc_s[j][r] * c2 : 0.f;
        sc[mt][j][r] = tv ? v : -INFINITY;
      }
    }
  }
  // online softmax per head column; the warp holds at least one valid token, so the running
  // max is finite after this tile and masked tokens get probability exp2(-inf) = 0
  float alpha[NT];
  bool moved = false;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    float mx = sc[0][j][0];
#pragma unroll
    for (int mt = 0; mt < MmaShape<D, G, PQ>::MT; ++mt) mx = fmaxf(mx, fmaxf(sc[mt][j][0], sc[mt][j][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mn = fmaxf(m2[j], mx);
    alpha[j] = ex2(m2[j] - mn);   // 0 on the first tile (old max -inf)
    moved |= mn != m2[j];
    m2[j] = mn;
    float ps = 0.f;
#pragma unroll
    for (int mt = 0; mt < MmaShape<D, G, PQ>::MT; ++mt)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float pr = ex2(sc[mt][j][r] - mn);
        sc[mt][j][r] = pr;
        ps += pr;
      }
    lsum[j] = lsum[j] * alpha[j] + ps;
  }
  // rescale the accumulators only when some column's running max moved (warp-uniform)
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
  if constexpr (PQ) {
    // PQ-coded V: per M-tile the warp decodes its 16 tokens into its fp16 tile (one code byte,
    // one 8-byte centroid and one 8-byte store per (token, sub-space)), then reads the A
    // operand transposed with ldmatrix: row g of block (s, mm) is channel 64s + 16mm + g, row
    // g + 8 channel 64s + 16mm + g + 8. B operand: the probability, the same in both group
    // parity columns (a PQ row has no scales). Codes past the tile's tokens index real
    // centroids (finite) and meet probability 0.
    using PC = PqCfg<D>;
    constexpr int SUBS = PC::SUBS;
    const uint32_t vt_ld = vt + ((lane & 7) + 8 * (lane >> 4)) * PC::VT_ROW + ((lane >> 3) & 1) * 16;
#pragma unroll
    for (int mt = 0; mt < MmaShape<D, G, PQ>::MT; ++mt) {
      const int r0 = wr0 + mt * 16;
#pragma unroll kPqDecodeUnroll
      for (int i = lane; i < 16 * SUBS; i += 32) {
        const int tk = i / SUBS, sub = i % SUBS, r = r0 + tk;
        uint32_t off;
        if constexpr (D == 128)  // 32-byte rows under the 32-byte swizzle of the TMA copy
          off = r * Cfg::VROW + ((((sub >> 4) ^ (r >> 2)) & 1) << 4) + (sub & 15);
        else                     // 16-byte rows, no swizzle
          off = r * Cfg::VROW + sub;
        const uint32_t code = lds_u8(stage + Cfg::V_OFF + off);
        sts64(vt + tk * PC::VT_ROW + sub * 8, lds64(cbs + (code * SUBS + sub) * 8));
      }
      __syncwarp();
      uint32_t pb[NT][2];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        pb[j][0] = movm_t(h2_as_u32(__float2half2_rn(sc[mt][j][0])));
        pb[j][1] = movm_t(h2_as_u32(__float2half2_rn(sc[mt][j][1])));
      }
#pragma unroll
      for (int s = 0; s < NHALF; ++s)
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(vt_ld + (64 * s + 16 * mm) * 2, a0, a1, a2, a3);
#pragma unroll
          for (int j = 0; j < NT; ++j) mma16816(o[s][mm][j], a0, a1, a2, a3, pb[j][0], pb[j][1]);
        }
      __syncwarp();  // the tile is read before the next M-tile overwrites it
    }
  } else {
  // PV over the warp's M-tiles (16 tokens each = one MMA k-step). B operand: the probability
  // (fp16) times the V scale of the column's group (fp16 multiply), transposed into place.
#pragma unroll
  for (int mt = 0; mt < MmaShape<D, G, PQ>::MT; ++mt) {
    const int r0 = wr0 + mt * 16;
    uint32_t vw_lo[NHALF], vw_hi[NHALF];
    scale_words<D>(stage + lo_.vs + mt * 16 * Cfg::SROW * 2, vw_lo);
    scale_words<D>(stage + lo_.vs + (mt * 16 + 8) * Cfg::SROW * 2, vw_hi);
    if (!FULL) {
      // past the tile's tokens the scale rows may never have been copied: use 0 so that a
      // zero probability cannot meet a non-finite leftover
#pragma unroll
      for (int s = 0; s < NHALF; ++s) {
        vw_lo[s] = (r0 + g < nt) ? vw_lo[s] : 0u;
        vw_hi[s] = (r0 + g + 8 < nt) ? vw_hi[s] : 0u;
      }
    }
    uint32_t X[2 * NHALF];  // INT2: (tokens 0-7 | 8-15) x (channel half)
    if constexpr (VB == 2) {
      if constexpr (D == 128)
        ldsm_x4_t(stage + lo_.v[0] + mt * 16 * Cfg::VROW, X[0], X[1], X[2], X[3]);
      else
        ldsm_x2_t(stage + lo_.v[0] + mt * 16 * Cfg::VROW, X[0], X[1]);
    }
    __half2 pg[NT], pg8[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      pg[j] = __float2half2_rn(sc[mt][j][0]);
      pg8[j] = __float2half2_rn(sc[mt][j][1]);
    }
#pragma unroll
    for (int s = 0; s < NHALF; ++s) {
      uint32_t pb[NT][2];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        pb[j][0] = movm_t(h2_as_u32(__hmul2(pg[j], u32_as_h2(vw_lo[s]))));
        pb[j][1] = movm_t(h2_as_u32(__hmul2(pg8[j], u32_as_h2(vw_hi[s]))));
      }
      if constexpr (VB == 4) {
        // INT4: X4 = (chunk 2s | 2s+1) x (tokens 0-7 | 8-15), each register two tokens' 16-bit
        // word g (channels 4g .. 4g+3 of the chunk's group). M-tile mm = chunk 2s + mm / 2,
        // nibbles 2 (mm % 2) (rows g) and 2 (mm % 2) + 1 (rows g + 8): all 16 rows in one
        // quantisation group, whose parity column is the one kept
        uint32_t X4[4];
        ldsm_x4_t(stage + lo_.v[s] + mt * 16 * Cfg::VROW, X4[0], X4[1], X4[2], X4[3]);
        const uint32_t x08 = X4[0] >> 8, x18 = X4[1] >> 8, x28 = X4[2] >> 8, x38 = X4[3] >> 8;
#define FADE_PV4(MM, XA, XA8, XB, XB8)                                                      \
  {                                                                                         \
    const uint32_t a0 = k_pair<2 * (MM % 2)>(XA, XA8), a1 = k_pair<2 * (MM % 2) + 1>(XA, XA8); \
    const uint32_t a2 = k_pair<2 * (MM % 2)>(XB, XB8), a3 = k_pair<2 * (MM % 2) + 1>(XB, XB8); \
    _Pragma("unroll") for (int j = 0; j < NT; ++j)                                          \
        mma16816(o[s][MM][j], a0, a1, a2, a3, pb[j][0], pb[j][1]);                          \
  }
        FADE_PV4(0, X4[0], x08, X4[1], x18) FADE_PV4(1, X4[0], x08, X4[1], x18)
        FADE_PV4(2, X4[2], x28, X4[3], x38) FADE_PV4(3, X4[2], x28, X4[3], x38)
#undef FADE_PV4
      } else {
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
  }
}

// Position of a global middle tile in the schedule: row b, KV head h, tile within the unit.
struct SkPos {
  int b, h, tile;
};
__device__ __forceinline__ SkPos sk_locate(const StreamK& k, int g) {
  if (g >= k.row_start[k.B]) return SkPos{k.B, 0, 0};
  int lo = 0, hi = k.B - 1;  // the last row whose start is <= g (rows without tiles are skipped)
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (k.row_start[mid] <= g) lo = mid; else hi = mid - 1;
  }
  const int rt = sk_row_tiles(k, lo), off = g - k.row_start[lo];
  return SkPos{lo, off / rt, off % rt};
}
// Move `run` tiles forward, where the run ends at or before the end of the current unit.
__device__ __forceinline__ void sk_advance(const StreamK& k, SkPos& p, int run) {
  p.tile += run;
  if (p.tile < sk_row_tiles(k, p.b)) return;
  p.tile = 0;
  if (++p.h < k.H) return;
  p.h = 0;
  ++p.b;
  while (p.b < k.B && sk_row_tiles(k, p.b) == 0) ++p.b;
}
// Segments (maximal runs inside one unit) among n tiles starting at p.
__device__ __forceinline__ int sk_count_segments(const StreamK& k, SkPos p, int n) {
  int count = 0;
  while (n > 0) {
    const int run = min(n, sk_row_tiles(k, p.b) - p.tile);
    ++count;
    n -= run;
    sk_advance(k, p, run);
  }
  return count;
}

// Bounded wait that also gives up as soon as another warp of the CTA has raised `abort`.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity, int32_t* status,
                                                   int code, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (clock64() - t0 > kWaitCycles) {
      atomicCAS(status, 0, code);
      *abort = 1;
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Persistent decode attention under a stream-K schedule: CTA c first takes the FP16-tier items
// of units c, c + P, ... (split 0), then its contiguous run of middle tiles [cta_start[c],
// cta_start[c+1]) in global tile order, which may cross unit boundaries: every maximal run
// inside one unit is a segment whose partial goes to split 1 + k (k = the CTA's rank among the
// CTAs touching that unit). Every item occupies one or more stages of the ring: the producer
// warp copies each stage's code and scale rows (TMA) and, with the item's first stage, the
// item's query rows (bulk copy); it writes what the stage holds into the stage info before
// arming it. The producer therefore runs ahead across item boundaries and the consumers never
// wait on global memory for metadata or queries. Consumer warps merge their partials in shared
// memory at the end of each item (named barrier 1, consumers only) and write its partial.
template <int D, int G, bool PQ, int VB, int KB>
__global__ void __launch_bounds__(MmaShape<D, G, PQ>::THREADS, MmaShape<D, G, PQ>::MINB)
attn_mid_mma_kernel(const __grid_constant__ CUtensorMap tk0, const __grid_constant__ CUtensorMap tk1,
                    const __grid_constant__ CUtensorMap tv0, const __grid_constant__ CUtensorMap tv1,
                    const __grid_constant__ CUtensorMap tsk, const __grid_constant__ CUtensorMap tsv,
                    const __grid_constant__ CUtensorMap trk, const __grid_constant__ CUtensorMap trv,
                    MmaArgs a, const __grid_constant__ StreamK sk) {
  using Cfg = MmaCfgOf<D, G, PQ, VB, KB>;
  constexpr int kConsumers = MmaShape<D, G, PQ>::CONS;
  constexpr int NT = (2 * G + 7) / 8;    // 8-column n-tiles of (head, group parity)
  constexpr int NHALF = D / 64;          // 64-channel halves (accumulator sets)
  constexpr int NSTAGE = Cfg::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, kept as an offset into the __shared__ array so that every access
  // through it compiles to a shared-memory (not a generic) load or store
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + Cfg::BAR_OFF;          // NSTAGE x 8 bytes
  const uint32_t bar_empty = bar_full + NSTAGE * 8;
  int* info = reinterpret_cast<int*>(smem + Cfg::INFO_OFF);  // [NSTAGE][kInfo]
  float* wm = reinterpret_cast<float*>(smem + Cfg::MERGE_OFF);  // [kConsumers][8]
  float* wl = wm + 64;                                          // [kConsumers][8]
  float* wf = wl + 64;                                          // [G][kConsumers]
  float* wo = wf + 64;                                  // [kConsumers][G][WO_ROW]
  static_assert(kConsumers * G <= 64, "warp-merge arrays of 64 (warp, head) entries");
  constexpr int WR = Cfg::WO_ROW;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int units = a.B * a.H;
  const bool f16_staged = a.f16_rreg > 0;  // FP16 tiers through the ring (the host decides)
  // this CTA's work: FP16 items of units c, c + P, ..., then middle tiles [g0, g1)
  const int cta = blockIdx.x, P = gridDim.x;
  const int n16 = cta < units ? (units - cta + P - 1) / P : 0;
  const int g0 = sk.cta_start[cta], g1 = sk.cta_start[cta + 1];
  const SkPos p0 = sk_locate(sk, g0);
  const int nseg = sk_count_segments(sk, p0, g1 - g0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kConsumers);
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if constexpr (PQ) {  // the layer's codebook, transposed to centroid-major, once per CTA
    constexpr int SUBS = PqCfg<D>::SUBS;
    const uint2* src = reinterpret_cast<const uint2*>(a.pq_cb);
    uint2* dst = reinterpret_cast<uint2*>(smem + PqCfg<D>::CB_OFF);
    for (int e = threadIdx.x; e < SUBS * kPqCentroids; e += blockDim.x)
      dst[(e % kPqCentroids) * SUBS + e / kPqCentroids] = src[e];
  }
  __syncthreads();
  volatile int* abort = &s_abort;
  // when launched as a programmatic dependent of the kernel before it (the append of the new
  // token; a layer with fewer middle tiles than CTAs): everything above reads only the schedule
  // and this CTA's shared memory; wait here until that grid has completed and its writes
  // (counts, ring rows, rotated queries) are visible (a no-op otherwise)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the combine kernel that follows is a programmatic dependent: let it be scheduled now (its
  // CTAs take SM slots as this grid's CTAs exit and wait on the device for this grid's end)
  asm volatile("griddepcontrol.launch_dependents;");

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      // one item: n_stage stages of unit `unit`; middle tiles tile0 .. tile0 + n_stage - 1
      auto issue_item = [&](int unit, int split, int tile0, int n_stage) {
        const int b = unit / a.H, hk = unit % a.H;
        const int32_t* m = a.meta + unit * kF;
        const int n_mid = m[FADE_META_N_MID], cur = m[FADE_META_CUR];
        const CUtensorMap* mk = cur ? &tk1 : &tk0;
        const CUtensorMap* mv = cur ? &tv1 : &tv0;
        const uint16_t* ksg = cur ? a.ks[1] : a.ks[0];
        const uint16_t* vsg = cur ? a.vs[1] : a.vs[0];
        for (int it = 0; it < n_stage; ++it) {
          const int s = issued % NSTAGE;
          if (issued >= NSTAGE &&
              !mbar_wait_or_abort(bar_empty + 8 * s, ((issued / NSTAGE) & 1) ^ 1, a.status, 2,
                                  abort))
            return false;
          const int tile = tile0 + it;
          int nt = split > 0 ? min(kTileTok, n_mid - tile * kTileTok) : 0;  // <= 0: q only
          if (FADE_DEBUG && nt > 0 && tile * kTileTok + nt > a.C) {  // past the unit's slots
            record_status(a.status, kCheckAttnTile);
            nt = 0;
          }
          int* inf = info + s * kInfo;
          inf[kInfoUnit] = unit;
          inf[kInfoSplit] = split;
          inf[kInfoNt] = max(nt, 0);
          inf[kInfoLast] = it == n_stage - 1;
          inf[kInfoTok0] = tile * kTileTok;
          inf[kInfoSink] = m[FADE_META_N_SINK];
          inf[kInfoRec] = m[FADE_META_N_RECENT];
          inf[kInfoHead] = m[FADE_META_HEAD];
          const uint32_t stage = sbase + s * Cfg::STAGE;
          // scale rows copied: rounded up so the copy is a multiple of 16 bytes (it stays inside
          // the unit: rows start at multiples of 4 and the slot stride is a multiple of 64)
          constexpr int kAlign = 16 / (Cfg::SROW * 2);
          const int ns = (max(nt, 0) + kAlign - 1) / kAlign * kAlign;
          uint32_t bytes = 0;
          // (PQ-coded V has no scale rows: only the K scales are copied)
          if (nt > 0) bytes += kTileTok * (Cfg::KROW + Cfg::VROW) + (PQ ? 1u : 2u) * ns * Cfg::SROW * 2;
          if (it == 0) bytes += G * D * 2;
          if (split == 0 && f16_staged) bytes += (a.S + a.W) * D * 2;
          mbar_expect_tx(bar_full + 8 * s, bytes);
          if (split == 0 && f16_staged) {  // K (first stage) or V rows: sinks, then the ring
            // each 64-channel half of the rows into its own region, 128-byte swizzled: the
            // sink region of half h at h * sreg, the ring region of half h at
            // NHALF * sreg + h * rreg (every region 1024-byte aligned)
            const CUtensorMap* ms = it == 0 ? &tsk : &tsv;
            const CUtensorMap* mr = it == 0 ? &trk : &trv;
#pragma unroll
            for (int hh = 0; hh < NHALF; ++hh) {
              if (a.S > 0)
                tma_load_2d(stage + hh * a.f16_sreg, ms, 64 * hh, unit * a.S, bar_full + 8 * s);
              tma_load_2d(stage + NHALF * a.f16_sreg + hh * a.f16_rreg, mr, 64 * hh,
                          unit * a.W, bar_full + 8 * s);
            }
          }
          if (nt > 0) {
            const size_t r = (size_t)unit * a.C + (size_t)tile * kTileTok;
            tma_load_2d(stage + Cfg::K_OFF, mk, 0, (int)r, bar_full + 8 * s);
            tma_load_2d(stage + Cfg::V_OFF, mv, 0, (int)r, bar_full + 8 * s);
            bulk_load_1d(stage + Cfg::KS_OFF, ksg + r * Cfg::SROW, ns * Cfg::SROW * 2,
                         bar_full + 8 * s);
            if (!PQ)
              bulk_load_1d(stage + Cfg::VS_OFF, vsg + r * Cfg::SROW, ns * Cfg::SROW * 2,
                           bar_full + 8 * s);
          }
          if (it == 0)
            bulk_load_1d(stage + Cfg::Q_OFF, a.q + (size_t)(b * a.Hq + hk * G) * D, G * D * 2,
                         bar_full + 8 * s);
          ++issued;
        }
        return true;
      };
      bool go = true;
      // every unit's partial count for the combine: 1 (split 0) for a unit without middle
      // tiles, written with its FP16 item; else 2 + k, written by the CTA (rank k) that holds
      // the unit's last tile
      for (int u = cta; u < units && go; u += P) {
        if (sk_row_tiles(sk, u / a.H) == 0) a.seg_count[u] = 1;
        go = issue_item(u, 0, 0, f16_staged ? 2 : 1);
      }
      SkPos pos = p0;
      for (int g = g0; g < g1 && go;) {
        const int rt = sk_row_tiles(sk, pos.b);
        const int run = min(g1 - g, rt - pos.tile);
        // this CTA's rank among the CTAs holding tiles of the unit
        const int k = sk_nonempty(sk, sk_cta_of(sk, g - pos.tile), cta - 1);
        if (pos.tile + run == rt) a.seg_count[pos.b * a.H + pos.h] = 2 + k;
        go = issue_item(pos.b * a.H + pos.h, 1 + k, pos.tile, run);
        g += run;
        sk_advance(sk, pos, run);
      }
      // never leave the CTA with copies in flight: wait (bounded) for the last issued stages
      for (int k = max(0, issued - NSTAGE); k < issued; ++k)
        mbar_wait(bar_full + 8 * (k % NSTAGE), (k / NSTAGE) & 1, a.status, 3);
    }
    // the producer warp takes part in no further barrier
    return;
  }

  // ------------------------------------------------------------ consumers
  const float c2 = a.inv_sqrt_d * kLog2e;
  const int wr0 = warp * MmaShape<D, G, PQ>::WARP_TOK;
  const LaneOffsets<D, VB> lo_ = lane_offsets<D, G, PQ, VB, KB>(wr0, lane);
  const bool want_logits = a.logits != nullptr;
  // PQ-coded V: this warp's decoded V tile and the codebook (unused otherwise)
  const uint32_t vt = sbase + PqCfg<D>::VT_OFF + warp * 16 * PqCfg<D>::VT_ROW;
  const uint32_t cbs = sbase + PqCfg<D>::CB_OFF;
  int used = 0;  // stages consumed so far (the producer's `issued` sequence)
  // the same number of items in every consumer warp (and so the same barriers), whatever waits
  // may fail: the count comes from the schedule, the rest from the stage info
  for (int item = 0; item < n16 + nseg; ++item) {
    int s_ = used % NSTAGE;
    bool ok = !*abort && mbar_wait_or_abort(bar_full + 8 * s_, (used / NSTAGE) & 1, a.status, 1,
                                            abort);
    const int* inf = info + s_ * kInfo;
    const int unit = ok ? inf[kInfoUnit] : 0, split = ok ? inf[kInfoSplit] : 0;
    const bool write_ok = ok;
    const int b = unit / a.H, hk = unit % a.H, hq0 = hk * G;
    const uint16_t* qs = reinterpret_cast<const uint16_t*>(smem + s_ * Cfg::STAGE + Cfg::Q_OFF);
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

    if (split == 0 && kF16Mma && f16_staged) {
      // ---------------------------------------------------------- FP16 tiers (tensor cores)
      // the item's two stages hold the K rows and the V rows: sinks (rows 0..S-1) then the
      // ring slots (rows S..S+W-1), fp16. Warp w takes the 16-row M-tiles w, w + kConsumers,
      // ...: QK^T with the K rows as A operand (ldmatrix) and the queries as B (column n =
      // head n), softmax per head column, PV with V^T as A (ldmatrix.trans) and the
      // probabilities as B (movmatrix). Rows that hold no token (unfilled sinks, empty ring
      // slots, padding past the staged rows) get logit -inf; V past the staged rows is zeroed.
      const int n_sink = ok ? inf[kInfoSink] : 0, n_rec = ok ? inf[kInfoRec] : 0;
      const int head_slot = ok ? inf[kInfoHead] : 0;
      const uint32_t st_k = sbase + s_ * Cfg::STAGE;
      const int s_v = (used + 1) % NSTAGE;
      const bool ok_v = ok && !*abort &&
                        mbar_wait_or_abort(bar_full + 8 * s_v, ((used + 1) / NSTAGE) & 1,
                                           a.status, 1, abort);
      const uint32_t st_v = sbase + s_v * Cfg::STAGE;
      const int R = a.S + a.W;
      const int nmt = (ok && ok_v) ? (R + 15) / 16 : 0;
      uint32_t qf[D / 16][2];  // B operand: (channels 16kk + 2t, +1 | +8, +9) of head g
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const bool hv = ok && g < G;
        const uint32_t qa = st_k + Cfg::Q_OFF + (g * D + 16 * kk + 2 * t) * 2;
        qf[kk][0] = hv ? lds32(qa) : 0u;
        qf[kk][1] = hv ? lds32(qa + 16) : 0u;
      }
      float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
      float of[NHALF][4][4];
#pragma unroll
      for (int s = 0; s < NHALF; ++s)
#pragma unroll
        for (int mm = 0; mm < 4; ++mm)
#pragma unroll
          for (int e = 0; e < 4; ++e) of[s][mm][e] = 0.f;
      for (int mt = warp; mt < nmt; mt += kConsumers) {
        const int r0 = mt * 16;
        float cacc[4] = {0.f, 0.f, 0.f, 0.f};
        // this lane's row in its region (sinks or ring) and the 128-byte swizzle of its
        // 16-byte chunks: chunk c of row rr sits at chunk c ^ (rr & 7)
        uint32_t k_row, k_reg, k_y;
        {
          const int r = r0 + (lane & 7) + 8 * ((lane >> 3) & 1);
          const bool sink = r < a.S;
          const int rr = sink ? r : r - a.S;
          k_reg = sink ? a.f16_sreg : a.f16_rreg;
          k_row = st_k + (sink ? 0u : NHALF * a.f16_sreg) + rr * 128;
          k_y = (uint32_t)((lane >> 4) ^ (rr & 7));
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(k_row + (kk >> 2) * k_reg + ((((2 * kk) & 7) ^ k_y) << 4), a0, a1, a2, a3);
          mma16816(cacc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        }
        // logits of rows r0 + g + 8e for the head columns 2t + cc
        float sc[2][2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = r0 + g + 8 * e;
          const bool tv = r < a.S ? r < n_sink
                                  : (r < R && (r - a.S - head_slot + a.W) % a.W < n_rec);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int h = 2 * t + cc;
            const bool v = tv && h < G;
            if (want_logits && v)
              a.logits[(size_t)(b * a.Hq + hq0 + h) * a.NS + (r < a.S ? r : a.C + r)] =
                  cacc[2 * e + cc] * a.inv_sqrt_d;
            sc[e][cc] = v ? cacc[2 * e + cc] * c2 : -INFINITY;
          }
        }
        float al[2];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float mx = fmaxf(sc[0][cc], sc[1][cc]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(mrun[cc], mx);
          const float mref = mn == -INFINITY ? 0.f : mn;  // no valid token yet: all terms 0
          al[cc] = ex2(mrun[cc] - mref);
          mrun[cc] = mn;
          sc[0][cc] = ex2(sc[0][cc] - mref);
          sc[1][cc] = ex2(sc[1][cc] - mref);
          lrun[cc] = lrun[cc] * al[cc] + sc[0][cc] + sc[1][cc];
        }
#pragma unroll
        for (int s = 0; s < NHALF; ++s)
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {
            of[s][mm][0] *= al[0];
            of[s][mm][1] *= al[1];
            of[s][mm][2] *= al[0];
            of[s][mm][3] *= al[1];
          }
        const uint32_t pb0 = movm_t(h2_as_u32(__floats2half2_rn(sc[0][0], sc[0][1])));
        const uint32_t pb1 = movm_t(h2_as_u32(__floats2half2_rn(sc[1][0], sc[1][1])));
        // V^T halves of tokens past the staged rows are zeroed (the stage may hold anything
        // there); masks for tokens (2t, 2t+1) and (2t+8, 2t+9) of the M-tile
        const int tk = r0 + 2 * t;
        const uint32_t mlo = (tk < R ? 0xFFFFu : 0u) | (tk + 1 < R ? 0xFFFF0000u : 0u);
        const uint32_t mhi = (tk + 8 < R ? 0xFFFFu : 0u) | (tk + 9 < R ? 0xFFFF0000u : 0u);
        uint32_t v_row, v_reg, v_y;
        {
          const int r = r0 + (lane & 7) + 8 * (lane >> 4);
          const bool sink = r < a.S;
          const int rr = sink ? r : r - a.S;
          v_reg = sink ? a.f16_sreg : a.f16_rreg;
          v_row = st_v + (sink ? 0u : NHALF * a.f16_sreg) + rr * 128;
          v_y = (uint32_t)(((lane >> 3) & 1) ^ (rr & 7));
        }
#pragma unroll
        for (int s = 0; s < NHALF; ++s)
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(v_row + s * v_reg + (((2 * mm) ^ v_y) << 4), a0, a1, a2, a3);
            mma16816(of[s][mm], a0 & mlo, a1 & mlo, a2 & mhi, a3 & mhi, pb0, pb1);
          }
      }
      __syncwarp();
      if (lane == 0) {  // both stages of the item are read: release them
        if (ok) mbar_arrive(bar_empty + 8 * s_);
        if (ok_v) mbar_arrive(bar_empty + 8 * s_v);
      }
      used += 2;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {  // the head columns' mass over the warp's rows
        lrun[cc] += __shfl_xor_sync(0xffffffffu, lrun[cc], 4);
        lrun[cc] += __shfl_xor_sync(0xffffffffu, lrun[cc], 8);
        lrun[cc] += __shfl_xor_sync(0xffffffffu, lrun[cc], 16);
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int h = 2 * t + cc;
        if (h < G) {
          if (g == 0) {
            wm[warp * 8 + h] = mrun[cc];
            wl[warp * 8 + h] = lrun[cc];
          }
#pragma unroll
          for (int s = 0; s < NHALF; ++s)
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
              const int c = 64 * s + 16 * mm + g;
              wo[(warp * G + h) * WR + c] = of[s][mm][cc];
              wo[(warp * G + h) * WR + c + 8] = of[s][mm][2 + cc];
            }
        }
      }
    } else if (split == 0) {
      // ---------------------------------------------------------- FP16 tiers (CUDA cores)
      // warp w takes tokens w, w + kConsumers, ...; lane l holds channels l*CPL .. +CPL-1
      constexpr int CPL = D / 32;
      float qr[G][CPL], acc[G][CPL], mm_[G], ll[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        mm_[h] = -INFINITY;
        ll[h] = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          qr[h][c] = ok ? __half2float(__ushort_as_half(qs[h * D + lane * CPL + c])) : 0.f;
          acc[h][c] = 0.f;
        }
      }
      const int n_sink = ok ? inf[kInfoSink] : 0, n_rec = ok ? inf[kInfoRec] : 0;
      const int head_slot = ok ? inf[kInfoHead] : 0;
      const uint32_t st_k = sbase + s_ * Cfg::STAGE;  // K rows (staged case)
      uint32_t st_v = 0;
      int s_v = 0;
      bool ok_v = false;
      if (f16_staged) {  // the V rows arrive in the item's second stage
        s_v = (used + 1) % NSTAGE;
        ok_v = ok && !*abort &&
               mbar_wait_or_abort(bar_full + 8 * s_v, ((used + 1) / NSTAGE) & 1, a.status, 1,
                                  abort);
        st_v = sbase + s_v * Cfg::STAGE;
      } else {
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(bar_empty + 8 * s_);  // q is in registers
        ++used;
      }
      const int n_tok = (!f16_staged || ok_v) ? n_sink + n_rec : 0;
      // two tokens per pass (u and u + kConsumers): both rows are loaded before either is used
      for (int u0 = warp; u0 < n_tok; u0 += 2 * kConsumers) {
        float kv[2][CPL], vv[2][CPL];
        int lidx[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int u = min(u0 + e * kConsumers, n_tok - 1);  // a duplicate is masked below
          const bool is_sink = u < n_sink;
          const int slot = is_sink ? u : (head_slot + u - n_sink) % a.W;
          if (f16_staged) {
            const uint32_t off = (is_sink ? u : a.S + slot) * D * 2 + lane * CPL * 2;
            lds_f16_lane<CPL>(st_k + off, kv[e]);
            lds_f16_lane<CPL>(st_v + off, vv[e]);
          } else {
            const size_t row =
                is_sink ? ((size_t)unit * a.S + u) * D : ((size_t)unit * a.W + slot) * D;
            load_f16_lane<CPL>((is_sink ? a.sink_k : a.rec_k) + row + lane * CPL, kv[e]);
            load_f16_lane<CPL>((is_sink ? a.sink_v : a.rec_v) + row + lane * CPL, vv[e]);
          }
          lidx[e] = is_sink ? u : a.S + a.C + slot;
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (u0 + e * kConsumers >= n_tok) break;  // warp-uniform
          float d[G];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            d[h] = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) d[h] = fmaf(qr[h][c], kv[e][c], d[h]);
          }
          warp_allreduce<G>(d, lane);
          if (want_logits && lane < G)
            a.logits[(size_t)(b * a.Hq + hq0 + lane) * a.NS + lidx[e]] =
                pick(d, lane) * a.inv_sqrt_d;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float s2 = d[h] * c2;
            const float mn = fmaxf(mm_[h], s2);
            const float al = ex2(mm_[h] - mn);   // 0 when the old max is -inf
            const float p = ex2(s2 - mn);
            ll[h] = ll[h] * al + p;
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[h][c] = fmaf(p, vv[e][c], acc[h][c] * al);
            mm_[h] = mn;
          }
        }
      }
      if (f16_staged) {  // both stages of the item are read: release them
        __syncwarp();
        if (lane == 0) {
          if (ok) mbar_arrive(bar_empty + 8 * s_);
          if (ok_v) mbar_arrive(bar_empty + 8 * s_v);
        }
        used += 2;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (lane == 0) {
          wm[warp * 8 + h] = mm_[h];
          wl[warp * 8 + h] = ll[h];
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) wo[(warp * G + h) * WR + lane * CPL + c] = acc[h][c];
      }
    } else {
      // ---------------------------------------------------------- packed middle tier (MMA)
      // query B operand: column n of n-tile j = (head 4j + n/2, parity n%2); thread (g, t)
      // holds column g, k-slots {2t, 2t+1} (group 2s of half s) and {2t+8, 2t+9} (group 2s+1)
      // one 16-byte load gives channels 8t .. 8t+7 of the lane's group; byte permutes pair
      // them as (c, c+4) for the four k-steps
      uint32_t qb[NHALF][4][NT][2];
      const uint32_t qs_addr = sbase + s_ * Cfg::STAGE + Cfg::Q_OFF;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int h = 4 * j + g / 2, par = g & 1;
        const bool valid = ok && h < G;
#pragma unroll
        for (int s = 0; s < NHALF; ++s) {
          if constexpr (KB == 4) {
            const uint4 v = valid ? lds128(qs_addr + (h * D + 64 * s + 32 * par + 8 * t) * 2)
                                  : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t pk[4] = {prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u),
                                    prmt(v.y, v.w, 0x5410u), prmt(v.y, v.w, 0x7632u)};
#pragma unroll
            for (int kp = 0; kp < 4; ++kp) {
              qb[s][kp][j][0] = par == 0 ? pk[kp] : 0u;   // group 2s
              qb[s][kp][j][1] = par == 1 ? pk[kp] : 0u;   // group 2s+1
            }
          } else {
            // INT2 K: lane t's k-slots are channels 64s + 16t .. 64s + 16t + 15 (group 2s + (t >=
            // 2)); step st pairs channels (2st, 8 + 2st) and (2st + 1, 9 + 2st) of them
            const bool mine = valid && par == (t >= 2 ? 1 : 0);
            const uint32_t qa = qs_addr + (h * D + 64 * s + 16 * t) * 2;
            const uint4 lo = mine ? lds128(qa) : make_uint4(0u, 0u, 0u, 0u);
            const uint4 hi = mine ? lds128(qa + 16) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int st = 0; st < 4; ++st) {
              qb[s][st][j][0] = prmt(w[st], w[4 + st], 0x5410u);
              qb[s][st][j][1] = prmt(w[st], w[4 + st], 0x7632u);
            }
          }
        }
      }
      float* logit_base =
          want_logits ? a.logits + (size_t)(b * a.Hq + hq0) * a.NS + a.S : nullptr;
      while (true) {
        const int nt = ok ? inf[kInfoNt] : 0;
        const bool last = ok ? inf[kInfoLast] != 0 : true;
        const uint32_t stage = sbase + s_ * Cfg::STAGE;
        float* logit_row = want_logits ? logit_base + (ok ? inf[kInfoTok0] : 0) : nullptr;
        if (ok) {
          if (want_logits) {
            if (nt == kTileTok)
              consume_tile<D, G, true, true, PQ, VB, KB>(a, stage, lo_, nt, wr0, lane, qb, m2, lsum, o,
                                             c2, logit_row, vt, cbs);
            else if (wr0 < nt)
              consume_tile<D, G, false, true, PQ, VB, KB>(a, stage, lo_, nt, wr0, lane, qb, m2, lsum, o,
                                              c2, logit_row, vt, cbs);
          } else {
            if (nt == kTileTok)
              consume_tile<D, G, true, false, PQ, VB, KB>(a, stage, lo_, nt, wr0, lane, qb, m2, lsum, o,
                                              c2, logit_row, vt, cbs);
            else if (wr0 < nt)
              consume_tile<D, G, false, false, PQ, VB, KB>(a, stage, lo_, nt, wr0, lane, qb, m2, lsum, o,
                                               c2, logit_row, vt, cbs);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_empty + 8 * s_);
          ++used;
        }
        if (last) break;
        s_ = used % NSTAGE;
        ok = !*abort && mbar_wait_or_abort(bar_full + 8 * s_, (used / NSTAGE) & 1, a.status, 1,
                                           abort);
        inf = info + s_ * kInfo;
      }
      // total probability mass of each head over the warp's tokens (lanes sharing t)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        lsum[j] += __shfl_xor_sync(0xffffffffu, lsum[j], 4);
        lsum[j] += __shfl_xor_sync(0xffffffffu, lsum[j], 8);
        lsum[j] += __shfl_xor_sync(0xffffffffu, lsum[j], 16);
      }
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
              if constexpr (PQ) {  // rows g, g + 8 = channels 64s + 16mm + g (+ 8); both
                                   // parity columns carry the same probability
                const int c = 64 * s + 16 * mm + g;
                wo[(warp * G + h) * WR + c] = o[s][mm][j][0];
                wo[(warp * G + h) * WR + c + 8] = o[s][mm][j][2];
              } else if constexpr (VB == 4) {  // rows g, g + 8 = nibbles 2 (mm % 2) (+ 1) of
                                                // word g of group 2s + mm / 2: its parity kept
                const int c = 64 * s + 32 * (mm >> 1) + 4 * g + 2 * (mm & 1);
                wo[(warp * G + h) * WR + c] = o[s][mm][j][mm >> 1];
                wo[(warp * G + h) * WR + c + 1] = o[s][mm][j][2 + (mm >> 1)];
              } else {
                const int c = 64 * s + 8 * g + 2 * mm;
                wo[(warp * G + h) * WR + c] = gsel ? o[s][mm][j][1] : o[s][mm][j][0];
                wo[(warp * G + h) * WR + c + 1] = gsel ? o[s][mm][j][3] : o[s][mm][j][2];
              }
            }
        }
      }
    }
    // ------------------------------------------------------------ merge the consumer warps
    consumer_bar<kConsumers>();
    const size_t pbase = ((size_t)(b * a.Hq + hq0)) * a.nsplit + split;
    if (warp == 0) {
      // entry e = base + lane is (head h, warp w) = (e / kConsumers, e % kConsumers): head h's
      // max over the warps, the weight 2^(m_w - M) of warp w, and the weighted mass, reduced
      // across the w lanes (whole heads per pass of 32 entries: kConsumers divides 32)
#pragma unroll
      for (int base = 0; base < G * kConsumers; base += 32) {
        const int e = base + lane;
        const int h = e / kConsumers, w = e % kConsumers;
        const bool act = e < G * kConsumers;
        const float mw = act ? wm[w * 8 + h] : -INFINITY;
        float M = mw;
#pragma unroll
        for (int o = kConsumers / 2; o; o >>= 1)
          M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
        float L = act ? wl[w * 8 + h] * f : 0.f;
#pragma unroll
        for (int o = kConsumers / 2; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (act) wf[h * kConsumers + w] = f;
        if (act && w == 0 && write_ok) {
          a.part_ml[(pbase + (size_t)h * a.nsplit) * 2] = M * kLn2;  // natural-log units
          a.part_ml[(pbase + (size_t)h * a.nsplit) * 2 + 1] = L;
        }
      }
    }
    consumer_bar<kConsumers>();
    for (int i = threadIdx.x; i < G * D; i += kConsumers * 32) {
      const int h = i / D, c = i % D;
      float O = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w)
        O = fmaf(wo[(w * G + h) * WR + c], wf[h * kConsumers + w], O);
      if (write_ok) a.part_acc[(pbase + (size_t)h * a.nsplit) * D + c] = O;
    }
    consumer_bar<kConsumers>();  // the merge area is rewritten by the next item
  }
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

// 2D map over fp16 rows of D channels ([rows][D]), boxes of 64 channels (128 bytes) x box_rows
// rows under the 128-byte swizzle: one box fills one region of staged FP16-tier rows.
fade_status_t encode_f16_rows(CUtensorMap* m, const void* base, unsigned long long rows, int D,
                              int box_rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return set_error(FADE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {(cuuint64_t)D, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(FADE_ERR_CUDA, "cuTensorMapEncodeTiled (fp16 rows) failed (%d)", (int)r);
  return FADE_OK;
}

// Tensor maps by their full set of inputs: a map holds only the base address, the sizes,
// strides, box and swizzle, so equal inputs give an equal map, and encoding is host work on
// every call otherwise. Bounded: cleared when it reaches kMapCacheMax entries.
struct MapKey {
  int dev;
  const void* base;
  unsigned long long rows;
  int inner;     // code rows: bytes per row; fp16 rows: channels
  int box_rows;  // fp16 rows only
  int kind;      // 0: code rows, 1: fp16 rows
  bool operator==(const MapKey& o) const {
    return dev == o.dev && base == o.base && rows == o.rows && inner == o.inner &&
           box_rows == o.box_rows && kind == o.kind;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    size_t h = std::hash<const void*>()(k.base);
    for (unsigned long long v : {(unsigned long long)k.dev, k.rows, (unsigned long long)k.inner,
                                 (unsigned long long)k.box_rows, (unsigned long long)k.kind})
      h = h * 1000003u ^ std::hash<unsigned long long>()(v);
    return h;
  }
};
constexpr size_t kMapCacheMax = 8192;
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

fade_status_t cached_map(CUtensorMap* out, const void* base, unsigned long long rows, int inner,
                         int box_rows, int kind) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  const MapKey k{dev, base, rows, inner, box_rows, kind};
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    const auto it = g_maps.find(k);
    if (it != g_maps.end()) {
      *out = it->second;
      return FADE_OK;
    }
  }
  const fade_status_t s = kind == 0 ? encode_rows(out, base, rows, inner)
                                    : encode_f16_rows(out, base, rows, inner, box_rows);
  if (s) return s;
  std::lock_guard<std::mutex> lk(g_map_mu);
  if (g_maps.size() >= kMapCacheMax) g_maps.clear();
  g_maps.emplace(k, *out);
  return FADE_OK;
}

template <int D, int G, bool PQ, int VB, int KB>
fade_status_t launch_mma(const fade_config_t* c, const fade_layer_t* L, MmaArgs a,
                         const StreamK& sk, cudaStream_t st) {
  using Cfg = MmaCfgOf<D, G, PQ, VB, KB>;
  constexpr int kSmem = PQ ? PqCfg<D>::SMEM : Cfg::SMEM;
  // the resident CTAs (each with 1 KB reserved by the system) fit the 228 KB of an SM
  static_assert(kSmem <= 227 * 1024 &&
                    MmaShape<D, G, PQ>::MINB * (kSmem + 1024) <= 228 * 1024,
                "shared memory of the resident CTAs");
  constexpr int NH = D / 64;
  const unsigned long long units = (unsigned long long)c->batch * c->num_kv_heads;
  const unsigned long long rows = units * a.C;
  CUtensorMap tk[2], tv[2];
  fade_status_t s;
  for (int i = 0; i < 2; ++i) {
    if ((s = cached_map(&tk[i], L->mid_k_codes[i], rows, Cfg::KROW, 0, 0))) return s;
    if ((s = cached_map(&tv[i], L->mid_v_codes[i], rows, Cfg::VROW, 0, 0))) return s;
  }
  // the FP16 tiers of an item go through the ring when their swizzled regions (1024-byte
  // aligned, one per 64-channel half of the sinks and of the ring), plus 16 rows of reads
  // past the last one (the padding of the last 16-row M-tile), fit before the query rows
  const int S = c->n_sink, W = c->recent_window;
  const int sreg = S > 0 ? (S * 128 + 1023) / 1024 * 1024 : 0;
  const int rreg = (W * 128 + 1023) / 1024 * 1024;
  const bool staged = kF16Mma && S <= 256 && W <= 256 && NH * (sreg + rreg) + 16 * 128 <= Cfg::Q_OFF;
  a.f16_sreg = staged ? sreg : 0;
  a.f16_rreg = staged ? rreg : 0;
  CUtensorMap tsk, tsv, trk, trv;
  if (staged) {
    if ((s = cached_map(&trk, L->recent_k, units * W, D, W, 1))) return s;
    if ((s = cached_map(&trv, L->recent_v, units * W, D, W, 1))) return s;
    if (S > 0) {
      if ((s = cached_map(&tsk, L->sink_k, units * S, D, S, 1))) return s;
      if ((s = cached_map(&tsv, L->sink_v, units * S, D, S, 1))) return s;
    } else {  // no sinks: never read
      tsk = trk;
      tsv = trv;
    }
  } else {  // not staged: never read
    tsk = tsv = trk = trv = tk[0];
  }
  auto kern = attn_mid_mma_kernel<D, G, PQ, VB, KB>;
  // the shared-memory opt-in, once per device for this instantiation (devices 0..63)
  static std::atomic<unsigned long long> smem_set{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 64;
  if (dev >= 64 || !((smem_set.load() >> dev) & 1ull)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
        cudaSuccess)
      return launch_status("fade_decode_attention (middle tier) shared-memory opt-in");
    if (dev < 64) smem_set.fetch_or(1ull << dev);
  }
  // persistent grid: the schedule's CTAs (as many as fit on the device at once). A layer with
  // fewer middle tiles than CTAs is bound by launch latency: its kernel is a programmatic
  // dependent of the kernel before it on the stream (its prologue overlaps that kernel's end)
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(sk.P);
  lc.blockDim = dim3(MmaShape<D, G, PQ>::THREADS);
  lc.dynamicSmemBytes = kSmem;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = sk.row_start[sk.B] < sk.P ? 1 : 0;
  lc.attrs = at;
  lc.numAttrs = 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&lc, kern, tk[0], tk[1], tv[0], tv[1], tsk, tsv, trk, trv, a, sk);
  if (e != cudaSuccess)
    return set_error(FADE_ERR_CUDA, "fade_decode_attention (middle tier): %s",
                     cudaGetErrorString(e));
  return launch_status("fade_decode_attention (middle tier)");
}

}  // namespace
}  // namespace fade
