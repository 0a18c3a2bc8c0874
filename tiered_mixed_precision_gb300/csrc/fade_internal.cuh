// Internal helpers shared by the libfade translation units (host error plumbing and the
// device arithmetic every kernel must take identically: exact quantisation and fp32 RoPE).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fade.h"

namespace fade {

// ---------------------------------------------------------------- host side
fade_status_t set_error(fade_status_t st, const char* fmt, ...);
void clear_error();
// Maps the last launch error (if any) to FADE_ERR_CUDA with its message.
fade_status_t launch_status(const char* what);
// Validates a layer configuration (shapes, bits, policy, RoPE parameters).
fade_status_t validate_config(const fade_config_t* cfg);
// Validates the non-null buffers of a layer for the given config.
fade_status_t validate_layer(const fade_config_t* cfg, const fade_layer_t* layer);

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// NVTX ranges around the entry points that enqueue device work (a profiler shows each C-ABI
// call as a named range; without a profiler attached a range costs a function-pointer test).
#ifndef FADE_NVTX
#define FADE_NVTX 1
#endif
#if FADE_NVTX
struct NvtxRange {
  explicit NvtxRange(const char* name);
  ~NvtxRange();
};
#define FADE_RANGE(name) ::fade::NvtxRange fade_nvtx_range_(name)
#else
#define FADE_RANGE(name)
#endif

// Device-side checks. Every kernel guards its indices against the device metadata; a guard
// that fails (a state the host-side checks should have excluded) records its code in the
// layer's status word (status[0], first failure wins) and skips the access; fade_check_status
// reports codes >= kDevCheckBase as FADE_ERR_DEVICE_CHECK. FADE_DEBUG=1 builds add the checks
// that cost instructions on the hot paths (every compacted row, every attention tile).
#ifndef FADE_DEBUG
#define FADE_DEBUG 0
#endif
constexpr int kDevCheckBase = 16;
enum DevCheck {
  kCheckDemoteSlot = kDevCheckBase,  // demote: no free middle slot or a bad ring head
  kCheckAppendSlot,                  // append: the recent window is full
  kCheckCompactRow,                  // compaction: a destination row outside the unit (debug)
  kCheckAttnTile,                    // attention: a tile past the unit's capacity (debug)
};
inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

constexpr int kGroup = FADE_GROUP;     // channels per quantisation group
constexpr int kChunk = 1024;           // slots per selection chunk (bitmap prefix unit)
constexpr float kSubnormalMin = 5.9604644775390625e-08f;  // 2^-24

// Rotated width of the configuration's RoPE (proportional RoPE: rotary_dim < d).
inline int rotary_width(const fade_config_t* c) {
  return (c->rope.rotary_dim > 0 && c->rope.rotary_dim < c->head_dim) ? c->rope.rotary_dim
                                                                       : c->head_dim;
}

// Middle slots per unit in every middle buffer: the capacity rounded up to 64 slots.
inline int mid_stride(const fade_config_t* c) { return (c->mid_capacity + 63) / 64 * 64; }

// Per-row lengths passed by value to kernels (rows <= FADE_MAX_BATCH).
struct RowLens {
  int32_t v[FADE_MAX_BATCH];
};

// Stream-K schedule of the persistent tensor-core attention (INT4 K / INT2 V). The middle tier
// of every unit is cut into 256-token tiles; tiles are numbered unit by unit (row-major over
// (row, KV head)); CTA c takes global tiles [cta_start[c], cta_start[c+1]) plus the FP16-tier
// items of units c, c + P, ... . A unit's tiles may span several CTAs: each CTA writes one
// partial per unit segment it covers (split 1 + k for the k-th CTA of the unit; split 0 is the
// FP16 tiers). The boundaries are weighted so that every CTA gets about the same work.
constexpr int kMaxCtaSK = 320;   // persistent CTAs at most
constexpr int kTileTokens = FADE_ATTN_TILE_TOKENS;
struct StreamK {
  int P;                               // persistent CTAs
  int B, H;
  int smax;                            // most middle segments of any unit
  int row_start[FADE_MAX_BATCH + 1];   // first global tile of row b's first unit
  int cta_start[kMaxCtaSK + 1];
};
// First global tile of row b's first unit, and the middle tiles of each unit of row b.
__host__ __device__ inline int sk_row_start(const StreamK& k, int b) { return k.row_start[b]; }
__host__ __device__ inline int sk_row_tiles(const StreamK& k, int b) {
  return (k.row_start[b + 1] - k.row_start[b]) / k.H;
}
// The CTA whose range holds global tile g: the largest c < P with cta_start[c] <= g.
__host__ __device__ inline int sk_cta_of(const StreamK& k, int g) {
  int lo = 0, hi = k.P - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (k.cta_start[mid] <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}
// CTAs c in [c_lo, c_hi] whose middle range is not empty.
__host__ __device__ inline int sk_nonempty(const StreamK& k, int c_lo, int c_hi) {
  int n = 0;
  for (int c = c_lo; c <= c_hi; ++c) n += k.cta_start[c + 1] > k.cta_start[c];
  return n;
}
// Number of middle segments (partials after split 0) of unit (b, h): the CTAs with tiles of
// the unit. The k-th of them (k = sk_nonempty(first, c - 1)) writes split 1 + k.
__host__ __device__ inline int sk_segments(const StreamK& k, int b, int h) {
  const int rt = sk_row_tiles(k, b);
  if (rt == 0) return 0;
  const int g0 = sk_row_start(k, b) + h * rt;
  return sk_nonempty(k, sk_cta_of(k, g0), sk_cta_of(k, g0 + rt - 1));
}

// Decode attention on the tensor cores (INT4 or INT2 K; INT2, INT4 or PQ-coded V): split 0
// covers the FP16 tiers, splits 1.. the segments of the middle tier. Defined in
// attention_mma.cu (kernels in attention_mma.cuh; INT2-K instantiations in attention_mma_k2.cu).
bool mid_mma_supported(const fade_config_t* c);
// Persistent CTAs the kernel runs with on the current device.
int mid_mma_ctas(const fade_config_t* c);
// The schedule for the layer's current middle-tier counts (host mirrors).
void build_stream_k(const fade_config_t* c, const fade_layer_t* L, int ctas, StreamK* k);
fade_status_t launch_mid_mma(const fade_config_t* c, const fade_layer_t* L, const uint16_t* q,
                             float* logits, float* part_ml, float* part_acc, int32_t* seg_count,
                             const StreamK& sk, int nsplit, cudaStream_t st);

// ---------------------------------------------------------------- device side
__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ uint16_t f2h(float f) { return __half_as_ushort(__float2half_rn(f)); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Quantise one 32-channel group held one value per lane (all 32 lanes active).
// s = fp16(absmax / qmax) with IEEE fp32 division; s = 2^-24 if it underflows; the code is
// rint(x / s) (fp32 IEEE division, ties to even) clamped to [-qmax, qmax].
__device__ __forceinline__ void quant_group_lane(float x, int qmax, uint16_t& s_bits, int& q) {
  const float a = warp_max(fabsf(x));
  float s = __half2float(__float2half_rn(__fdiv_rn(a, (float)qmax)));
  if (a > 0.f && s == 0.f) s = kSubnormalMin;
  s_bits = f2h(s);
  q = 0;
  if (s > 0.f) {
    float r = rintf(__fdiv_rn(x, s));
    r = fminf(fmaxf(r, (float)-qmax), (float)qmax);
    q = (int)r;
  }
}

// Pack the group's codes (one per lane) and store them as 32-bit words: INT4 puts 8 lanes in
// a word (nibble i = lane 8w+i, written by lane 8w), INT2 puts 16 (crumb i = lane 16w+i,
// written by lane 16w). This is the little-endian byte layout of the codec. `dst` points at
// the group's first code byte and must be 4-byte aligned.
template <int BITS>
__device__ __forceinline__ void pack_group_store(int q, uint8_t* dst) {
  const int lane = threadIdx.x & 31;
  constexpr int per = 32 / BITS;   // codes per 32-bit word
  uint32_t v = (uint32_t(q) & ((1u << BITS) - 1u)) << (BITS * (lane % per));
#pragma unroll
  for (int o = 1; o < per; o <<= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  if (lane % per == 0) reinterpret_cast<uint32_t*>(dst)[lane / per] = v;
}

// Sign-extended code of channel c of a packed row.
template <int BITS>
__device__ __forceinline__ int unpack_code(const uint8_t* row, int c) {
  constexpr int per = 8 / BITS;
  const uint32_t b = row[c / per];
  const uint32_t u = (b >> (BITS * (c % per))) & ((1u << BITS) - 1u);
  return int(u) - (int(u >> (BITS - 1)) << BITS);
}

// ---- product quantisation of V (FADE-zh §产品量化): 256 centroids per 4-channel sub-space.
constexpr int kPqSub = 4, kPqCentroids = 256;

// Squared distance between a sub-vector x (fp16 values held as fp32) and the centroid whose
// four fp16 channels are packed in `c`, in one fixed order: ((e0^2 + e1^2) + e2^2) + e3^2,
// e_j = x_j - c_j, every operation rounded on its own (the intrinsics keep the compiler
// from fusing them), so that every caller takes the same integer decision.
__device__ __forceinline__ float pq_dist(const float x[4], uint2 c) {
  const float2 c01 = __half22float2(*reinterpret_cast<const __half2*>(&c.x));
  const float2 c23 = __half22float2(*reinterpret_cast<const __half2*>(&c.y));
  const float e0 = __fsub_rn(x[0], c01.x), e1 = __fsub_rn(x[1], c01.y);
  const float e2 = __fsub_rn(x[2], c23.x), e3 = __fsub_rn(x[3], c23.y);
  float acc = __fadd_rn(__fmul_rn(e0, e0), __fmul_rn(e1, e1));
  acc = __fadd_rn(acc, __fmul_rn(e2, e2));
  return __fadd_rn(acc, __fmul_rn(e3, e3));
}

// Index of the nearest of the 256 centroids `cb` of one sub-space; a strict comparison in
// increasing index order gives the lowest index on ties.
__device__ __forceinline__ int pq_nearest(const float x[4], const uint2* cb) {
  float best = __int_as_float(0x7f800000);  // +inf
  int bi = 0;
#pragma unroll 8
  for (int c = 0; c < kPqCentroids; ++c) {
    const float d = pq_dist(x, cb[c]);
    if (d < best) {
      best = d;
      bi = c;
    }
  }
  return bi;
}

// Encode one fp16 row of D channels with one warp: lane s < D/4 codes sub-space s. The V
// scale slots of a PQ row are written as zeros.
template <int D>
__device__ __forceinline__ void warp_pq_encode_row(const uint16_t* x, const uint16_t* codebook,
                                                   uint8_t* codes, uint16_t* scales) {
  const int lane = threadIdx.x & 31;
  if (lane < D / kPqSub) {
    const uint2 raw = *reinterpret_cast<const uint2*>(x + kPqSub * lane);
    const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    const float xv[4] = {x01.x, x01.y, x23.x, x23.y};
    const uint2* cb = reinterpret_cast<const uint2*>(codebook) + (size_t)lane * kPqCentroids;
    codes[lane] = (uint8_t)pq_nearest(xv, cb);
  }
  if (lane < D / kGroup) scales[lane] = 0;
}

// fp32 rotation of one pair with every product and sum rounded separately.
__device__ __forceinline__ void rotate_pair(float x1, float x2, float c, float s, float& y1,
                                            float& y2) {
  y1 = __fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, s));
  y2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
}

// RoPE table layout: per position, d/2 rotation pairs grouped two by two; block b holds
// (cos_{2b}, cos_{2b+1}, sin_{2b}, sin_{2b+1}) as one float4, so a 16-byte load gives the
// cosines and sines of two adjacent pairs as ready-made fp32x2 operands.
__device__ __forceinline__ float rope_cos(const float* table, int half, int pos, int i) {
  return table[(size_t)pos * 2 * half + (i >> 1) * 4 + (i & 1)];
}
__device__ __forceinline__ float rope_sin(const float* table, int half, int pos, int i) {
  return table[(size_t)pos * 2 * half + (i >> 1) * 4 + 2 + (i & 1)];
}

// Re-position one pair: un-rotate at `pold`, rotate at `pnew`.
__device__ __forceinline__ void reposition_pair(const float* __restrict__ table, int half,
                                                int i, int pold, int pnew, float x1, float x2,
                                                float& y1, float& y2) {
  float t1, t2;
  rotate_pair(x1, x2, rope_cos(table, half, pold, i), -rope_sin(table, half, pold, i), t1, t2);
  rotate_pair(t1, t2, rope_cos(table, half, pnew, i), rope_sin(table, half, pnew, i), y1, y2);
}

// Re-position a whole fp32 key held as pairs by a warp and write it quantised (middle tier)
// or as fp16. Lane l owns channels c1 = 32*gp + l and c2 = c1 + d/2 for gp < d/64.
template <int D>
struct WarpKey {
  float lo[D / 64];  // channel 32*gp + lane
  float hi[D / 64];  // channel 32*gp + lane + D/2
};

template <int D, int BITS>
__device__ __forceinline__ void warp_store_quantized(const WarpKey<D>& k, uint8_t* codes_row,
                                                     uint16_t* scales_row) {
  const int lane = threadIdx.x & 31;
  constexpr int qmax = (1 << (BITS - 1)) - 1;
  constexpr int bytes_per_group = kGroup * BITS / 8;
#pragma unroll
  for (int gp = 0; gp < D / 64; ++gp) {
    // group gp holds channels [32gp, 32gp+32) -> the `lo` values
    uint16_t sb;
    int q;
    quant_group_lane(__half2float(__float2half_rn(k.lo[gp])), qmax, sb, q);
    pack_group_store<BITS>(q, codes_row + gp * bytes_per_group);
    if (lane == 0) scales_row[gp] = sb;
    // group gp + D/64 holds channels [D/2 + 32gp, ...) -> the `hi` values
    quant_group_lane(__half2float(__float2half_rn(k.hi[gp])), qmax, sb, q);
    pack_group_store<BITS>(q, codes_row + (gp + D / 64) * bytes_per_group);
    if (lane == 0) scales_row[gp + D / 64] = sb;
  }
}

// ---- packed fp32 pairs (Blackwell f32x2 arithmetic). Each instruction rounds each element to
// nearest like its scalar form, but the assembler may fuse a packed product into a following
// packed sum even with an explicit rounding mode: use these only where such a fusion cannot
// change a result (exact steps, or steps whose error analysis covers it). Separately rounded
// products and sums use the scalar __fmul_rn / __fadd_rn intrinsics.
typedef unsigned long long f2x;  // low 32 bits = first element
__device__ __forceinline__ f2x f2_pack(float lo, float hi) {
  f2x r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(f2x v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2x f2_mul(f2x a, f2x b) {
  f2x d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2x f2_add(f2x a, f2x b) {
  f2x d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2x f2_sub(f2x a, f2x b) {
  f2x d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2x f2_fma(f2x a, f2x b, f2x c) {  // a*b + c, one rounding
  f2x d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// Round both elements to fp16 and back (the cast through the model dtype).
__device__ __forceinline__ f2x f2_round_f16(f2x v) {
  float lo, hi;
  f2_unpack(v, lo, hi);
  const float2 f = __half22float2(__floats2half2_rn(lo, hi));
  return f2_pack(f.x, f.y);
}

// round_half_even(x / s) for fp16-valued x and s > 0, exactly (equal to rint of the IEEE fp32
// quotient, which cannot land on or cross a half-integer for fp16 operands): a reciprocal
// estimate gives a candidate within one of the answer, the residual x - q*s is exact in fp32
// (a 3-bit integer times an 11-bit significand, then a difference spanning under 24 bits), and
// comparing it with s/2 corrects the candidate and resolves exact ties to the even integer.
__device__ __forceinline__ float rint_div_exact(float x, float s) {
  float q = rintf(x * __frcp_rn(s));
  const float e = fmaf(-q, s, x);
  const float h = 0.5f * s;
  const float ae = fabsf(e);
  if (ae > h) {
    q += copysignf(1.f, e);
  } else if (ae == h) {
    const float q2 = q + copysignf(1.f, e);
    if ((int)q & 1) q = q2;  // exact tie: keep the even neighbour (q is a small integer)
  }
  return q;
}

// Quantise one 32-value group held by one thread; writes the packed codes (4 words for INT4,
// 2 for INT2) and returns the fp16 scale bits.
template <int BITS>
__device__ __forceinline__ uint16_t quant_group_thread(const float (&x)[32], uint32_t* words) {
  constexpr int qmax = (1 << (BITS - 1)) - 1;
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(x[i]));
  float s = __half2float(__float2half_rn(__fdiv_rn(a, (float)qmax)));
  if (a > 0.f && s == 0.f) s = kSubnormalMin;
  constexpr int per = 32 / BITS;
#pragma unroll
  for (int w = 0; w < 32 / per; ++w) {
    uint32_t v = 0;
#pragma unroll
    for (int e = 0; e < per; ++e) {
      float q = 0.f;
      if (s > 0.f) q = fminf(fmaxf(rint_div_exact(x[w * per + e], s), (float)-qmax), (float)qmax);
      v |= (uint32_t((int)q) & ((1u << BITS) - 1u)) << (BITS * e);
    }
    words[w] = v;
  }
  return __half_as_ushort(__float2half_rn(s));
}

// Two rotation pairs at once: (x1, x2) <- (x1*c - x2*s, x2*c + x1*s) elementwise, with the
// four products as packed multiplies and the sums as scalar IEEE adds, so that every product
// and every sum is rounded on its own (no packed sum reads a packed product).
__device__ __forceinline__ void rotate2(f2x& X1, f2x& X2, f2x C, f2x S) {
  float a0, a1, b0, b1, c0, c1, d0, d1;
  f2_unpack(f2_mul(X1, C), a0, a1);
  f2_unpack(f2_mul(X2, S), b0, b1);
  f2_unpack(f2_mul(X2, C), c0, c1);
  f2_unpack(f2_mul(X1, S), d0, d1);
  X1 = f2_pack(__fsub_rn(a0, b0), __fsub_rn(a1, b1));
  X2 = f2_pack(__fadd_rn(c0, d0), __fadd_rn(c1, d1));
}

// The inverse rotation of rotate2 with the same (c, s): (x1*c + x2*s, x2*c - x1*s). Equal bit
// for bit to rotate2 with the sines negated (a product with -s is the negated product, and
// subtracting a negated value is adding it), without the negations.
__device__ __forceinline__ void rotate2_inv(f2x& X1, f2x& X2, f2x C, f2x S) {
  float a0, a1, b0, b1, c0, c1, d0, d1;
  f2_unpack(f2_mul(X1, C), a0, a1);
  f2_unpack(f2_mul(X2, S), b0, b1);
  f2_unpack(f2_mul(X2, C), c0, c1);
  f2_unpack(f2_mul(X1, S), d0, d1);
  X1 = f2_pack(__fadd_rn(a0, b0), __fadd_rn(a1, b1));
  X2 = f2_pack(__fsub_rn(c0, d0), __fsub_rn(c1, d1));
}

// Correctly rounded fp32 a / QMAX for fp16-valued a >= 0 (QMAX = 7 or 1), the scale division
// of the quantiser. For QMAX = 7: Markstein's correction step (q0 = a * RN(1/7), e = a - q0 * 7
// exact by FMA, q1 = RN(q0 + e * RN(1/7))); an exhaustive check over every non-negative finite
// fp16 a shows q1 equal to the IEEE quotient.
template <int QMAX>
__device__ __forceinline__ float div_by_qmax(float a) {
  if constexpr (QMAX == 1) {
    return a;
  } else {
    constexpr float r = 1.0f / (float)QMAX;
    const float q0 = a * r;
    const float e = fmaf(-q0, (float)QMAX, a);
    return fmaf(e, r, q0);
  }
}

// Byte permute: output byte i = byte sel[4i+2:4i] of {b, a} (a = bytes 0-3, b = bytes 4-7).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Exact dequantisation of INT4 codes, one packed pair at a time. The two little-endian words
// of a half group (channel j at bits 4j) are first split into offset-binary nibbles, even
// channels in ev[w] and odd ones in od[w] (byte b of word w = channel 8w + 2b (+1)); a byte
// permute then moves a nibble into the low mantissa byte of 2^23, so the float is
// 2^23 + code + 8, and subtracting 2^23 + 8 and multiplying by s are exact.
__device__ __forceinline__ void split_int4(const uint32_t (&w)[2], uint32_t (&ev)[2],
                                           uint32_t (&od)[2]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    ev[h] = (w[h] & 0x0F0F0F0Fu) ^ 0x08080808u;
    od[h] = ((w[h] >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
  }
}
// Pair k (channels 2k, 2k+1 of the half group; k a constant once the caller's loop is unrolled).
__device__ __forceinline__ f2x dequant_pair_int4(const uint32_t (&ev)[2], const uint32_t (&od)[2],
                                                 int k, f2x S) {
  const uint32_t magic = 0x4B000000u;
  const float lo = __uint_as_float(prmt(ev[k >> 2], magic, 0x7650u + (k & 3)));
  const float hi = __uint_as_float(prmt(od[k >> 2], magic, 0x7650u + (k & 3)));
  return f2_mul(f2_sub(f2_pack(lo, hi), f2_pack(8388616.f, 8388616.f)), S);
}
// Same for BITS-bit codes in general (here used for INT2), pair k of the little-endian words w.
template <int BITS>
__device__ __forceinline__ f2x dequant_pair_bits(const uint32_t* w, int k, f2x S) {
  constexpr int per = 32 / BITS;
  constexpr uint32_t msk = (1u << BITS) - 1u, flip = 1u << (BITS - 1);
  const int j0 = 2 * k, j1 = 2 * k + 1;
  const uint32_t c0 = ((w[j0 / per] >> (BITS * (j0 % per))) & msk) ^ flip;
  const uint32_t c1 = ((w[j1 / per] >> (BITS * (j1 % per))) & msk) ^ flip;
  const float off = 8388608.f + (float)flip;   // 2^23 + 2^(bits-1)
  return f2_mul(f2_sub(f2_pack(__uint_as_float(0x4B000000u | c0), __uint_as_float(0x4B000000u | c1)),
                       f2_pack(off, off)),
                S);
}

// The exact scalar path of codes_half_group (rare: exact ties, a candidate off by one, subnormal
// scales), kept out of line so that the callers' unrolled code stays small; the 16 values come
// in registers (two uint4 of half2 words) and the packed codes go back in registers.
template <int BITS>
__device__ __noinline__ uint2 codes_half_group_exact(uint4 lo, uint4 hi, float s) {
  constexpr int per = 32 / BITS;
  constexpr uint32_t mask = (1u << BITS) - 1u;
  constexpr int qmax = (1 << (BITS - 1)) - 1;
  const uint32_t H[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int w = 0; w < 16 / per; ++w) {
    uint32_t o = 0u;
#pragma unroll
    for (int e = 0; e < per; ++e) {
      const int j = w * per + e;
      const __half2 hp = *reinterpret_cast<const __half2*>(&H[j >> 1]);
      const float x = (j & 1) ? __high2float(hp) : __low2float(hp);
      const float q = fminf(fmaxf(rint_div_exact(x, s), (float)-qmax), (float)qmax);
      o |= (uint32_t((int)q) & mask) << (BITS * e);
    }
    out[w] = o;
  }
  return make_uint2(out[0], out[1]);
}

// Codes of 16 fp16 values (8 half2 words) of one group whose scale s (> 0) is already
// known, packed little-endian from bit 0 of out[0] (INT4: two words, INT2: one): exact
// round_half_even(x/s). Fast path: x * (1/s) + 1.5 * 2^23 leaves a candidate code in the low
// bits (two's complement); the exact residual x - q*s, below s/2 for every value, confirms all
// 16 candidates, which are then packed with byte permutes (INT4). Otherwise (an exact tie, a
// candidate off by one, or a subnormal scale where the clamp can bind) every code is redone by
// the exact scalar path with the clamp.
template <int BITS>
__device__ __forceinline__ void codes_half_group(const uint32_t (&H)[8], float s, uint32_t* out) {
  constexpr uint32_t mask = (1u << BITS) - 1u;
  // any reciprocal estimate serves: the exact residual below confirms or rejects the candidates
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  const float h = 0.5f * s;
  const f2x R = f2_pack(r, r), M = f2_pack(12582912.f, 12582912.f), NS = f2_pack(-s, -s);
  uint32_t qb[16];
  float emax = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&H[k]));
    const f2x X = f2_pack(f.x, f.y);
    const f2x QM = f2_add(f2_mul(X, R), M);
    const f2x E = f2_fma(f2_sub(QM, M), NS, X);
    float e0, e1, qm0, qm1;
    f2_unpack(E, e0, e1);
    f2_unpack(QM, qm0, qm1);
    qb[2 * k] = __float_as_uint(qm0);
    qb[2 * k + 1] = __float_as_uint(qm1);
    emax = fmaxf(emax, fmaxf(fabsf(e0), fabsf(e1)));
  }
  if (s >= 6.103515625e-05f && emax < h) {
    if constexpr (BITS == 4) {
      // word v: channels 8v..8v+7; A = bytes of the even channels' codes, B = the odd ones
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

// ---------------------------------------------------------------- async copies, mbarriers
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz: a wait that never ends
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
__device__ __forceinline__ void record_status(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Bounded wait: gives up after `limit` cycles and records the failure (`code`) in status[0]
// unless an earlier failure is recorded there.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, int32_t* status,
                                                int code, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) {
      atomicCAS(status, 0, code);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status,
                                          int code) {
  return mbar_wait_limit(bar, parity, status, code, kWaitCycles);
}
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                             uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Shared -> global bulk copy (both 16-byte aligned, bytes a multiple of 16), bulk async-group.
__device__ __forceinline__ void bulk_store_1d(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the committed bulk stores have read their shared-memory sources.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until the committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Order this thread's generic shared-memory writes before later async-proxy (bulk copy) reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace fade
