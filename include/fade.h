/*
 * fade.h — C ABI of libfade: the decode-attention hot path of the FADE tiered KV cache on
 * one NVIDIA GB300 (sm_103a).
 *
 * Sources cited below:
 *   FADE-zh  page "FADE：面向LLM推理的注意力感知分层KV缓存压缩技术"
 *   FADE-en  page "FADE: Attention-Aware Hierarchical KV Cache Compression for LLM Inference"
 *   KVLong   page "探秘Transformer系列之（25）--- KV Cache优化之处理长文本序列"
 *
 * The cache of one layer holds, per (row, KV head) "unit":
 *   - FP16 sinks: the first n_sink tokens (FADE-zh §第一层);
 *   - FP16 recent window: the last recent_window tokens, stored as a ring (FADE-zh §第一层);
 *   - the middle tier: symmetric absmax codes, K at middle_k_bits and V at middle_v_bits
 *     (4 or 2), one fp16 scale per 32 channels, packed little-endian into bytes
 *     (FADE-zh §第二层, §第三层, §量化与Bit-Packing), in two buffers used alternately by
 *     eviction (live buffer = meta field CUR);
 *   - one fp32 importance score per held token (FADE-zh §四种驱逐策略详解).
 * Keys are stored RoPE'd at their cache index (StreamingLLM positions, KVLong §1.2.2).
 *
 * Conventions for every call:
 *   - All device memory is allocated and owned by the caller; sizes come from fade_layout().
 *     The library allocates no device memory and keeps no global state except the
 *     thread-local error string.
 *   - Calls are asynchronous on the given stream (cudaStream_t passed as void*; NULL = the
 *     legacy default stream). Argument, shape and capacity errors are detected on the host
 *     before any launch and returned synchronously; nothing is enqueued then. A launch
 *     failure returns FADE_ERR_CUDA. fade_last_error() describes the last failure of the
 *     calling thread.
 *   - fp16 data is passed as raw IEEE binary16 (uint16 bits). Row-major layouts throughout.
 *   - The host keeps a mirror of per-row tier counts in the fade_layer_t (h_* arrays); each
 *     call updates it as it enqueues work, so the caller never synchronises to learn sizes.
 *   - Kernels never trap and never spin without a limit: a wait inside a kernel (an
 *     mbarrier of a bulk-copy pipeline) gives up after about 2 s, records a code in the
 *     layer's status words and returns; fade_check_status reports it.
 */
#ifndef FADE_H_
#define FADE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FADE_OK = 0,
  FADE_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad shape, out-of-range value */
  FADE_ERR_UNSUPPORTED = 2,      /* a valid configuration this build does not implement */
  FADE_ERR_CAPACITY = 3,         /* a tier or workspace would overflow its buffer */
  FADE_ERR_CUDA = 4,             /* a CUDA call or kernel launch failed */
  FADE_ERR_TIMEOUT = 5,          /* a kernel gave up a bounded wait (fade_check_status) */
  FADE_ERR_DEVICE_CHECK = 6      /* a device-side index check failed (fade_check_status) */
} fade_status_t;

/* RoPE schemes (FADE-zh §RoPE方案兼容性: standard RoPE and the scaling types llama3, linear,
 * ntk, yarn, dynamic and proportional; ALiBi models make re-positioning a no-op:
 * FADE_ROPE_NONE). Every scheme is a set of inverse frequencies inv_i (rotate-half pairs
 * i, i + r/2 over the rotated width r = fade_rope_t.rotary_dim, d by default: proportional
 * RoPE is any scheme with r < d); base_i = base^(-2i/r), and d below reads r:
 *   DEFAULT  inv_i = base_i
 *   LLAMA3   base_i blended by the number of rotations r_i = L / (2 pi / base_i) over the
 *            original context L = original_max_position: r_i > high_freq_factor keeps base_i,
 *            r_i < low_freq_factor uses base_i / factor, otherwise
 *            (1 - t) base_i / factor + t base_i with t = (r_i - low) / (high - low)
 *   LINEAR   inv_i = base_i / factor (position interpolation: positions divided by factor)
 *   NTK      inv_i = (base * factor^(d / (d - 2)))^(-2i/d) (NTK-aware base scaling)
 *   YARN     the LLAMA3 blend with low_freq_factor = alpha and high_freq_factor = beta of the
 *            YaRN ramp (1 and 32 in its paper); YaRN's attention temperature is not part of
 *            the table (it would scale every rotation, and un-RoPE / re-RoPE with it)
 *   DYNAMIC  dynamic NTK: the NTK rule with the factor taken from the sequence length L,
 *            base' = base * (factor * L / original_max_position - (factor - 1))^(d / (d - 2))
 *            when L > original_max_position, the default table otherwise. L is the length the
 *            table is built for (max_pos of fade_rope_table_init), so every key is rotated and
 *            re-positioned with one table; re-basing every step as the sequence grows is not
 *            done (it would re-rotate every cached key). */
typedef enum {
  FADE_ROPE_NONE = 0,
  FADE_ROPE_DEFAULT = 1,
  FADE_ROPE_LLAMA3 = 2,
  FADE_ROPE_LINEAR = 3,
  FADE_ROPE_NTK = 4,
  FADE_ROPE_YARN = 5,
  FADE_ROPE_DYNAMIC = 6
} fade_rope_kind_t;

/* Eviction policies (FADE-zh §四种驱逐策略详解 1-3). NONE = safe mode (no eviction). */
typedef enum {
  FADE_EVICT_NONE = 0,
  FADE_EVICT_H2O = 1,
  FADE_EVICT_EMA = 2,
  FADE_EVICT_POSITION = 3
} fade_policy_t;

typedef struct {
  int32_t kind;                  /* fade_rope_kind_t */
  int32_t original_max_position; /* llama3, yarn: the original context L */
  double base;                   /* theta base, e.g. 10000, 500000 */
  double factor;                 /* llama3, linear, ntk, yarn: the scaling factor (> 0) */
  double low_freq_factor;        /* llama3; yarn: alpha */
  double high_freq_factor;       /* llama3; yarn: beta (> low_freq_factor) */
  int32_t rotary_dim;            /* proportional RoPE (FADE-zh §RoPE方案兼容性: Gemma 4,
                                    partial_rotary_factor): only channels 0..rotary_dim-1
                                    rotate, paired (i, i + rotary_dim/2), with every
                                    scheme's frequencies computed for a rotary_dim-wide head
                                    (base^(-2i/rotary_dim)); channels rotary_dim..d-1 pass
                                    through. 0 or d: every channel (standard RoPE). Otherwise
                                    a multiple of 4 in [4, d). */
} fade_rope_t;

/* One layer's cache configuration (FADE-zh §自定义配置: n_sink, recent_window, int4_budget,
 * eviction_policy, middle_k_bits, middle_v_bits). */
typedef struct {
  int32_t batch;          /* rows, 1..FADE_MAX_BATCH; fixed for the cache's lifetime */
  int32_t num_q_heads;    /* Hq; a multiple of num_kv_heads, Hq/Hkv <= 8 */
  int32_t num_kv_heads;   /* Hkv */
  int32_t head_dim;       /* d: 64 or 128 */
  int32_t n_sink;         /* FP16 sink tokens kept per unit, >= 0 */
  int32_t recent_window;  /* FP16 recent tokens kept per unit, >= 1 */
  int32_t int4_budget;    /* middle tokens kept per unit when evicting; < 0: unbounded */
  int32_t middle_k_bits;  /* 4 (2 is accepted too) */
  int32_t middle_v_bits;  /* 2 or 4 */
  int32_t mid_capacity;   /* middle slots allocated per unit (>= budget + 1 when evicting);
                             batch x num_kv_heads x mid_stride must stay below 2^31
                             (FADE_ERR_UNSUPPORTED otherwise) */
  int32_t policy;         /* fade_policy_t */
  float ema_decay;        /* EMA decay delta in [0, 1) */
  int32_t shared_rows;    /* 0: tier decisions per (row, KV head); 1: the rows share them
                             (FADE-zh §批处理支持: one allocation for all rows). Victims are
                             then chosen per KV head by the row-summed scores (H2O, EMA; the
                             prefill mass for H2O) and applied to every row; every row must hold
                             equal tier counts (equal prompt lengths at prefill), otherwise
                             FADE_ERR_INVALID_ARGUMENT. Each row keeps its own scores. */
  int32_t v_codec;        /* fade_v_codec_t: how the middle tier stores V. FADE_V_PQ needs
                             middle_v_bits = 2 (a PQ row has the INT2 row's d/4 bytes) and
                             fade_layer_t.pq_codebook */
  fade_rope_t rope;
} fade_config_t;

/* Middle-tier V codec. FADE_V_PQ (FADE-zh §产品量化, the alternative to INT2 at about 2 bits
 * per element): each 4-channel sub-vector of V is stored as the uint8 index of its nearest
 * centroid in a per-layer codebook (see fade_pq_encode); the V scale slots are then written
 * as zeros and carry nothing. */
typedef enum { FADE_V_INT = 0, FADE_V_PQ = 1 } fade_v_codec_t;

#define FADE_MAX_BATCH 256
#define FADE_STATUS_WORDS 4
#define FADE_NOALLOC_SCRATCH_BYTES (8u << 20) /* see fade_decode_attention_noalloc */
#define FADE_GROUP 32

/* Per-unit device metadata: int32 [batch][num_kv_heads][FADE_META_FIELDS]. */
enum {
  FADE_META_N_SINK = 0,   /* sinks held */
  FADE_META_N_MID = 1,    /* middle tokens held (slots 0..N_MID-1 of buffer CUR) */
  FADE_META_N_RECENT = 2, /* recent tokens held */
  FADE_META_HEAD = 3,     /* ring slot of the oldest recent token */
  FADE_META_CUR = 4,      /* live middle buffer, 0 or 1 */
  FADE_META_N_EV = 5,     /* evictions chosen and not yet committed (internal) */
  FADE_META_SYNC = 6,     /* internal: middle slots below this index hold the same K/V codes
                             and scales in both buffers (0 after prefill or reset) */
  FADE_META_P1 = 7,       /* internal (prefill) */
  FADE_META_FIELDS = 8
};

/* Caller-owned buffers of one layer. Device pointers unless marked host. Shapes use
 * B = batch, H = num_kv_heads, S = n_sink, W = recent_window, d, and C = the middle slot
 * stride: mid_capacity rounded up to a multiple of 64 (fade_layout_t.mid_stride), so every
 * unit's rows start 16-byte aligned for bulk copies. Only the first mid_capacity slots of a
 * unit are ever used. */
typedef struct {
  uint16_t* sink_k;          /* fp16 [B][H][S][d] */
  uint16_t* sink_v;          /* fp16 [B][H][S][d] */
  uint16_t* recent_k;        /* fp16 [B][H][W][d], ring */
  uint16_t* recent_v;        /* fp16 [B][H][W][d], ring */
  uint8_t* mid_k_codes[2];   /* u8 [B][H][C][d*middle_k_bits/8] */
  uint16_t* mid_k_scales[2]; /* fp16 [B][H][C][d/32] */
  uint8_t* mid_v_codes[2];   /* u8 [B][H][C][d*middle_v_bits/8] */
  uint16_t* mid_v_scales[2]; /* fp16 [B][H][C][d/32] */
  float* sink_scores;        /* f32 [B][H][S] */
  float* mid_scores[2];      /* f32 [B][H][C] */
  float* recent_scores;      /* f32 [B][H][W], indexed by ring slot */
  int32_t* meta;             /* i32 [B][H][FADE_META_FIELDS] */
  uint32_t* victims;         /* scratch: u32 [B][H][victim_words] */
  int32_t* chunk_base;       /* scratch: i32 [B][H][chunk_slots] */
  int32_t victim_words;      /* from fade_layout_t: sizes the longest prompt / middle tier */
  int32_t chunk_slots;       /* from fade_layout_t */
  int32_t* status;           /* i32 [FADE_STATUS_WORDS]: device-side error status, 0 = ok;
                                zeroed by fade_cache_reset; nonzero after a kernel gave up a
                                bounded wait (the call's results are then invalid); read by
                                fade_check_status */
  int32_t* h_n_sink;         /* HOST i32 [B]: mirror of N_SINK (same for every head) */
  int32_t* h_n_mid;          /* HOST i32 [B]: mirror of N_MID */
  int32_t* h_n_recent;       /* HOST i32 [B]: mirror of N_RECENT */
  const uint16_t* pq_codebook; /* FADE_V_PQ only: fp16 [d/4][256][4], this layer's codebook
                                  (shared by every row and KV head); NULL otherwise */
} fade_layer_t;

/* Byte sizes of every buffer of a layer and of the per-call workspaces. */
typedef struct {
  size_t sink_k, sink_v, recent_k, recent_v;
  size_t mid_k_codes, mid_k_scales, mid_v_codes, mid_v_scales; /* each of the two buffers */
  size_t sink_scores, mid_scores, recent_scores, meta, victims, chunk_base, status;
  size_t logits_ws;   /* f32 [B][Hq][S + C + W]: per-token logits for H2O / EMA */
  int32_t mid_stride;  /* C: middle slots per unit in every middle buffer */
  size_t ml_ws;       /* f32 [B][Hq][2]: final (max, sum) of each query head's softmax */
  size_t attn_ws;     /* split-KV partials for fade_decode_attention (and one i32 partial
                         count per unit) */
  int32_t victim_words;  /* u32 words per unit in `victims` */
  int32_t chunk_slots;   /* i32 entries per unit in `chunk_base` */
  int32_t max_prompt;    /* the prompt length the scratch sizes were computed for */
  int32_t max_splits;    /* split-KV partial slots per (row, query head) */
  size_t prefill_mass_ws; /* workspace of fade_prefill_mass for prompts of max_prompt */
} fade_layout_t;

/* Validate `cfg` and return the sizes of a layer's buffers for prompts of up to
 * `max_prompt` tokens per row. Host only, no CUDA calls. */
fade_status_t fade_layout(const fade_config_t* cfg, int32_t max_prompt, fade_layout_t* out);

/* RoPE table (FADE-zh §RoPE重计算: float32 RoPE math; FADE-zh §RoPE方案兼容性: the schemes
 * above). Writes f32 [max_pos][d/4][4]: block b < r/4 of position pos holds (cos_{2b},
 * cos_{2b+1}, sin_{2b}, sin_{2b+1}) of rotation pairs 2b and 2b+1 (r = the rotated width;
 * blocks r/4..d/4-1 are not written), for
 * angle = fp32(pos) * inv_freq_i (one fp32 multiply), inv_freq_i = base^(-2i/d) in fp64
 * (llama3-adjusted in fp64) rounded to fp32, cos/sin evaluated in fp64 and rounded to fp32.
 * `table` is device memory of max_pos*d*4 bytes, 16-byte aligned. Not valid for
 * FADE_ROPE_NONE. */
fade_status_t fade_rope_table_init(const fade_config_t* cfg, float* table, int32_t max_pos,
                                   void* stream);

/* Rotate fp16 vectors to their positions (the model's RoPE of q and k; KVLong §1.2.2: the
 * position of a token is its index in the cache). x, y: fp16 [n_groups][group_len][d]
 * (y may alias x). Vector j of group g is rotated to position
 * (pos_start ? pos_start[g] : 0) + j * pos_step, with pos_start a device i32 [n_groups].
 * Rotation pairs channel i with i + r/2 for i < r/2 (r = the rotated width, d by default);
 * channels r..d-1 are copied unchanged; every product and sum is rounded to fp32 (no fused
 * multiply-add); the result is rounded to fp16. Positions must lie in [0, max_pos). */
fade_status_t fade_rope_apply(const fade_config_t* cfg, const float* table, int32_t max_pos,
                              const uint16_t* x, uint16_t* y, int64_t n_groups,
                              int32_t group_len, const int32_t* pos_start, int32_t pos_step,
                              void* stream);

/* Quantise and pack (FADE-zh §量化与Bit-Packing: symmetric quantisation with bit-packing).
 * x: fp16 [n_vec][dim], dim a multiple of 32. Per 32-channel group: a = max|x|,
 * s = fp16(a / qmax) with qmax = 2^(bits-1)-1 (fp32 IEEE division, round to nearest even);
 * s = 2^-24 if a > 0 and s rounds to 0; q = clamp(rint(x / s), -qmax, qmax) (fp32
 * division, ties to even), 0 when a = 0. codes: u8 [n_vec][dim*bits/8], INT4 byte j =
 * q[2j] | q[2j+1] << 4, INT2 byte j = sum_r q[4j+r] << 2r, two's complement fields.
 * scales: fp16 [n_vec][dim/32]. bits is 2 or 4. */
fade_status_t fade_quantize_pack(const uint16_t* x, int64_t n_vec, int32_t dim, int32_t bits,
                                 uint8_t* codes, uint16_t* scales, void* stream);

/* Inverse codec: out[n][c] = q * s as f32 (exact). Same layouts as fade_quantize_pack. */
fade_status_t fade_dequantize(const uint8_t* codes, const uint16_t* scales, int64_t n_vec,
                              int32_t dim, int32_t bits, float* out, void* stream);

/* Product quantisation of V (FADE-zh §产品量化: a codebook trained from calibration vectors
 * with 256 centroids; vectors encoded to uint8 codes and decoded back). A vector of `dim`
 * channels (a multiple of 4, at most 1024) is cut into dim/4 sub-vectors of 4 consecutive
 * channels; sub-space s has its own 256 centroids. codebook: fp16 [dim/4][256][4].
 *
 * fade_pq_encode: codes[n][s] = the centroid c of sub-space s with the smallest squared
 * distance to x[n][4s..4s+3], the distance taken in fp32 as ((e0^2 + e1^2) + e2^2) + e3^2
 * with e_j = x_j - c_j and every difference, square and sum rounded on its own (no fused
 * operations); the lowest index wins a tie. x: fp16 [n_vec][dim], finite; codes: u8
 * [n_vec][dim/4]. */
fade_status_t fade_pq_encode(const uint16_t* codebook, const uint16_t* x, int64_t n_vec,
                             int32_t dim, uint8_t* codes, void* stream);

/* out[n][4s + j] = codebook[s][codes[n][s]][j]: fp16 [n_vec][dim], exact. */
fade_status_t fade_pq_decode(const uint16_t* codebook, const uint8_t* codes, int64_t n_vec,
                             int32_t dim, uint16_t* out, void* stream);

#define FADE_PQ_SUB 4
#define FADE_PQ_CENTROIDS 256
#define FADE_PQ_MAX_CALIB 8192
/* Workspace of fade_pq_train: i64 member sums, i32 member counts and the copied indices. */
#define FADE_PQ_TRAIN_WS_BYTES(dim) ((size_t)(dim) * 2304u + 1024u)

/* Train a codebook by Lloyd's k-means in every sub-space. Centroid c starts at the
 * sub-vectors of calibration row h_init_idx[c] (HOST i32 [256], each in [0, n_vec): the
 * caller's random draw); each of `iters` rounds assigns every calibration sub-vector by the
 * fade_pq_encode rule and sets each centroid to the mean of its members: the member sum is
 * exact (taken in integers of 2^-24), divided once in fp64 and rounded to fp16 (nearest
 * even); a centroid without members keeps its value. calib: fp16 [n_vec][dim], finite,
 * 1 <= n_vec <= FADE_PQ_MAX_CALIB. codebook (out): fp16 [dim/4][256][4]. ws: device,
 * FADE_PQ_TRAIN_WS_BYTES(dim) bytes, 16-byte aligned. */
fade_status_t fade_pq_train(const uint16_t* calib, int64_t n_vec, int32_t dim,
                            const int32_t* h_init_idx, int32_t iters, uint16_t* codebook,
                            void* ws, size_t ws_bytes, void* stream);

/* Host mirror only: apply to h_n_sink / h_n_mid / h_n_recent the tier-count changes of one
 * decode step (fade_cache_demote, fade_evict_rerope, fade_cache_append in that order), with
 * their capacity checks, without enqueuing any work. For a caller that replays a captured
 * step (a CUDA graph), whose kernels advance the device-side metadata themselves. On an error
 * (FADE_ERR_CAPACITY: a full middle tier or recent window) the mirror is left unchanged. */
fade_status_t fade_cache_advance_host(const fade_config_t* cfg, fade_layer_t* layer);

/* fade_cache_advance_host for n_layers layers of one configuration in one call (layers: HOST
 * array of n_layers layer pointers, n_layers >= 0): every layer's rows are checked before any
 * count is stored, so on an error no mirror changes. For a caller replaying a captured step of
 * many layers, whose host work per step this keeps to one call. */
fade_status_t fade_cache_advance_host_layers(const fade_config_t* cfg, fade_layer_t* const* layers,
                                             int32_t n_layers);

/* Empty the cache: zero the device metadata and the host mirror. */
fade_status_t fade_cache_reset(const fade_config_t* cfg, fade_layer_t* layer, void* stream);

/* Build the tiers from a prompt (FADE-zh §核心机制, §驱逐策略, §四种驱逐策略详解 1: H2O
 * scores come from prefill attention). k_rot: fp16 [B][H][max_prompt][d], already RoPE'd
 * at positions 0..P-1; v: fp16 [B][H][max_prompt][d]; h_prompt_len: HOST i32 [B] with
 * row lengths P (<= max_prompt). Sinks = first n_sink tokens, recent = last recent_window,
 * the rest are middle candidates. When the candidates exceed int4_budget and the policy
 * evicts, the excess with the smallest (key, index) is dropped: key = mass (H2O), 0 (EMA,
 * so the oldest go first) or the index (position). Survivors are re-positioned in fp32 to
 * contiguous indices and cast to fp16; the middle tier is then quantised once. H2O scores
 * start at the survivors' mass (mass: device f32 [B][H][max_prompt], required for H2O,
 * ignored otherwise); other scores start at 0. The cache must be empty (after reset).
 * `table` may be NULL only for FADE_ROPE_NONE. Uses the layer's scratch buffers. */
fade_status_t fade_cache_prefill(const fade_config_t* cfg, fade_layer_t* layer,
                                 const uint16_t* k_rot, const uint16_t* v,
                                 int32_t max_prompt, const int32_t* h_prompt_len,
                                 const float* mass, const float* table, int32_t max_pos,
                                 void* stream);

/* Prefill attention mass (FADE-zh §四种驱逐策略详解 1: H2O needs the attention captured at
 * prefill; KVLong §1.3.1 H2O: a token's importance is the column sum of the attention
 * matrix). q_rot: fp16 [B][Hq][max_prompt][d] and k_rot: fp16 [B][H][max_prompt][d], both
 * RoPE'd at positions 0..P-1; h_prompt_len: HOST i32 [B]. Writes mass: f32
 * [B][H][max_prompt], mass[b][h][j] = sum over the query heads of KV head h and over the
 * queries i >= j of softmax_j(q_i . k_j / sqrt(d)) (causal), 0 past a row's length. fp32
 * arithmetic in one fixed order (no atomics): the result is identical on every run. ws:
 * device workspace of fade_layout_t.prefill_mass_ws bytes (B * Hq * max_prompt * 8: each
 * query row's softmax max and sum), 8-byte aligned; FADE_ERR_CAPACITY if ws_bytes is
 * smaller. The result is the `mass` argument of fade_cache_prefill. */
fade_status_t fade_prefill_mass(const fade_config_t* cfg, const uint16_t* q_rot,
                                const uint16_t* k_rot, int32_t max_prompt,
                                const int32_t* h_prompt_len, float* mass, void* ws,
                                size_t ws_bytes, void* stream);

/* Demote (FADE-zh §第二层: mid-aged tokens go to the quantised tier): in every unit whose
 * recent window is full, the oldest recent token is quantise-packed (K at middle_k_bits, V
 * at middle_v_bits, or with FADE_V_PQ V encoded by the fade_pq_encode rule against
 * layer->pq_codebook, its scale slots set to 0) into the next middle slot of the live buffer
 * and its score moves with it; its cache index is unchanged. FADE_ERR_CAPACITY if a middle
 * slot would overflow. fade_cache_prefill codes its middle tier the same way. */
fade_status_t fade_cache_demote(const fade_config_t* cfg, fade_layer_t* layer, void* stream);

/* Evict and re-position (FADE-zh §驱逐策略: on reaching INT4_BUDGET tokens are evicted and
 * keys are un-RoPE'd at the old position and re-RoPE'd at the contiguous StreamingLLM
 * position; FADE-zh §RoPE重计算: fp32 math, cast through fp16; FADE-zh §四种驱逐策略详解).
 * In every unit holding more than int4_budget middle tokens, the excess middle tokens with
 * the smallest key (score, index) — (index) for the position policy — are dropped (equal
 * scores: the lower index goes first). Survivors are compacted into the other middle
 * buffer, which becomes live; every survivor whose index drops is re-positioned: a middle
 * key is dequantised, rotated back from its old index and forward to its new one in fp32,
 * cast to fp16 and re-quantised; recent keys are re-positioned in place; V codes, V scales
 * and scores move unchanged. A no-op for FADE_EVICT_NONE or a negative budget. */
fade_status_t fade_evict_rerope(const fade_config_t* cfg, fade_layer_t* layer,
                                const float* table, int32_t max_pos, void* stream);

/* Append (FADE-zh §第一层): the new token of every unit: k_rot, v fp16 [B][H][d], the key
 * already RoPE'd at fade_next_position(). It becomes a sink while fewer than n_sink sinks
 * are held, else the newest recent token; its score starts at 0. FADE_ERR_CAPACITY if the
 * recent window is full (demote first). */
fade_status_t fade_cache_append(const fade_config_t* cfg, fade_layer_t* layer,
                                const uint16_t* k_rot, const uint16_t* v, void* stream);

/* A decode step's RoPE and append in one launch (FADE-zh §第一层 and §RoPE方案兼容性): the
 * result of fade_rope_apply on q_raw (fp16 [B][Hq][d]) into q_rot and on k_raw (fp16
 * [B][H][d]), every vector of row b at position pos[b] (pos: DEVICE i32 [B]; group_len Hq
 * resp. H, pos_step 0), followed by fade_cache_append of the rotated key and v (fp16
 * [B][H][d]), bit for bit; the rotated key goes straight into its slot (no k_rot buffer).
 * demote != 0: fade_cache_demote first, in the same launch (for a step in which no eviction
 * separates the demotion from the append: a cache that does not evict, or whose middle tier
 * stays within its budget). table / max_pos as for fade_rope_apply (unused for
 * FADE_ROPE_NONE: a copy). Errors as for the calls it replaces (FADE_ERR_CAPACITY: the recent
 * window full without demotion, or the middle tier full), before any launch. */
fade_status_t fade_rope_append(const fade_config_t* cfg, fade_layer_t* layer, const float* table,
                               int32_t max_pos, const uint16_t* q_raw, const uint16_t* k_raw,
                               const uint16_t* v, const int32_t* pos, uint16_t* q_rot,
                               int32_t demote, void* stream);

/* Decode attention (FADE-zh §项目结构与代码质量, kernels/: fused INT4 dequant + SDPA; KVLong
 * §1.2: softmax-weighted average of V). q_rot: fp16 [B][Hq][d] RoPE'd at the new token's
 * position; out: fp16 [B][Hq][d]. Every query head h attends, with scale 1/sqrt(d), to
 * every token held by its KV head h / (Hq/Hkv): sinks, middle (dequantised in registers;
 * with FADE_V_PQ the middle V is each sub-space's centroid from layer->pq_codebook) and
 * recent. Split-KV over SMs: partials go to `ws` (ws_bytes >= fade_layout().attn_ws),
 * then a combine writes out and ml_ws = f32 [B][Hq][2] (max logit M, sum L of exp(s - M)).
 * If logits_ws is not NULL (f32 [B][Hq][S + C + W]) the scaled logits s are stored at the
 * token's storage slot: sink i at i, middle slot m at S + m, ring slot r at S + C + r. */
fade_status_t fade_decode_attention(const fade_config_t* cfg, const fade_layer_t* layer,
                                    const uint16_t* q_rot, uint16_t* out, float* logits_ws,
                                    float* ml_ws, void* ws, size_t ws_bytes, void* stream);

/* Tokens per middle tile of the tensor-core attention kernel's schedule. */
#define FADE_ATTN_TILE_TOKENS 256

/* Host: 1 if fade_decode_attention's launch is scheduled by middle tiles (the tensor-core
 * kernel, which every valid configuration runs: INT4 or INT2 middle K with INT2, INT4 or
 * PQ-coded V), 0 otherwise, -1 for an invalid configuration (fade_last_error says why). The
 * launch is scheduled (stream-K) from every row's number of FADE_ATTN_TILE_TOKENS-token middle
 * tiles as the host mirror holds them at the call, and reads every other count on the device:
 * a captured call (CUDA graph) stays valid while those tile counts are unchanged. */
int32_t fade_attention_tiled(const fade_config_t* cfg);

/* Decode attention for callers that cannot allocate device memory. The pages have no
 * counterpart to this call; it exists for code that may not call cudaMalloc (or any
 * allocator) where attention runs: an allocator-free region of a serving loop, a plugin that
 * is handed only its inputs and outputs, or code that must not touch a memory pool it does not
 * own. It computes exactly what fade_decode_attention computes, with the same arguments except
 * the workspace: the split-KV partials go to a fixed array inside the library, of
 * FADE_NOALLOC_SCRATCH_BYTES (8 MiB) per GPU, which every GPU that loads the library holds
 * until the process exits.
 *   - The first call on a device looks up the array's device address with that device current
 *     (cudaGetSymbolAddress); make the first call on each device before any stream capture.
 *   - All calls on a device share the one array, which keeps the last call's contents. Calls
 *     that overlap on the GPU (unordered streams) race; order them, e.g. on one stream. No part
 *     of the array needs to start at zero: each call writes every partial before reading it.
 *   - A shape whose partials (B * Hq * splits * (d + 2) * 4 bytes, plus 4 bytes per unit)
 *     exceed the array is
 *     rejected on the host with FADE_ERR_CAPACITY and a message naming the limit.
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library routine. */
fade_status_t fade_decode_attention_noalloc(const fade_config_t* cfg, const fade_layer_t* layer,
                                            const uint16_t* q_rot, uint16_t* out,
                                            float* logits_ws, float* ml_ws, void* stream);

/* Accumulate attention mass (FADE-zh §四种驱逐策略详解 1 H2O, 2 EMA; KVLong §1.3.1 H2O: the
 * score of a token sums its attention). With p[h][j] = exp(s[h][j] - M[h]) / L[h] from the
 * preceding fade_decode_attention's logits_ws and ml_ws: H2O adds sum over the unit's query
 * heads of p to every held token's score; EMA sets score = delta*score + (1-delta)*sum p.
 * A no-op for the position and none policies. */
fade_status_t fade_h2o_accumulate(const fade_config_t* cfg, fade_layer_t* layer,
                                  const float* logits_ws, const float* ml_ws, void* stream);

/* Host: cache position of row `row`'s next token = held tokens after the next step's
 * demotion and eviction (KVLong §1.2.2: positions inside the cache). -1 on bad arguments. */
int32_t fade_next_position(const fade_config_t* cfg, const fade_layer_t* layer, int32_t row);

/* Host: the layer's tier counts from the host mirror (FADE-zh §遥测与调试: tokens per tier):
 * out = HOST i32 [B][3] = (sinks, middle, recent) of every row (the same for all KV heads). */
fade_status_t fade_tier_counts(const fade_config_t* cfg, const fade_layer_t* layer,
                               int32_t* out);

/* Host: KV bytes held by the layer (FADE-zh §使用注意事项 3, compressed_storage_bytes: KV
 * storage only): FP16 tokens at 4d bytes, middle tokens at d*(kb+vb)/8 code bytes plus two
 * fp16 scales per 32 channels. */
uint64_t fade_compressed_bytes(const fade_config_t* cfg, const fade_layer_t* layer);

/* Host, synchronising: wait for the work queued on `stream`, then read the layer's device
 * status words. FADE_ERR_TIMEOUT if a kernel of this layer gave up a bounded wait since the
 * last fade_cache_reset (every wait on an mbarrier or a bulk copy is bounded, about 2 s; the
 * kernel then records a code in status[0] and returns instead of hanging);
 * FADE_ERR_DEVICE_CHECK if a kernel's index guard failed (codes >= 16: the guard skips the
 * access and records its code; a library built with FADE_DEBUG=1 adds such guards on every
 * compacted row and attention tile); in both cases the results of the calls since are
 * invalid. FADE_ERR_CUDA if the stream reports an error; FADE_OK otherwise. The asynchronous
 * calls never read the status words: this is the call that turns them into an error. */
fade_status_t fade_check_status(const fade_layer_t* layer, void* stream);

/* Self-test of the bounded waits: one kernel in which a consumer waits on an mbarrier with
 * the same bounded wait the attention kernel uses, for at most `limit_cycles` SM clock cycles
 * (1 .. the kernels' own limit of 4e9), while a producer warp arrives on it only if
 * `producer_arrives` is nonzero. On a timeout the kernel writes code 1 into status[0]
 * (device i32, unless status[0] is already nonzero) and returns. Lets a test make a wait run
 * out without a fault or a hang and check that fade_check_status reports it. */
fade_status_t fade_selftest_bounded_wait(int32_t* status, int32_t producer_arrives,
                                         int64_t limit_cycles, void* stream);

/* Measurement helper (no counterpart in the pages; it serves the roofline of
 * fade_evict_rerope, whose cost is fp32 arithmetic): launches `blocks` CTAs of 256 threads in
 * which every thread runs `iters` rounds of eight independent chains of packed fp32 multiplies
 * (mul.rn.f32x2, two separately rounded fp32 operations per lane per instruction) on
 * registers. *ops_out (host, may be NULL) receives the fp32 operations the launch performs;
 * timed with events on `stream` this is the device's rate of separately rounded fp32
 * operations. sink: device f32 [256], never written in practice (keeps the chains alive). */
fade_status_t fade_measure_fp32_rate(int32_t blocks, int32_t iters, float* sink,
                                     double* ops_out, void* stream);

/* The calling thread's last error message ("" if none). */
const char* fade_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FADE_H_ */
