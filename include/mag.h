/*
 * mag -- the single-token decode step of a GQA transformer with 4-bit
 * group-quantised weights (W4A16) and a block-pooled KV cache in FP16, INT8
 * or INT4, on one GB300 (sm_103a). C ABI.
 *
 * Pages this interface follows (cited by title and section):
 *   [Magnitude] "Magnitude: on-device AI-agent inference engine --
 *               self-optimising scheduling and elastic memory pools"
 *               (0539edu.com): 4.3 engine config and construction,
 *               4.4 inference calls, 5.1 context overflow, 5.2 memory stats.
 *   [Core]      "5. Core modules: format, runtime, scheduling, memory and
 *               routing" (ai-infra.cypggs.com): 5.1 packager (W4A16, merged
 *               QKV and gate-up, pre-generated RoPE table, shapes in the
 *               package), 5.2 runtime (preallocated KV pool, static shapes,
 *               allocation-free decode loop), 5.4 KV capacity planning.
 *   [TFLite]    "TFLite memory planner" (pwwt.cn): 2.1-2.2 lifetime analysis
 *               and greedy-by-size arena, 3.2 preserve-all debug mode and
 *               externally owned I/O buffers.
 *
 * Conventions for every call:
 *   - Ownership: the library owns every device allocation it makes (weights,
 *     KV pool, block tables, RoPE table, activation arena, graphs). The caller
 *     owns the CUDA stream and every input/output buffer it passes; those are
 *     never placed in the arena ([TFLite] 3.2, external buffers).
 *   - Ordering: calls are ordered on the context's stream (given at create);
 *     except where stated they return without synchronising the host.
 *   - Errors: every call returns mag_status. Argument and capacity errors are
 *     found on the host before anything is launched and leave the context
 *     unchanged (no partial append). mag_last_error() gives a message.
 *   - Threads: one context is used by one host thread at a time.
 *   - Pointers named *_dev are device pointers; *_host are host pointers.
 */
#ifndef MAG_H
#define MAG_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MAG_OK = 0,
  MAG_ERR_INVALID_ARG = 1,  /* bad shape, pointer, id, size or format */
  MAG_ERR_OOM = 2,          /* a device or pinned-host allocation failed */
  MAG_ERR_KV_FULL = 3,      /* the block pool has too few free blocks */
  MAG_ERR_CONTEXT_FULL = 4, /* a session would pass max_context (never truncated) */
  MAG_ERR_NOT_LOADED = 5,   /* a step was asked for before every weight was loaded */
  MAG_ERR_CUDA = 6,         /* a CUDA runtime call failed (message says which) */
  MAG_ERR_TIMEOUT = 7,      /* a bounded device-side wait gave up */
  MAG_ERR_UNSUPPORTED = 8,  /* a shape or mode this build does not handle */
  MAG_ERR_CORRUPT = 9       /* a device-side check found a write outside an arena tensor (MAG_FLAG_DEBUG_CANARY)
                               or a block-table entry outside the pool; the message says which */
} mag_status;

typedef enum { MAG_KV_FP16 = 0, MAG_KV_INT8 = 1, MAG_KV_INT4 = 2 } mag_kv_dtype;

/* Flags. */
#define MAG_FLAG_NO_GRAPH ((uint64_t)1)        /* launch kernels one by one instead of replaying a CUDA graph */
#define MAG_FLAG_ARENA_NO_REUSE ((uint64_t)2)  /* give every arena tensor its own bytes ([TFLite] 3.2 preserve-all) */
#define MAG_FLAG_NO_PDL ((uint64_t)4)          /* no programmatic dependent launch between kernels */
/* Elastic KV pool ([Magnitude] 2.2 layer 1, 3.2 hot / cold pool): pool_blocks becomes a reserved virtual
 * range (rounded up to whole mapping groups); device memory is mapped a group at a time (zeroed), the
 * lowest groups up to the hot size stay mapped, a group above it is mapped when the free blocks run out
 * and returned to the device once wholly free (after the stream has passed its last use). The hot size
 * is one group, or, with the adaptive runtime on, hot_pool_slack x the P90 need (mag_set_adaptive).
 * Free blocks go out lowest id first. pool_order_host must be NULL. */
#define MAG_FLAG_ELASTIC_POOL ((uint64_t)8)
/* Time every step with a pair of CUDA events around its launches (mag_get_step_stats.last_ms). */
#define MAG_FLAG_STEP_TIMING ((uint64_t)16)
/* Debug: 64-byte canary bands before and after every decode-arena tensor (the arena then reuses no bytes,
 * as with MAG_FLAG_ARENA_NO_REUSE), checked by one more kernel at the end of every decode or verify step;
 * a changed band makes the next mag_sync return MAG_ERR_CORRUPT naming the tensor, and the bands are
 * rewritten. (Every step also checks each pool block id it reads from a block table against the pool: an
 * id outside it is not used, the step's results are wrong, and mag_sync returns MAG_ERR_CORRUPT; the
 * device tables are then rewritten from the host's copy.) */
#define MAG_FLAG_DEBUG_CANARY ((uint64_t)32)

/* Model shape and capacities ([Core] 5.1: the shape travels with the model;
 * [Core] 5.2: everything sized once, up front; [Magnitude] 4.3: EngineConfig). */
typedef struct mag_config {
  int32_t n_layers;
  int32_t hidden;     /* D */
  int32_t n_heads;    /* Hq */
  int32_t n_kv_heads; /* Hkv; Hq % Hkv == 0, query head h reads KV head h / (Hq/Hkv) */
  int32_t head_dim;   /* d: 64 or 128 */
  int32_t ffn;        /* F */
  int32_t vocab;      /* V; 0 = no LM head, the step outputs the fp16 hidden state */
  float rms_eps;
  float rope_base;
  int32_t kv_dtype;     /* mag_kv_dtype */
  int32_t block_tokens; /* tokens per KV block; must be 16 */
  int32_t pool_blocks;  /* P, blocks in the pool (each covers every layer) */
  int32_t max_sessions;
  int32_t max_batch;   /* sessions per decode step, 1..16 */
  int32_t max_chunk;   /* tokens per prefill chunk; 0 = prefill not used */
  int32_t max_context; /* tokens a session may hold */
  const int32_t* pool_order_host; /* initial free-list order, a permutation of 0..P-1; NULL = 0,1,..,P-1 */
  uint64_t flags;                 /* MAG_FLAG_* */
} mag_config;

typedef struct mag_ctx mag_ctx;

/* Create a context: validates the shape, plans the activation arena
 * ([TFLite] 2.1-2.2, 64-byte aligned offsets), allocates the weight region,
 * the KV pool of pool_blocks blocks ([Core] 5.2) and the block tables, and
 * builds the RoPE cos/sin table on the host in double, stored as fp32
 * ([Core] 5.1, rope table pre-generation). `cuda_stream` is a cudaStream_t
 * on which all work of the context is ordered (NULL: the context creates and
 * owns a stream that synchronises with the legacy default stream).
 * Errors: INVALID_ARG, UNSUPPORTED, OOM, CUDA; *out is NULL on error. */
mag_status mag_create(const mag_config* cfg, void* cuda_stream, mag_ctx** out);

/* Free everything the context owns (synchronises its stream first). NULL is a no-op. */
void mag_destroy(mag_ctx* ctx);

/* Tensors of mag_load_weights. Projections are merged as [Core] 5.1 rewrites
 * them: QKV rows [q (Hq*d); k (Hkv*d); v (Hkv*d)], gate-up rows [gate (F); up (F)]. */
typedef enum {
  MAG_W_QKV = 0,      /* [(Hq+2Hkv)d, D] */
  MAG_W_O = 1,        /* [D, Hq*d] */
  MAG_W_GATE_UP = 2,  /* [2F, D] */
  MAG_W_DOWN = 3,     /* [D, F] */
  MAG_NORM_ATTN = 4,  /* gain [D] before attention */
  MAG_NORM_FFN = 5,   /* gain [D] before the FFN */
  MAG_NORM_FINAL = 6, /* gain [D] before the LM head (layer ignored) */
  MAG_LM_HEAD = 7     /* [V, D] fp16 (layer ignored) */
} mag_tensor;

/* Source formats. W4G32 is the packed 4-bit group-32 layout ([Core] 5.1
 * W4A16; the byte layout is this library's): a matrix [N, K] has G =
 * ceil(K/32) groups per row; its bytes are the codes u8 [N][16G] (byte j of a
 * group holds code 2j in the low nibble and code 2j+1 in the high nibble,
 * ragged last group padded with code 0) immediately followed by the fp16
 * (scale, min) pairs [N][G][2]; element k of a row is scale*code + min. */
typedef enum {
  MAG_FMT_F32_DENSE = 0, /* fp32 row-major [N, K]; quantised to W4G32 on the device (projections only) */
  MAG_FMT_W4G32 = 1,     /* already packed (projections only) */
  MAG_FMT_F16 = 2        /* fp16 (norm gains, LM head) */
} mag_format;

/* Load one tensor from device memory `src_dev` of `bytes` bytes (which must
 * equal the size the format and shape imply). FP32_DENSE is quantised on the
 * device by the rule of mag_quantize_w4g32. Ordered on the stream; src_dev
 * may be reused once the stream reaches this point.
 * Errors: INVALID_ARG (id, layer, format, size), CUDA. */
mag_status mag_load_weights(mag_ctx* ctx, int32_t tensor, int32_t layer, const void* src_dev, int32_t src_format,
                            size_t bytes);

/* Load one fp32 projection (MAG_W_QKV..MAG_W_DOWN; [N, K] row-major, bytes =
 * N*K*4, device memory) like mag_load_weights with MAG_FMT_F32_DENSE, to the
 * same bytes, but without allocating device memory. The pages have no
 * counterpart: it is for callers that cannot allocate at load time -- a
 * process whose KV pool was sized to take the HBM left after the weights, or
 * one that forbids device allocation after start-up -- where the ordinary
 * path's transient W4G32 copy of the whole projection (up to N*K*5/8 bytes)
 * would fail. The projection goes through one 4 MiB scratch buffer that is part
 * of the library image, one per device, in slabs of whole 16-row tiles
 * (QKV: whole heads); nothing in the scratch needs to start at zero.
 * A tile of rows of K values takes 16 * ceil(K/32) * 20 bytes: a projection
 * whose smallest slab (one tile; QKV: one head of d/16 tiles) exceeds 4 MiB
 * -- K above 419,424; QKV K above 52,416 (d = 128) or 104,832 (d = 64) -- is
 * rejected with INVALID_ARG. The context's device must be current. The first call on each
 * device looks the scratch's address up, and so does the first call after the
 * device's context was replaced (a device reset); make those calls before any
 * stream capture begins. Ordered on the context's stream; src_dev may be reused once the
 * stream reaches this point. Calls that overlap in time on one device (other
 * streams, threads or contexts) race on the shared scratch: order them.
 * Errors: INVALID_ARG (id, layer, size, scratch limit, device), CUDA. */
mag_status mag_load_weights_f32_noalloc(mag_ctx* ctx, int32_t tensor, int32_t layer, const void* src_dev,
                                        size_t bytes);

/* Sessions: each holds its own block table and length. Close returns its
 * blocks to the back of the free list. Errors: INVALID_ARG, and OOM-like
 * MAG_ERR_INVALID_ARG when max_sessions are open. */
mag_status mag_session_open(mag_ctx* ctx, int32_t* session_out);
mag_status mag_session_close(mag_ctx* ctx, int32_t session);
mag_status mag_session_length(mag_ctx* ctx, int32_t session, int32_t* length_out);

/* Shorten a session to `length` tokens (0..its length), e.g. to drop draft
 * tokens that mag_verify_tokens appended and the caller rejected. Blocks
 * wholly past the new length go back to the free list; the tokens past it are
 * never read again and the next append overwrites them. The pages have no
 * counterpart (their speculative controller, [Core] 5.6, is out of scope;
 * only this step of it is built). Host-only, no launch. Errors: INVALID_ARG. */
mag_status mag_session_truncate(mag_ctx* ctx, int32_t session, int32_t length);

/* Append n_tokens of already-rotated K and V to a session's cache, fp16
 * [L][n_tokens][Hkv][d] each, quantised on store to the pool precision
 * (INT8: one fp16 scale per token and head, s = fp16(max|x|/127), q =
 * rint(x/s) clamped to +-127; INT4: the W4G32 rule along head_dim). Blocks
 * are taken from the free list when a token index is a multiple of 16.
 * Errors: INVALID_ARG, CONTEXT_FULL, KV_FULL (nothing is appended), CUDA. */
mag_status mag_kv_append(mag_ctx* ctx, int32_t session, int32_t n_tokens, const void* k_dev, const void* v_dev);

/* One decode step ([Magnitude] 4.4 infer, one token; [Core] 5.2 tight decode
 * loop): for each of `batch` distinct sessions, take the fp16 hidden state
 * hidden_in_dev[b][D] of its next token, run every layer (RMSNorm, W4 QKV,
 * RoPE at the session's position, KV append, attention over the pool, W4 O +
 * residual, RMSNorm, W4 gate-up + SwiGLU, W4 down + residual) and write
 * out_dev[b][V] fp16 logits (or [b][D] fp16 hidden state when vocab == 0).
 * The session's length grows by one. Replays a CUDA graph captured on the
 * first step of each batch size. The residual stream is kept in fp32.
 * Errors: INVALID_ARG, CONTEXT_FULL, KV_FULL, NOT_LOADED, CUDA. */
mag_status mag_decode_step(mag_ctx* ctx, int32_t batch, const int32_t* session_ids_host, const void* hidden_in_dev,
                           void* out_dev);

/* The same step with HOST buffers: copies hidden_in_host to the device,
 * runs the step, copies the output back into out_host and synchronises. */
mag_status mag_decode_step_host(mag_ctx* ctx, int32_t batch, const int32_t* session_ids_host,
                                const void* hidden_in_host, void* out_host);

/* Chunked prefill ("5. Core modules" 5.1 W4A16 model, 5.2 block pool): append
 * n_tokens (1..max_chunk) of one session at its next positions, with causal
 * attention over the session's cache and the chunk itself, and write the fp16
 * output (logits, or the hidden state when vocab == 0) of the chunk's last
 * token to last_out_dev. hidden_in_dev is fp16 [n_tokens][D]; the chunk's K/V
 * are stored in the pool like mag_kv_append's (the same quantisers). The
 * projections run as tensor-core GEMMs that read the W4 weights the decode
 * step reads and expand them in shared memory to fp16(s q + m), one rounding
 * per weight (no weight copy is kept; mag_get_memory_stats reports 0 for it).
 * Stream-ordered.
 * Errors: INVALID_ARG, CONTEXT_FULL, KV_FULL, NOT_LOADED, UNSUPPORTED (created
 * with max_chunk = 0), CUDA. */
mag_status mag_prefill_chunk(mag_ctx* ctx, int32_t session, int32_t n_tokens, const void* hidden_in_dev,
                             void* last_out_dev);

/* Chunked prefill of several sessions in one pass (the batched form of mag_prefill_chunk): session
 * session_ids_host[i] appends n_tokens_host[i] >= 1 tokens at its next positions; the sessions' rows
 * follow each other in hidden_in_dev (fp16 [sum n_tokens][D], session 0's first), the total at most
 * max_chunk, 1..16 distinct sessions. Each session's tokens attend causally to its own cache and to
 * its own earlier tokens of the chunk; the projections run once over all rows. last_out_dev receives
 * the fp16 output of every session's last token, [n_sessions][V] (or [n_sessions][D] when
 * vocab == 0), in the order given. Errors: as mag_prefill_chunk, and INVALID_ARG for a repeated
 * session; nothing is appended on error. */
mag_status mag_prefill_batch(mag_ctx* ctx, int32_t n_sessions, const int32_t* session_ids_host,
                             const int32_t* n_tokens_host, const void* hidden_in_dev, void* last_out_dev);

/* Multi-token verify step (draft tokens of speculative decoding checked in
 * one pass, [Core] 5.6): n_tokens tokens of one session at its next
 * positions, writing the fp16 output of every token, out_dev[n_tokens][V] (or
 * [n_tokens][D] when vocab == 0): token j attends causally to the session's
 * cache and tokens 0..j. hidden_in_dev is fp16 [n_tokens][D]. All n_tokens
 * are appended; mag_session_truncate drops the rejected ones. With
 * n_tokens <= max_batch it runs as a decode step whose rows are the tokens
 * (each W4 matrix read once for all of them; one captured graph per count);
 * otherwise, with n_tokens <= min(4, max_chunk), through the prefill chunk
 * path. Errors: INVALID_ARG (count outside both ranges, session, buffers),
 * CONTEXT_FULL, KV_FULL, NOT_LOADED, CUDA. */
mag_status mag_verify_tokens(mag_ctx* ctx, int32_t session, int32_t n_tokens, const void* hidden_in_dev,
                             void* out_dev);

/* Wait for the context's stream and read the device error word
 * (MAG_ERR_TIMEOUT if a bounded device wait gave up). */
mag_status mag_sync(mag_ctx* ctx);

typedef struct mag_memory_stats {
  uint64_t weight_bytes;       /* packed W4 + scales + norm gains + LM head */
  uint64_t kv_pool_bytes;      /* L * P * block bytes */
  uint64_t kv_block_bytes;     /* bytes of one (layer, block) */
  int32_t pool_blocks_total;
  int32_t pool_blocks_free;
  uint64_t arena_bytes;        /* planned activation arena */
  uint64_t arena_unshared_bytes; /* sum of the arena tensors' sizes (no reuse) */
  uint64_t other_device_bytes; /* block tables, RoPE table, counters, step arguments */
  int32_t sessions_open;
  uint64_t prefill_weight_bytes; /* weight copies kept for the prefill GEMM: 0 (it reads the W4 tiles) */
  uint64_t prefill_arena_bytes;  /* planned prefill activation arena (max_chunk rows) */
  /* KV pool memory: a fixed pool has it all mapped; an elastic one (MAG_FLAG_ELASTIC_POOL) maps groups of
   * pool_group_blocks blocks: the hot ones (pool_blocks_hot) stay, others come and go with demand */
  uint64_t kv_pool_mapped_bytes;
  int32_t pool_blocks_mapped;
  int32_t pool_blocks_hot;
  int32_t pool_group_blocks;
} mag_memory_stats;

/* [Magnitude] 5.2 get_memory_stats: weights, pool, arena. */
mag_status mag_get_memory_stats(mag_ctx* ctx, mag_memory_stats* out);

/* Statistics of the context's steps ([Magnitude] 4.4 InferenceResult timing, per step): the last decode,
 * verify or prefill call and the running count. last_bytes models the step's device traffic: the weights
 * read once (packed W4, scales, norm gains, LM head), every row's KV up to the keys it attends, and the
 * hidden states in and the logits (or hidden states) out. */
typedef struct mag_step_stats {
  int64_t steps;             /* decode, verify and prefill calls that launched work since create */
  int32_t last_kind;         /* 0 decode step, 1 verify on the decode kernels, 2 the chunk path (prefill / verify) */
  int32_t last_rows;         /* token rows of the last call (batch, drafts or chunk tokens) */
  int32_t last_launches;     /* kernel launches of the last call */
  int32_t last_max_keys;     /* most keys one row of the last call attends */
  uint64_t last_bytes;       /* modelled device bytes of the last call */
  double last_ms;            /* device time of the last call (MAG_FLAG_STEP_TIMING), else -1 */
} mag_step_stats;

/* Statistics of the last call; with MAG_FLAG_STEP_TIMING this waits for that call to finish.
 * Errors: INVALID_ARG (null), CUDA. */
mag_status mag_get_step_stats(mag_ctx* ctx, mag_step_stats* out);

/* Message of the last error on this context (never NULL; "" if none). */
const char* mag_last_error(mag_ctx* ctx);

/* [Core] 5.4 KV capacity planning: bytes one token adds to the pool over all
 * layers, 2 * L * Hkv * d * bytes per value, plus this library's per-token
 * scale metadata for INT8 (2 B per head) and INT4 (4 B per 32 values). */
uint64_t mag_kv_bytes_per_token(const mag_config* cfg);

/* Stateless quantiser ([Core] 5.1 W4A16 packing): fp32 [rows, cols] on the
 * device -> codes u8 [rows][16G] and (scale, min) fp16 [rows][G][2], G =
 * ceil(cols/32). Per group of 32 consecutive values: m = fp16(min), s =
 * fp16((max - min)/15) (fp32 subtract, IEEE divide), code = clamp(rint((x -
 * m)/s), 0, 15) in fp32 (0 when s == 0). Ordered on `cuda_stream`.
 * Errors: INVALID_ARG, CUDA. */
mag_status mag_quantize_w4g32(const void* src_dev, int64_t rows, int64_t cols, void* codes_dev, void* scale_min_dev,
                              void* cuda_stream);

/* ---- adaptive runtime: load profile, plan switching, hot pool size ----
 * [Magnitude] 2.1-2.2, 3.1-3.3, 4.3 and 6.1-6.2: a profile of recent
 * inferences (sliding window, sampled) whose P90 length picks one of three
 * preset plans (short / medium / long sequences) and sizes the hot KV pool.
 * Here an "inference" is one session row of a decode or verify step, and its
 * length is the context that row attends to (its position + 1). A plan is a
 * decode-attention split count (the thread-block cluster size over a
 * session's keys); each plan has its own captured graphs, and a switch swaps
 * which graphs the step launches. */
typedef struct mag_adapt_config {
  int32_t enable_adaptive;       /* 0: the profile and every policy are off (the default state) */
  int32_t adaptive_window_size;  /* recorded inferences in the window; the pages' default 64 */
  int32_t adaptive_sample_rate;  /* one inference in this many is recorded; default 4 */
  int32_t plan_short_below;      /* P90 below this: short plan (0); default 128 */
  int32_t plan_long_above;       /* P90 above this: long plan (2); between the two, medium (1); default 512 */
  int32_t plan_splits[3];        /* attention splits of plans 0, 1, 2 for one session, 0..64 (0 = the
                                    default: about 2 blocks per SM, at most one cluster of 16); a
                                    batch of B is capped at 4 x SMs / (B x Hkv); more splits than the
                                    device's largest co-scheduled cluster run as up to 8 clusters of 8
                                    whose outputs the last block to finish merges */
  int32_t plan_wide[3];          /* 1: plan p runs the wide attention blocks (8 warps at head_dim 128,
                                    16 at 64; one block per SM) instead of 4-warp blocks */
  int32_t force_plan;            /* -1: plans follow the profile; 0..2: that plan, always */
  int32_t async_switch;          /* 1: a new plan's graphs are captured on a background thread and the
                                    step keeps the old plan until they are ready */
  float hot_pool_slack;          /* hot pool = slack x the blocks of the P90 length per open session;
                                    default 1.2 */
} mag_adapt_config;

/* The pages' defaults (enable_adaptive = 1, window 64, rate 4, thresholds 128 / 512, no forced plan,
 * no async switch, slack 1.2) and split counts 4 / 8 / 16 measured on GB300 for the three plans. */
void mag_adapt_defaults(mag_adapt_config* out);

/* Turn the adaptive runtime on (or off with enable_adaptive = 0) and reset its profile. The plan in use
 * stays until the first decision. Errors: INVALID_ARG (window or rate < 1, thresholds out of order,
 * split or plan out of range). */
mag_status mag_set_adaptive(mag_ctx* ctx, const mag_adapt_config* cfg);

typedef struct mag_profile {
  int64_t seen;        /* inferences offered to the profile */
  int32_t recorded;    /* in the window (<= adaptive_window_size) */
  int32_t p50, p90, p99; /* nearest-rank quantiles of the window; -1 while it is empty */
  int32_t plan;        /* plan the next step launches */
  int32_t pending_plan; /* plan whose graphs a background capture is building; -1 if none */
  int32_t plan_splits; /* attention split count of `plan` */
  int32_t plan_wide;   /* whether `plan` runs the wide attention blocks */
  int32_t switches;    /* plan changes so far */
  int64_t hot_blocks;  /* hot pool target from the last full window; -1 before one */
} mag_profile;
mag_status mag_get_profile(mag_ctx* ctx, mag_profile* out);

/* The profile on its own (host only, no context or GPU), for callers that keep their own statistics:
 * observe returns 1 when the value was recorded (the first observation, then every sample_every-th);
 * quantile is nearest-rank over the window (the ceil(q n)-th smallest, q in (0, 1]; -1 if empty). */
typedef struct mag_profiler mag_profiler;
mag_status mag_profiler_create(int32_t window, int32_t sample_every, mag_profiler** out);
void mag_profiler_destroy(mag_profiler* p);
int32_t mag_profiler_observe(mag_profiler* p, int32_t length);
mag_status mag_profiler_quantile(const mag_profiler* p, double q, int32_t* out);
int32_t mag_profiler_count(const mag_profiler* p);
/* The two policies as pure functions: plan of a P90 length (0 below short_below, 2 above long_above,
 * else 1), and the hot pool in blocks, ceil(slack x n_sessions x ceil(p90 / 16)) with slack taken to
 * six decimals (0 when p90 or n_sessions is not positive). */
int32_t mag_plan_for(int32_t p90, int32_t short_below, int32_t long_above);
int64_t mag_hot_pool_blocks(int32_t p90, int32_t n_sessions, float slack);

/* ---- debug and test hooks ---- */

/* Copy a loaded projection back in W4G32 bytes (codes then pairs) into dst_dev. */
mag_status mag_debug_read_weights(mag_ctx* ctx, int32_t tensor, int32_t layer, void* dst_dev, size_t bytes);

/* Byte offsets in the pool of token `token` of a session at `layer`, for KV
 * head 0: out[0] K data, out[1] V data, out[2] K meta, out[3] V meta (meta =
 * -1 for FP16); head h adds h * 16 * (bytes of one vector or its meta).
 * out[4] is the physical block id. */
mag_status mag_debug_kv_locate(mag_ctx* ctx, int32_t session, int32_t layer, int32_t token, int64_t out[5]);

/* Device pointer and size of the KV pool, for reading stored bytes. */
mag_status mag_debug_pool(mag_ctx* ctx, void** pool_dev, uint64_t* bytes);

typedef struct mag_arena_tensor {
  char name[24];
  uint64_t size;   /* bytes */
  int32_t first;   /* first op index (producer) */
  int32_t last;    /* last op index (last consumer), closed interval */
  uint64_t offset; /* planned offset, multiple of 64 */
} mag_arena_tensor;

/* The activation arena plan of phase 0 (decode step at max_batch) or 1
 * (prefill chunk at max_chunk): up to `cap` tensors into out, their count into
 * n_out and the arena size into arena_bytes. */
mag_status mag_debug_arena_plan(mag_ctx* ctx, int32_t phase, mag_arena_tensor* out, int32_t cap, int32_t* n_out,
                                uint64_t* arena_bytes);

/* Debug: write one entry of a session's block table on the device only (the host keeps its own copy), to
 * test the block-id checks of MAG_ERR_CORRUPT. Synchronous. Errors: INVALID_ARG (session not open, index
 * past the session's blocks), CUDA. */
mag_status mag_debug_set_table_entry(mag_ctx* ctx, int32_t session, int32_t index, int32_t value);

/* Debug: the decode activation arena's device address and size (the offsets of mag_debug_arena_plan phase
 * 0 are relative to it; with MAG_FLAG_DEBUG_CANARY a tensor's bytes start kCanaryBand = 64 bytes into its
 * planned slot, after its leading band). */
mag_status mag_debug_arena(mag_ctx* ctx, void** ptr, uint64_t* bytes);

/* Kernel launches of the last decode step (0 if none ran yet). */
int32_t mag_debug_last_step_launches(mag_ctx* ctx);

/* Kinds of kernel launch reported by mag_debug_profile_step. */
typedef enum {
  MAG_OP_STEP_BEGIN = 0, /* block-table writes, fp16 input -> fp32 residual, RMSNorm of layer 0 */
  MAG_OP_QKV = 1,        /* W4 QKV GEMV + RoPE of q and k */
  MAG_OP_ATTENTION = 2,  /* K/V append into the pool + split-K attention + split merge */
  MAG_OP_O = 3,          /* W4 O GEMV + residual + RMSNorm (last block) */
  MAG_OP_GATE_UP = 4,    /* W4 gate-up GEMV + SwiGLU */
  MAG_OP_DOWN = 5,       /* W4 down GEMV + residual + next RMSNorm or output (last block) */
  MAG_OP_LM_HEAD = 6     /* fp16 LM head GEMV */
} mag_op;

/* One decode step like mag_decode_step but launched kernel by kernel (no
 * graph, no programmatic dependent launch) with a CUDA event pair around each
 * launch on the context's stream; synchronises, then writes the launch count
 * to n_out and, for the first `cap` launches, kinds[i] (mag_op) and ms[i]
 * (device time between the pair). The session lengths advance as in a step. */
mag_status mag_debug_profile_step(mag_ctx* ctx, int32_t batch, const int32_t* session_ids_host,
                                  const void* hidden_in_dev, void* out_dev, int32_t* kinds, float* ms, int32_t cap,
                                  int32_t* n_out);

/* One decode step like mag_decode_step, launched kernel by kernel (no graph, no programmatic dependent
 * launch), that also copies the fp32 residual stream of every row into resid_dev (device memory, fp32
 * [L+1][batch][D], caller-owned): row 0 is the input hidden state widened to fp32, row l+1 the residual
 * after layer l (after its down projection). Lets a test check the step one layer at a time against a
 * reference fed the same residual ([Core] 5.1: the pre-norm residual stream the layers share). The
 * session lengths advance as in a step; synchronises the context's stream.
 * Errors: as mag_decode_step; INVALID_ARG for a null resid_dev; TIMEOUT as mag_sync. */
mag_status mag_debug_step_residuals(mag_ctx* ctx, int32_t batch, const int32_t* session_ids_host,
                                    const void* hidden_in_dev, void* out_dev, void* resid_dev);

/* Step timeline ([Magnitude] 3.1: the load profile times each operator through built-in timing hooks;
 * here per kernel phase): one decode step like
 * mag_decode_step, its launches made one by one (with programmatic dependent launch, as in the step graph)
 * with a record buffer in their arguments. The GEMV and attention blocks append records of four uint64
 * {tag, block, event, time} to recs_dev (device memory, caller-owned, room for `cap` records = 32 cap
 * bytes): tag (1 << 60) | n_mtiles << 32 | n_chunks << 8 | batch for a GEMV, (2 << 60) | layer for
 * attention; block = blockIdx.x | y << 20 | z << 40; time = the GPU's global timer in ns. GEMV events: 0
 * block entry, 1 before its wait on the previous kernel (its first weight copies issued), 2 activations
 * staged. Attention events: 0 entry, 1 after the wait, 2 keys done, 3 end. Records past cap are dropped;
 * *n_out = the records attempted. The session lengths advance as in a step; synchronises the stream.
 * Errors: as mag_decode_step; INVALID_ARG for a null buffer or count, cap < 0. */
mag_status mag_debug_timeline(mag_ctx* ctx, int32_t batch, const int32_t* session_ids_host, const void* hidden_in_dev,
                              void* out_dev, void* recs_dev, int32_t cap, int32_t* n_out);

/* Failure injection for tests ([Magnitude] 5.1-5.2: the engine's error behaviour): the number of polls a
 * decode GEMV's pipeline wait (for its weight copies to land in shared memory) makes before it gives up.
 * polls < 0 restores the built-in limit (2^22); 0 makes every such wait give up at once, as if the copies
 * were stuck: the kernel then sets its bit in the error word, waits (within the built-in limit) for the
 * copies it has in flight, skips its arithmetic and returns, so the step's outputs are meaningless, the
 * next mag_sync returns MAG_ERR_TIMEOUT and the context stays usable (drop the step's token with
 * mag_session_truncate). Synchronises the stream; graphs captured under another limit are captured again.
 * Errors: INVALID_ARG (null context), CUDA. */
mag_status mag_debug_set_wait_limit(mag_ctx* ctx, int64_t polls);

/* Failure injection for tests ([Magnitude] 5.2: memory errors): process-wide, the next `skip` allocations
 * the library makes succeed and the `count` after them fail as if the device (or pinned host memory) were
 * full: device and pinned-host allocations, the stream-ordered scratch of an fp32 load, and the physical
 * memory of an elastic KV pool group. Each call that meets one returns MAG_ERR_OOM (an elastic pool that
 * can map no new group: MAG_ERR_OOM from the call that needed it) with the context unchanged and usable;
 * mag_create returns it with *out NULL, everything it had allocated freed. count <= 0 turns it off. */
void mag_debug_fail_allocations(int32_t skip, int32_t count);

/* A prefill chunk like mag_prefill_chunk, launched without programmatic dependent launch, that also copies
 * the fp32 residual of all n_tokens rows into resid_dev (device memory, fp32 [L+1][n_tokens][D],
 * caller-owned): row 0 the chunk's input widened to fp32, row l+1 the residuals after layer l. For checking
 * the chunk one layer at a time against a reference ([Core] 5.1, 5.2). Synchronises the context's stream.
 * Errors: as mag_prefill_chunk; INVALID_ARG for a null resid_dev; TIMEOUT as mag_sync. */
mag_status mag_debug_prefill_residuals(mag_ctx* ctx, int32_t session, int32_t n_tokens, const void* hidden_in_dev,
                                       void* last_out_dev, void* resid_dev);

#ifdef __cplusplus
}
#endif
#endif
