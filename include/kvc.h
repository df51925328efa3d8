/*
 * kvc.h -- compressed-KV-cache attention on one GB300 (sm_103a): the C ABI.
 *
 * Two halves of one serving path:
 *   prefill   score every prompt key by the attention a trailing observation
 *             window of queries pays it, max-pool the scores, keep a per-head
 *             top-k under a per-layer budget, and store the survivors as 2- or
 *             4-bit group-quantized codes (keys per channel, values per token,
 *             groups of 32, fp16 scale + zero-point per group);
 *   decode    append each new key/value to a bf16 recent window that is
 *             quantized group by group as it fills, and attend one query per
 *             head (GQA-aware) over packed codes + window in one softmax.
 *
 * Sources of the method (page title, section):
 *   PyramidKV: Dynamic KV Cache Compression based on Pyramidal Information
 *     Funneling -- §4.2 (per-layer budgets, arithmetic sequence, bottom layers
 *     get more), §4.2.2 KV Cache Selection (instruction-token scores, pooling,
 *     per-head top-k, the last alpha tokens always kept).
 *   MiniKV: Pushing the Limits of LLM Inference via 2-Bit Layer-Discriminative
 *     KV Cache -- §2 eq. (1) and Definition 2.1 (the co-compression problem:
 *     layers, heads, head dim, budget, bits), §4.1 (selection frozen after
 *     prefill), §4.2 (uniform / pyramid budgets), §4.4 and Algorithm 1
 *     (quantize the selected tokens, pack codes into INT32 words with FP16 scale
 *     and zero-point, streaming 16-bit buffer, one softmax over packed + buffer).
 *   KV Cache Compression: Eviction and Quantization (blog) -- "Quantization:
 *     keep each token in fewer bits" and "Measured on a real model" (zero-point
 *     = group min, scale = (max - min)/(2^b - 1), keys per channel, values per
 *     token, exact recent window).
 *
 * Conventions for every call
 *   - Device pointers are caller-owned (e.g. PyTorch tensors). They are only
 *     borrowed until the work enqueued on `stream` completes; the library never
 *     frees them. `stream` is a cudaStream_t (NULL = legacy default stream).
 *   - All work is stream-ordered. One cache must be used from one stream at a
 *     time; calls on one cache must not overlap.
 *   - Arguments are validated on the host before anything is enqueued; a
 *     failing call returns a status and enqueues nothing (or, for a launch
 *     failure, KVC_E_CUDA). Calls never abort, exit or trap.
 *   - Every device-side wait is bounded. A wait that gives up sets the cache's
 *     error word and its kernel winds down (its output is then undefined).
 *     Where the device has native atomics on host memory (e.g. a Grace-hosted
 *     GPU) the word lives in mapped pinned host memory, and the next call on the
 *     cache made after the word was set returns KVC_E_TIMEOUT (KVC_E_DEVICE_CHECK
 *     when a device-side check of the checked build set it), enqueues nothing
 *     and clears it; elsewhere kvc_check_device reports it. After KVC_E_TIMEOUT
 *     the cache's contents are undefined: kvc_cache_reset and prefill again.
 *   - Tensors are dense, row-major, bf16 unless stated; outputs are fp32.
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvc_status {
  KVC_OK = 0,
  KVC_E_ARG = 1,          /* null pointer or argument value out of range        */
  KVC_E_SHAPE = 2,        /* dimensions unsupported or inconsistent             */
  KVC_E_OOM = 3,          /* device allocation failed                           */
  KVC_E_CUDA = 4,         /* a CUDA runtime call or kernel launch failed        */
  KVC_E_STATE = 5,        /* call out of order (e.g. decode before prefill)     */
  KVC_E_CAPACITY = 6,     /* more appended tokens than max_new_tokens allows    */
  KVC_E_TIMEOUT = 7,      /* a bounded device-side wait gave up                 */
  KVC_E_DEVICE_CHECK = 8  /* a device-side check recorded an error              */
} kvc_status;

/* Per-layer budget schedules (PyramidKV §4.2; MiniKV §4.2). */
typedef enum kvc_schedule {
  KVC_SCHED_NONE = 0,     /* keep every prompt token (quantize-only cache)      */
  KVC_SCHED_UNIFORM = 1,  /* every layer keeps avg_budget tokens per head       */
  KVC_SCHED_PYRAMID = 2   /* linear: layer 0 gets 2x - x/d, the top layer x/d   */
} kvc_schedule;

/* Optional allocator hooks (e.g. a framework's caching allocator). When
 * `alloc` is NULL the library uses cudaMalloc / cudaFree. */
typedef void* (*kvc_alloc_fn)(size_t bytes, void* stream, void* ctx);
typedef void (*kvc_free_fn)(void* ptr, void* stream, void* ctx);

/* Size limits of kvc_dims (KVC_E_SHAPE beyond them): every token count and
 * per-head capacity the library forms on the host then stays inside int32. */
#define KVC_MAX_PROMPT_LEN (1 << 30)     /* prompt_len                          */
#define KVC_MAX_NEW_TOKENS (1 << 24)     /* max_new_tokens                      */
#define KVC_MAX_QUERY_HEADS (1 << 24)    /* batch * n_q_heads                   */

/* The problem statement (MiniKV Definition 2.1 plus the selection and window
 * parameters of PyramidKV §4.2.2 and MiniKV §4.4). */
typedef struct kvc_dims {
  int32_t n_layers;       /* transformer layers (1..256)                           */
  int32_t batch;          /* independent sequences (batch * n_q_heads at most      */
                          /*   KVC_MAX_QUERY_HEADS)                                */
  int32_t n_q_heads;      /* query heads; a multiple of n_kv_heads                 */
  int32_t n_kv_heads;     /* key/value heads (GQA group g = n_q_heads/n_kv_heads,  */
                          /*   g in {1, 2, 4, 8})                                  */
  int32_t head_dim;       /* 64 or 128                                             */
  int32_t prompt_len;     /* n, tokens in the prompt (1..KVC_MAX_PROMPT_LEN)       */
  int32_t obs_window;     /* alpha, trailing observation/instruction tokens;       */
                          /*   0 only with KVC_SCHED_NONE budgets (no scoring)     */
  int32_t pool_kernel;    /* w, odd max-pool width (1 = no pooling)                */
  int32_t bits;           /* 2 or 4; or 16: no quantization, every kept token     */
                          /*   stays exact in the bf16 window (no packed store,    */
                          /*   no flush); R must then hold the kept, observation   */
                          /*   and max_new_tokens appended tokens of every layer   */
                          /*   (with the full budget: plain dense attention)       */
  int32_t group_size;     /* G, quantization group; must be 32                     */
  int32_t window_len;     /* R, bf16 recent window; a multiple of G, 32..1024      */
                          /*   (up to 65536 with bits == 16)                       */
  int32_t max_new_tokens; /* decode steps the cache is sized for                   */
                          /*   (0..KVC_MAX_NEW_TOKENS)                             */
  kvc_alloc_fn alloc;     /* optional; NULL = cudaMalloc                           */
  kvc_free_fn free;       /* optional; must be set when alloc is                   */
  void* alloc_ctx;        /* passed to alloc/free                                  */
} kvc_dims;

typedef struct kvc_cache kvc_cache;   /* opaque; owns its device storage */

/* ---------------------------------------------------------------------------
 * kvc_plan_budgets -- per-layer token budgets (host only, no device work).
 *   PyramidKV §4.2 / MiniKV §4.2. For KVC_SCHED_PYRAMID the budgets run linearly
 *   from 2x - x/d (layer 0) down to x/d (top layer), x = avg_budget and
 *   d = pyramid_depth, in whole groups of G tokens: unit budgets are floored and
 *   the leftover units go to the largest remainders (ties to the lower layer),
 *   so they sum to exactly n_layers * avg_budget. UNIFORM gives avg_budget to
 *   every layer; NONE gives prompt_len (keep all). Every budget is finally
 *   clipped to prompt_len - obs_window.
 *   budgets_out: host array of n_layers int32 (written).
 *   Errors: KVC_E_ARG (null pointer, avg_budget not a positive multiple of G,
 *   pyramid_depth < 1), KVC_E_SHAPE (invalid dims).
 * ------------------------------------------------------------------------- */
kvc_status kvc_plan_budgets(const kvc_dims* dims, kvc_schedule schedule,
                            int32_t avg_budget, int32_t pyramid_depth,
                            int32_t* budgets_out);

/* ---------------------------------------------------------------------------
 * kvc_plan_budgets_weighted -- per-layer token budgets in proportion to given
 *   positive weights (host only, no device work). MiniKV §4.2 "Layer-Specific
 *   Selectivity", the variance policies: Var-prop (weights = the layers'
 *   variance scores, see kvc_score_variance) and Var-inv (weights = their
 *   inverses). Budgets are whole groups of G tokens; every layer gets one group
 *   and the remaining n_layers * avg_budget / G - n_layers groups are shared in
 *   proportion to the weights: each weight is scaled to the integer
 *   q_l = max(1, rint(w_l / max(w) * 2^30)), layer l's quota is
 *   spare * q_l / sum(q), quotas are floored and the leftover groups go one each
 *   to the largest remainders (ties to the lower layer), so the budgets sum to
 *   exactly n_layers * avg_budget. Every budget is finally clipped to
 *   prompt_len - obs_window.
 *   weights:     host array of n_layers doubles (read).
 *   budgets_out: host array of n_layers int32 (written).
 *   Errors: KVC_E_ARG (null pointer, a weight not positive and finite,
 *   avg_budget not a positive multiple of G), KVC_E_SHAPE (invalid dims).
 * ------------------------------------------------------------------------- */
kvc_status kvc_plan_budgets_weighted(const kvc_dims* dims, int32_t avg_budget,
                                     const double* weights, int32_t* budgets_out);

/* ---------------------------------------------------------------------------
 * kvc_prefill_compress -- compress one layer's prompt into the cache.
 *   PyramidKV §4.2.2; MiniKV §4.1, §4.4 and Algorithm 1 (prefill part).
 *   If *cache is NULL a cache is created for `dims` and `budgets` (host,
 *   n_layers int32, as from kvc_plan_budgets) and returned in *cache (the
 *   call's arguments are checked first: a call rejected by them creates
 *   nothing); later calls must pass the same dims. Each layer is compressed once.
 *   q_obs: device bf16 [batch][n_q_heads][obs_window][head_dim], the queries of
 *          the last obs_window prompt positions (may be NULL when the layer's
 *          budget keeps every token).
 *   k, v:  device bf16 [batch][n_kv_heads][prompt_len][head_dim] (post-RoPE keys).
 *   Computes, per (sequence, kv head): causal softmax of q_obs.k^T/sqrt(d) per
 *   observation row, summed over rows and over the g query heads of the group,
 *   for keys [0, n - alpha); a max-pool of width pool_kernel; the
 *   min(budget, n - alpha) largest pooled scores (ties to the lower index);
 *   whole groups of 32 kept tokens (ascending position) are quantized into the
 *   packed store; the remaining kept tokens and then the alpha observation
 *   tokens start the bf16 window.
 *   Errors: KVC_E_ARG (null k, v or cache; q_obs NULL for a scoring layer;
 *   layer out of range), KVC_E_SHAPE (dims unlike the cache's, or as
 *   kvc_cache_create), KVC_E_STATE (layer already compressed), KVC_E_OOM,
 *   KVC_E_CUDA.
 * ------------------------------------------------------------------------- */
kvc_status kvc_prefill_compress(const kvc_dims* dims, const int32_t* budgets,
                                int32_t layer, const void* q_obs, const void* k,
                                const void* v, kvc_cache** cache, void* stream);

/* ---------------------------------------------------------------------------
 * kvc_prefill_acumul -- like kvc_prefill_compress with MiniKV's full-prompt
 *   cumulated attention as the selection score (MiniKV §4.3 "selective
 *   flash-attention", Figure 9; Algorithm 1, prefill). Per (sequence, kv head),
 *   every prompt query of each of the g query heads sharing the kv head attends
 *   causally to the prompt keys; keys are visited in blocks of 128 from the
 *   first on, each row keeps a running maximum m over the blocks seen so far,
 *   and exp(q.k/sqrt(d) - m) is added into the key's score -- rows are never
 *   normalised. Scores of positions [0, n - alpha) then go through the same
 *   max-pool (width pool_kernel; 1 leaves them unchanged) and per-head top-k as
 *   kvc_prefill_compress, and the kept tokens are stored the same way.
 *   The cache must exist (kvc_cache_create or an earlier prefill call).
 *   q_full: device bf16 [batch][n_q_heads][prompt_len][head_dim], every prompt
 *           query (may be NULL when the layer's budget keeps every token).
 *   k, v:   device bf16 [batch][n_kv_heads][prompt_len][head_dim].
 *   Needs 128 % (n_q_heads / n_kv_heads) == 0 and n_q_heads / n_kv_heads <= 16.
 *   The scores stay readable through kvc_scores_layer / kvc_score_variance until
 *   the next scoring call. The row blocks' contributions are added as 64-bit
 *   fixed-point integers (units of 2^-40), so the scores and kept sets are the
 *   same on every run. Allocates, on first use, 8 bytes per score for them.
 *   Errors: KVC_E_ARG, KVC_E_SHAPE (group size, or initial window not shorter
 *   than R), KVC_E_STATE (layer already compressed), KVC_E_CUDA.
 * ------------------------------------------------------------------------- */
kvc_status kvc_prefill_acumul(kvc_cache* cache, int32_t layer, const void* q_full, const void* k,
                              const void* v, void* stream);

/* ---------------------------------------------------------------------------
 * kvc_prefill_attention -- the selective flash-attention of MiniKV §4.3 and
 *   Figure 9: one pass over the layer's prompt that returns the causal attention
 *   output X_O of every prompt query and, from the same tiles, the cumulated
 *   attention A_cumul by which the layer is then compressed exactly as
 *   kvc_prefill_acumul compresses it (same scores, kept sets and packing).
 *   x_out: device bf16 [batch][n_q_heads][prompt_len][head_dim], 16-byte aligned
 *          (written): X_O[i] = sum over keys j <= i of softmax(q_i . k_j /
 *          sqrt(head_dim)) v_j, accumulated in fp32 on the tensor cores with the
 *          weights rounded to bf16 (|error| <= 2^-8 of the largest |v| of the
 *          row's keys, plus the bf16 rounding of the output).
 *   q_full, k, v as for kvc_prefill_acumul (v is read by the attention too).
 *   With a budget that keeps every token no scores are formed; X_O still is.
 *   Errors: KVC_E_ARG (null pointer, misaligned x_out), KVC_E_SHAPE, KVC_E_STATE,
 *   KVC_E_CUDA, KVC_E_TIMEOUT (a wait of an earlier call on the cache gave up).
 * ------------------------------------------------------------------------- */
kvc_status kvc_prefill_attention(kvc_cache* cache, int32_t layer, const void* q_full,
                                 const void* k, const void* v, void* x_out, void* stream);

/* ---------------------------------------------------------------------------
 * kvc_prefill_sinks -- like kvc_prefill_compress with the attention-sink +
 *   recent-token selection in place of the scored one (blog "KV Cache
 *   Compression: Eviction and Quantization", "Measured on a real model": the first
 *   4 tokens plus the most recent ones within the budget; PyramidKV's StreamingLLM
 *   baseline, the first k - alpha and the last alpha tokens, is n_sinks = k).
 *   Per (sequence, kv head), with k = min(the layer's budget, n - alpha) and
 *   s = min(n_sinks, k): positions [0, s) and [n - alpha - (k - s), n - alpha) are
 *   kept (ascending); whole groups of 32 go to the packed store and the rest,
 *   then the alpha observation tokens, start the bf16 window, as for every
 *   selection. No scoring: no observation queries are read. One launch (the
 *   kept positions are formed and stored, for kvc_export_layer, by the packing
 *   kernel). The cache must exist (kvc_cache_create or an earlier prefill call).
 *   n_sinks >= 0.
 *   Errors: KVC_E_ARG, KVC_E_SHAPE (initial window not shorter than R),
 *   KVC_E_STATE (layer already compressed), KVC_E_OOM, KVC_E_CUDA.
 * ------------------------------------------------------------------------- */
kvc_status kvc_prefill_sinks(kvc_cache* cache, int32_t layer, int32_t n_sinks, const void* k,
                             const void* v, void* stream);

/* ---------------------------------------------------------------------------
 * kvc_prefill_selected -- like kvc_prefill_compress, but with the kept
 *   positions supplied by the caller instead of scored (any selection policy:
 *   e.g. attention sinks + recent tokens, StreamingLLM-style).
 *   kept: device int32 [batch][n_kv_heads][n_kept], strictly ascending, each in
 *   [0, prompt_len - obs_window) (may be NULL when n_kept == 0: only the
 *   observation window is kept); n_kept <= the layer's budget. The cache must
 *   exist (created by kvc_prefill_compress or kvc_cache_create).
 *   Errors: as kvc_prefill_compress; KVC_E_CAPACITY if n_kept > budget. Index
 *   order/range is the caller's contract; the checked build (kvc_build_checked)
 *   tests the range on the device, skips an index outside it (position 0 is read
 *   instead) and the next call on the cache returns KVC_E_DEVICE_CHECK.
 * ------------------------------------------------------------------------- */
kvc_status kvc_prefill_selected(kvc_cache* cache, int32_t layer, const int32_t* kept,
                                int32_t n_kept, const void* k, const void* v,
                                void* stream);

/* kvc_cache_create -- create an empty cache for dims/budgets (what
 * kvc_prefill_compress does when *cache is NULL); budgets: host int32
 * [n_layers], each clipped to prompt_len - obs_window. Errors: KVC_E_ARG (null
 * pointer, a negative budget, invalid argument values of dims), KVC_E_SHAPE
 * (unsupported dims or beyond the size limits, an initial window that does not
 * fit its ring, g * obs_window > 256 for a scoring layer), KVC_E_OOM, KVC_E_CUDA. */
kvc_status kvc_cache_create(const kvc_dims* dims, const int32_t* budgets,
                            kvc_cache** cache);

/* ---------------------------------------------------------------------------
 * kvc_cache_create_layers -- create an empty cache whose layers differ in
 *   precision: MiniKV Figure 1's layer-discriminative cache (16-bit top layers,
 *   2-bit lower layers; §4.1's 16-bit buffer holds the exact tokens).
 *   layer_bits: host array of n_layers entries, each 2, 4 or 16. A 2/4-bit layer
 *   is stored as kvc_cache_create stores it at that precision, with a window of
 *   dims->window_len slots. A 16-bit layer keeps every token exact: when
 *   dims->bits is 2 or 4 its bf16 ring is sized to hold its kept, observation
 *   and max_new_tokens appended tokens (rounded up to 32); when dims->bits is 16
 *   the ring has dims->window_len slots, which must hold them. dims->bits must
 *   still be 2, 4 or 16. Every other call works on such a cache unchanged, and
 *   one decode launch attends over all its layers, whatever their precision.
 *   Errors: KVC_E_ARG (null pointer, an entry not 2/4/16), KVC_E_SHAPE (a
 *   16-bit ring longer than 65,536 slots, or an initial window that does not
 *   fit), KVC_E_OOM.
 * ------------------------------------------------------------------------- */
kvc_status kvc_cache_create_layers(const kvc_dims* dims, const int32_t* budgets,
                                   const int32_t* layer_bits, kvc_cache** cache);

/* ---------------------------------------------------------------------------
 * kvc_append -- append one token per (sequence, kv head) to one layer.
 *   MiniKV Algorithm 1 (decoding: concatenate into the 16-bit buffer; quantize
 *   when it fills). k_new, v_new: device bf16 [batch][n_kv_heads][head_dim].
 *   When the window reaches window_len tokens its oldest 32 are quantized as
 *   one key group (per channel) and 32 value rows (per token) and leave it.
 *   Errors: KVC_E_STATE (layer not prefilled), KVC_E_CAPACITY (more than
 *   max_new_tokens appends), KVC_E_ARG, KVC_E_CUDA.
 * ------------------------------------------------------------------------- */
kvc_status kvc_append(kvc_cache* cache, int32_t layer, const void* k_new,
                      const void* v_new, void* stream);

/* kvc_append_layers -- kvc_append over layers [layer_begin, +layer_count) in
 * one launch; k_new, v_new: device bf16 [layer_count][batch][n_kv_heads][head_dim]. */
kvc_status kvc_append_layers(kvc_cache* cache, int32_t layer_begin, int32_t layer_count,
                             const void* k_new, const void* v_new, void* stream);

/* ---------------------------------------------------------------------------
 * kvc_decode_attn -- decode attention of one query per head.
 *   MiniKV §2 eq. (1), Algorithm 1 (one softmax over dequantized packed keys
 *   and the window's keys; output = A_quant.dequant(V) + A_window.V_window);
 *   blog "Measured on a real model" (exact window, rounded rest).
 *   q:   device bf16 [layer_count][batch][n_q_heads][head_dim].
 *   out: device fp32 [layer_count][batch][n_q_heads][head_dim] (written).
 *   Query head j reads kv head j / g. q and out must be 16-byte aligned. The token
 *   axis of every (layer, sequence, kv head) of the call is cut into chunks (16
 *   window tokens, or the packed groups of the same bytes), and the chunks of
 *   all of them are shared out evenly over every warp of the grid; a unit
 *   spread over several warps is merged with a log-sum-exp combine, in a fixed
 *   order, by the warp that finishes it last (same launch).
 *   Errors: KVC_E_STATE (a layer not prefilled), KVC_E_ARG, KVC_E_CUDA.
 * ------------------------------------------------------------------------- */
kvc_status kvc_decode_attn(kvc_cache* cache, int32_t layer_begin, int32_t layer_count,
                           const void* q, float* out, void* stream);

/* kvc_decode_step -- one decode step of Algorithm 1 on layers [layer_begin,
 * +layer_count): append k_new/v_new (as kvc_append_layers, with the group flush
 * when the window reaches R) and attend q (as kvc_decode_attn); the results equal
 * those two calls made in sequence. One launch, or two in the steps where some
 * layer's window fills (the append with its group flush runs first). Shapes as in
 * those calls. Errors: KVC_E_STATE (a layer not prefilled), KVC_E_CAPACITY (more
 * than max_new_tokens appends), KVC_E_ARG (null pointer, q or out not 16-byte
 * aligned, layers out of range), KVC_E_CUDA. */
kvc_status kvc_decode_step(kvc_cache* cache, int32_t layer_begin, int32_t layer_count,
                           const void* q, const void* k_new, const void* v_new,
                           float* out, void* stream);

/* kvc_check_device -- synchronize `stream` and report device-side failures
 * recorded since the last check: KVC_E_DEVICE_CHECK if a check of the checked
 * build found an index out of range, else KVC_E_TIMEOUT if a bounded wait inside
 * a kernel gave up (that kernel then skipped the affected work), KVC_OK otherwise.
 * The error word is cleared. */
kvc_status kvc_check_device(kvc_cache* cache, void* stream);

/* ---------------------------------------------------------------------------
 * kvc_build_checked -- 1 if this library was compiled with device-side checks
 *   (KVC_CHECKED=1 at build time: caller-supplied indices are range-checked on the
 *   device and reported as KVC_E_DEVICE_CHECK by the next call on the cache, in
 *   place of an out-of-range access), else 0.
 * ------------------------------------------------------------------------- */
int32_t kvc_build_checked(void);

/* kvc_set_wait_limit -- bound every staging wait of this cache's decode launches
 * to `polls` polls of its mbarrier (0: each wait gives up at once); a negative
 * value restores the default bound (2^20 polls). A testing aid: it lets a test
 * drive the timeout path (the kernel winds down, lets its copies land, hands its
 * partial units over so the arrival counters return to zero, and the error is
 * reported) without faulting anything. Errors: KVC_E_ARG. */
kvc_status kvc_set_wait_limit(kvc_cache* cache, int64_t polls);

/* kvc_free -- release the cache and all device storage it owns. The caller
 * must ensure no enqueued work still uses it (synchronize the stream first).
 * NULL is accepted. */
kvc_status kvc_free(kvc_cache* cache);

/* ---------------------------------------------------------------------------
 * Inspection (tests, tools).
 * ------------------------------------------------------------------------- */
typedef struct kvc_layer_info {
  int32_t prefilled;      /* 1 once the layer is compressed                      */
  int32_t budget;         /* clipped budget (tokens per head)                     */
  int32_t n_kept;         /* prompt tokens selected (excluding the obs window)   */
  int32_t packed_tokens;  /* tokens in the packed store (multiple of 32)         */
  int32_t capacity_tokens;/* packed capacity (tokens per head)                   */
  int32_t window_tokens;  /* tokens in the bf16 window                           */
  int32_t appended;       /* tokens appended since prefill                       */
  int64_t packed_bytes;   /* device bytes of this layer's packed store           */
  int32_t bits;           /* storage precision of the layer: 2, 4 or 16          */
  int32_t window_capacity;/* slots of the layer's bf16 ring                      */
} kvc_layer_info;

kvc_status kvc_layer_info_get(const kvc_cache* cache, int32_t layer, kvc_layer_info* out);

/* kvc_export_layer -- unpack one layer into plain device arrays (caller-owned;
 * any pointer may be NULL to skip that array). T = packed_tokens, W =
 * window_tokens, K = n_kept, B = batch, H = n_kv_heads, d = head_dim.
 *   kept    int32  [B][H][K]       selected prompt positions (ascending)
 *   k_codes uint8  [B][H][T][d]    key codes (token-major)
 *   k_scale, k_zero  fp16 [B][H][T/32][d]   per-channel key groups
 *   v_codes uint8  [B][H][T][d]
 *   v_scale, v_zero  fp16 [B][H][T][d/32]   per-token value groups
 *   win_k, win_v     bf16 [B][H][W][d]      window, oldest first
 * The packed layout itself is internal; this is the only way to read it. */
typedef struct kvc_export {
  int32_t* kept;
  uint8_t* k_codes;
  void* k_scale;
  void* k_zero;
  uint8_t* v_codes;
  void* v_scale;
  void* v_zero;
  void* win_k;
  void* win_v;
} kvc_export;

kvc_status kvc_export_layer(kvc_cache* cache, int32_t layer, const kvc_export* dst,
                            void* stream);

/* kvc_score_variance -- the variance score of the last scored layer (MiniKV
 * §4.2, Figure 7: the variance of cumulated attention), per (sequence, kv head):
 * the population variance, over the prompt_len - obs_window selectable
 * positions, of the selection scores (before pooling): the observation-window
 * scores after kvc_prefill_compress, the cumulated attention A_cumul after
 * kvc_prefill_acumul or kvc_prefill_attention. Compensated fp32 sums per thread,
 * the block's and the slices' partials combined in double-float and fp64 in a
 * fixed order (the result does not depend on timing), written as fp32 to
 * var_out (device, [B][H]). The mean over (B, H) is the layer's weight for
 * Var-prop / Var-inv budgets. One launch on `stream`. Only valid right after the
 * scoring call (the scratch is reused by the next one); kvc_prefill_compress does
 * not score a layer kept whole (budget >= prompt_len - obs_window). Errors:
 * KVC_E_ARG (null pointer), KVC_E_STATE (no layer scored since create or reset),
 * KVC_E_CUDA. */
kvc_status kvc_score_variance(kvc_cache* cache, float* var_out, void* stream);

/* kvc_scores_layer -- copy the last scored layer's selection scores (fp32,
 * device [B][H][prompt_len - obs_window]) and pooled scores (same shape);
 * either pointer may be NULL. Only valid right after kvc_prefill_compress of a
 * scoring layer (the scratch is reused by the next one). */
kvc_status kvc_scores_layer(kvc_cache* cache, float* scores, float* pooled, void* stream);

/* ---------------------------------------------------------------------------
 * kvc_select_noalloc -- the prefill selection of one layer (observation-window
 *   scores, max-pool, per-head top-k; the same kernels and results as
 *   kvc_prefill_compress) for callers that cannot allocate device memory, e.g.
 *   runtimes that carve all GPU memory into their own arena, or latency-critical
 *   loops where a cudaMalloc is not allowed. The pages have no counterpart: this
 *   is an interface variant, not a step of the method.
 *   Allocates nothing: intermediates live in one static device array of
 *   KVC_NOALLOC_SCRATCH_BYTES (32 MiB) that every GPU loading this library holds
 *   until exit. All calls share it (it keeps the last call's contents; every
 *   value a call reads is written by that call first), so calls that overlap on
 *   the GPU race: serialize them. A second static array, zero at load, holds
 *   the scoring launch's 1 + B*H counters (B*H <= 8192); every launch leaves
 *   them at zero. The first call on a device looks up the device addresses;
 *   make it before any stream capture.
 *   Scratch needed: B*H*(4*ceil(n/128)+4)*g*alpha*8 + B*H*(n-alpha)*4 bytes
 *   (+ the same again for scores when `scores` is NULL), each part rounded up
 *   to 256 bytes.
 *   q_obs: device bf16 [B][Hq][alpha][d]; k: device bf16 [B][H][n][d];
 *   kept:  device int32 [B][H][min(budget, n - alpha)] (written, ascending);
 *   scores: optional device fp32 [B][H][n - alpha] (written when not NULL).
 *   Only the fields n_layers..pool_kernel of dims are read.
 *   The static arrays are committed on a device by the first call made on it
 *   (the runtime loads their module lazily): make that call before an arena
 *   reserves the rest of the device's memory.
 *   A bounded wait inside the scoring launch that gives up sets the entry
 *   point's own error word; the top-k launch then writes every kept index as
 *   -1 (never a stale selection), and kvc_select_noalloc_check reports it.
 *   Errors: KVC_E_ARG, KVC_E_SHAPE, KVC_E_CAPACITY (the sizes need more than
 *   the static scratch, or B*H > 8192; nothing is enqueued), KVC_E_OOM (the
 *   static arrays could not be committed on this device), KVC_E_CUDA.
 * ------------------------------------------------------------------------- */
#define KVC_NOALLOC_SCRATCH_BYTES (32u << 20)
kvc_status kvc_select_noalloc(const kvc_dims* dims, int32_t budget, const void* q_obs,
                              const void* k, int32_t* kept, float* scores, void* stream);

/* kvc_select_noalloc_check -- synchronize `stream` and report whether a bounded
 * wait of a kvc_select_noalloc call on the current device gave up since the
 * last check (KVC_E_TIMEOUT; those calls wrote -1 kept indices), then clear the
 * word. KVC_OK when none did or no call was made on this device. Allocates
 * nothing. Errors: KVC_E_CUDA. */
kvc_status kvc_select_noalloc_check(void* stream);

/* kvc_cache_reset -- forget every layer's contents (host-side state only; the
 * device storage is kept) so the cache can take the next prompt with the same
 * dims and budgets. Enqueued work must have completed or be stream-ordered
 * before the next call on the cache. */
kvc_status kvc_cache_reset(kvc_cache* cache);

/* kvc_launch_count -- number of kernels this library has launched in the
 * process so far (all caches, all threads). */
uint64_t kvc_launch_count(void);

/* kvc_status_string -- static description of a status code. */
const char* kvc_status_string(kvc_status status);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H_ */
