/*
 * smol.h - C ABI of libsmol, a GB300 (sm_103a) implementation of the forward
 * pass of a pre-norm LLaMA-style decoder (SmolLM2-135M and relatives).
 *
 * Sources (web pages describing the method, cited by title and section):
 *   [M1] "model.py", minimal SmolLM2-135M style model (Sualeh77 Space):
 *        1 Config, 2 RMSNorm, 3 RoPE, 4 Attention, 5 MLP (SwiGLU),
 *        6 Transformer Block, 7 Top-level SmolLM2-135M (forward, generate).
 *   [M3] "SmolLM3" (nnterp encyclopedia): "The block, in order",
 *        "Grouped-query attention", "The readout, the embeddings and the tokenizer".
 *   [M4] "model.py", complete SmolLM2-135M implementation (abi96062):
 *        SmolLM2Model.forward (position_ids).
 *   [M5] "components.py" (abi96062): RMSNorm, RotaryEmbedding,
 *        GroupedQueryAttention, SwiGLU_FFN, TransformerBlock.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument marked "device" is a CUDA device pointer on the
 *     current device; "host" pointers are ordinary host memory read before
 *     the call returns.  Tensors are dense, row-major (last index fastest),
 *     bf16 unless stated; weight matrices use the nn.Linear layout [out, in].
 *   - Device buffers must be 16-byte aligned (SMOL_ERR_MISALIGNED otherwise).
 *   - The caller owns every buffer and the stream.  No entry point allocates,
 *     frees or synchronises: all work is enqueued asynchronously on `stream`
 *     (a cudaStream_t passed as void*; NULL = the legacy default stream).
 *   - Return value: SMOL_OK (0) or a negative smol_status.  On an argument
 *     error nothing is launched.  SMOL_ERR_CUDA reports a launch error; the
 *     text of the last one is available through smol_status_string.
 *   - Kernels never spin without a bound.  A bounded wait that gives up
 *     writes a nonzero code into the workspace's status word and the kernel
 *     returns; smol_workspace_status reads that word.
 *   - Numeric range: the residual stream between and inside blocks and every
 *     tensor-core operand are f16 (fp32 accumulation), so activations must
 *     stay below 65504 in magnitude (SmolLM2-shaped activations are orders of
 *     magnitude smaller).  A value that would round to infinity when the
 *     input is converted or a residual sum is written, or a non-finite row,
 *     is recorded in the status word (SMOL_ERR_RANGE); the outputs of that
 *     call are then not defined.
 *   - Input values that kernels clamp (a token id outside [0, V), a cache
 *     length or left-padding start outside its stated range) are recorded in
 *     the status word (SMOL_ERR_INPUT); the rows concerned are not defined.
 *   - The status word keeps the first code written until
 *     smol_workspace_status reads and clears it.
 *   - Supported shapes: head_dim in {64, 128}; hidden == n_heads * head_dim;
 *     n_heads % n_kv_heads == 0 with a group of at most 8; hidden, intermediate
 *     and vocab multiples of 64; T >= 1; rows (B*T) up to 2^31-1.
 */
#ifndef SMOL_H
#define SMOL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Model dimensions ([M1] section 1 Config). */
typedef struct smol_config {
  int hidden;          /* d */
  int n_heads;         /* H, query heads */
  int n_kv_heads;      /* KV, key/value heads */
  int head_dim;        /* hd */
  int intermediate;    /* I, SwiGLU width */
  int n_layers;        /* L */
  int vocab;           /* V (0 if no embedding/head is used) */
  int max_pos;         /* max_position_embeddings: RoPE table rows and length guard */
  float rms_eps;       /* RMSNorm epsilon */
  float rope_theta;    /* RoPE base */
  /* Per-block variants of SmolLM3 ([M3] "Every fourth block has no rotary",
   * "A sliding window the 3B checkpoints leave off").  Both are HOST arrays
   * of n_layers entries, indexed by the block's layer index, read during the
   * call; NULL leaves every block as SmolLM2's.
   * no_rope_layers[l]: 1 = block l rotates q and k (RoPE), 0 = a NoPE block
   *                    (q and k enter attention as projected; the k_out/k_new
   *                    and cache keys of that block are unrotated too).
   * sliding_window[l]: 0 = full causal attention; w > 0 = query t sees only
   *                    keys j with t - w < j <= t (its own and the w - 1
   *                    before it); in decode the new token at position L sees
   *                    cache slots j >= L - w + 1 and itself. */
  const int32_t *no_rope_layers;
  const int32_t *sliding_window;
} smol_config;

/* One block's weights, device pointers, bf16, nn.Linear layout [out, in]. */
typedef struct smol_block_weights {
  const void *attn_norm; /* [d]          RMSNorm before attention            */
  const void *wq;        /* [H*hd, d]                                        */
  const void *wk;        /* [KV*hd, d]                                       */
  const void *wv;        /* [KV*hd, d]                                       */
  const void *wo;        /* [d, H*hd]                                        */
  const void *mlp_norm;  /* [d]          RMSNorm before the MLP              */
  const void *wgate;     /* [I, d]                                           */
  const void *wup;       /* [I, d]                                           */
  const void *wdown;     /* [d, I]                                           */
} smol_block_weights;

/* Whole-model weights.  `layers` is a HOST array of n_layers structs holding
 * device pointers.  `embed` [V, d] is also the tied lm_head ([M1] section 7,
 * "tie weights"; [M3] "The readout").  embed/final_norm may be NULL when only
 * blocks are packed. */
typedef struct smol_model_weights {
  const smol_block_weights *layers;
  const void *embed;       /* [V, d] device, bf16 */
  const void *final_norm;  /* [d]    device, bf16 */
} smol_model_weights;

typedef enum smol_status {
  SMOL_OK = 0,
  SMOL_ERR_INVALID_ARG = -1,       /* NULL pointer, non-positive size, bad layer index */
  SMOL_ERR_UNSUPPORTED_SHAPE = -2, /* see "Supported shapes" above                   */
  SMOL_ERR_MISALIGNED = -3,        /* a device buffer is not 16-byte aligned         */
  SMOL_ERR_TOO_LONG = -4,          /* positions exceed max_pos ([M1] section 7 assert) */
  SMOL_ERR_WORKSPACE = -5,         /* workspace or packed buffer too small           */
  SMOL_ERR_CUDA = -6,              /* a CUDA runtime call or launch failed           */
  SMOL_ERR_DEVICE = -7,            /* current device is not a compute-capability 10.3 GPU */
  SMOL_ERR_TIMEOUT = -8,           /* a kernel's bounded wait gave up (status word)  */
  SMOL_ERR_RANGE = -9,             /* a value beyond the f16 range (status word)     */
  SMOL_ERR_INPUT = -10             /* an input value out of range (status word)      */
} smol_status;

/* Operation selector for smol_workspace_bytes. */
enum { SMOL_OP_BLOCK = 1, SMOL_OP_MODEL = 2, SMOL_OP_DECODE = 3 };

/* Element type of the residual stream (x and out) of smol_block_forward.
 * SMOL_ACT_F32 keeps the residual stream in fp32 across block calls (the
 * projections still read an f16 copy as their tensor-core operand, and the
 * residual h inside the block is f16). */
enum { SMOL_ACT_BF16 = 0, SMOL_ACT_F32 = 1 };

/* ---------------------------------------------------------------------------
 * Packed weights.
 * smol_prepare_weights converts raw weights into the library's layout, once,
 * on `stream`:
 *   - the attention and MLP RMSNorm weights are folded into the columns of
 *     the projections that consume them (W'[j,k] = W[j,k] * w_norm[k],
 *     rounded to f16, the tensor-core operand type of every projection), and
 *     the final-norm weight into an f16 copy of the tied head, so each norm
 *     reduces to a per-row scale rsqrt(mean(x^2)+eps)
 *     ([M1] section 2; [M5] RMSNorm formula);
 *   - Wq, Wk, Wv are stacked into one [(H+2KV)*hd, d] matrix;
 *   - Wgate and Wup are interleaved in groups of 64 rows;
 *   - a cos/sin table of the RoPE angles pos * theta^(-2i/hd) for
 *     pos < max_pos is computed in double precision and stored as fp32
 *     ([M1] section 3; [M5] RotaryEmbedding).
 * n_layers <= cfg->n_layers layers are packed (layers[0..n_layers)).  With
 * w->embed non-NULL the embedding and head are packed too (needs vocab > 0).
 * `packed` (device) must hold smol_packed_bytes(cfg, n_layers, with_embed)
 * bytes; it is written asynchronously and owned by the caller.
 * ------------------------------------------------------------------------- */
size_t smol_packed_bytes(const smol_config *cfg, int n_layers, int with_embed);
int smol_prepare_weights(const smol_config *cfg, const smol_model_weights *w, int n_layers,
                         void *packed, size_t packed_bytes, void *stream);

/* Workspace bytes needed by one call of `op` with batch B and T tokens per
 * sequence (decode: T is ignored).  0 for an unsupported configuration. */
size_t smol_workspace_bytes(const smol_config *cfg, int op, int B, int T);

/* ---------------------------------------------------------------------------
 * smol_block_forward: one decoder block, layer `layer` of a packed set.
 *   h   = x + O(GQA-attention(RoPE(Q), RoPE(K), V)),  Q,K,V = RMSNorm1(x) W^T
 *   out = h + Down(SiLU(Gate(RMSNorm2(h))) * Up(RMSNorm2(h)))
 * [M1] sections 4-6 (MultiHeadSelfAttention, SmolMLP, SmolBlock);
 * [M3] "The block, in order"; [M5] TransformerBlock.
 *   x            device [B, T, d] input (read only), bf16 or fp32 per act_dtype.
 *   out          device [B, T, d] output of the same type; may equal x.
 *   act_dtype    SMOL_ACT_BF16 or SMOL_ACT_F32.
 *   valid_start  device int32 [B] or NULL.  Sequence b is left-padded: tokens
 *                t < valid_start[b] are padding.  A key j is visible to query t
 *                iff valid_start[b] <= j <= t (causal plus padding mask, [M1]
 *                section 4), and the position id of token t is
 *                t - valid_start[b] ([M4] position_ids).  Padding rows get an
 *                attention output of 0; their `out` rows are finite but are
 *                not defined by the method.  Each value must lie in [0, T]
 *                (a value outside is clamped and recorded as SMOL_ERR_INPUT).
 *   k_out,v_out  device [B, KV, T, hd] bf16 or NULL: post-RoPE keys and the
 *                values, the per-layer cache entries of [M1] section 4.
 *   ws           device workspace of at least
 *                smol_workspace_bytes(cfg, SMOL_OP_BLOCK, B, T) bytes.
 * Positions must stay below cfg->max_pos (else SMOL_ERR_TOO_LONG).
 * ------------------------------------------------------------------------- */
int smol_block_forward(const smol_config *cfg, const void *packed, int layer,
                       const void *x, void *out, int act_dtype, int B, int T,
                       const int32_t *valid_start,
                       void *k_out, void *v_out, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * smol_block_forward_masked: smol_block_forward with a key mask in place of
 * left padding: the additive attention_mask of [M1] section 4 (0 where a key
 * may be attended, -inf where not), given as bytes.
 *   key_mask  device uint8 [B, T], required: key j of sequence b is visible
 *             iff key_mask[b*T + j] != 0, on top of the causal mask.  Position
 *             ids stay t (the page derives none from the mask).  A query row
 *             that sees no key gets an attention output of 0.
 * All other arguments as in smol_block_forward.
 * ------------------------------------------------------------------------- */
int smol_block_forward_masked(const smol_config *cfg, const void *packed, int layer,
                              const void *x, void *out, int act_dtype, int B, int T,
                              const uint8_t *key_mask, void *k_out, void *v_out, void *ws,
                              size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * smol_model_forward: embedding -> cfg->n_layers blocks -> final RMSNorm ->
 * tied lm_head ([M1] section 7 SmolLM2.forward; [M4] SmolLM2Model.forward).
 *   ids          device int32 [B, T], each in [0, V) (an out-of-range id is
 *                clamped into range by the gather and recorded as
 *                SMOL_ERR_INPUT in the status word).
 *   valid_start  device int32 [B] or NULL (as in smol_block_forward).
 *   logits       device [B, T, V] bf16.
 *   ws           >= smol_workspace_bytes(cfg, SMOL_OP_MODEL, B, T) bytes.
 * Needs a packed set with all cfg->n_layers layers and the embedding.
 * ------------------------------------------------------------------------- */
int smol_model_forward(const smol_config *cfg, const void *packed, const int32_t *ids,
                       int B, int T, const int32_t *valid_start, void *logits,
                       void *ws, size_t ws_bytes, void *stream);

/* smol_model_forward with the key mask of smol_block_forward_masked (device
 * uint8 [B, T], required) in place of valid_start; every block uses it. */
int smol_model_forward_masked(const smol_config *cfg, const void *packed, const int32_t *ids,
                              int B, int T, const uint8_t *key_mask, void *logits,
                              void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * smol_prefill_with_cache: T new tokens per sequence on top of a KV cache
 * (chunked prefill; [M1] section 4 with past_key_value and T > 1, section 7
 * with past_key_values).  New token t of sequence b sits at position
 * cache_len[b] + t and attends over its cache_len[b] cached entries and the
 * new tokens 0 .. t (the causal mask offset by the past; the page's model.py
 * drops the mask whenever a past exists, which would let a token see later
 * ones).  Per-block NoPE flags and windows apply as in the other calls.
 *   ids        device int32 [B, T].
 *   cache_len  device int32 [B], each in [0, min(S_max, max_pos - T)]
 *              (clamped into that range on the device; a value outside is
 *              recorded as SMOL_ERR_INPUT in the status word).
 *   k_cache, v_cache  device [L, B, KV, S_max, hd] bf16, post-RoPE keys; read only.
 *   k_new, v_new      device [L, B, KV, T, hd] bf16 outputs: the new tokens'
 *              post-RoPE keys and values per layer, for the caller to append
 *              at slots cache_len[b] .. cache_len[b] + T - 1.
 *   logits     device [B, T, V] bf16.
 *   ws         >= smol_prefill_cache_workspace_bytes(cfg, B, T, S_max) bytes.
 * Supported: head_dim 64 and 128, as the other calls; T < max_pos (SMOL_ERR_TOO_LONG).
 * ------------------------------------------------------------------------- */
size_t smol_prefill_cache_workspace_bytes(const smol_config *cfg, int B, int T, int S_max);
int smol_prefill_with_cache(const smol_config *cfg, const void *packed, const int32_t *ids, int B,
                            int T, const int32_t *cache_len, const void *k_cache,
                            const void *v_cache, int S_max, void *k_new, void *v_new,
                            void *logits, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * smol_decode_step: one new token per sequence with a KV cache
 * ([M1] section 4, the past_key_value branch, and section 7 generate).
 *   ids        device int32 [B], the new tokens.
 *   cache_len  device int32 [B]: sequence b has cache_len[b] cached entries
 *              (slots [0, cache_len[b]) of its cache rows); its new token is
 *              at position cache_len[b] and attends over those entries plus
 *              its own key/value, with no other mask.  Each value must lie in
 *              [0, S_max] and cache_len[b] < max_pos (not checked on the host:
 *              values are clamped to [0, min(S_max, max_pos-1)] on the device,
 *              and a clamped value is recorded as SMOL_ERR_INPUT in the status
 *              word).
 *   k_cache,v_cache device [L, B, KV, S_max, hd] bf16, post-RoPE keys (stored
 *              "after RoPE, before GQA expansion", [M1] section 4).  Read only.
 *   k_new,v_new device [L, B, KV, hd] bf16 outputs: this token's post-RoPE key
 *              and its value per layer.  The cache is not written; appending
 *              them at slot cache_len[b] is left to the caller (the slot may
 *              not exist when cache_len[b] == S_max).
 *   logits     device [B, V] bf16, next-token logits.
 *   ws         >= smol_workspace_bytes(cfg, SMOL_OP_DECODE, B, 1) bytes.
 * ------------------------------------------------------------------------- */
int smol_decode_step(const smol_config *cfg, const void *packed, const int32_t *ids,
                     const int32_t *cache_len, int B, const void *k_cache, const void *v_cache,
                     int S_max, void *k_new, void *v_new, void *logits,
                     void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * smol_decode_step_noalloc: smol_decode_step without a caller workspace.
 * The pages have no counterpart; this exists for callers that cannot give the
 * library scratch memory at the moment they decode: a serving loop that
 * forbids device allocation after start-up, a host whose allocator is not
 * reachable from where the step is issued, or code that must not call
 * cudaMalloc because it may synchronise the whole device.
 *   Arguments and results are those of smol_decode_step, minus ws/ws_bytes.
 *   Scratch: a fixed 8 MiB device array inside the library (every GPU that
 *   loads the library holds one until the process exits).  Calls for which
 *   smol_workspace_bytes(cfg, SMOL_OP_DECODE, B, 1) exceeds 8 MiB return
 *   SMOL_ERR_WORKSPACE and launch nothing (SmolLM2-135M needs about 5.1 MiB
 *   at B = 64).
 *   Each call made outside stream capture looks up the array's device address
 *   (a host call, cudaGetSymbolAddress, with the device current), so the
 *   first call on a device must come before any stream capture on it; a call
 *   made while `stream` is capturing reuses the address of the last uncaptured
 *   call on that device (SMOL_ERR_INVALID_ARG if there was none).  Nothing is
 *   allocated or freed, ever.
 *   All calls share the one array: calls whose work overlaps on the GPU
 *   (different streams, or different host threads) race on it and give
 *   wrong results; serialise them.  Each call clears what must start at
 *   zero, so back-to-back calls on one stream are safe.
 *   The array's first word is the status word of these calls' bounded waits:
 *   read it with smol_decode_noalloc_status.
 * ------------------------------------------------------------------------- */
int smol_decode_step_noalloc(const smol_config *cfg, const void *packed, const int32_t *ids,
                             const int32_t *cache_len, int B, const void *k_cache,
                             const void *v_cache, int S_max, void *k_new, void *v_new,
                             void *logits, void *stream);

/* Reads (synchronising `stream`) and clears the status word that
 * smol_decode_step_noalloc's kernels write into the library's scratch array on
 * the current device, with the codes of smol_workspace_status: SMOL_OK,
 * SMOL_ERR_TIMEOUT, SMOL_ERR_RANGE or SMOL_ERR_INPUT (the first one recorded
 * since the last read; the outputs of that call are not valid), or
 * SMOL_ERR_CUDA.
 * No counterpart on the pages.  Not meant for the hot path, nor for use while
 * `stream` is capturing. */
int smol_decode_noalloc_status(void *stream);

/* ---------------------------------------------------------------------------
 * smol_decode_next: smol_decode_step followed by the next-token choice of
 * smol_sample ([M1] section 7 generate: logits of the last position, then
 * argmax or a draw).  Arguments as in smol_decode_step and smol_sample:
 *   logits     device [B, V] bf16; may be NULL for a greedy choice.
 *   temperature, top_k, top_p, do_sample, uniform: as in smol_sample (uniform,
 *              device fp32 [B], is needed only when sampling).
 *   next       device int32 [B] output.  It may be the same buffer as `ids`
 *              (ids are read by the step's first kernel, next written by its
 *              last), so a generate loop can feed it back.
 * Greedy (do_sample == 0 or temperature <= 0): the choice is taken inside the
 * tied head's GEMM epilogue -- every output tile keeps each row's largest
 * bf16-rounded logit and its first column, combined across tiles by a 64-bit
 * atomic maximum -- so the logits need not be written or read again.
 * Sampling: the step writes the logits and the choice kernel of smol_sample
 * reads them.  Errors as smol_decode_step; SMOL_ERR_INVALID_ARG also for a
 * NULL `next`, a NaN temperature or top_p, or, when sampling, a NULL logits
 * or uniform.
 * ------------------------------------------------------------------------- */
int smol_decode_next(const smol_config *cfg, const void *packed, const int32_t *ids,
                     const int32_t *cache_len, int B, const void *k_cache, const void *v_cache,
                     int S_max, void *k_new, void *v_new, void *logits, float temperature, int top_k,
                     float top_p, int do_sample, const float *uniform, int32_t *next,
                     void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * smol_append_kv: appends a decode step's new keys and values to the caches,
 * the caller's part of [M1] section 4 (the cache grows by the new token's
 * post-RoPE key and its value):
 *   k_cache[l, b, kv, cache_len[b], :] = k_new[l, b, kv, :] (and v alike) for
 *   every layer l and kv head, then cache_len[b] += 1.
 *   k_new, v_new      device [L, B, KV, hd] bf16 (smol_decode_step's outputs).
 *   k_cache, v_cache  device [L, B, KV, S_max, hd] bf16.
 *   cache_len         device int32 [B], read and incremented.  A row whose
 *                     length is outside [0, S_max) (a full cache) is left as
 *                     it is, its length unchanged.
 * Two kernel launches on `stream`, no workspace.
 * ------------------------------------------------------------------------- */
int smol_append_kv(const smol_config *cfg, int B, const void *k_new, const void *v_new, void *k_cache,
                   void *v_cache, int S_max, int32_t *cache_len, void *stream);

/* ---------------------------------------------------------------------------
 * smol_sample: the next token of each row of logits, chosen the way the pages'
 * generate loop chooses it ([M1] section 7 generate; [M4] generate).
 *   Greedy when do_sample == 0 or temperature <= 0: the first index of the row
 *   maximum.  Otherwise, with z = logits / temperature:
 *     top_k > 0   tokens whose z is below the k-th largest z are removed
 *                 (values equal to the k-th stay; top_k >= V removes nothing);
 *     top_p < 1   in descending z order (equal values by ascending index), the
 *                 tokens after the first one at which the cumulative softmax
 *                 probability of the top-k survivors exceeds top_p are removed
 *                 (top_p <= 0: only the first token in that order survives);
 *     the draw    the first index i, in vocabulary order, at which the
 *                 cumulative probability of the survivors exceeds uniform[b]
 *                 (the inverse CDF; the pages call a multinomial sampler).
 *   logits      device bf16 [B, ld], rows of V finite values (ld >= V elements).
 *   uniform     device fp32 [B], each in [0, 1): the caller's random numbers
 *               (unused, may be NULL, when greedy).
 *   next        device int32 [B] output.
 * One kernel launch on `stream`, no workspace.  SMOL_ERR_INVALID_ARG for a NULL
 * pointer, B < 1, V < 1, ld < V, or a NaN temperature/top_p.
 * ------------------------------------------------------------------------- */
int smol_sample(const void *logits, int B, int V, long long ld, float temperature, int top_k,
                float top_p, int do_sample, const float *uniform, int32_t *next, void *stream);

/* Reads (synchronising `stream`) and clears the workspace status word.
 * Returns SMOL_OK, SMOL_ERR_TIMEOUT (a bounded wait gave up), SMOL_ERR_RANGE
 * (a value beyond the f16 range), SMOL_ERR_INPUT (an input value out of
 * range) -- whichever a kernel recorded first since the last read -- or
 * SMOL_ERR_CUDA.  Not meant for the hot path. */
int smol_workspace_status(void *ws, void *stream);

/* Number of kernels the most recent forward/decode call on this thread
 * launched (0 after an argument error). */
int smol_last_launch_count(void);

/* For tests of the failure path only (no counterpart on the pages): the limit,
 * in nanoseconds, of the bounded waits of the prefill attention kernel in
 * launches made from now on by any thread (0 restores the default of 1 s).  A
 * limit shorter than the kernel's own latencies makes a wait give up: the
 * kernel drains the copies and MMAs it issued (those drains keep the 1 s
 * limit), records SMOL_ERR_TIMEOUT in the status word and returns, leaving its
 * outputs undefined; the device stays usable. */
void smol_set_wait_limit_ns(unsigned long long ns);

/* ---------------------------------------------------------------------------
 * Per-launch timing, for measurement only (off unless started; not for use
 * inside CUDA graph capture).  Kernel kinds: */
enum {
  SMOL_K_EMBED = 0,      /* embedding gather + row statistics            */
  SMOL_K_ROWSTATS = 1,   /* block input row statistics + f16 copy         */
  SMOL_K_QKV = 2,        /* RMSNorm + QKV GEMM + RoPE                     */
  SMOL_K_ATTN = 3,       /* causal GQA flash attention                    */
  SMOL_K_OPROJ = 4,      /* O GEMM + residual                             */
  SMOL_K_GATEUP = 5,     /* RMSNorm + gate/up GEMM + SwiGLU               */
  SMOL_K_DOWN = 6,       /* down GEMM + residual                          */
  SMOL_K_HEAD = 7,       /* final RMSNorm + tied lm_head GEMM             */
  SMOL_K_DEC_ATTN = 8,   /* decode attention over the KV cache            */
  SMOL_K_OTHER = 9,      /* packing and bookkeeping kernels               */
  SMOL_K_SAMPLE = 10,    /* next-token choice (smol_sample)               */
  SMOL_K_COUNT = 11
};
/* From now on (this host thread), every launch whose kind bit is set in
 * `kind_mask` is bracketed by CUDA events on its stream, up to `capacity`
 * launches (events are created here, before the timed work).  Returns
 * SMOL_OK or SMOL_ERR_CUDA. */
int smol_profile_begin(unsigned kind_mask, int capacity);
/* Stops recording, waits for the recorded events and writes, per recorded
 * launch in order, its kind (kinds[i]) and duration in milliseconds (ms[i]),
 * up to cap entries (host arrays).  Returns the number written, or a
 * negative status. */
int smol_profile_end(int *kinds, float *ms, int cap);

/* Static text for a status code; for SMOL_ERR_CUDA, the last CUDA error text. */
const char *smol_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* SMOL_H */
