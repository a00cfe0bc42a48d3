/*
 * dflash.h — C ABI of libdflash: the DFlash block-diffusion draft path on
 * one GB300 (sm_103a).
 *
 * The method (DFlash, "Block Diffusion for Flash Speculative Decoding"):
 *   1. fuse:    H_t = RMSNorm(W_c [H^(l1); ...; H^(l5)])  — the hidden states of
 *               five uniformly spaced target layers, concatenated on the hidden
 *               axis and projected by W_c (D x 5D).  (A3-dflash tutorial
 *               §2.1.1; txtmix source reading §5.)
 *   2. inject:  every draft layer turns H_t into K/V entries through its own
 *               k_proj (+ k_norm, RoPE) and v_proj, appended to that layer's
 *               persistent draft KV cache; H_t never enters Q, o_proj or the
 *               FFN.  (A3-dflash tutorial §2.1.2; txtmix §5.)
 *   3. draft:   one forward pass of the block [anchor, mask x (B-1)] through
 *               every draft layer, bidirectional attention over
 *               [context KV ; block KV] with grouped K/V heads, SwiGLU FFN,
 *               then the target's shared LM head with argmax on rows 1..B-1.
 *               (txtmix §6 and §9.)
 *   4. verify:  greedy longest matching prefix plus one bonus token; the
 *               target cache is trimmed to start + accepted + 1.  (txtmix §8.)
 *
 * Conventions for every call:
 *   - Pointers named "device" are CUDA device pointers; "host" are host
 *     memory.  All tensors are dense row-major with the stated shapes.
 *   - Linear weights are stored out x in (y = x W^T).  RMSNorm gains are fp32.
 *   - Weights, K/V caches, fused features and activations use the handle's
 *     dtype (DFLASH_F32 or DFLASH_BF16); accumulation is always fp32.
 *   - The library borrows every caller pointer (weights, caches, outputs,
 *     workspace) and never frees them.  A handle owns only a device status
 *     word and a RoPE cos/sin table, allocated in dflash_create.
 *   - Calls are asynchronous on the given stream (NULL = legacy default
 *     stream) and do not synchronise the host, except dflash_get_status.
 *   - A handle must not be used from two streams at once.
 *   - Return value: DFLASH_OK or an error code.  Argument errors are
 *     detected on the host before anything is launched.  Errors only the
 *     device can see (a sequence outgrowing its cache, a token id out of
 *     range, a position beyond the RoPE table) skip the offending writes and
 *     set the handle's device status word, read by dflash_get_status.
 *   - An argmax over a row whose logits hold no maximum (all NaN or all
 *     -inf: an overflow upstream) writes id 0 and gap 0 and records
 *     DFLASH_ERR_DEVICE_BOUNDS, so no id past the vocabulary reaches the
 *     caller.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* dflash_stream_t;

enum dflash_status {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, negative size */
  DFLASH_ERR_SHAPE = 2,         /* shape outside what the handle supports */
  DFLASH_ERR_ALIGNMENT = 3,     /* a pointer is not 16-byte aligned */
  DFLASH_ERR_CAPACITY = 4,      /* a K/V cache would overflow (device-detected) */
  DFLASH_ERR_UNSUPPORTED = 5,   /* dtype / head_dim / device architecture */
  DFLASH_ERR_CUDA = 6,          /* a CUDA runtime call or launch failed */
  DFLASH_ERR_DEVICE_TIMEOUT = 7,/* a bounded device-side wait gave up */
  DFLASH_ERR_DEVICE_BOUNDS = 8, /* token id or position out of range (device-detected) */
  DFLASH_ERR_WORKSPACE = 9,     /* workspace smaller than dflash_workspace_bytes */
  DFLASH_ERR_STATIC_LIMIT = 10  /* request larger than a fixed internal scratch array */
};

enum dflash_dtype { DFLASH_F32 = 0, DFLASH_BF16 = 1 };

#define DFLASH_MAX_LAYERS 16
#define DFLASH_MAX_PICK 8
#define DFLASH_SEL_KMAX 16   /* candidates per position of dflash_select_candidates */

/* Model shape.  One struct serves the draft (qk_norm = 1, bidirectional
 * block) and the small causal target used by the end-to-end loop
 * (qk_norm = 0).  Fields follow the draft checkpoint's dflash_config
 * (txtmix §11: block size, target_layer_ids, mask_token_id,
 * input_embedding_scale) plus the Qwen3/Llama layer shape. */
typedef struct dflash_config {
  int32_t hidden;            /* D */
  int32_t n_heads;           /* H query heads */
  int32_t n_kv_heads;        /* G key/value heads; H % G == 0 */
  int32_t head_dim;          /* d: 64 or 128 */
  int32_t ffn;               /* F, SwiGLU intermediate size */
  int32_t vocab;             /* V, shared embedding / LM head rows */
  int32_t n_layers;          /* decoder layers, <= DFLASH_MAX_LAYERS */
  int32_t n_target_layers;   /* depth of the target the features come from */
  int32_t n_pick;            /* fused target layers (5), <= DFLASH_MAX_PICK */
  int32_t target_layer_ids[DFLASH_MAX_PICK]; /* informational */
  int32_t mask_token_id;
  int32_t max_pos;           /* RoPE table covers positions 0 .. max_pos-1 */
  int32_t qk_norm;           /* 1: per-head RMSNorm on q and k before RoPE */
  int32_t dtype;             /* enum dflash_dtype */
  float rope_theta;
  float rms_eps;
  float embed_scale;         /* input_embedding_scale */
  /* Draft layer types (txtmix §6): a sliding_attention layer is causal and
   * keeps a window of sliding_window keys, a full_attention layer is
   * bidirectional.  Block row i sits at position p = L + i after the L
   * context entries; a causal layer's row sees keys at positions <= p, a
   * windowed layer's row keys at positions > p - sliding_window (context
   * included).  0 everywhere: every layer bidirectional over all keys. */
  int32_t causal_layers;     /* bit l: layer l is causal */
  int32_t window_layers;     /* bit l: layer l keeps sliding_window keys */
  int32_t sliding_window;    /* >= 1 when window_layers != 0 */
  /* DFlash 2's grouped dynamic causal conv (txtmix §13-§14): > 0 gives
   * every draft layer two conv modules (around attention and around the
   * FFN; weights in dflash_layer_weights), one dynamic correction per
   * conv_group channels (16 in DFlash 2); D % conv_group == 0.  0: none. */
  int32_t conv_group;
} dflash_config;

/* One decoder layer's weights (device, borrowed). */
typedef struct dflash_layer_weights {
  const void* wq;            /* [H*d, D] */
  const void* wk;            /* [G*d, D] */
  const void* wv;            /* [G*d, D] */
  const void* wo;            /* [D, H*d] */
  const void* wg;            /* [F, D]  gate */
  const void* wu;            /* [F, D]  up */
  const void* wd;            /* [D, F]  down */
  const float* g_in;         /* [D] input RMSNorm gain */
  const float* g_post;       /* [D] post-attention RMSNorm gain */
  const float* q_norm;       /* [d] (qk_norm only) */
  const float* k_norm;       /* [d] (qk_norm only) */
  /* conv modules (conv_group > 0 only), one per sublayer.  A module's
   * kernel projection kp [2*2*(D/conv_group), D] (handle dtype, no bias)
   * maps the residual entering the sublayer to corrections read as
   * [call, tap, group]; base [2 (call), 2 (tap), D] fp32.  Coefficient of
   * channel c, tap k, call n at row t: base[n][k][c] + corr_t[n][k][c /
   * conv_group]; conv_t(y) = coef_0 * y_t + coef_1 * y_(t-1), with no
   * predecessor for a block's first row.  Call 0 (prepare) convolves the
   * residual before the sublayer's norm, call 1 (finish) the sublayer's
   * output before the residual add. */
  const void* conv_att_kp;
  const float* conv_att_base;
  const void* conv_mlp_kp;
  const float* conv_mlp_base;
} dflash_layer_weights;

typedef struct dflash_weights {
  const void* wc;            /* [D, n_pick*D] fusion projection (draft only) */
  const float* g_c;          /* [D] hidden_norm gain (draft only) */
  const float* g_f;          /* [D] final RMSNorm gain before the LM head */
  const void* embed;         /* [V, D] shared embedding */
  const void* lm_head;       /* [V, D] shared LM head */
  dflash_layer_weights layers[DFLASH_MAX_LAYERS];
} dflash_weights;

/* Per-layer K/V cache (device, borrowed).  k[l], v[l]: [batch_cap, G, cap, d]
 * in the handle's dtype; len: device int32 [batch_cap], the number of filled
 * positions of each sequence (entry t holds position t). */
typedef struct dflash_kv {
  void* k[DFLASH_MAX_LAYERS];
  void* v[DFLASH_MAX_LAYERS];
  int32_t* len;
  int32_t cap;
  int32_t batch_cap;
} dflash_kv;

typedef struct dflash_handle dflash_handle;

/* Create a handle for one model.  Validates the shape, copies cfg and the
 * weight pointers, allocates the device status word and a RoPE table of
 * max_pos x d/2 (cos, sin) pairs computed on the host in double precision.
 * Requires a device of compute capability 10.3. */
int dflash_create(const dflash_config* cfg, const dflash_weights* w, dflash_handle** out);
int dflash_destroy(dflash_handle* h);

/* Bytes of workspace any call of this handle needs: draft blocks of up to
 * max_batch sequences of max_block rows, and fuse / inject / target-forward
 * calls of up to max_rows rows (a forward pass over batch*T rows counts as
 * batch*T).  The caller allocates it (256-byte aligned) and passes it with
 * its size; a call given less returns DFLASH_ERR_WORKSPACE. */
size_t dflash_workspace_bytes(const dflash_handle* h, int32_t max_batch, int32_t max_block,
                              int64_t max_rows);

/* Target layers whose hidden states are fused (host, integer only):
 * n_pick ids spread uniformly over 0-based [1, n_target_layers-3],
 * rounding half up; n_pick == 1 takes the middle layer n_target_layers/2.
 * (txtmix §5, build_target_layer_ids.)  ids_out: host int32[n_pick]. */
int dflash_build_target_layer_ids(int32_t n_target_layers, int32_t n_pick, int32_t* ids_out);

/* Step 1 — context fusion.  hidden: host array of n_pick device pointers,
 * each [T, D] (handle dtype), in ascending layer order.  h_t_out: device
 * [T, D] (handle dtype).  H_t = RMSNorm(concat(hidden) W_c^T; g_c). */
int dflash_fuse_context(dflash_handle* h, const void* const* hidden, int64_t T,
                        void* h_t_out, void* ws, size_t ws_bytes, dflash_stream_t s);

/* Step 2 — K/V injection.  h_t: device [n_rows, D].  Rows
 * seq_row0[b] .. seq_row0[b]+seq_rows[b]-1 of h_t belong to sequence b
 * (device int32 [batch] each) and are appended to sequence b of every
 * layer's cache at positions len[b] .. len[b]+seq_rows[b]-1:
 *   K = RoPE(k_norm(h_t W_k^T), pos), V = h_t W_v^T.
 * kv->len is advanced by seq_rows on the device.  A sequence that would
 * exceed kv->cap is skipped and flags DFLASH_ERR_CAPACITY. */
int dflash_inject_kv(dflash_handle* h, const void* h_t, int64_t n_rows,
                     const int32_t* seq_row0, const int32_t* seq_rows, int32_t batch,
                     const dflash_kv* kv, void* ws, size_t ws_bytes, dflash_stream_t s);

/* Step 3 — one block draft forward.  anchor: device int32 [batch].  The
 * block of sequence b is [anchor[b], mask x (B-1)] at positions
 * len[b] .. len[b]+B-1 and attends (no mask) to its own B rows and to the
 * len[b] cached context entries of each layer.  The cache is only read:
 * the block's own K/V live in the workspace.
 *   draft_ids: device int32 [batch, B]; column 0 = anchor, columns 1..B-1 =
 *              argmax (lowest index on ties) of the fp32 logits.  May be
 *              NULL when hidden_out is given: the LM head is skipped (a
 *              caller that samples at T > 0 takes the residual, then
 *              dflash_lm_head_logits and dflash_sample_rows).
 *   top2_gap:  nullable device fp32 [batch, B-1], top-1 minus top-2 logit.
 *   hidden_out: nullable device fp32 [batch*B, D], the residual stream after
 *              the last layer (before the final norm). */
int dflash_draft_block(dflash_handle* h, const int32_t* anchor, int32_t batch, int32_t B,
                       const dflash_kv* kv, int32_t* draft_ids, float* top2_gap,
                       float* hidden_out, void* ws, size_t ws_bytes, dflash_stream_t s);

/* Steps 1-3 of one speculative round in one call: context fusion of the
 * n_rows pending target features (hidden, as for dflash_fuse_context, into
 * h_t_out), their K/V injection (seq_row0 / seq_rows as for
 * dflash_inject_kv; kv->len advances by seq_rows), then the block draft of
 * dflash_draft_block over the grown caches.  The result equals the three
 * calls in that order.  Blocks of at most 16 rows with at most 16 pending
 * rows (bf16, head dim 128) run as one persistent launch; other shapes run
 * the three calls.  n_rows == 0 skips fusion and injection.  draft_ids may
 * be NULL when hidden_out is given, as for dflash_draft_block (a round that
 * samples or selects its drafts from the residual). */
int dflash_draft_round(dflash_handle* h, const void* const* hidden, int32_t n_rows,
                       const int32_t* seq_row0, const int32_t* seq_rows, void* h_t_out,
                       const int32_t* anchor, int32_t batch, int32_t B, const dflash_kv* kv,
                       int32_t* draft_ids, float* top2_gap, float* hidden_out, void* ws,
                       size_t ws_bytes, dflash_stream_t s);

/* Step 4 — greedy verification (integer only, no handle).
 * draft, post: device int32 [batch, B]; post[b, j] is the target's argmax at
 * block position j.  accept[b] = number of leading j in 1..B-1 with
 * draft[b, j] == post[b, j-1]; bonus[b] = post[b, accept[b]];
 * out_tokens[b] = draft[b, 1..accept], bonus, then -1 padding;
 * tau[b] = accept[b] + 1 (nullable); new_len[b] = start[b] + accept[b] + 1,
 * the trimmed target-cache length (nullable; may alias start). */
int dflash_verify_greedy(const int32_t* draft, const int32_t* post, int32_t batch, int32_t B,
                         const int32_t* start, int32_t* accept, int32_t* tau, int32_t* bonus,
                         int32_t* out_tokens, int32_t* new_len, dflash_stream_t s);

/* Device-side bookkeeping of a round, so a loop of rounds needs no host read
 * in between (txtmix §9: the emitted tokens of a round are the accepted
 * drafts and the bonus).  out_tokens, tau: device int32 [batch, B] and
 * [batch] as written by dflash_verify_greedy.  For each sequence b the first
 * tau[b] tokens are appended to out_buf[b, out_len[b] ..] (device int32
 * [batch, out_cap]; tokens past out_cap are counted but not stored) and
 * out_len[b] (device int32 [batch]) advances by tau[b].  tau_log (nullable,
 * device int32 [batch, log_cap]) records tau at index n_rounds[b] (device
 * int32 [batch], advanced by one).  The handle only supplies the status word:
 * a tau outside [1, B] flags DFLASH_ERR_DEVICE_BOUNDS and emits nothing. */
int dflash_emit_tokens(dflash_handle* h, const int32_t* out_tokens, const int32_t* tau,
                       int32_t batch, int32_t B, int32_t* out_buf, int32_t out_cap,
                       int32_t* out_len, int32_t* tau_log, int32_t log_cap, int32_t* n_rounds,
                       dflash_stream_t s);

/* One greedy round from and to host memory (txtmix §9: draft a block from
 * the new target features, verify it against the target's argmax): the
 * round's inputs are copied in, dflash_draft_round and dflash_verify_greedy
 * run, and the results are copied out, all queued on stream s with one
 * cudaMemcpyAsync per buffer and direction.  The call returns once the work
 * is queued; host_out holds the results after the stream is synchronised.
 *   host_features: host [n_pick, n_rows, D] in the handle's dtype, pinned
 *     for an asynchronous copy (NULL when n_rows == 0); dev_features: device
 *     buffer of the same size, 16-byte aligned; slice i becomes hidden[i]
 *     of dflash_draft_round.
 *   host_in: host int32 [batch + batch*B], anchor [batch] then post
 *     [batch, B] (the target's argmax, as for dflash_verify_greedy);
 *     dev_in: device int32 of the same size.
 *   host_out, dev_out: host and device int32 [dflash_round_out_len(batch,
 *     B)]: draft_ids [batch, B] at 0, out_tokens [batch, B] at batch*B, then
 *     accept, tau and bonus [batch] at 2*batch*B, 2*batch*B + P and
 *     2*batch*B + 2P, P = batch rounded up to a multiple of 4.
 *   seq_row0, seq_rows, h_t_out, kv, ws: as for dflash_draft_round; start
 *     and new_len (nullable): as for dflash_verify_greedy, device int32.
 * Errors: those of the two calls; DFLASH_ERR_CUDA when a copy cannot be
 * queued.  All buffers are the caller's; nothing is allocated. */
int dflash_round_host(dflash_handle* h, const void* host_features, void* dev_features,
                      int32_t n_rows, const int32_t* host_in, int32_t* dev_in, int32_t* host_out,
                      int32_t* dev_out, const int32_t* seq_row0, const int32_t* seq_rows,
                      void* h_t_out, int32_t batch, int32_t B, const dflash_kv* kv,
                      const int32_t* start, int32_t* new_len, void* ws, size_t ws_bytes,
                      dflash_stream_t s);

/* Entries of dflash_round_host's result buffer: 2*batch*B + 3*P, P = batch
 * rounded up to a multiple of 4.  Host only; -1 for batch < 1 or B < 1. */
int64_t dflash_round_out_len(int32_t batch, int32_t B);

/* Final RMSNorm + shared LM head + fused argmax over rows of an fp32
 * residual stream.  x: device fp32 [rows, D]; norm_gain: device fp32 [D];
 * ids: device int32 [rows]; top2_gap: nullable device fp32 [rows]. */
int dflash_lm_head_argmax(dflash_handle* h, const float* x, int32_t rows, const float* norm_gain,
                          int32_t* ids, float* top2_gap, void* ws, size_t ws_bytes,
                          dflash_stream_t s);

/* fp32 logits of rows of an fp32 residual stream through the final RMSNorm
 * (norm_gain, device fp32 [D]) and the shared LM head.  x: device fp32;
 * logits: device fp32 [rows, V] (16-byte aligned).  skip_first_of = 0 reads
 * x as [rows, D]; skip_first_of = B > 1 reads x as blocks of B rows and
 * skips the first row of each (the anchors), so rows = batch * (B - 1). */
int dflash_lm_head_logits(dflash_handle* h, const float* x, int32_t rows, const float* norm_gain,
                          int32_t skip_first_of, float* logits, void* ws, size_t ws_bytes,
                          dflash_stream_t s);

/* Bytes of device scratch dflash_sample_rows needs for rows rows of the
 * vocabulary (and dflash_verify_rejection for batch = rows sequences):
 * per row 16 bytes for each chunk of 2048 vocabulary entries plus 48, and
 * 512 more.  0 for a negative rows or vocab < 1.  Host only. */
size_t dflash_sampling_ws_bytes(int32_t rows, int32_t vocab);

/* Sampling at temperature T > 0 (txtmix §8, the T = 1 setting of the
 * paper's experiments).  For each row of logits (device fp32 [rows, vocab])
 * p = softmax(logits / T); probs (nullable, device fp32 [rows, vocab])
 * receives p; ids (nullable, device int32) receives the inverse-CDF draw
 * with u[r] (device fp64 [rows], uniform in [0, 1)): the smallest index
 * whose running sum of p in index order exceeds u[r] times the total.  Row r
 * goes to ids[r]; ids_skip_first_of = k > 1 reads ids as blocks of k and
 * fills their slots 1..k-1 in order (row r at block r / (k-1), slot
 * 1 + r % (k-1)), so the draws of dflash_lm_head_logits(skip_first_of = B)
 * land in draft_ids[batch, B] behind the anchors; 1 or negative is
 * DFLASH_ERR_INVALID_ARG.  At least one of ids and probs is required; probs
 * may be the logits buffer itself (the softmax is then taken in place).
 * ws: device scratch of dflash_sampling_ws_bytes(rows, vocab) bytes,
 * 256-byte aligned (DFLASH_ERR_ALIGNMENT, DFLASH_ERR_WORKSPACE otherwise);
 * the call owns it until it completes on s. */
int dflash_sample_rows(dflash_handle* h, const float* logits, int32_t rows, int32_t vocab,
                       float temperature, const double* u, int32_t* ids,
                       int32_t ids_skip_first_of, float* probs, void* ws, size_t ws_bytes,
                       dflash_stream_t s);

/* Speculative sampling verification (txtmix §8: acceptance probability p/q,
 * the prefix ends at the first rejection, the token after it is drawn from
 * max(p - q, 0) renormalised).  draft: device int32 [batch, B] =
 * [anchor, d_1 .. d_{B-1}]; q_probs: device fp32 [batch, B-1, vocab], the
 * draft's distribution at block positions 1..B-1 (d_j was drawn from row
 * j-1); p_probs: device fp32 [batch, B, vocab], the target's distribution of
 * the token after block position j.  d_j is accepted when
 * u_accept[b, j-1] * q(d_j) < p(d_j) (device fp64 [batch, B-1]); with a
 * drafts accepted, the token after them is drawn with u_sample[b] (device
 * fp64 [batch]) from max(p[a] - q[a], 0) when d_{a+1} was rejected, from
 * p[B-1] when all were accepted.  Outputs as dflash_verify_greedy
 * (token: nullable device int32 [batch], the drawn token).  ws: device
 * scratch of dflash_sampling_ws_bytes(batch, vocab) bytes, 256-byte
 * aligned. */
int dflash_verify_rejection(dflash_handle* h, const int32_t* draft, const float* q_probs,
                            const float* p_probs, int32_t vocab, const double* u_accept,
                            const double* u_sample, int32_t batch, int32_t B,
                            const int32_t* start, int32_t* accept, int32_t* tau, int32_t* token,
                            int32_t* out_tokens, int32_t* new_len, void* ws, size_t ws_bytes,
                            dflash_stream_t s);

/* DFlash 2 candidate selection, greedy (txtmix §13-§14: top-k candidates
 * per draft position, an adjacent-pair score, a greedy walk from the
 * anchor).  Rows are block positions 1..B-1 of each sequence.
 *   logits:    device fp32 [batch*(B-1), vocab], the draft's LM-head logits
 *              (dflash_lm_head_logits with skip_first_of = B).
 *   hidden:    device fp32 [batch*B, D], the residual stream after the last
 *              layer (dflash_draft_block's hidden_out); rows 1..B-1 of each
 *              block pass the final RMSNorm with norm_gain (device fp32 [D]).
 *   Each position t keeps its top_k tokens (largest logit first, the lower
 *   id first among equal logits) with unary score U_t = their logit.  The
 *   context gate is H_t = W_h xhat_t (w_h: device [rank, D], handle dtype,
 *   no bias).  From a = anchor[b] the walk takes, at every position, the
 *   candidate c maximising U_t(c) + sum_r code_pred[a, r] H_t[r]
 *   code_succ[c, r] (the earlier candidate on a tie) and continues from it.
 *   code_pred, code_succ: device [n_codes, rank] (handle dtype), n_codes >=
 *   vocab.  1 <= top_k <= DFLASH_SEL_KMAX and top_k <= vocab; rank a positive
 *   multiple of 32.
 *   draft_ids: device int32 [batch, B] = [anchor, path].  candidates
 *   (nullable): device int32 [batch*(B-1), top_k] in that order.  scores
 *   (nullable): device fp32 [batch*(B-1)], the chosen pair scores.
 *   ws: device scratch of dflash_select_ws_bytes(h, batch, B, top_k, rank)
 *   bytes, 256-byte aligned.  An anchor id outside [0, n_codes) reads code
 *   row 0 and sets DFLASH_ERR_DEVICE_BOUNDS. */
size_t dflash_select_ws_bytes(const dflash_handle* h, int32_t batch, int32_t B, int32_t top_k,
                              int32_t rank);
int dflash_select_candidates(dflash_handle* h, const float* logits, const float* hidden,
                             const float* norm_gain, const int32_t* anchor, int32_t batch,
                             int32_t B, int32_t top_k, const void* w_h, int32_t rank,
                             const void* code_pred, const void* code_succ, int32_t n_codes,
                             int32_t* draft_ids, int32_t* candidates, float* scores, void* ws,
                             size_t ws_bytes, dflash_stream_t s);

/* Causal forward of a target model (qk_norm == 0 handle) over T new tokens
 * per sequence, appended to its cache.  tokens: device int32 [batch, T] at
 * positions len[b] .. len[b]+T-1; every row attends to cache entries
 * 0 .. its own position.  kv->len advances by T.
 *   tap_ids: host int32 [n_taps], 0-based layer ids; taps_out (nullable):
 *            device [n_taps, batch*T, D] (handle dtype), the residual
 *            stream after each listed layer.
 *   argmax_out: device int32 [batch*T], greedy next token of every row
 *            (final RMSNorm with g_f, shared LM head). */
int dflash_target_forward(dflash_handle* h, const int32_t* tokens, int32_t batch, int32_t T,
                          const dflash_kv* kv, const int32_t* tap_ids, int32_t n_taps,
                          void* taps_out, int32_t* argmax_out, void* ws, size_t ws_bytes,
                          dflash_stream_t s);

/* LM-head argmax that allocates nothing and takes no workspace.
 * The paper has no counterpart to this call: it exists for callers that cannot
 * give the library device memory at call time, such as a serving loop whose
 * device memory is entirely reserved up front by its own pool, or a
 * latency-critical path that must not call cudaMalloc (which may synchronise
 * the device and has no latency bound).  Same result as dflash_lm_head_argmax
 * (final RMSNorm with norm_gain, shared LM head, lowest-index argmax and
 * top-2 gap per row); same arguments minus the workspace.
 *   - Scratch lives in one file-scope device array of about 5.8 MB that every
 *     GPU which loads the library keeps until the process exits.  Limits:
 *     rows <= 16, hidden <= 8192, vocab <= 262144, and the handle must be a
 *     bf16 handle whose weights tile for the streaming kernel (otherwise
 *     DFLASH_ERR_UNSUPPORTED); larger requests return DFLASH_ERR_STATIC_LIMIT.
 *   - The first call on a device looks up the array's device address (set-up,
 *     once per device, with that device current); make that first call before
 *     any stream capture.
 *   - All calls share the one array and it keeps the last call's contents;
 *     nothing in it needs to start at zero.  Calls that overlap on the GPU
 *     (different streams, or different handles at once) race on it: order
 *     them. */
int dflash_lm_head_argmax_noalloc(dflash_handle* h, const float* x, int32_t rows,
                                  const float* norm_gain, int32_t* ids, float* top2_gap,
                                  dflash_stream_t s);

/* Test of the failure handling (the paper has no counterpart).  Every wait
 * inside the kernels is bounded: on running out it records
 * DFLASH_ERR_DEVICE_TIMEOUT in the handle's status word and returns instead
 * of hanging the GPU.  This call launches one thread that waits, at most
 * limit_ns nanoseconds (1000 .. 1e9), with the kernels' own wait routines on
 * something nothing will complete — which = 0: an mbarrier no thread
 * arrives at; which = 1: a device counter nothing raises (the grid
 * barrier's wait) — so the next dflash_get_status returns
 * DFLASH_ERR_DEVICE_TIMEOUT, and the handle stays usable.  Asynchronous on
 * s; DFLASH_ERR_INVALID_ARG for another which or limit. */
int dflash_selftest_wait(dflash_handle* h, int32_t which, int64_t limit_ns, dflash_stream_t s);

/* Synchronise stream s, then read and clear the handle's device status word.
 * Returns DFLASH_OK or the first device-detected error code. */
int dflash_get_status(dflash_handle* h, dflash_stream_t s);

const char* dflash_strerror(int code);

/* Number of kernels this library has launched in this process. */
int64_t dflash_launch_count(void);

/* Per-kernel device timing.  While enabled, every launch of this handle is
 * bracketed by CUDA events on its stream; dflash_timing_read synchronises,
 * then returns for kernel class `kclass` the summed milliseconds and the
 * launch count since the last reset (and resets that class). */
enum dflash_kernel_class {
  DFLASH_K_WEIGHT_GEMM = 0,   /* skinny weight-streaming projections */
  DFLASH_K_ATTENTION = 1,
  DFLASH_K_LM_HEAD = 2,
  DFLASH_K_DENSE_GEMM = 3,    /* fuse / inject / prefill projections */
  DFLASH_K_ELEMENTWISE = 4,   /* norms, embedding, RoPE, SwiGLU, bookkeeping */
  DFLASH_K_VERIFY = 5,
  DFLASH_K_DRAFT_CHAIN = 6,   /* whole draft block in one persistent launch (<= 16 rows) */
  DFLASH_K_NCLASS = 7
};
int dflash_timing_enable(dflash_handle* h, int on);
int dflash_timing_read(dflash_handle* h, int32_t kclass, double* total_ms, int64_t* launches);

/* Phase timeline of the persistent draft-block kernel (class
 * DFLASH_K_DRAFT_CHAIN).  While enabled (a small device buffer owned by the
 * handle), each such launch records for every phase (embed; per layer q/k/v,
 * attention, combine, o_proj, gate/up, down; LM head) eight device-clock
 * times in ns (%globaltimer): the first and the last CTA to begin it, the
 * first and the last CTA to finish it, the last CTA to finish its
 * multiply-adds, and the latest split-K fix-up start, fix-up sum and
 * epilogue end (the last three only for projection phases; 0 elsewhere).
 * dflash_chain_trace_read synchronises the device and writes these eight
 * values for min(n, phases) phases of the handle's latest traced launch into
 * the host array out[8 * n]; *n_phases gets the phase count (0: none). */
int dflash_chain_trace_enable(dflash_handle* h, int on);
int dflash_chain_trace_read(dflash_handle* h, int64_t* out, int32_t n, int32_t* n_phases);
/* Raw per-CTA event log of the latest traced launch: 4 sampled CTAs x 164
 * phases x 50 words (times are the CTA's SM cycle counter, comparable within
 * one CTA only; 0 = no event): phase start, phase end, then for the CTA's
 * first 12 projection units: data ready, multiply done, weight load issued,
 * activation load issued.  Recorded only by builds compiled with
 * -DDFLASH_CH_EVLOG=1 (a profiling build); otherwise all zero.  Copies
 * min(n, total) words to the host array out; *count gets the number copied. */
int dflash_chain_trace_events(dflash_handle* h, int64_t* out, int64_t n, int64_t* count);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
