/*
 * blockdrafter.h -- C ABI of a GB300 (sm_103a) library that runs one proposal round of
 * a DFlash-style parallel block drafter with DSpine's adjacent gated causal injection.
 *
 * Sources the operations follow (page title and section):
 *   [DFlash-notes] NInfer maintainer page "dflash.md": conditioning equations, context
 *                  K/V projection, draft input table, local-window attention rule,
 *                  per-layer equations, proposal head, ring storage.
 *   [Bridge]       "DSpine for Qwen3.8-27B: Causal Features Through Depth", section
 *                  "The bridge: read 1,024 features, write through rank 512".
 *   [Gate]         "DSpine 完全拆解", sections "相邻因果注入" and "门控与写回".
 *   [BlockCausal]  "DSpine 完全拆解", section "块因果注意力".
 *
 * Conventions shared by every entry point:
 *   - Every pointer marked "dev" is a device pointer the CALLER allocated and owns; the
 *     library never allocates, frees or synchronises.  It enqueues kernels on `stream`
 *     (a cudaStream_t passed as void*; NULL = legacy default stream) and returns.
 *   - Matrices are row-major [out, in] (PyTorch nn.Linear layout), contiguous, in the
 *     config's element type (bf16 or fp32), 16-byte aligned base addresses.
 *   - Every call returns a bd_status and never aborts; bd_last_error() gives a
 *     thread-local message for the last non-OK status.  Invalid arguments are
 *     rejected on the host before anything is enqueued.
 *   - `workspace` is caller-owned device scratch of at least bd_workspace_bytes(...)
 *     bytes, 256-byte aligned; its contents need not be initialised and are
 *     clobbered.  Calls that share a workspace must be ordered on one stream.
 *   - Device-side waits are bounded; a wait that gives up sets a device error word
 *     that bd_sync_status() reports as BD_ERR_DEVICE_TIMEOUT.
 */
#ifndef BLOCKDRAFTER_H
#define BLOCKDRAFTER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BD_ABI_VERSION 8
#define BD_MAX_LAYERS 16

typedef enum {
  BD_OK = 0,
  BD_ERR_INVALID_ARG = -1,     /* null pointer, bad size, out-of-range id, misalignment  */
  BD_ERR_UNSUPPORTED = -2,     /* geometry the kernels do not implement (never a fallback) */
  BD_ERR_CUDA = -3,            /* a CUDA runtime/driver call failed                        */
  BD_ERR_DEVICE_TIMEOUT = -4,  /* a bounded device-side wait gave up                       */
  BD_ERR_WORKSPACE = -5,       /* workspace too small or misaligned                        */
  BD_ERR_RANGE = -6            /* a value met an fp16 conversion beyond +-65504 (or not
                                  finite): a weight while packing, or an activation on its
                                  way into an fp16 tensor-core operand (bd_sync_status)     */
} bd_status;

typedef enum { BD_BF16 = 0, BD_F32 = 1 } bd_dtype;

/* Block attention among the W block rows.  [DFlash-notes] is bidirectional;
 * [BlockCausal] lets row i see block rows 0..i only.  Context keys are unaffected. */
typedef enum { BD_BLOCK_BIDIRECTIONAL = 0, BD_BLOCK_CAUSAL = 1 } bd_block_mask;

/* Draft geometry; the fields mirror a DFlash draft config ([DFlash-notes], config
 * fields: layer count, dimensions, eps, RoPE theta, layer attention types, sliding
 * window, target block ids, mask token id) plus the DSpine bridge widths ([Bridge]). */
typedef struct {
  int hidden;                        /* H                                                  */
  int n_layers;                      /* L <= BD_MAX_LAYERS                                 */
  int n_q_heads, n_kv_heads;         /* Hq, Hkv (Hq % Hkv == 0)                            */
  int head_dim;                      /* D: 64 or 128                                       */
  int ffn;                           /* SwiGLU intermediate width I                        */
  int vocab;                         /* V rows of the tied embedding / LM head             */
  int n_target_layers;               /* captured target layers; W_feature is [H, n*H]      */
  int window[BD_MAX_LAYERS];         /* sliding window S of layer l; 0 = full context      */
  int ring_capacity[BD_MAX_LAYERS];  /* ring slots of layer l (>= window; full: max ctx)   */
  float eps;                         /* RMSNorm eps, also the bridge's numerical floor     */
  float rope_theta;                  /* split-half RoPE base                               */
  int mask_token_id;                 /* MASK id fed to the K proposal rows                 */
  int code_width;                    /* Rc; 0 disables the bridge (plain DFlash)           */
  int msg_width;                     /* Mc                                                 */
  int block_mask;                    /* bd_block_mask                                      */
  int dtype;                         /* bd_dtype of weights, rings and activations         */
  int conv_group;                    /* DFlash2 dynamic grouped convolution: group width   */
                                     /* gw (a multiple of 4 dividing H), or 0 for none     */
} bd_config;

/* Per-layer weights (dev, caller-owned, row-major [out, in], config dtype). */
typedef struct {
  const void *in_norm;   /* [H]                                                          */
  const void *wq;        /* [Hq*D, H]                                                    */
  const void *wk;        /* [Hkv*D, H]  used for block AND context keys                  */
  const void *wv;        /* [Hkv*D, H]  used for block AND context values                */
  const void *q_norm;    /* [D] per-head query RMSNorm gain                              */
  const void *k_norm;    /* [D] per-head key RMSNorm gain                                */
  const void *wo;        /* [H, Hq*D]                                                    */
  const void *post_norm; /* [H]                                                          */
  const void *w_gate;    /* [I, H]                                                       */
  const void *w_up;      /* [I, H]                                                       */
  const void *w_down;    /* [H, I]                                                       */
  const void *r_read;    /* [Rc, H]  DSpine per-layer code read R_l (bridge only)        */
  const void *w_write;   /* [H, Mc]  DSpine per-layer write W_l (bridge only)            */
  /* DFlash2 convolution (conv_group = gw > 0 only): per branch (a = attention, m = MLP)
   * the delta projection [4*H/gw, H], rows ordered (side, tap, group), and the base
   * coefficients [2 sides][2 taps][H]. */
  const void *conv_delta_a, *conv_base_a;
  const void *conv_delta_m, *conv_base_m;
} bd_layer_weights;

typedef struct {
  const void *w_feature;    /* [H, n_target_layers*H], bias-free                          */
  const void *context_norm; /* [H]                                                        */
  const void *final_norm;   /* [H]                                                        */
  const void *embed_head;   /* [V, H] tied target embedding and LM head                   */
  const void *codebook;     /* [V, Rc] token-code table (bridge only)                     */
  const void *g_recv;       /* [Mc, Rc] receiver gate G, shared by all layers             */
  const void *g_pred;       /* [Mc, Rc] predecessor gate G_p, shared                      */
  const void *a_val;        /* [Mc, Rc] predecessor value map A, shared                   */
  const void *gate_bias;    /* [Mc] gate bias b, or NULL for b = 0                        */
  bd_layer_weights layer[BD_MAX_LAYERS];
  /* Optional packed image of every projection matrix written by bd_pack_weights (dev,
   * caller-owned), or NULL.  When set, the tensor-core products stream weight tiles from
   * it (one contiguous copy per pipeline stage); the row-major matrices above are still
   * required (embedding rows, norm gains, codebook and the raw layout are read from them). */
  const void *packed;
} bd_weights;

/* Context K/V rings ([DFlash-notes], ring storage): layer l holds
 * k[l], v[l] = dev [b_max][Hkv][ring_capacity[l]][D] in the config dtype.  Absolute
 * position p of request b lives in slot p mod ring_capacity[l]; a ring whose request
 * has context frontier F holds the live interval [max(0, F - cap), F).  Request b of
 * a round or a materialisation uses ring row b. */
typedef struct {
  void *k[BD_MAX_LAYERS];
  void *v[BD_MAX_LAYERS];
  int b_max;
} bd_kv_cache;

/* Library ABI version (BD_ABI_VERSION). */
int bd_abi_version(void);

/* Bytes of workspace any entry point below needs for rounds of up to `b_max`
 * requests with up to `max_masks` masks (K) and materialisations of up to
 * `max_ctx_rows` rows per call (a round's own pending rows, up to 16 per request, are
 * always covered).  Returns 0 for an invalid or unsupported config. */
size_t bd_workspace_bytes(const bd_config *cfg, int b_max, int max_masks, int max_ctx_rows);

/* Bytes of the packed weight image for `cfg` (0 for an invalid config). */
size_t bd_packed_bytes(const bd_config *cfg);

/*
 * Writes the packed image of every projection matrix of `w` into `packed` (dev,
 * caller-owned, >= bd_packed_bytes(cfg) bytes, 1024-byte aligned).  The image holds each
 * matrix as 128-row x 128-byte tiles, each tile contiguous and already in the 128-byte
 * swizzled order the tensor cores read from shared memory (the SwiGLU gate and up
 * matrices interleaved 64 rows each per tile); out-of-range rows/columns are zero.  Run it
 * once after loading the weights, then set w->packed = packed.
 *
 * The image is not only a permutation.  In a bf16 config it stores the attention-branch
 * matrices (W_q, W_k, W_v, W_o, and with conv_group > 0 the attention branch's W_delta),
 * the MLP matrices (W_gate, W_up, W_down, and the MLP branch's W_delta), the bridge
 * matrices (R_l, W_l, G, G_p, A) and the LM head as fp16, and the products that read them
 * then take fp16 activations (see bd_ctx_kv_materialize, bd_draft_round, bd_lm_head_argmax
 * and bd_refine_tail); W_feature stays bf16, bit for bit.  The
 * conversion is exact for every bf16 value of magnitude 2^-14 .. 65504; smaller values
 * become fp16 subnormals with an absolute error of at most 2^-25; a value beyond
 * +-65504 makes the next bd_sync_status return BD_ERR_RANGE.  Results with and without
 * the image therefore differ by these roundings and the activations' fp16 rounding
 * (about 1e-3 of max|h| at the 27B geometry; context K/V by up to one bf16 unit), not bit
 * for bit.  In an fp32 config the
 * image is a pure permutation.
 */
bd_status bd_pack_weights(const bd_config *cfg, const bd_weights *w, void *packed,
                          size_t packed_bytes, void *stream);

/*
 * Context K/V materialisation (S1 + S2).  [DFlash-notes], conditioning and context K/V:
 *   c_t = plain_rmsnorm(W_feature s_t, context_norm)
 *   for each layer l:  k = rope_1d(plain_head_rmsnorm(W_k^l c_t, k_norm^l), t)
 *                      v = W_v^l c_t
 * stored (bf16 round-to-nearest in a bf16 config) into ring row `row_request[r]` at
 * slot row_pos[r] mod ring_capacity[l].  In a bf16 config c_t enters the K/V products as
 * bf16, or as fp16 with the packed image (whose W_k, W_v are fp16; see bd_pack_weights).
 *
 *   target_feats  dev [n_rows, n_target_layers*H]  captured residual rows s_t (the
 *                 target layers' residual outputs concatenated in recorded order)
 *   row_request   dev int32 [n_rows]  ring row (request) of each feature row, < b_max
 *   row_pos       dev int64 [n_rows]  absolute context position t of each row (>= 0)
 *   ctx_frontier  dev int64 [b_max]   each request's context frontier F AFTER this call.
 *                 A row is stored in layer l only if row_pos >= F - ring_capacity[l]
 *                 (the final live window); older rows of a long chunk are computed
 *                 but not stored, while the frontier still covers the whole chunk.
 *   n_rows        1 .. max_ctx_rows given to bd_workspace_bytes
 * Rows of one request must have distinct positions.  Rows are independent: any split
 * of a chunk into calls stores the same ring contents.
 */
bd_status bd_ctx_kv_materialize(const bd_config *cfg, const bd_weights *w,
                                const bd_kv_cache *kv, const void *target_feats,
                                const int32_t *row_request, const int64_t *row_pos,
                                const int64_t *ctx_frontier, int n_rows, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * Pending context rows a round materialises before it drafts (the decode-step catch-up,
 * [DFlash-notes] paragraph on the processed-token frontier: feature rows the target has
 * committed but the drafter has not yet turned into context K/V are converted first, so
 * that the draft context extends to F when the block is proposed).
 * The rows' context K/V are computed and stored exactly as bd_ctx_kv_materialize would
 * (c_t enters the K/V products as bf16 in a bf16 config), but inside the round: the
 * feature projection runs first and every layer's context K/V products share the weight
 * tiles of that layer's block Q/K/V product (one read of W_k and W_v per layer).
 *
 *   feats    dev [n_rows, n_target_layers*H]  captured residual rows s_t
 *   request  dev int32 [n_rows]  request (ring row) of each row, < B of the round
 *   pos      dev int64 [n_rows]  absolute position t of each row, one of the 16 newest:
 *            frontier[request] - 16 <= t < frontier[request] (a row outside that range is
 *            skipped and reported by bd_sync_status); stored in layer l only if
 *            t >= frontier[request] - ring_capacity[l]
 *   n_rows   0 .. 16*B (0 = nothing pending)
 * Rows of one request must have distinct positions.
 */
typedef struct {
  const void *feats;
  const int32_t *request;
  const int64_t *pos;
  int n_rows;
} bd_pending;

/*
 * One masked-block draft forward (S3 .. S9 and the final norm) for B requests.
 * Numerics (bf16 config): the residual stream, norms, softmax statistics and every
 * accumulator are fp32; context K/V are used as stored (bf16).
 *   Without the packed image (w->packed NULL) the weights are used as stored and every
 *   activation that feeds a tensor-core product (normed rows, attention output, SwiGLU
 *   product, codes, messages, queries, softmax weights, the block's own keys/values)
 *   enters as a bf16 hi+lo pair (about 16 significant bits).
 *   With the packed image the Q/K/V, W_o, MLP and bridge products read fp16 weights (see
 *   bd_pack_weights) and take fp16 activations (the normed rows, the attention output,
 *   the SwiGLU product, the codes and messages: 11 significant bits; for B * W <= 32
 *   the one-launch bridge also takes the raw residual rows, unnormalised, as fp16).  An
 *   activation beyond the fp16 range on its way into an fp16 operand is still stored (as
 *   +-inf) and makes the next bd_sync_status return BD_ERR_RANGE.
 *   The attention always takes the queries, softmax weights and the block's own keys/values
 *   as bf16 hi+lo pairs against the ring's bf16 keys/values as stored.
 * [DFlash-notes] draft input table and per-layer equations; [Bridge] and [Gate] for
 * the injection after every layer when code_width > 0:
 *   row (b, 0) = embed(anchor_ids[b]) at position F_b; rows (b, i>=1) = embed(MASK) at
 *   F_b + i.  Each layer: rmsnorm -> Q/K/V (+ head norm, RoPE) -> attention over the
 *   request's ring context and its own block -> W_o + residual -> rmsnorm -> SwiGLU +
 *   residual -> [bridge read, anchor code, gated predecessor message, RMS-scaled write;
 *   the anchor row receives no write].  Then final plain_rmsnorm.
 *   With conv_group = gw > 0 (DFlash2, [DFlash-notes] dynamic grouped convolution) each
 *   branch works on Conv_0 of its normalised input X and adds Conv_1 of its output, both
 *   with delta = W_delta X as [2 sides][2 taps][H/gw] per row:
 *     Conv_s(Y)[i, c] = (base[s,0,c] + delta[i,s,0,c/gw]) Y[i, c]
 *                       + [i >= 1] (base[s,1,c] + delta[i,s,1,c/gw]) Y[i-1, c]
 *   over the block rows i of each request (no history across requests or rounds).
 *
 *   anchor_ids  dev int32 [B]  anchor token a_b (< vocab)
 *   frontier    dev int64 [B]  committed context length F_b >= 1 of request b; ring row b
 *               must hold the live interval of every layer at that frontier
 *   B           1 .. 8 requests;  n_masks  K in 1 .. 15 (block width W = K + 1)
 *   head_in     dev fp32 [B*K, H] OUT: final-normed mask rows, row b*K + (i-1) for block
 *               row i >= 1 -- the input of bd_lm_head_argmax
 *   hidden_out  dev fp32 [B*W, H] OUT final-normed rows of every block row, or NULL
 *   layers_out  dev fp32 [L, B*W, H] OUT post-injection residual after each layer, or
 *               NULL (a debugging/parity output; it adds device-to-device copies)
 *   tail_state  dev fp32 OUT, or NULL: the last layer's state the last-write refinement
 *               redoes its injection from (input of bd_refine_tail), T = B*W rows:
 *               [T*H] pre-injection residual u, then [T] its RMS r, then [T*Mc] the
 *               receiver gate term G c.  Requires code_width > 0.
 *   pending     host pointer to a bd_pending (its arrays are dev), or NULL: context rows
 *               to materialise first; frontier[] is then the frontier they complete
 */
bd_status bd_draft_round(const bd_config *cfg, const bd_weights *w, const bd_kv_cache *kv,
                         const int32_t *anchor_ids, const int64_t *frontier, int B,
                         int n_masks, float *head_in, float *hidden_out, float *layers_out,
                         float *tail_state, const bd_pending *pending, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * Tied LM head with per-row argmax (S10).  [DFlash-notes], proposal head:
 *   logits = embed_head . hidden_r ;  token_out[r] = argmax_v logits[v]
 * Ties resolve to the lowest token id.  fp32 accumulation.  In a bf16 config without
 * the packed image each hidden row enters the tensor cores as a bf16 hi+lo pair (about
 * 16 significant bits) against the bf16 head as stored; with the packed image the head
 * is its fp16 copy (see bd_pack_weights) and each hidden row enters as fp16 (11
 * significant bits; a value beyond +-65504 makes bd_sync_status return BD_ERR_RANGE).
 * An fp32 config uses tf32 tensor-core products on the fp32 rows and head.
 *
 *   hidden         dev fp32 [rows, H] (e.g. bd_draft_round's head_in)
 *   rows           1 .. 8*15
 *   token_out      dev int32 [rows]  OUT
 *   max_logit_out  dev fp32 [rows]   OUT the winning logit, or NULL
 */
bd_status bd_lm_head_argmax(const bd_config *cfg, const bd_weights *w, const float *hidden,
                            int rows, int32_t *token_out, float *max_logit_out,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Tied LM head with the k best candidates per row (k <= 16; the candidate sets of the
 * last-write refinement).  "DSpine for Qwen3.8-27B: Causal Features Through Depth",
 * section "The last write is refined using discrete candidates": the released drafter
 * keeps 16 candidates per proposal row, and its fallback path scores them with the BF16
 * vocabulary head -- the exact version computed here (no FP8 pre-selection):
 *   logits = embed_head . hidden_r ;  the k largest logits of row r, by descending
 *   score, equal scores to the lower token id.
 * Arithmetic as in bd_lm_head_argmax; candidate r*k + 0 is bd_lm_head_argmax's token.
 *
 *   hidden     dev fp32 [rows, H];  rows 1 .. 8*15;  k 1 .. BD_TOPK_MAX (and <= vocab)
 *   token_out  dev int32 [rows, k]  OUT candidate ids, best first
 *   score_out  dev fp32 [rows, k]   OUT their logits, or NULL
 * Errors: BD_ERR_INVALID_ARG for k, rows or pointers out of range; the workspace is the
 * one bd_workspace_bytes sizes (it covers both head entry points).
 */
#define BD_TOPK_MAX 16
bd_status bd_lm_head_topk(const bd_config *cfg, const bd_weights *w, const float *hidden, int rows,
                          int k, int32_t *token_out, float *score_out, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * FP8 retrieval head.  "DSpine for Qwen3.8-27B: Causal Features Through Depth", section
 * "The last write is refined using discrete candidates": the released drafter's optimized
 * path scores the whole vocabulary approximately with a row-scaled FP8 copy of the head,
 * takes 128 candidates, rescores them with the BF16 head and keeps 16.
 *   image:      each head row v as e4m3(E_v / s_v), s_v = max|E_v| / 448 (round to nearest
 *               even; fp32 division), stored in the GEMM's packed tile layout, then the V
 *               fp32 scales s_v.  bd_pack_head_fp8 writes it from w->embed_head (a bf16
 *               config with hidden % 16 == 0); its size is bd_head_fp8_bytes(cfg) (0 if
 *               the config has no FP8 head), `image` 1024-byte aligned, caller-owned.
 *   retrieval:  each hidden row is coded the same way (scale max|h| / 448); approximate
 *               score of row v = s_v * (codes_v . codes_h) (the hidden row's common scale
 *               is left out); each 128-row vocabulary tile keeps its 16 best, and the row
 *               the n_cand best of those (a tile holding more than 16 of them loses its
 *               excess; equal scores to the lower id).
 *   rescoring:  the exact logits embed_head[c] . hidden_r of the n_cand candidates (bf16 head
 *               rows, fp32 hidden, fp32 sums); the k best, by descending score, equal
 *               scores to the lower id (the order of bd_lm_head_topk).
 *
 *   hidden     dev fp32 [rows, H];  rows 1 .. 8*15;  k 1 .. BD_TOPK_MAX;  n_cand k .. 256
 *              (and <= vocab);  the pages' value is 128
 *   token_out  dev int32 [rows, k]  OUT;  score_out  dev fp32 [rows, k] OUT or NULL
 * The rescoring gives each returned id its exact logit; whether the exact top k were all
 * among the candidates is not guaranteed (candidate generation, not an exact head).
 * Errors: BD_ERR_UNSUPPORTED for an fp32 config or hidden % 16 != 0; BD_ERR_INVALID_ARG
 * for out-of-range sizes or pointers.  Workspace as sized by bd_workspace_bytes.
 */
size_t bd_head_fp8_bytes(const bd_config *cfg);
bd_status bd_pack_head_fp8(const bd_config *cfg, const bd_weights *w, void *image,
                           size_t image_bytes, void *stream);
bd_status bd_lm_head_topk_fp8(const bd_config *cfg, const bd_weights *w, const void *head_fp8,
                              const float *hidden, int rows, int n_cand, int k,
                              int32_t *token_out, float *score_out, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * Last-write refinement, transition tables and greedy walk (the DSpine tail).
 * "DSpine for Qwen3.8-27B: Causal Features Through Depth", section "The last write is
 * refined using discrete candidates", and "DSpine 完全拆解", section on predecessor-
 * conditioned decoding and the transition cache.  For block row i >= 2 of request b and
 * each candidate s of row i-1 the last layer's injection into row i is redone from
 * tail_state with the predecessor code replaced by sqrt(Rc) * codebook[s]:
 *   g = sigmoid(G c_i + G_p c_s + b),  m = g * (A c_s),  x' = u_i + r_i W_L m,
 *   h' = plain_rmsnorm(x', final_norm),  table[b][i-2][p][j] = embed_head[cand_j] . h'
 * over row i's candidates j.  Row 1 keeps its own scores (its predecessor is the anchor,
 * which the round already used).  The greedy walk takes row 1's lowest-rank best
 * candidate, then for i = 2..K the lowest-rank best of the table row of row i-1's choice.
 * With the packed image the products read its fp16 G_p, A and W_L and take the codebook
 * rows and messages as fp16; without it, bf16 weights with exact bf16 codebook rows and
 * bf16 hi+lo messages.
 *
 *   tail_state   dev fp32, from bd_draft_round of the same B and n_masks
 *   cand_ids     dev int32 [B*K, kc]  candidates of the mask rows (e.g. bd_lm_head_topk)
 *   cand_scores  dev fp32 [B*K, kc]   their scores (row 1 of each request is read)
 *   B 1..8;  n_masks K 2..15;  kc 1..BD_TOPK_MAX
 *   token_out    dev int32 [B*K]  OUT the walk's tokens
 *   pick_out     dev int32 [B*K]  OUT the chosen candidate indices, or NULL
 *   table_out    dev fp32 [B, K-1, kc, kc]  OUT the transition tables, or NULL
 * Errors: BD_ERR_INVALID_ARG (ranges, NULL inputs, no bridge); out-of-range candidate
 * ids are reported by bd_sync_status.  Workspace as sized by bd_workspace_bytes.
 */
bd_status bd_refine_tail(const bd_config *cfg, const bd_weights *w, const float *tail_state,
                         const int32_t *cand_ids, const float *cand_scores, int B, int n_masks,
                         int kc, int32_t *token_out, int32_t *pick_out, float *table_out,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * bd_lm_head_argmax without a workspace, for callers that cannot allocate device
 * memory (no counterpart in the papers; it computes exactly what bd_lm_head_argmax
 * computes, with the same kernels).  Callers such as a serving engine whose pool owns
 * all device memory after start-up, or a plugin host that gives the library no
 * allocation hook, cannot hand over a workspace; this entry point allocates nothing.
 *
 * Its scratch is one file-scope device array of BD_NOALLOC_SCRATCH_BYTES that every GPU
 * loading the library holds until the process exits.  Limits: rows <= 32, hidden <=
 * 8192, vocab <= 262144; larger sizes return BD_ERR_INVALID_ARG with a message.
 * All calls share the array and it keeps the previous call's contents (the counters
 * that must start at zero are cleared by every call), so calls that overlap on the GPU
 * -- on two streams or from two threads -- race and must be ordered by the caller.
 * The first call on a device looks up the array's device address (with that device
 * current) and caches it; make that first call before any stream capture.  The cached
 * address belongs to the device's context of that moment: after cudaDeviceReset on that
 * device, do not call this entry point again in the same process.
 * The configuration is checked as bd_lm_head_argmax checks it (BD_ERR_INVALID_ARG).
 */
#define BD_NOALLOC_MAX_ROWS 32
#define BD_NOALLOC_MAX_HIDDEN 8192
#define BD_NOALLOC_MAX_VOCAB 262144
#define BD_NOALLOC_SCRATCH_BYTES (12u << 20)
bd_status bd_lm_head_argmax_noalloc(const bd_config *cfg, const bd_weights *w,
                                    const float *hidden, int rows, int32_t *token_out,
                                    float *max_logit_out, void *stream);

/*
 * Measurement hook (no counterpart in the papers): brackets single kernel launches with
 * caller-created CUDA events (cudaEvent_t passed as void*, timing enabled), so that a
 * benchmark can time one kernel of a round, also inside a captured graph.  While a kind
 * is set on the calling thread, the i-th launch of that kind within each later
 * bd_draft_round call (or bd_lm_head_argmax call, for BD_TIME_HEAD) is preceded by
 * cudaEventRecord(begin[i]) and followed by cudaEventRecord(end[i]) on the call's
 * stream, for i < n; further launches of the kind are not bracketed.  The events stay
 * owned by the caller and must outlive every call (or graph replay) that records them.
 * An event between two launches removes their programmatic overlap, so a bracketed
 * round runs slightly slower than an unbracketed one.  kind BD_TIME_NONE clears the
 * setting (begin, end and n are then ignored).
 * Errors: BD_ERR_INVALID_ARG for an unknown kind, n outside 1..BD_TIMING_MAX or a NULL
 * event.
 */
#define BD_TIMING_MAX 32
typedef enum {
  BD_TIME_NONE = 0,
  BD_TIME_QKV = 1,        /* the Q/K/V product of each layer                    */
  BD_TIME_ATTENTION = 2,  /* the block attention of each layer                  */
  BD_TIME_WO = 3,         /* the output projection of each layer                */
  BD_TIME_GATE_UP = 4,    /* the SwiGLU gate/up product of each layer           */
  BD_TIME_DOWN = 5,       /* the down projection of each layer                  */
  BD_TIME_BRIDGE = 6,     /* the one-launch DSpine bridge of each layer         */
  BD_TIME_HEAD = 7        /* the LM-head product of bd_lm_head_argmax           */
} bd_time_kind;
bd_status bd_set_timing_events(int kind, void *const *begin, void *const *end, int n);

/* Number of kernels this library has enqueued (all threads) since it was loaded.
 * Graph replays do not pass through the library and are not counted. */
uint64_t bd_kernel_launches(void);

/* Failure-path self-test: enqueues one thread that waits, with the bounded inter-CTA wait
 * the split-tile reductions and attention splits use, for the dev uint32 *flag (4-byte
 * aligned, caller-owned) to become >= 1, giving up after limit_us microseconds
 * (1 .. 2,000,000; those kernels use 2 s).  A wait that gives up flags the device error
 * word, so the next bd_sync_status returns BD_ERR_DEVICE_TIMEOUT, and ends: nothing hangs
 * and the context stays usable. */
bd_status bd_selftest_wait(const unsigned *flag, int limit_us, void *stream);

/* Thread-local description of the last non-OK status returned on this thread. */
const char *bd_last_error(void);

/* Synchronises `stream`, then reads and clears the device error word.  Returns
 * BD_ERR_DEVICE_TIMEOUT if a bounded device wait gave up since the last check,
 * BD_ERR_INVALID_ARG if a kernel met an out-of-range id or position, BD_ERR_RANGE if a
 * value met an fp16 conversion beyond +-65504 (or was not finite), BD_ERR_CUDA if the
 * stream reports an error, BD_OK otherwise. */
bd_status bd_sync_status(void *stream);

#ifdef __cplusplus
}
#endif
#endif /* BLOCKDRAFTER_H */
