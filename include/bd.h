/*
 * bd.h -- C ABI of the block-diffusion denoise-step library (libbd.so).
 *
 * One denoise step of block-wise masked-diffusion decoding, as described in
 * "MinerU-Diffusion: Rethinking Document OCR as Inverse Rendering via
 * Diffusion Decoding" (paper.rainbus.top summary), method steps 2-4:
 *   the output is split into blocks of L' tokens decoded in order; in every
 *   denoise step the current block attends bidirectionally to itself and
 *   causally to every earlier block and the visual/prompt prefix (kept in a
 *   KV cache, novelty paragraph: "KV-cache reuse"), never to later blocks;
 *   each still-masked position whose prediction confidence reaches the
 *   threshold T (0.95) is confirmed, the others are denoised again.
 *
 * Conventions shared by every call:
 *   - All pointers to tensors are DEVICE pointers unless stated otherwise.
 *     The caller owns every buffer, workspace and stream; the library never
 *     allocates, frees or synchronises.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream).  Host-side argument checks run first;
 *     on failure the call returns a non-OK status and launches nothing.
 *   - Kernels that meet a bad value in device memory (a page id outside the
 *     pool, a context longer than the page table covers, a token id outside
 *     the vocabulary) skip the offending access and write BD_ERR_DEVICE_CHECK
 *     into *dev_status (first error wins; 0 means OK).  dev_status is a
 *     device int32 the caller zeroes and reads when it chooses.  No device
 *     code traps or asserts.
 *   - Element types: BD_F32 (float) or BD_BF16 (bfloat16, accumulation in
 *     fp32).  All tensors of one call share the dtype.
 *   - Token state: int32, BD_MASK (-1) marks a still-masked position
 *     ("yellow" in the pages' Fig. 1); any other value is a confirmed token.
 */
#ifndef BD_H
#define BD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BD_MASK (-1)
#define BD_PAGE_SIZE 64

typedef enum {
  BD_OK = 0,
  BD_ERR_INVALID_ARG = 1,  /* host-side check failed, nothing launched      */
  BD_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head_dim)     */
  BD_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed          */
  BD_ERR_DEVICE_CHECK = 4, /* device-side bounds check (via *dev_status)    */
  BD_ERR_TIMEOUT = 5,      /* a bounded device wait gave up (via dev_status)*/
  BD_ERR_WORKSPACE = 6     /* workspace pointer/size too small or misaligned*/
} bd_status;

typedef enum { BD_F32 = 0, BD_BF16 = 1 } bd_dtype;

/*
 * Paged KV cache of ONE attention layer.
 *   k_pool, v_pool: [num_pages][num_kv_heads][page_size][head_dim], dtype.
 *   page_table:     [batch][max_pages_per_seq] int32 physical page ids; token
 *                   position p of sequence b lives in page
 *                   page_table[b][p / page_size], slot p % page_size.
 * page_size must be BD_PAGE_SIZE.  The pool base pointers must be 16-byte
 * aligned.  The struct itself is read on the host only (it may live on the
 * caller's stack).
 */
typedef struct {
  bd_dtype dtype;
  int32_t num_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t max_pages_per_seq;
  void *k_pool;
  void *v_pool;
  const int32_t *page_table;
} bd_paged_kv;

/* ------------------------------------------------------------------------
 * bd_block_attention -- block attention of the current block (method step 3,
 * "block-attention diffusion decoding"; also the training figure's mask in
 * "MinerU-Diffusion reads documents with diffusion decoding instead of left
 * to right", section "The idea").
 *
 * For sequence b, query position i < block_len and query head h (KV head
 * g = h / (num_q_heads / num_kv_heads)):
 *   keys   = cache tokens [0, ctx_len[b]) of head g   (prefix + earlier blocks)
 *            followed by the block's own block_len keys k_blk[b, :, g]
 *   out[b,i,h] = softmax_j(softmax_scale * q[b,i,h] . key_j) @ value_j
 * Every block position attends to every block position (masked or not); no
 * later block exists at decode time, so no further mask applies.
 *
 *   ctx_len   [batch] int32, device: cached tokens per sequence (<= max_ctx and
 *             <= max_pages_per_seq * page_size, checked on the device).  Pool
 *             rows past a sequence's context (the rest of its last page) may
 *             hold anything, NaN included: they never reach the output.
 *   tokens    [batch][block_len] int32 or NULL.  When given, a sequence with
 *             no BD_MASK position is skipped (its out rows are not written).
 *   q         [batch][block_len][num_q_heads][head_dim]
 *   k_blk,v_blk [batch][block_len][num_kv_heads][head_dim]
 *   out       [batch][block_len][num_q_heads][head_dim], dtype
 *   max_ctx   host-side upper bound on ctx_len (sizes the KV split).
 *   ws        device workspace of at least bd_block_attention_workspace() bytes,
 *             256-byte aligned; its contents need no initialisation.  Calls
 *             that share a workspace must be ordered on the GPU (one stream).
 * Limits: head_dim 64 or 128; block_len 1..32; num_q_heads % num_kv_heads == 0;
 *         block_len * (num_q_heads / num_kv_heads) <= 128.
 * ------------------------------------------------------------------------ */
size_t bd_block_attention_workspace(int32_t batch, int32_t block_len, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t max_ctx);

bd_status bd_block_attention(const bd_paged_kv *kv, const int32_t *ctx_len,
                             const int32_t *tokens, int32_t batch, int32_t block_len,
                             int32_t num_q_heads, int32_t max_ctx, const void *q,
                             const void *k_blk, const void *v_blk, float softmax_scale,
                             void *out, void *ws, size_t ws_bytes, int32_t *dev_status,
                             void *stream);

/* ------------------------------------------------------------------------
 * bd_confidence_commit -- vocabulary projection, confidence and threshold
 * commit for one denoise step (method steps 4 and 6).
 *
 * For every still-masked position (b, i) (tokens[b][i] == BD_MASK):
 *   logits_v  = hidden_states[b,i,:] . lm_head[v,:]      (v < vocab)
 *   p_max     = max_v softmax(logits)_v = 1 / sum_v exp(logits_v - max logits)
 *   argmax    = lowest v attaining max logits
 * Full logits never leave the chip.  Then, per sequence b:
 *   S = { masked i : p_max[b,i] >= threshold }; if S is empty and a position is
 *   masked, S = { the masked i with the largest p_max, lowest i on ties };
 *   tokens[b,i] = argmax[b,i] for i in S.  Confirmed tokens are never changed.
 *
 *   hidden_states [batch][block_len][hidden], lm_head [vocab][hidden], dtype.
 *   tokens     [batch][block_len] int32, in/out.
 *   p_max      [batch][block_len] float out (-1 at positions not masked on entry)
 *   argmax     [batch][block_len] int32 out (-1 likewise)
 *   n_committed[batch] int32 out: positions confirmed in this step
 *   n_masked   [batch] int32 out: positions still masked after this step
 *   ws         device workspace of at least bd_confidence_commit_workspace()
 *              bytes, 256-byte aligned; no initialisation needed.
 * Limits: block_len 1..32; hidden % 64 == 0 (bf16) or % 16 == 0 (f32);
 *         1 <= vocab < 2^31; threshold not NaN.
 * ------------------------------------------------------------------------ */
size_t bd_confidence_commit_workspace(bd_dtype dtype, int32_t batch, int32_t block_len,
                                      int32_t hidden, int32_t vocab);

bd_status bd_confidence_commit(bd_dtype dtype, int32_t batch, int32_t block_len,
                               int32_t hidden, int32_t vocab, const void *hidden_states,
                               const void *lm_head, float threshold, int32_t *tokens,
                               float *p_max, int32_t *argmax, int32_t *n_committed,
                               int32_t *n_masked, void *ws, size_t ws_bytes,
                               int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * bd_confidence_commit_regions -- bd_confidence_commit with one threshold per
 * block position.  The pages suggest, as future work, thresholds that adapt
 * to the region of the page being decoded (text, table, formula); here a
 * region is any set of positions the caller gives the same value.
 *
 *   thresholds [batch][block_len] float, DEVICE pointer, 4-byte aligned, read
 *              in stream order: position (b, i) qualifies when masked and
 *              p_max[b,i] >= thresholds[b,i] (a NaN entry never qualifies);
 *              if no masked position of b qualifies, the single most
 *              confident one is committed, as in bd_confidence_commit.
 *   all other arguments, results, workspace (bd_confidence_commit_workspace)
 *   and limits as bd_confidence_commit; thresholds NULL or misaligned:
 *   BD_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------ */
bd_status bd_confidence_commit_regions(bd_dtype dtype, int32_t batch, int32_t block_len,
                                       int32_t hidden, int32_t vocab, const void *hidden_states,
                                       const void *lm_head, const float *thresholds,
                                       int32_t *tokens, float *p_max, int32_t *argmax,
                                       int32_t *n_committed, int32_t *n_masked, void *ws,
                                       size_t ws_bytes, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * bd_confidence_commit_noalloc -- bd_confidence_commit without a caller
 * workspace.  The paper has no counterpart to this call: it exists for
 * callers that cannot allocate device memory when they run a step (serving
 * runtimes that forbid allocation while a request is in flight, plugins with
 * no access to their host's allocator, embedded callers whose device memory
 * is all handed out at start-up).
 *
 * Same arguments, results and limits as bd_confidence_commit, minus ws and
 * ws_bytes.  The scratch space comes from one 8 MiB array in device memory
 * that the library reserves on every GPU that loads it, for the life of the
 * process.  Shapes whose bd_confidence_commit_workspace() exceeds 8 MiB are
 * rejected with BD_ERR_WORKSPACE before any launch (at hidden 2048 and vocab
 * 151936 on a 152-SM GPU this allows batch * block_len up to about 1400).
 * The first call on a device looks up the array's address while that device
 * is current; make that first call before any stream capture starts.  The
 * address is cached per device, so every call must run in that device's
 * primary context (the runtime API's), and the process must not call
 * cudaDeviceReset after the first call.  All
 * calls on a device share the array and leave its contents behind: nothing in
 * it needs to start at zero, but calls whose executions overlap on the GPU
 * (unordered streams) race on it.  It allocates and frees nothing.
 * ------------------------------------------------------------------------ */
bd_status bd_confidence_commit_noalloc(bd_dtype dtype, int32_t batch, int32_t block_len,
                                       int32_t hidden, int32_t vocab, const void *hidden_states,
                                       const void *lm_head, float threshold, int32_t *tokens,
                                       float *p_max, int32_t *argmax, int32_t *n_committed,
                                       int32_t *n_masked, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * bd_sample_commit -- bd_confidence_commit under the sampling reading of the
 * inference settings (method step 6 lists top-k 0, temperature 1.0, top-p
 * 1.0; read as sampling, each masked position draws its token from
 * softmax(logits / temperature) with no top-k or nucleus truncation).
 *
 * For every still-masked position (b, i), with pos = b * block_len + i:
 *   z_v      = (hidden_states[b,i,:] . lm_head[v,:]) / temperature
 *   U_v      = (f + 1/2) / 2^23, f = a 23-bit field of word ((pos / 2) % 4)
 *              of Philox-4x64-10 (Salmon et al., SC'11) at counter
 *              (v, pos / 8, n, 0) under key (seed, 0): bits 63..41 of the
 *              word for even pos, bits 31..9 for odd pos
 *   sampled  = lowest v attaining max_v (z_v - ln(-ln U_v))   (Gumbel-max)
 *   p_sel    = softmax(z)[sampled]
 * then the commit rule of bd_confidence_commit with p_sel as the confidence
 * and sampled as the token.
 *
 *   offset     DEVICE pointer to a uint64 draw counter n (8-byte aligned),
 *              owned by the caller.  The call draws with the value it finds
 *              there (in stream order) and adds 1 to it, so consecutive
 *              steps on a stream, including replays of a captured CUDA
 *              graph, draw fresh noise.  Equal (seed, n, inputs) give equal
 *              results.
 *   p_sel      [batch][block_len] float out (-1 at positions not masked on entry)
 *   sampled    [batch][block_len] int32 out (-1 likewise)
 *   other arguments, workspace rules and limits as bd_confidence_commit, with
 *   bd_sample_commit_workspace() in place of its workspace query;
 *   1e-6 <= temperature <= 1e6 and offset non-NULL, else BD_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------ */
size_t bd_sample_commit_workspace(bd_dtype dtype, int32_t batch, int32_t block_len,
                                  int32_t hidden, int32_t vocab);

bd_status bd_sample_commit(bd_dtype dtype, int32_t batch, int32_t block_len, int32_t hidden,
                           int32_t vocab, const void *hidden_states, const void *lm_head,
                           float threshold, float temperature, uint64_t seed, uint64_t *offset,
                           int32_t *tokens, float *p_sel, int32_t *sampled,
                           int32_t *n_committed, int32_t *n_masked, void *ws, size_t ws_bytes,
                           int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * bd_sample_commit_truncated -- bd_sample_commit with the other two settings
 * of method step 6 switched on: top-k and top-p (nucleus) truncation, applied
 * in that order to z = logits / temperature.
 *
 * Per masked position (b, i), pos = b * block_len + i:
 *   theta_k  = the top_k-th largest z_v            (top_k > 0 and < vocab)
 *   theta_p  = over the entries with z >= theta_k, sorted by z descending with
 *              masses exp(z - max z): the z of the first entry at which the
 *              running mass reaches top_p * (their total mass)  (top_p < 1)
 *   kept     = { v : z_v >= max(theta_k, theta_p) }  (boundary ties kept)
 *   sampled  = lowest v in kept attaining max (z_v - ln(-ln U_v)), U_v as in
 *              bd_sample_commit (same counter, key and draw counter)
 *   p_sel    = exp(z_sampled) / sum_{v in kept} exp(z_v)
 * then the commit rule with p_sel as the confidence.  The boundary search is
 * exact in the GPU's fp32 z; the masses it accumulates are exp(z - max z)
 * rounded down to multiples of 2^-40.
 *
 *   top_k      >= 0; 0 (or >= vocab) disables it.
 *   top_p      in (0, 1]; 1 disables it.  With both disabled this is
 *              bd_sample_commit.
 *   ws         at least bd_sample_commit_truncated_workspace() bytes: the
 *              truncation needs each masked row's full distribution, so the
 *              fp32 logits of the masked rows (batch * block_len * vocab * 4
 *              bytes) pass through the workspace.
 *   other arguments, results and limits as bd_sample_commit; top_k < 0 or
 *   top_p outside (0, 1] (or NaN): BD_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------ */
size_t bd_sample_commit_truncated_workspace(bd_dtype dtype, int32_t batch, int32_t block_len,
                                            int32_t hidden, int32_t vocab);

bd_status bd_sample_commit_truncated(bd_dtype dtype, int32_t batch, int32_t block_len,
                                     int32_t hidden, int32_t vocab, const void *hidden_states,
                                     const void *lm_head, float threshold, float temperature,
                                     int32_t top_k, float top_p, uint64_t seed,
                                     uint64_t *offset, int32_t *tokens, float *p_sel,
                                     int32_t *sampled, int32_t *n_committed, int32_t *n_masked,
                                     void *ws, size_t ws_bytes, int32_t *dev_status,
                                     void *stream);

/* ------------------------------------------------------------------------
 * bd_append_block_kv -- append a finished block's K/V to the paged cache
 * (novelty paragraph: block-causal structure lets earlier blocks' K/V be
 * reused).  For every sequence b with n_masked[b] == 0 (NULL = all):
 *   cache position ctx_len[b] + i  <-  k_blk[b, i], v_blk[b, i]  (i < block_len)
 *   ctx_len[b] += block_len
 * Call it once per finished block.  The block may straddle two pages.
 *   k_blk, v_blk [batch][block_len][num_kv_heads][head_dim], dtype.
 *   ctx_len [batch] int32 device, in/out.
 * ------------------------------------------------------------------------ */
bd_status bd_append_block_kv(const bd_paged_kv *kv, int32_t batch, int32_t block_len,
                             const void *k_blk, const void *v_blk, int32_t *ctx_len,
                             const int32_t *n_masked, int32_t *dev_status, void *stream);

/* ========================================================================
 * Decoder layer stack (the long-context workload's 28-layer decoder).
 *
 * "Rethinking Document OCR as Inverse Rendering via Diffusion Decoding"
 * (paper.rainbus.top summary), reproduction paragraph: the diffusion decoder
 * is initialised from SDAR-1.7B-Chat-b32 (hidden 2048, 16 query / 8 KV heads
 * of 128).  The pages give no layer internals; these calls compute the
 * plainest reading, one layer being
 *   xn = bf16(x / sqrt(mean(x^2) + eps))      (RMSNorm, no gain)
 *   [q | k | v] = bf16(xn Wqkv^T)             (bd_qkv_projection)
 *   a = bf16(block attention)                 (bd_block_attention)
 *   x = x + a Wo^T; next xn                   (bd_out_projection_residual)
 * with no MLP.  x (the residual stream) is fp32 [rows][hidden]; every other
 * activation is bf16.  rows = batch * block_len, row r = b * block_len + i.
 * Weights are bf16, row-major [out_features][in_features].  These calls need
 * a GPU with tcgen05 (sm_100 family) and return BD_ERR_UNSUPPORTED elsewhere.
 * ======================================================================== */

/* bd_embed_rmsnorm -- decoder input: x[r] = E[tokens[r]] for a confirmed
 * position, mask_embed for tokens[r] == BD_MASK; xn[r] = RMSNorm(x[r]).
 *   tokens [rows] int32; embed [vocab][hidden] bf16; mask_embed [hidden] bf16;
 *   x [rows][hidden] float out; xn [rows][hidden] bf16 out.
 * A token outside [0, vocab) sets BD_ERR_DEVICE_CHECK and uses mask_embed.
 * Limits: hidden % 4 == 0, hidden <= 4096; pointers 16-byte aligned. */
bd_status bd_embed_rmsnorm(int32_t rows, int32_t hidden, int32_t vocab, const int32_t *tokens,
                           const void *embed, const void *mask_embed, float eps, float *x,
                           void *xn, int32_t *dev_status, void *stream);

/* bd_qkv_projection -- [q | k | v] = bf16(xn Wqkv^T).
 *   xn [rows][hidden] bf16; w_qkv [(Hq + 2 Hkv) D][hidden] bf16 (rows: the
 *   query heads, then the key heads, then the value heads);
 *   q [rows][Hq][D], k and v [rows][Hkv][D] bf16 out.
 *   ws: at least bd_qkv_projection_workspace() bytes, 256-byte aligned.
 * Limits: hidden % 64 == 0; (Hq + 2 Hkv) D % 128 == 0. */
size_t bd_qkv_projection_workspace(int32_t rows, int32_t hidden, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim);
bd_status bd_qkv_projection(int32_t rows, int32_t hidden, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, const void *xn,
                            const void *w_qkv, void *q, void *k, void *v, void *ws,
                            size_t ws_bytes, int32_t *dev_status, void *stream);

/* bd_out_projection_residual -- x += attn Wo^T, then xn = RMSNorm(x) (the
 * next layer's input).
 *   attn [rows][in_features] bf16; w_o [hidden][in_features] bf16;
 *   x [rows][hidden] float in/out; xn [rows][hidden] bf16 out.
 *   ws: at least bd_out_projection_workspace() bytes, 256-byte aligned.
 * Limits: in_features % 64 == 0; hidden % 128 == 0, hidden <= 4096. */
size_t bd_out_projection_workspace(int32_t rows, int32_t in_features, int32_t hidden);
bd_status bd_out_projection_residual(int32_t rows, int32_t in_features, int32_t hidden,
                                     const void *attn, const void *w_o, float eps, float *x,
                                     void *xn, void *ws, size_t ws_bytes, int32_t *dev_status,
                                     void *stream);

/* bd_mlp_residual -- optional gated MLP of a decoder layer, after the
 * attention residual.  The pages give no layer internals; the decoder starts
 * from SDAR-1.7B-Chat (reproduction paragraph), a Qwen3-family model, whose
 * MLP is SwiGLU:
 *   [g | u] = xn w_gate_up^T     (xn = bf16(RMSNorm(x)), as
 *                                 bd_out_projection_residual leaves it)
 *   a       = bf16(silu(g) * u), silu(g) = g / (1 + exp(-g))
 *   x      += a w_down^T         (fp32), then xn_out = bf16(RMSNorm(x))
 *   xn [rows][hidden] bf16 in; xn_out [rows][hidden] bf16 out (may be xn);
 *   w_gate_up [2 inter][hidden] bf16, gate rows first; w_down [hidden][inter]
 *   bf16; x [rows][hidden] float in/out.
 *   ws: at least bd_mlp_workspace() bytes, 256-byte aligned.
 * Limits: inter % 64 == 0, 64 <= inter <= 32768; hidden % 128 == 0,
 *         hidden <= 4096; pointers 16-byte aligned. */
size_t bd_mlp_workspace(int32_t rows, int32_t hidden, int32_t inter);
bd_status bd_mlp_residual(int32_t rows, int32_t hidden, int32_t inter, const void *xn,
                          const void *w_gate_up, const void *w_down, float eps, float *x,
                          void *xn_out, void *ws, size_t ws_bytes, int32_t *dev_status,
                          void *stream);

/* bd_append_block_kv_layers -- bd_append_block_kv for num_layers layers that
 * share one page table and one ctx_len (kv: host array of num_layers structs
 * with equal dtype, geometry and page_table; only the pools differ).
 *   k_blk, v_blk [num_layers][batch][block_len][num_kv_heads][head_dim].
 * Every done sequence's block goes to positions ctx_len[b] .. + block_len - 1
 * of every layer, then ctx_len[b] += block_len once.  num_layers <= 64. */
bd_status bd_append_block_kv_layers(const bd_paged_kv *kv, int32_t num_layers, int32_t batch,
                                    int32_t block_len, const void *k_blk, const void *v_blk,
                                    int32_t *ctx_len, const int32_t *n_masked,
                                    int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Splitting one sequence across GPUs (the path otherwise shards by sequence
 * with no exchange).  Each split needs one exchange, done by the caller with
 * its collective library; these calls produce what is exchanged and combine
 * what was gathered (method steps 3-4: the block's attention and each masked
 * position's confidence are the quantities split).
 *
 * bd_conf_record: the online-softmax state of one position over a slice of
 * the vocabulary: m = max logit, s = sum of exp(l - m) over the slice, idx =
 * lowest vocabulary id (whole-vocabulary numbering) attaining m.  A position
 * that is not masked holds m = -inf, s = 0, idx = INT32_MAX.  12 bytes.
 * ------------------------------------------------------------------------ */
typedef struct {
  float m;
  float s;
  int32_t idx;
} bd_conf_record;

/* Vocabulary-parallel LM head: this GPU's slice lm_head_shard = rows
 * [vocab_offset, vocab_offset + vocab_shard) of W ([vocab_shard][hidden],
 * bf16).  For every position of tokens (BD_MASK = masked) writes
 * records[b * block_len + i] over the slice; no logit reaches memory and
 * nothing is committed.  Workspace from bd_confidence_shard_workspace()
 * (256-byte aligned).  bf16 only. */
size_t bd_confidence_shard_workspace(bd_dtype dtype, int32_t batch, int32_t block_len,
                                     int32_t hidden, int32_t vocab_shard);
bd_status bd_confidence_shard(bd_dtype dtype, int32_t batch, int32_t block_len, int32_t hidden,
                              int32_t vocab_shard, int32_t vocab_offset,
                              const void *hidden_states, const void *lm_head_shard,
                              const int32_t *tokens, bd_conf_record *records, void *ws,
                              size_t ws_bytes, int32_t *dev_status, void *stream);

/* The commit of bd_confidence_commit from gathered records: records is
 * DEVICE memory [num_shards][batch * block_len] (the concatenation of every
 * slice's records, in any shard order); vocab is the whole vocabulary size.
 * Merges each position's states (p_max = 1 / s, argmax = idx) and applies the
 * commit rule; outputs as bd_confidence_commit. */
bd_status bd_commit_shards(int32_t batch, int32_t block_len, int32_t vocab, int32_t num_shards,
                           const bd_conf_record *records, float threshold, int32_t *tokens,
                           float *p_max, int32_t *argmax, int32_t *n_committed,
                           int32_t *n_masked, int32_t *dev_status, void *stream);

/* Host-side merge of gathered records (HOST memory [num_shards][n] -> [n]),
 * the same rule as the device merge.  No CUDA call. */
bd_status bd_merge_conf_records_host(int32_t num_shards, int64_t n,
                                     const bd_conf_record *records, bd_conf_record *out);

/* KV-split attention: merge per-row partials of num_shards key slices,
 * m and l [num_shards][rows] (max in natural-log units, sum of exp(s - m)),
 * o [num_shards][rows][head_dim] unnormalised: out[r] = sum_s e^(m_s - M)
 * o_s[r] / sum_s e^(m_s - M) l_s[r].  A slice with no key of a row holds
 * m = -inf, l = 0.  The host version takes HOST pointers and calls no CUDA
 * function; the device version takes DEVICE pointers and writes out
 * [rows][head_dim] as fp32 or bf16 (head_dim <= 256), async on stream. */
bd_status bd_merge_attention_partials_host(int32_t num_shards, int64_t rows, int32_t head_dim,
                                           const float *m, const float *l, const float *o,
                                           float *out);
bd_status bd_merge_attention_partials(int32_t num_shards, int64_t rows, int32_t head_dim,
                                      const float *m, const float *l, const float *o,
                                      bd_dtype out_dtype, void *out, void *stream);

/* Human-readable name of a status code (static string, never NULL). */
const char *bd_status_string(bd_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t bd_version(void);

/* Diagnostic: number of kernels this process has launched through the
 * library so far (all devices, all threads).  Reading it never synchronises. */
uint64_t bd_kernel_launches(void);

/* ------------------------------------------------------------------------
 * bd_debug_force_attention_kernel -- TEST HOOK, not part of the method.
 * bd_block_attention picks its kernel from the call's shape and dtype alone
 * (BD_ATTN_AUTO, the default).  A test that wants to check each kernel on the
 * same inputs forces one of them for every later bd_block_attention call in
 * this process; a kernel that cannot serve a shape falls back to the one the
 * shape would pick.  Returns BD_ERR_INVALID_ARG for an unknown value.
 * Process-wide and not synchronised with calls in flight: set it only
 * between calls, and set BD_ATTN_AUTO again afterwards.
 * ------------------------------------------------------------------------ */
typedef enum {
  BD_ATTN_AUTO = 0,      /* by shape                                        */
  BD_ATTN_PAIR = 1,      /* tcgen05 head-pair kernel, also on small problems */
  BD_ATTN_MMA = 2,       /* mma.sync kernel (bf16), tile ranges or splits   */
  BD_ATTN_SIMT = 3,      /* SIMT kernel                                     */
  BD_ATTN_CLUSTER = 4,   /* mma.sync kernel, one cluster per segment (bf16), *
                          * also on large problems                          */
  BD_ATTN_PAIR_CLUSTER = 5 /* tcgen05 head-pair kernel, one cluster per head  *
                            * pair, also on large problems                   */
} bd_attention_kernel;

bd_status bd_debug_force_attention_kernel(int32_t which);

/* ------------------------------------------------------------------------
 * bd_debug_wait_timeout_selftest -- TEST HOOK, not part of the method.
 * Every device-side wait of the library (mbarrier waits of the tcgen05/TMA
 * kernels) gives up after one second of wall time; the kernel then writes
 * BD_ERR_TIMEOUT into *dev_status, stops issuing work, frees its tensor
 * memory and returns, leaving the context usable.  This call launches one
 * CTA that takes exactly that path: it allocates tensor memory, waits on a
 * barrier nothing arrives at, and unwinds.  After about one second the
 * caller's *dev_status holds BD_ERR_TIMEOUT (if it held 0 before).  No copy
 * or MMA is in flight at the wait.  Asynchronous on `stream`.
 * ------------------------------------------------------------------------ */
bd_status bd_debug_wait_timeout_selftest(int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BD_H */
