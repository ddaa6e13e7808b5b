/*
 * ds4a.h -- C ABI of the compressed sparse multi-query attention path of
 * DeepSeek-V4-Flash, as the "DS4 (DwarfStar 4)" page describes it, built as
 * hand-written CUDA kernels for GB300 (sm_103a).
 *
 * The path ("DS4 (DwarfStar 4)", Key Techniques, "KV attention compression";
 * Architecture, fixed model shape):
 *   - layers 0-1 attend the raw 128-token sliding window only;
 *   - even layers from 2 pool every 4 tokens into one compressed row and keep
 *     the 512 compressed rows a learned indexer ranks highest;
 *   - odd layers pool every 128 tokens and attend every compressed row;
 *   - attention is multi-query (64 query heads share one KV head) and runs as
 *     one softmax over the union of the raw window and the compressed rows.
 * The compressor keeps a rolling score/KV state and appends a pooled row each
 * time a block of `ratio` tokens completes; prefill runs it over a whole chunk
 * (2048 tokens by default, Architecture, "Whole-model graph execution"),
 * decode one token at a time.
 *
 * Conventions for every call:
 *   - fp16 arrays are IEEE binary16 bit patterns (uint16_t), row-major, rows
 *     of `head_dim` (or `d_idx`) elements, base 16-byte aligned.  float and
 *     int32 arrays are 4-byte aligned.
 *   - Every array pointer is a DEVICE pointer owned by the caller.  The
 *     library allocates, frees and synchronises nothing (except
 *     ds4a_last_device_error, which synchronises the given stream, and
 *     ds4a_decode_layer_step, which takes host inputs and waits for its output).
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.  Work is enqueued on it and returns before it runs.
 *   - Positions are absolute token indices, 0-based.  The compressed row j
 *     pools tokens j*ratio .. j*ratio+ratio-1 and becomes visible to the query
 *     at position p once its block is complete: (j+1)*ratio <= p+1.
 *   - Return value: DS4A_OK, or an error code below.  On an argument error
 *     nothing is enqueued.  Errors found by a kernel while it runs (a gathered
 *     row index out of range, a bounded wait that gave up) do not fail the
 *     call; the kernel skips the access and records the first such error in
 *     a per-device error word read by ds4a_last_device_error.
 *   - Launch order: kernels are launched with programmatic dependent launch.
 *     A kernel may start once the kernel ahead of it on the stream has started
 *     its own dependent phase, reads a few named inputs early (each call lists
 *     them: cache state such as key rows and window rows, and its queries), and
 *     waits for the kernel ahead to finish before it reads anything else or
 *     writes anything.  So the kernel directly ahead on the stream must not
 *     write those early inputs.  The calls of this library never write another
 *     call's early inputs; a kernel that does not use programmatic launch
 *     finishes before the next call starts.  With the environment variable
 *     DS4A_PDL=0 (read once per process) every kernel waits for the kernel
 *     ahead before it starts.
 */
#ifndef DS4A_H
#define DS4A_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DS4A_OK               0
#define DS4A_ERR_ARG          1  /* null or misaligned pointer, bad size */
#define DS4A_ERR_CAPACITY     2  /* output rows exceed the caller's capacity */
#define DS4A_ERR_UNSUPPORTED  3  /* head_dim / heads / sizes not compiled */
#define DS4A_ERR_CUDA         4  /* a CUDA launch or runtime call failed */
#define DS4A_ERR_TIMEOUT      5  /* a bounded device wait gave up */
#define DS4A_ERR_WORKSPACE    6  /* workspace missing or too small */
#define DS4A_ERR_DEVICE_INDEX 7  /* a kernel met a row index out of range */

/* Human-readable name of a status code (static string). */
const char *ds4a_status_str(int status);

/* Synchronises `stream`, then returns and clears the first error recorded by a
 * kernel on the current device since the last call (DS4A_OK if none). */
int ds4a_last_device_error(void *stream);

/*
 * ds4a_test_set_wait_limit -- TEST HOOK, not part of the attention path; the
 * pages have no counterpart.  With limit_ns > 0, every decode attention launch
 * enqueued afterwards by this process (ds4a_attn_decode,
 * ds4a_compress_attn_decode) makes CTA 0 of its cluster, once every partial sent
 * to it has arrived, also wait on a barrier that nothing completes.  That wait
 * gives up after limit_ns, records DS4A_ERR_TIMEOUT in the device error word and
 * the launch finishes with its normal output, so a test can drive the bounded
 * wait's give-up path without any fault.  0 (the default) turns it off.
 * Returns DS4A_ERR_ARG for a limit outside 0 .. 10 s.
 */
int ds4a_test_set_wait_limit(long long limit_ns);

/*
 * ds4a_compress_append -- feed n_new tokens to the KV compressor of one layer.
 * ("DS4 (DwarfStar 4)", Key Techniques, "KV attention compression": rolling
 * score/KV state, pooled rows appended at ratio boundaries.)
 *
 * The pooled row of block b is sum_t a_t k_t and sum_t a_t v_t over the block's
 * tokens, with a = softmax over the block of the score s_t = score_w . k_t
 * (the same weights for K and V).  Decode (n_new = 1) updates the open block's
 * running state online; a longer chunk pools its complete blocks directly.
 *
 *   k, v       [n_new, head_dim] fp16: tokens at positions pos .. pos+n_new-1.
 *   head_dim   multiple of 8, 8 .. 256.
 *   score_w    [head_dim] float: the layer's learned score vector.
 *   ratio      tokens per pooled row, 1 .. 1024.
 *   pos        tokens this layer's compressor has already been fed.
 *   state      [2 + 2*head_dim] float, caller-owned, persistent per layer:
 *              (running max, running sum, weighted K sum, weighted V sum) of the
 *              open block.  Read when pos % ratio != 0, written when
 *              (pos + n_new) % ratio != 0; no reset is ever needed.
 *   comp_k, comp_v [cap, head_dim] fp16: the layer's compressed rows.  Rows
 *              floor(pos/ratio) .. floor((pos+n_new)/ratio)-1 are written.
 *   cap        rows allocated; DS4A_ERR_CAPACITY if the last row written
 *              would be >= cap.
 * n_new = 0 is a no-op.  Early reads: k and score_w.
 */
int ds4a_compress_append(const uint16_t *k, const uint16_t *v, int n_new, int head_dim,
                         const float *score_w, int ratio, long long pos, float *state,
                         uint16_t *comp_k, uint16_t *comp_v, long long cap, void *stream);

/*
 * ds4a_compress_append_keys -- ds4a_compress_append that also pools per-token
 * indexer keys: each compressed row's indexer key is the same softmax-weighted
 * sum over the block, sum_t a_t kidx_t, with a = softmax over the block of
 * score_w . k_t.  ("DS4 (DwarfStar 4)", Key Techniques, "KV attention
 * compression": the compressor keeps a rolling score/KV state and appends pooled
 * rows at ratio boundaries, and the ratio-4 layers rank those rows with a
 * learned indexer.  The pages do not say where an indexer key comes from; this
 * call is the reading in which the compressor pools it from per-token keys, the
 * alternative to ds4a_indexer_topk's caller-supplied key per row.)
 *
 *   Arguments as ds4a_compress_append, and:
 *   k_idx_tok  [n_new, d_idx] fp16: the indexer keys of tokens pos .. pos+n_new-1.
 *   d_idx      multiple of 8, 8 .. 256.
 *   state      [2 + 2*head_dim + d_idx] float: the state of ds4a_compress_append
 *              followed by the open block's weighted indexer-key sum.
 *   comp_kidx  [cap, d_idx] fp16: pooled indexer keys, row j beside comp_k's row j.
 * The pooled K and V rows are the same bits ds4a_compress_append writes.  An
 * ds4a_indexer_topk call may follow it directly on the stream: the indexer reads
 * the key rows this call can write only after the call has finished.
 */
int ds4a_compress_append_keys(const uint16_t *k, const uint16_t *v, const uint16_t *k_idx_tok, int n_new,
                              int head_dim, int d_idx, const float *score_w, int ratio, long long pos, float *state,
                              uint16_t *comp_k, uint16_t *comp_v, uint16_t *comp_kidx, long long cap, void *stream);

/*
 * ds4a_indexer_topk -- rank compressed rows for n_q queries and keep the top k.
 * ("DS4 (DwarfStar 4)", Key Techniques, "KV attention compression": a learned
 * indexer selects the top-512 compressed rows on ratio-4 layers.)
 *
 * Query i sits at position q_pos0 + i and sees rows
 * j < n_vis_i = min(n_rows, floor((q_pos0+i+1)/ratio)).  Its score for row j
 * is q_idx_i . k_idx_j, computed from the exact fp16 products and rounded once
 * to binary32; rows are ranked by that score, ties to the lower index.
 *
 *   q_idx      [n_q, d_idx] fp16 indexer queries.
 *   k_idx      [n_rows, d_idx] fp16, one indexer key per compressed row.
 *   d_idx      multiple of 8, 8 .. 256.
 *   k          rows kept per query, 1 .. 2048.
 *   out_idx    [n_q, k] int32: the kept rows in ascending order, then -1 for
 *              every slot past min(k, n_vis_i).
 *   out_n      [n_q] int32, or NULL: min(k, n_vis_i).
 *   ws         workspace of ds4a_indexer_workspace_bytes(n_q, n_rows, k) bytes,
 *              zero-filled by the caller once before its first use (the call
 *              leaves its counters at zero again).  Calls that share one
 *              workspace must be stream-ordered.
 * Early reads (see "Launch order" above): the queries and the key rows
 * j < floor(q_pos0 / ratio), the rows complete before the first query's token.
 * Key rows from floor(q_pos0 / ratio) on, which a compressor call for the same
 * tokens may write (ds4a_compress_append_keys), are read only after the kernel
 * ahead has finished.
 */
int ds4a_indexer_topk(const uint16_t *q_idx, int n_q, const uint16_t *k_idx, long long n_rows,
                      int d_idx, long long q_pos0, int ratio, int k, int32_t *out_idx,
                      int32_t *out_n, void *ws, size_t ws_bytes, void *stream);

size_t ds4a_indexer_workspace_bytes(int n_q, long long n_rows, int k);

/*
 * ds4a_indexer_topk_compress -- one decode step's indexer query and the
 * compressor update for the step's token, in a single kernel launch.
 * ("DS4 (DwarfStar 4)", Key Techniques, "KV attention compression": both are
 * per-token steps of a ratio-4 layer; the indexer reads the caller's indexer
 * keys, the compressor reads the new token, and neither reads what the other
 * writes.)
 *
 * Same results as ds4a_indexer_topk(q_idx, 1, k_idx, n_rows, d_idx, q_pos,
 * ratio, k, out_idx, out_n, ws, ws_bytes, stream) followed by
 * ds4a_compress_append(k_new, v_new, 1, head_dim, score_w, ratio, q_pos, state,
 * comp_k, comp_v, cap, stream): the same kernels' arithmetic, bit for bit.  One
 * launch instead of two takes a kernel boundary off a decode step's chain.
 *
 *   Indexer arguments as ds4a_indexer_topk with n_q = 1 and q_pos0 = q_pos.
 *   Compressor arguments as ds4a_compress_append with n_new = 1 and pos = q_pos
 *   (k_new, v_new: [1, head_dim] fp16, the token at position q_pos).
 *   Errors: the union of the two calls' checks; nothing is enqueued on error.
 *   Early reads: the union of the two calls' early reads.
 *   L2 prefetch: with at most 8192 visible rows, the launch also asks L2 for the
 *   comp_k / comp_v rows (below the visible count, hence inside the cap rows
 *   passed) that its query most likely keeps, before its dependency wait, so
 *   that the attention call which gathers them next finds them there.  A
 *   prefetch returns no data: it reads nothing the results depend on.
 */
int ds4a_indexer_topk_compress(const uint16_t *q_idx, const uint16_t *k_idx, long long n_rows, int d_idx,
                               long long q_pos, int ratio, int k, int32_t *out_idx, int32_t *out_n, void *ws,
                               size_t ws_bytes, const uint16_t *k_new, const uint16_t *v_new, int head_dim,
                               const float *score_w, float *state, uint16_t *comp_k, uint16_t *comp_v,
                               long long cap, void *stream);

/*
 * ds4a_indexer_topk_noalloc -- ds4a_indexer_topk for one query (n_q = 1) with no
 * workspace argument and no allocation.  The pages have no counterpart: this is
 * a convenience of this library.
 *
 * For callers that cannot allocate device memory at the point of the call --
 * plugin or callback hosts whose enqueue step may not allocate (allocation
 * there can synchronise the device, or the host forbids it) and programs that
 * run inside a fixed, pre-reserved memory budget.  The scratch lives in a
 * statically sized device array inside the library (256 KiB + 256 bytes), held
 * by every GPU that loads the library until the process exits.
 *
 *   Arguments as ds4a_indexer_topk with n_q = 1 and q_pos0 = q_pos.
 *   The limit counts the rows the query sees, min(n_rows, floor((q_pos+1)/ratio)):
 *   at most 65536; more returns DS4A_ERR_WORKSPACE and enqueues nothing.
 *   The first call on each device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   Each call enqueues the indexer kernel only: the array starts at zero and the
 *   kernel leaves its completion ticket at zero when it finishes.  All calls
 *   share the one array and it keeps the last call's contents: calls whose work
 *   overlaps on the GPU (different streams, or different host threads, without
 *   ordering between them) race and give wrong results.
 */
int ds4a_indexer_topk_noalloc(const uint16_t *q_idx, const uint16_t *k_idx, long long n_rows,
                              int d_idx, long long q_pos, int ratio, int k, int32_t *out_idx,
                              int32_t *out_n, void *stream);

/*
 * ds4a_indexer_topk_compress_keys -- one decode step's indexer query and the
 * compressor update for its token on a layer whose compressor pools per-token
 * indexer keys, in one launch.  Same results as ds4a_compress_append_keys(k_new,
 * v_new, k_idx_tok, 1, head_dim, d_idx, score_w, ratio, q_pos, state, comp_k, comp_v,
 * k_idx, cap, stream) followed by ds4a_indexer_topk(q_idx, 1, k_idx, n_rows, d_idx,
 * q_pos, ratio, k, out_idx, out_n, ws, ws_bytes, stream), bit for bit.  When the
 * token completes a row, the launch's compressor CTA writes the row (K, V and its
 * pooled indexer key into k_idx), scores that key against q_idx exactly as the
 * indexer scores a row, and joins the indexer's completion count, so the row is
 * ranked in the same launch.  ("DS4 (DwarfStar 4)", Key Techniques, "KV attention
 * compression": the learned indexer ranks the compressed rows.)
 *   Arguments as the two calls; k_idx is written (the pooled key rows).  Errors: the
 *   union of the two calls' checks; DS4A_ERR_CAPACITY when the row the token
 *   completes is >= min(cap, n_rows).  Nothing is enqueued on error.
 *   Early reads: q_idx, k_new, k_idx_tok, score_w and the rows j < floor(q_pos/ratio)
 *   of k_idx.
 */
int ds4a_indexer_topk_compress_keys(const uint16_t *q_idx, uint16_t *k_idx, long long n_rows, int d_idx,
                                    long long q_pos, int ratio, int k, int32_t *out_idx, int32_t *out_n, void *ws,
                                    size_t ws_bytes, const uint16_t *k_new, const uint16_t *v_new,
                                    const uint16_t *k_idx_tok, int head_dim, const float *score_w, float *state,
                                    uint16_t *comp_k, uint16_t *comp_v, long long cap, void *stream);

/*
 * ds4a_attn_decode -- one decode query: multi-query attention over the raw
 * window and the selected (or all) compressed rows, as one softmax.
 * ("DS4 (DwarfStar 4)", Architecture: 64 heads, 1 KV head, 128-token window;
 * Key Techniques, "KV attention compression".)
 *
 * For each head h: out_h = sum_j softmax_j(scale * q_h . K_j) V_j, the union
 * of the n_win window rows and the compressed rows listed by sel.
 *
 *   q          [H, D] fp16; H multiple of 8, 8 .. 64; D = 64 or 128.
 *   win_k, win_v [n_win, D] fp16: the raw window rows, in any order
 *              (a ring buffer can be passed as it is); 1 <= n_win <= 4096.
 *   comp_k, comp_v [n_comp, D] fp16: the layer's compressed rows.
 *   sel        [n_sel] int32 device array of row indices into comp_k/comp_v
 *              (negative entries are skipped, entries >= n_comp are skipped
 *              and recorded as DS4A_ERR_DEVICE_INDEX), or NULL to attend rows
 *              0 .. n_sel-1 (then n_sel <= n_comp).  n_sel may be 0.
 *   scale      softmax scale, 1/sqrt(D) in the model.
 *   out        [H, D] fp16.
 *   ws, ws_bytes  unused by this kernel design (pass NULL, 0); reserved.
 * Early reads: q and up to 64 window rows.  Each CTA also asks L2, before the
 * dependency wait, for the window rows it gathers after it and, with sel NULL,
 * for its compressed rows (a prefetch returns no data).
 */
int ds4a_attn_decode(const uint16_t *q, int H, int D, const uint16_t *win_k,
                     const uint16_t *win_v, int n_win, const uint16_t *comp_k,
                     const uint16_t *comp_v, long long n_comp, const int32_t *sel, int n_sel,
                     float scale, uint16_t *out, void *ws, size_t ws_bytes, void *stream);

/*
 * ds4a_compress_attn_decode -- one decode step of a layer that attends every
 * compressed row (no indexer: the ratio-128 layers): the compressor update for
 * the step's token and the attention, in a single kernel launch.
 * ("DS4 (DwarfStar 4)", Key Techniques, "KV attention compression".)
 *
 * Same results as ds4a_compress_append(k_new, v_new, 1, D, score_w, ratio, pos,
 * state, comp_k, comp_v, cap, stream) followed by ds4a_attn_decode(q, H, D,
 * win_k, win_v, n_win, comp_k, comp_v, cap, NULL, floor((pos+1)/ratio), scale,
 * out, NULL, 0, stream), bit for bit.  When the token completes a block, its
 * pooled row is the last row attended and the one CTA that attends it writes
 * it first; otherwise the compressor's state is updated off the critical path.
 *
 *   Compressor arguments as ds4a_compress_append with n_new = 1 and head_dim = D
 *   (k_new, v_new: [1, D] fp16, the token at position pos).
 *   Attention arguments as ds4a_attn_decode; the window must hold the token at pos.
 *   Errors: the union of the two calls' checks; nothing is enqueued on error.
 *   Early reads: k_new, score_w, q and up to 64 window rows; L2 prefetches as
 *   ds4a_attn_decode with sel NULL.
 */
int ds4a_compress_attn_decode(const uint16_t *k_new, const uint16_t *v_new, const float *score_w, int ratio,
                              long long pos, float *state, uint16_t *comp_k, uint16_t *comp_v, long long cap,
                              const uint16_t *q, int H, int D, const uint16_t *win_k, const uint16_t *win_v,
                              int n_win, float scale, uint16_t *out, void *stream);

/*
 * ds4a_attn_prefill -- causal attention for a prefill chunk of T queries at
 * positions q_pos0 .. q_pos0+T-1.
 *
 * Query i at p = q_pos0+i attends, in one softmax, the raw rows of positions
 * max(0, p-window+1) .. p and: nothing more if ratio == 0; the rows of its sel
 * row if sel is given; otherwise every visible compressed row
 * j < min(n_comp, floor((p+1)/ratio)).
 *
 *   q          [T, H, D] fp16 (H, D as in ds4a_attn_decode).
 *   raw_k, raw_v [n_prior + T, D] fp16: positions q_pos0-n_prior .. q_pos0+T-1
 *              (the prefix's last n_prior tokens, then the chunk).  n_prior must
 *              be >= min(window-1, q_pos0).
 *   window     raw window length, 1 .. 4096.
 *   comp_k, comp_v [n_comp, D] fp16, may be NULL when ratio == 0.
 *   sel        [T, k_stride] int32 (as written by ds4a_indexer_topk), or NULL.
 *   out        [T, H, D] fp16.
 *   ws, ws_bytes  unused by this kernel design (pass NULL, 0); reserved.
 * Early reads: none.
 */
int ds4a_attn_prefill(const uint16_t *q, int T, int H, int D, const uint16_t *raw_k,
                      const uint16_t *raw_v, int n_prior, int window, const uint16_t *comp_k,
                      const uint16_t *comp_v, long long n_comp, const int32_t *sel, int k_stride,
                      long long q_pos0, int ratio, float scale, uint16_t *out, void *ws,
                      size_t ws_bytes, void *stream);

/*
 * Batched decode: B independent sessions of one layer per call.
 * ("DwarfStar (ds4) Deep Dive", Step-by-Step Tutorial, "Start the Server": the
 * CUDA server's --batched-session 16 serves 16 decode sessions at once; the
 * "ds4 antirez DeepSeek V4 Flash local engine 2026 guide" page, Use Cases That
 * Fit, "A multi-user box on CUDA cards".)
 * Each session is one decode step as the single-session calls define it, at its
 * own position; a call amortises the per-launch latency over the sessions and
 * streams all of their key and KV rows at once.
 *
 * Layout: session s's arrays sit at fixed strides from session 0's:
 *   pos        [B] int64, DEVICE memory: session s decodes the token at pos[s]
 *              (which the caller has written into slot pos[s] % W of its ring).
 *   q          [B, H, D] fp16;   out [B, H, D] fp16.
 *   q_idx      [B, d_idx] fp16;  k_idx [B, cap, d_idx] fp16 (one key per row).
 *   ring_k, ring_v [B, W, D] fp16: each session's raw window ring, token t in
 *              slot t % W; the window is its min(W, pos+1) slots 0 .. W-1.
 *   comp_k, comp_v [B, cap, D] fp16; state [B, 2 + 2D] float.
 *   out_idx    [B, k] int32 kept rows (as ds4a_indexer_topk); out_n [B] or NULL.
 * Rows of a session that would reach past cap are not written: the compressor
 * update is skipped and DS4A_ERR_CAPACITY is recorded in the device error word
 * (the positions are in device memory, so the host cannot check them).
 * Early reads: pos, plus each single-session call's early reads.
 */

/* Workspace bytes of ds4a_indexer_topk_compress_batched: one 256-byte aligned
 * region per session (ticket + one key per row).  Zero-filled once by the caller;
 * the calls leave it at zero. */
size_t ds4a_decode_batched_workspace_bytes(int B, long long cap);

/*
 * ds4a_indexer_topk_compress_batched -- for every session, the indexer query of
 * its token at pos[s] over its visible rows min(cap, floor((pos[s]+1)/ratio)),
 * and the compressor update for that token (read from ring slot pos[s] % W), in
 * one launch: per session the same results as ds4a_indexer_topk_compress.
 *   W          ring length, 1 .. 4096; head_dim, d_idx, ratio, k as the
 *              single-session call; score_w [head_dim] float, shared by the
 *              sessions (one layer's weights).
 *   ws         ds4a_decode_batched_workspace_bytes(B, cap) bytes, 256-byte aligned.
 */
int ds4a_indexer_topk_compress_batched(int B, const uint16_t *q_idx, const uint16_t *k_idx, long long cap,
                                       int d_idx, const long long *pos, int ratio, int k, int32_t *out_idx,
                                       int32_t *out_n, void *ws, size_t ws_bytes, const uint16_t *ring_k,
                                       const uint16_t *ring_v, int W, int head_dim, const float *score_w,
                                       float *state, uint16_t *comp_k, uint16_t *comp_v, void *stream);

/*
 * ds4a_attn_decode_batched -- for every session, one decode query's attention
 * over its window and compressed rows, as ds4a_attn_decode: the rows listed in
 * its sel row (sel [B, n_sel] int32, -1 entries skipped), or with sel = NULL
 * every visible row min(cap, floor((pos[s]+1)/ratio)) (ratio = 0: window only).
 */
int ds4a_attn_decode_batched(int B, const uint16_t *q, int H, int D, const uint16_t *ring_k, const uint16_t *ring_v,
                             int W, const long long *pos, const uint16_t *comp_k, const uint16_t *comp_v,
                             long long cap, const int32_t *sel, int n_sel, int ratio, float scale, uint16_t *out,
                             void *stream);

/*
 * ds4a_compress_attn_decode_batched -- for every session of a layer that attends
 * every compressed row, the compressor update for its token and the attention,
 * in one launch: per session the same results as ds4a_compress_attn_decode.
 */
int ds4a_compress_attn_decode_batched(int B, const float *score_w, int ratio, float *state, uint16_t *comp_k,
                                      uint16_t *comp_v, long long cap, const uint16_t *q, int H, int D,
                                      const uint16_t *ring_k, const uint16_t *ring_v, int W, const long long *pos,
                                      float scale, uint16_t *out, void *stream);

/*
 * One decode step of one layer from host memory.
 * ("DS4 (DwarfStar 4)", Key Techniques, "KV attention compression" and "KV cache
 * with disk as first-class citizen": the raw 128-token window and the compressor
 * fed one token at a time.)
 *
 * ds4a_decode_layer_t names a layer's persistent device arrays once -- the arrays
 * the single-session calls above take -- and ds4a_decode_layer_step runs the
 * decode step of the token at position pos from host buffers.  It copies the
 * token's inputs into the layer's device arrays, enqueues the launches the device
 * calls make, copies the output to the host and waits for it.  The launches, by
 * layer kind:
 *   - indexer layer (topk > 0): ds4a_indexer_topk_compress, then ds4a_attn_decode
 *     over the kept rows;
 *   - indexer layer with pooled keys: ds4a_indexer_topk_compress_keys, then
 *     ds4a_attn_decode;
 *   - layer that attends every row (ratio > 0, topk = 0): ds4a_compress_attn_decode;
 *   - window-only layer (ratio = 0): ds4a_attn_decode over the window.
 * The window is the ring's min(W, pos+1) rows; the indexer ranks, and the
 * compressor writes, up to cap rows.  The results are those calls' results, bit
 * for bit.  The compressor state must hold the open block's tokens before pos
 * (the layer has decoded pos-1, or was fed up to pos-1).
 *
 * This call is the exception to the conventions above: the pointers of
 * ds4a_decode_host_inputs_t and out_host are HOST pointers, and the call waits for
 * the stream when out_host is not NULL.  When every given input is page-locked
 * (or registered) host memory, one kernel reads them over the host link and writes
 * the device arrays; on an indexer layer the indexer (and compressor) launch reads
 * its own inputs from the host buffers and runs beside that kernel, on the other
 * layers the next launch starts when it has finished.  Otherwise each input is one
 * cudaMemcpyAsync (pageable memory works, staged by the runtime).  A page-locked out_host is written by the attention kernel directly
 * and the layer's out array is then left as it was; any other out_host receives a
 * copy of out.  The host buffers must not change until the call has returned
 * (with out_host = NULL: until the stream has reached the step's end).
 */
typedef struct ds4a_decode_layer {
    int H, D;                    /* heads and head dim, as ds4a_attn_decode */
    int W;                       /* ring rows, 1 .. 4096: token t in slot t % W */
    int ratio;                   /* 0: window only; else tokens per compressed row, 1 .. 1024 */
    int topk;                    /* 0: attend every visible row; else rows the indexer keeps, 1 .. 2048 */
    int d_idx;                   /* indexer key width (topk > 0), multiple of 8, 8 .. 256 */
    int pooled_keys;             /* 1: the compressor pools per-token indexer keys (topk > 0) */
    float scale;                 /* softmax scale */
    long long cap;               /* rows of comp_k, comp_v and k_idx */
    uint16_t *ring_k, *ring_v;   /* [W, D] fp16 */
    const float *score_w;        /* [D] float (ratio > 0) */
    float *state;                /* [2 + 2D] float, + d_idx with pooled keys (ratio > 0) */
    uint16_t *comp_k, *comp_v;   /* [cap, D] fp16 (ratio > 0) */
    uint16_t *k_idx;             /* [cap, d_idx] fp16 (topk > 0) */
    uint16_t *q;                 /* [H, D] fp16: the step's query */
    uint16_t *q_idx;             /* [d_idx] fp16: the step's indexer query (topk > 0) */
    uint16_t *k_idx_tok;         /* [d_idx] fp16: the token's indexer key (pooled keys) */
    int32_t *out_idx;            /* [topk] int32 kept rows (topk > 0) */
    int32_t *out_n;              /* [1] int32 kept-row count, or NULL */
    void *ws;                    /* ds4a_indexer_workspace_bytes(1, cap, topk) bytes (topk > 0) */
    size_t ws_bytes;
    uint16_t *out;               /* [H, D] fp16 (not written when out_host is page-locked) */
} ds4a_decode_layer_t;

/* The step's host inputs.  A NULL pointer leaves that device array as it is (its
 * input is already there). */
typedef struct ds4a_decode_host_inputs {
    const uint16_t *k, *v;       /* [D] fp16: the token's K and V, copied to ring slot pos % W */
    const uint16_t *q;           /* [H, D] fp16, copied to q */
    const uint16_t *q_idx;       /* [d_idx] fp16, copied to q_idx (topk > 0) */
    const uint16_t *k_idx_row;   /* [d_idx] fp16: the indexer key of the row the token completes,
                                    copied to k_idx row (pos+1)/ratio - 1; used only on an indexer
                                    layer without pooled keys, when (pos+1) % ratio == 0 */
    const uint16_t *k_idx_tok;   /* [d_idx] fp16, copied to k_idx_tok (pooled keys) */
} ds4a_decode_host_inputs_t;

/*
 * ds4a_decode_layer_step -- the decode step of the token at pos (>= 0) of the
 * layer `layer`, inputs from `in` (may be NULL: every input already on the
 * device), output copied to out_host ([H, D] fp16, host) and the stream waited
 * for; with out_host = NULL the call returns once the work is enqueued.
 * Errors: every check of the calls it makes, done before anything is enqueued
 * (DS4A_ERR_ARG for a NULL layer, a NULL or misaligned array its kind needs, or
 * topk > 0 with ratio = 0 or pooled_keys with topk = 0; DS4A_ERR_CAPACITY when
 * row (pos+1)/ratio - 1 is >= cap; DS4A_ERR_WORKSPACE for a missing or small
 * workspace).  A failed copy or launch returns DS4A_ERR_CUDA; the device arrays
 * may then hold the step's inputs.
 */
int ds4a_decode_layer_step(const ds4a_decode_layer_t *layer, long long pos, const ds4a_decode_host_inputs_t *in,
                           uint16_t *out_host, void *stream);

/*
 * ds4a_probe_gather -- MEASUREMENT CALL, not a step of the attention path; the
 * pages have no counterpart.  Gathers the n_idx rows table[idx[i]] (D fp16 each,
 * D a multiple of 8, 8 .. 256) into shared memory with 16-byte asynchronous copies,
 * two 128-row tiles in flight per CTA, and adds one word of the result to *sink
 * (a device u32).  Prefill attention is bound by gathering its rows, so the
 * benchmark states the attention kernel's gather rate against this call's rate
 * on the same rows.  Indices outside [0, n_table) are skipped and recorded as
 * DS4A_ERR_DEVICE_INDEX.
 */
int ds4a_probe_gather(const uint16_t *table, long long n_table, int D, const int32_t *idx, long long n_idx,
                      unsigned int *sink, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DS4A_H */
