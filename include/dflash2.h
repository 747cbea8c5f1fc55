/*
 * dflash2.h -- C ABI of the DFlash2 candidate-selector head for GB300 (sm_103a).
 *
 * The selector head turns a block of drafter hidden states into a draft
 * block.  For every draft position t of every sequence b (row r = b*T + t):
 *
 *   logits_r   = W_vocab . h_r                      LM head (float32 accumulate)
 *   cand_r, U_r = top-k of logits_r                  ties: lower token id first
 *   g_r        = W_sel . h_r                         selector gate (linear, no bias)
 *   S_r[i][j]  = U_r[j] + < A(prev_i) (.) g_r , B(cand_r[j]) >
 *                prev = cand_{r-1} for t > 0, the anchor token for t = 0
 *   draft      = greedy walk: j_0 = argmax_j S_(b,0)[0][j],
 *                j_t = argmax_j S_(b,t)[j_(t-1)][j], emit cand[j_t]
 *
 * Sources: "DFlash 2: Keep Drafting Parallel" (inco.ai), section "A
 * Lightweight Path Selector" (the score S_t(a,b) = U_t(b) + <A(a) (.) H(h_t),
 * B(b)>, the top-16 candidates, the rank-256 codebooks A and B, greedy from
 * the last verified token); "DFlash2 Lands in llama.cpp: What PR #27342
 * Actually Changes", sections "The Central Insight" (edge = unary +
 * pairwise) and "What llama.cpp Actually Builds for the Selector"
 * (candidates = top_k(logits), the gathered unary scores, the selector hidden
 * projection, the predecessor/successor codebook gathers, rows packed as
 * candidate ids followed by transition scores, and the walk that starts with
 * predecessor = anchor).
 *
 * Conventions shared by every entry point:
 *  - Every tensor pointer is a DEVICE pointer owned by the caller (except
 *    the *_host arguments of dflash2_select_host).  The library allocates
 *    nothing, frees nothing, and never synchronises a stream (except
 *    dflash2_check_device_status and dflash2_select_host, which say so).
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  The returned status covers argument
 *    validation and launch errors (cudaGetLastError after enqueue); it does
 *    not wait for the kernels.  Some kernels are launched as programmatic
 *    dependents: they may begin under the tail of the kernel before them on
 *    the stream, but read their inputs and write their outputs only after it
 *    has completed, so stream order holds as for ordinary launches.
 *  - bf16 tensors are IEEE bfloat16, row-major and contiguous.  Tensors read
 *    by the tensor-memory-accelerator or by 16-byte vector loads (hidden,
 *    W_vocab, W_sel, pred_cb, succ_cb, logits) must be 16-byte aligned; the
 *    workspace must be 256-byte aligned; every other pointer 4-byte aligned.
 *  - Limits: B >= 1, T >= 1, 1 <= k <= 32 and k <= V, V < 2^24 (candidate
 *    ids are stored as exact floats in the lattice), H >= 8 and H % 8 == 0,
 *    8 <= D <= 1024 and D % 8 == 0, B*T <= 2^20.  Outside them a call returns
 *    DF2_ERR_INVALID_ARG (malformed) or DF2_ERR_UNSUPPORTED (well formed but
 *    beyond what the kernels implement) and enqueues nothing.
 *  - anchor values and W-row indices must lie in [0, V); this is a
 *    precondition (out-of-range anchors are clamped to 0 on the device so
 *    that no read leaves the codebooks, and the result is then unspecified).
 *  - Hidden rows are already aligned to the draft positions: row b*T + t
 *    scores draft position t of sequence b (the export slices the seed
 *    position off upstream; "How to Convert and Run DFlash Models with
 *    OpenVINO", defect 1 of "Three ways ...").
 *
 * Packed lattice row r (float32, width k + k*k):
 *    [ cand_0 .. cand_{k-1} | S[0][0..k-1] | S[1][0..k-1] | ... | S[k-1][0..k-1] ]
 *  candidate ids are stored as exact float values; S is predecessor-major.
 *  At t = 0 the single predecessor is the anchor and all k predecessor rows
 *  hold the same anchor-conditioned scores; the walk reads row 0.
 */
#ifndef DFLASH2_H
#define DFLASH2_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DF2_API __attribute__((visibility("default")))
#else
#define DF2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum df2_status {
    DF2_OK = 0,
    DF2_ERR_INVALID_ARG = 1, /* null pointer, bad dimension, misalignment                    */
    DF2_ERR_UNSUPPORTED = 2, /* valid request outside the implemented limits                 */
    DF2_ERR_WORKSPACE = 3,   /* workspace pointer null/misaligned or smaller than required   */
    DF2_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed                         */
    DF2_ERR_TIMEOUT = 5      /* a device-side pipeline wait gave up (see device status)      */
} df2_status;

/* Problem dimensions: B sequences x T draft positions, hidden size H, vocabulary V,
 * candidates per position k, selector rank D. */
typedef struct df2_dims {
    int32_t B, T, H, V, k, D;
} df2_dims;

/* Bytes of device workspace the calls below need for `dims` (0 if dims are invalid).
 * Independent of the device.  The workspace starts with a control block (the sticky
 * device status word, one completion counter per sequence, and the LM head's per-row-group
 * counters and per-row bound slots) that must be zero before the first call:
 * dflash2_workspace_init zeroes it (a zero-filled allocation also works).
 * Calls leave the control block at zero, so a workspace is reused without re-initialising;
 * after a DF2_ERR_TIMEOUT, initialise it again.  One workspace serves one stream at a time. */
DF2_API size_t dflash2_workspace_bytes(const df2_dims *dims);

/* Zeroes the control block at the start of `workspace` for `dims` (cudaMemsetAsync on stream). */
DF2_API df2_status dflash2_workspace_init(const df2_dims *dims, void *workspace, size_t workspace_bytes,
                                          void *stream);

/*
 * The whole selector head (LM head + top-k, gate, lattice, walk) for B*T rows.
 *   hidden   bf16 [B*T, H]   drafter hidden state of each draft position
 *   W_vocab  bf16 [V, H]     LM-head / output-embedding rows
 *   W_sel    bf16 [D, H]     selector projection (the context gate)
 *   pred_cb  bf16 [V, D]     predecessor codebook A
 *   succ_cb  bf16 [V, D]     successor codebook B
 *   anchor   int32 [B]       last verified token of each sequence
 * outputs:
 *   lattice  float [B*T, k + k*k]   packed rows (layout above)
 *   draft_ids int32 [B, T]          the greedy walk's tokens
 *   topk_ids int32 [B*T, k], topk_logits float [B*T, k], gate float [B*T, D]:
 *            optional copies of the candidates (sorted by logit desc, id asc), their
 *            logits (the unary scores) and the gate; NULL to skip.
 * Two launches: the tensor-core LM head (which also computes the gate; CTA pairs with
 * tcgen05.mma.cta_group::2 from 129 to 1024 rows) and one kernel for the merge, lattice and walk.  The full float32 logits never reach global memory:
 * each CTA of the LM head keeps a per-row top-k of its vocabulary slice in registers.
 */
DF2_API df2_status dflash2_select(const df2_dims *dims, const void *hidden, const void *W_vocab, const void *W_sel,
                          const void *pred_cb, const void *succ_cb, const int32_t *anchor, float *lattice,
                          int32_t *draft_ids, int32_t *topk_ids, float *topk_logits, float *gate,
                          void *workspace, size_t workspace_bytes, void *stream);

/* Options of the walk at the end of dflash2_select_walk. */
typedef struct df2_walk_opts {
    float temperature;     /* > 0 and finite: p = softmax(S / temperature) on the row the walk reads */
    float p_min;           /* the walk stops at the first position whose p is below it; <= 0 never stops */
    const float *uniforms; /* [B, T] in [0, 1): inverse-CDF sampling; NULL: greedy (first maximum) */
    int32_t *n_draft;      /* [B] tokens emitted per sequence, or NULL */
    float *confidence;     /* [B, T] p of the chosen transition up to and including a stop, 0 after; or NULL */
} df2_walk_opts;

/*
 * dflash2_select with the walk's confidence, the p_min early stop and sampling computed in
 * the same launches: the last CTA of each sequence in the merge/lattice kernel walks the
 * rows with the softmax of each row it reads, instead of the stored argmax ("DFlash2 Lands in
 * llama.cpp", section "p_min Means Something Different Under DFlash2": the confidence is the
 * softmax of the current transition row at the chosen candidate, and a low one stops the
 * draft; "DFlash 2: Keep Drafting Parallel", section "A Lightweight Path Selector": sampling
 * draws from the same scores).  The results are those of dflash2_walk_sample on the lattice
 * this call writes, bit for bit: draft_ids is -1 from a stop on.  walk == NULL is
 * dflash2_select.  The caller supplies the random numbers (uniforms), so a draw is
 * reproducible.  Probabilities are float32 with expf.
 */
DF2_API df2_status dflash2_select_walk(const df2_dims *dims, const df2_walk_opts *walk, const void *hidden,
                                       const void *W_vocab, const void *W_sel, const void *pred_cb,
                                       const void *succ_cb, const int32_t *anchor, float *lattice,
                                       int32_t *draft_ids, int32_t *topk_ids, float *topk_logits, float *gate,
                                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * Same path from given float32 logits [B*T, V] instead of the LM head: the top-k,
 * lattice and walk see exactly these logits (the unary score of a candidate is its
 * given logit), so the candidates and draft can be compared bit for bit.
 */
DF2_API df2_status dflash2_select_from_logits(const df2_dims *dims, const float *logits, const void *hidden,
                                      const void *W_sel, const void *pred_cb, const void *succ_cb,
                                      const int32_t *anchor, float *lattice, int32_t *draft_ids,
                                      int32_t *topk_ids, float *topk_logits, float *gate, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * dflash2_select for a caller whose step inputs and results live in host memory (the
 * drafting loop of a serving engine that feeds hidden states in and reads the draft out
 * each step).  One call enqueues, on `stream`: the copy of hidden to device staging
 * inside the workspace, the same two launches as dflash2_select, and the return of the
 * results; it then waits for the stream.  When anchor_host, draft_ids_host, lattice_host
 * (if not NULL) and status_host are all page-locked memory mapped into the current
 * device's address space (cudaHostAlloc / cudaMallocHost, or cudaHostRegister with
 * cudaHostRegisterMapped) and 4-byte aligned, the finish kernel reads the anchors from
 * and writes the draft ids, lattice rows and device status word into them directly, with
 * no copies (each copy on a stream costs about 3 us on GB300, whatever its size).
 * Otherwise the anchors are copied in and the results and status word copied back.
 * Unlike every other call it returns only when the results are in host memory, and it
 * also reports DF2_ERR_TIMEOUT from the device status word (then re-initialise the
 * workspace).
 *   hidden_host    bf16 [B*T, H], host memory
 *   anchor_host    int32 [B], host memory
 *   W_vocab, W_sel, pred_cb, succ_cb   device memory, as for dflash2_select
 *   lattice_host   float [B*T, k + k*k] host memory, or NULL to skip its copy
 *   draft_ids_host int32 [B*T] host memory
 *   status_host    optional uint32 in page-locked host memory that receives the device
 *                  status word (NULL: a pageable word on the stack and the copy path)
 * Host buffers should be page-locked: hidden_host so that its copy runs asynchronously,
 * the others for the direct path; pageable memory works but serialises the host on each
 * copy.
 * The workspace must hold dflash2_select_host_workspace_bytes(dims): the
 * dflash2_workspace_bytes layout followed by the device staging of hidden, anchor,
 * lattice and draft.  Nothing is allocated.
 */
DF2_API size_t dflash2_select_host_workspace_bytes(const df2_dims *dims);
DF2_API df2_status dflash2_select_host(const df2_dims *dims, const void *hidden_host, const void *W_vocab,
                                       const void *W_sel, const void *pred_cb, const void *succ_cb,
                                       const int32_t *anchor_host, float *lattice_host, int32_t *draft_ids_host,
                                       uint32_t *status_host, void *workspace, size_t workspace_bytes, void *stream);

/* ---- single steps of the path (the device code of the calls above), for stage-by-stage checks.
 * dflash2_lattice scores in the 128-thread layout; for 9 to 16 candidates dflash2_select scores
 * in two-warp CTAs, so its lattice sums in another order (both within the float32 bound). ---- */

/* LM head alone: logits float [B*T, V] = hidden . W_vocab^T with float32 accumulation
 * (tensor cores, same main loop as dflash2_select; this variant stores the tile instead
 * of reducing it to a top-k).  dims.k and dims.D are validated but unused. */
DF2_API df2_status dflash2_lm_head_logits(const df2_dims *dims, const void *hidden, const void *W_vocab, float *logits,
                                  void *workspace, size_t workspace_bytes, void *stream);

/* Top-k of given float32 logits [B*T, V]: topk_ids int32 [B*T, k], topk_logits float [B*T, k],
 * ordered by (logit desc, id asc).  "DFlash2 Lands in llama.cpp", candidates = top_k(logits).
 * At few rows one launch: the CTA that completes a row's last column slice merges the row,
 * counting slices in the workspace's control block (left at zero, like every call). */
DF2_API df2_status dflash2_topk(const df2_dims *dims, const float *logits, int32_t *topk_ids, float *topk_logits,
                        void *workspace, size_t workspace_bytes, void *stream);

/* Top-k of given float32 logits without a workspace, for callers that cannot allocate
 * device memory (an engine that plans all device memory itself and gives plugins no
 * allocator; a decode loop that cannot afford cudaMalloc's implicit synchronisation).
 * Same kernels and results as dflash2_topk; the per-slice partial lists live in an
 * 8 MiB array inside the library's device image (held by every GPU that loads the
 * library until exit), so B*T*KP must not exceed 4096 (KP = k rounded up to 4, 8, 16 or
 * 32); larger requests return DF2_ERR_UNSUPPORTED.  The first call on a device (per CUDA
 * context) looks up that array's device address (cudaGetSymbolAddress) with the device
 * current; make that first call before any stream capture.  The address is kept for the
 * life of the context: do not call across a device reset (cudaDeviceReset), which may
 * bring the context back under the same handle.  All calls share the array: calls that overlap on
 * the GPU (other streams, other host threads) race and must be serialised by the caller.
 * Every entry the kernels read is written earlier in the same call, so nothing needs
 * clearing.  The method pages have no counterpart: this is a deployment variant. */
DF2_API df2_status dflash2_topk_noalloc(const df2_dims *dims, const float *logits, int32_t *topk_ids,
                                        float *topk_logits, void *stream);

/* Gate alone: gate float [B*T, D] = hidden . W_sel^T, float32 accumulation on tensor cores. */
DF2_API df2_status dflash2_gate(const df2_dims *dims, const void *hidden, const void *W_sel, float *gate, void *workspace,
                        size_t workspace_bytes, void *stream);

/* Lattice alone, from candidates, their unary scores and the gate: writes the packed rows. */
DF2_API df2_status dflash2_lattice(const df2_dims *dims, const int32_t *topk_ids, const float *topk_logits,
                           const float *gate, const void *pred_cb, const void *succ_cb, const int32_t *anchor,
                           float *lattice, void *stream);

/* Walk alone over packed rows: one warp per sequence; ties go to the lowest candidate index. */
DF2_API df2_status dflash2_walk(const df2_dims *dims, const float *lattice, int32_t *draft_ids, void *stream);

/* Walk with confidence, p_min early stop and optional sampling, over packed rows (the
 * lattice dflash2_select writes).  On the row the walk reads, p = softmax(S / temperature).
 * uniforms == NULL: greedy (first maximum, as dflash2_walk).  Otherwise uniforms float
 * [B, T] in [0, 1): position t takes the first candidate whose running sum of p (in
 * candidate order) exceeds uniforms[b, t] -- the draw comes from the same scores ("DFlash 2:
 * Keep Drafting Parallel", section "A Lightweight Path Selector"); the caller supplies the
 * random numbers.  The chosen transition's p is its confidence; when it is below p_min the
 * walk stops ("DFlash2 Lands in llama.cpp", section "p_min Means Something Different Under
 * DFlash2"): draft_ids is -1 from that position on and n_draft[b] (optional) counts the
 * tokens emitted.  confidence float [B, T] (optional) holds p up to and including the stop,
 * 0 after.  temperature must be finite and > 0; p_min <= 0 never stops.  Probabilities are
 * float32 with expf. */
DF2_API df2_status dflash2_walk_sample(const df2_dims *dims, const float *lattice, float temperature, float p_min,
                                       const float *uniforms, int32_t *draft_ids, int32_t *n_draft,
                                       float *confidence, void *stream);

/* Dimensions of the dynamic local convolution: B blocks of T positions, C channels, G
 * channels per dynamic group. */
typedef struct df2_conv_dims {
    int32_t B, T, C, G;
} df2_conv_dims;

/* Grouped two-tap dynamic depthwise convolution of the drafter's hidden states ("DFlash 2:
 * Keep Drafting Parallel", section "A Lightweight Local Convolution": Conv_k(x)_t =
 * k_{t,0} (.) x_t + k_{t,1} (.) x_{t-1}; "DFlash2 Lands in llama.cpp", section "Dynamic
 * Local Convolution"):
 *   y[r,c] = (base[0,c] + dyn[r,0,c/G]) * xn(x[r])[c] + (base[1,c] + dyn[r,1,c/G]) * xn(prev)[c]
 * with prev = x[r-1] inside a block and x_prev[b] (the last verified token's row) at the
 * first position; no row of another block is ever read.  xn is the identity, or with gamma
 * the RMS normalisation v / sqrt(mean(v^2) + eps) * gamma (an all-zero row stays zero).
 *   x      bf16 [B*T, C]      the block's hidden states (row b*T + t)
 *   x_prev bf16 [B, C]        last verified token of each block, or NULL for a zero row
 *   base   bf16 [2, C]        learned per-channel taps (0: the position, 1: its predecessor)
 *   dyn    float [B*T, 2, C/G] per-group corrections, already projected from the hidden state
 *   gamma  bf16 [C] or NULL   RMS-normalisation weight (NULL: no normalisation)
 *   y      bf16 [B*T, C]      output (round to nearest even); must not overlap x or x_prev
 * Limits: C % G == 0, G % 8 == 0, 8 <= C <= 8192, eps >= 0.  x, x_prev, base, gamma and y
 * 16-byte aligned, dyn 4-byte aligned.  float32 arithmetic. */
DF2_API df2_status dflash2_dynamic_conv(const df2_conv_dims *dims, const void *x, const void *x_prev,
                                        const void *base, const float *dyn, const void *gamma, float eps, void *y,
                                        void *stream);

/* Synchronises `stream`, reads and clears the sticky device status word in `workspace`.
 * Returns DF2_ERR_TIMEOUT if a pipeline wait inside any kernel gave up since the last
 * check (the kernel then skipped its remaining work and its outputs are invalid). */
DF2_API df2_status dflash2_check_device_status(void *workspace, size_t workspace_bytes, void *stream);

/* Self-test of the device-side failure detection (no counterpart in the pages): one
 * thread waits, through the bounded-wait helper that every pipeline wait of the LM-head
 * kernel uses, on an mbarrier that nothing arrives on.  After limit_us microseconds
 * (1 .. 1,000,000) the wait gives up and raises a bit of the workspace's status word, as a
 * stalled pipeline would; dflash2_check_device_status then returns DF2_ERR_TIMEOUT (and
 * clears the word).  Enqueued on `stream`; nothing else is touched. */
DF2_API df2_status dflash2_selftest_wait_timeout(uint32_t limit_us, void *workspace, size_t workspace_bytes,
                                                 void *stream);

/* Timing hook: on this host thread, every following dflash2_select /
 * dflash2_select_from_logits call records `begin` on its stream just before the
 * LM-head (or logits top-k) launch and `end` just after it, so the caller can read
 * that kernel's duration with cudaEventElapsedTime.  Both are cudaEvent_t handles
 * created by the caller; pass NULL, NULL to stop.  Nothing is recorded otherwise. */
DF2_API df2_status dflash2_profile_events(void *begin, void *end);

/* Static description of a status code. */
DF2_API const char *dflash2_status_string(df2_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH (0.3.0: dflash2_select_walk, the
 * confidence / p_min / sampling walk inside the selector call). */
DF2_API int32_t dflash2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH2_H */
