// internal.h -- launchers shared by the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace df2 {

// Partial top-k lists hold at most this many vocabulary splits per row.
constexpr int kMaxSplits = 256;

// Splits per row that a launch over R rows may use, whatever the device: the LM head makes
// about SMs / ceil(R / 128) column slices and the top-k of given logits about 4 * SMs / R,
// so with at most 1024 SMs neither exceeds ceil(131072 / R).  Workspaces are sized by it.
inline int max_splits_for(long long R)
{
    const long long b = R > 0 ? (131072 + R - 1) / R : 1;
    return static_cast<int>(b < 1 ? 1 : b > kMaxSplits ? kMaxSplits : b);
}

// Capacity of the per-row candidate lists for a requested k (4, 8, 16 or 32).
inline int kp_for(int k) { return k <= 4 ? 4 : k <= 8 ? 8 : k <= 16 ? 16 : 32; }

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// Opts `kernel` in to at least `bytes` of dynamic shared memory on the current device; the
// attribute is set once per kernel, device and size (remembered per host thread).
cudaError_t ensure_dynamic_smem(const void *kernel, int bytes);

// LM head (and gate) in one tensor-core launch: C = hidden[R, K] . [W_vocab; W_store]^T
// (bf16 in, float32 accumulate).  The first V columns are reduced on the fly to per-row
// top-KP lists over each CTA's column slice, pval/pid [R, n_split, KP] (value desc, id
// asc; *n_split_out receives n_split); the next n_store columns (W_store rows) are stored
// as float32 out[r * ldo + n].  V = 0 or n_store = 0 drops that segment.  bound [R, KP] and
// group_done [lm_head_max_groups(R)] are scratch that is zero before the launch and zero
// again after it: a lower bound on each row's KP-th best logit that the CTAs share.
// dependent: launch as a programmatic dependent of the grid before it on the stream (one
// row tile per CTA, or CTA pairs); the kernel then sets up (and, with one tile per CTA,
// brings its first weight boxes into L2) and waits for that grid before it reads hidden or
// writes anything.
cudaError_t launch_lm_head(const void *hidden, int R, int K, const void *W_vocab, int V, int KP, float *pval,
                           int32_t *pid, int *n_split_out, const void *W_store, int n_store, float *out,
                           long long ldo, uint32_t *bound, unsigned *group_done, uint32_t *status,
                           bool dependent, cudaStream_t stream);

// Row groups of the LM head at R rows (at most one per 128-row tile).
inline int lm_head_max_groups(long long R) { return static_cast<int>((R + 127) / 128); }

// C = A[R, K] . B[N, K]^T stored as float32 out[r * ldo + n] (the store segment alone).
cudaError_t launch_gemm_store(const void *A, const void *B, int R, int K, int N, float *out, long long ldo,
                              uint32_t *status, cudaStream_t stream);

// Optional finish of the top-k of given logits inside the slice launch: row_done [R] counters
// (zero before, zero after), and where the rows' top-k go.
struct TopkFinish {
    unsigned *row_done = nullptr;
    int k = 0;
    int32_t *ids = nullptr;
    float *vals = nullptr;
};

// Per-row partial top-KP of given float32 logits [R, V] over n_split column slices.  With
// fin.row_done set, the launch may also merge the rows into fin.ids / fin.vals (the slice
// kernel for few rows does): *merged (if not null) then says so and no merge launch is needed.
cudaError_t launch_logits_topk_partial(const float *logits, int R, int V, int KP, float *pval, int32_t *pid,
                                       int *n_split_out, cudaStream_t stream, const TopkFinish &fin = TopkFinish{},
                                       bool *merged = nullptr);

// Merge [R, n_split, KP] partial lists into the top-k of each row (value desc, id asc).
cudaError_t launch_topk_merge(const float *pval, const int32_t *pid, int R, int n_split, int KP, int k,
                              int32_t *topk_ids, float *topk_vals, cudaStream_t stream);

// Device-visible pointers into a caller's page-locked host buffers, written by the finish
// kernel in place of copies after it (each may be null).
struct HostMirrors {
    float *lattice = nullptr;            // [B*T, k + k*k]
    int32_t *draft = nullptr;            // [B*T]
    uint32_t *status = nullptr;          // one word: receives *status_dev
    const uint32_t *status_dev = nullptr;
};

// The walk the finish kernel runs: with `sample` false the greedy walk over each row's stored
// argmax (no confidence); otherwise the walk with the chosen transition's softmax confidence,
// the p_min stop and, given uniforms, inverse-CDF sampling (walk_sample_rows).
struct WalkOpts {
    bool sample = false;
    float temperature = 1.f;
    float p_min = 0.f;
    const float *uniforms = nullptr;  // [B*T] in [0, 1), or null: greedy
    int32_t *n_draft = nullptr;       // [B] or null
    float *confidence = nullptr;      // [B*T] or null
};

// Everything after the lists in one launch (programmatic dependent launch): merge of
// the [R, n_split, KP] lists, lattice rows, and the walk by the last CTA of each
// sequence (best [R, k] is scratch for the walk's choices).  counters [B] must be zero
// before the call and are zero after it.  anchor is read before the kernel waits for the
// one before it, so no kernel of the same call may write it.
cudaError_t launch_finish(int B, int T, int k, int V, int D, int KP, int n_split, const float *pval,
                          const int32_t *pid, const float *gate, const uint16_t *pred_cb, const uint16_t *succ_cb,
                          const int32_t *anchor, float *lattice, int32_t *draft_ids, int32_t *topk_ids,
                          float *topk_vals, int32_t *best, unsigned *counters, const HostMirrors &mirrors,
                          const WalkOpts &walk, cudaStream_t stream);

// Packed lattice rows [B*T, k + k*k] from candidates, unary scores, gate and codebooks.
cudaError_t launch_lattice(int B, int T, int k, int V, int D, const int32_t *topk_ids, const float *topk_vals,
                           const float *gate, const uint16_t *pred_cb, const uint16_t *succ_cb,
                           const int32_t *anchor, float *lattice, cudaStream_t stream);

// Walk with confidence, p_min stop and optional sampling (uniforms [B*T] or null).
cudaError_t launch_walk_sample(int B, int T, int k, const float *lattice, float temperature, float p_min,
                               const float *uniforms, int32_t *draft_ids, int32_t *n_draft, float *confidence,
                               cudaStream_t stream);

// Two-tap dynamic depthwise conv of B blocks of T rows (bf16 [B*T, C] in and out).
cudaError_t launch_dynamic_conv(int B, int T, int C, int G, const uint16_t *x, const uint16_t *x_prev,
                                const uint16_t *base, const float *dyn, const uint16_t *gamma, float eps, uint16_t *y,
                                cudaStream_t stream);

// Greedy walk, one warp per sequence: draft_ids [B, T].
cudaError_t launch_walk(int B, int T, int k, const float *lattice, int32_t *draft_ids, cudaStream_t stream);

// Launches `kernel` as a programmatic dependent of the kernel before it on `stream`: it may
// start under that kernel's tail, and must wait for it (griddep_wait in every CTA, before
// anything it reads or writes) so that its own completion still implies that kernel's.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// selftest.cu
cudaError_t launch_wait_selftest(uint32_t *status, unsigned long long limit_ns, cudaStream_t stream);

}  // namespace df2
