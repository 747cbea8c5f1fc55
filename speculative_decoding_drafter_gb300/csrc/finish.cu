// finish.cu -- everything after the LM head, in one launch: merge of the per-slice
// top-k lists, the lattice row of each draft position, and the greedy walk.
//
// One CTA per draft position r = b*T + t (128 threads: small CTAs keep many positions in
// flight at large batch -- measured on GB300, 24.0 vs 30.7 us after the LM head at 512 rows,
// the same at batch 1):
//   1. warp 0 merges the partial lists of row r into its top-k (candidates and unary
//      scores), warp 1 those of row r-1 (the predecessors; the anchor at t = 0): lane l
//      takes lists l, l+32, ... (each already sorted); the entries at or above a bound on
//      the row's KP-th best are then gathered and sorted across the warp (bounded_merge),
//      or, when more than 32 are, a warp butterfly of bitonic merges finishes.  Warps 2-3
//      meanwhile fetch the gate row;
//   2. the lattice row (lattice.cuh), plus the walk's choice for every predecessor row;
//   3. the CTA counts itself done for sequence b; the last CTA of the sequence loads the
//      T choice rows and candidate ids into shared memory and follows j_t = best[t][j_(t-1)]
//      -- or, when the caller asked for confidences, a p_min stop or sampling, one warp walks
//      the sequence's rows with the softmax of each row it reads (walk_sample_rows).  The
//      counter returns to zero.
// Launched with programmatic stream serialisation: its prologue overlaps the tail of the
// kernel that produced the lists, and griddep_wait() orders the reads after it (the anchor,
// which no earlier kernel of the call writes, is read before).
// Host mirrors (the host-buffer call with page-locked buffers): the lattice rows and draft
// ids are written to the caller's host buffers as well, and the device status word, final
// once the LM head is done, to the caller's host status word; no copies follow the kernel.
#include <cstdint>

#include "internal.h"
#include "lattice.cuh"
#include "ptx.cuh"
#include "topk.cuh"

namespace df2 {
namespace {

struct FinishArgs {
    int T, k, V, D, n_split;
    const float *pval;
    const int32_t *pid;
    const float *gate;
    const uint16_t *pred_cb;
    const uint16_t *succ_cb;
    const int32_t *anchor;
    float *lattice;
    int32_t *draft;
    int32_t *topk_ids;   // optional copies (may be null)
    float *topk_vals;
    int32_t *best;       // [B*T, k] walk choices
    unsigned *counters;  // [B], zero between calls
    int walk_in_smem;    // the sequence's choice table fits the dynamic shared memory
    float *lattice_mirror;          // optional host mirrors (may be null)
    int32_t *draft_mirror;
    const uint32_t *status;         // device status word, copied to status_mirror if set
    uint32_t *status_mirror;
    int sample_walk;                // the confidence / p_min / sampling walk instead of the greedy one
    float temperature, p_min;
    const float *uniforms;          // [B*T] or null
    int32_t *n_draft;               // [B] or null
    float *confidence;              // [B*T] or null
};

constexpr int kFinishThreads = 128;

template <int KP>
__global__ void __launch_bounds__(kFinishThreads) finish_kernel(const FinishArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_cand[32];
    __shared__ int s_prev[32];
    __shared__ float s_unary[32];
    __shared__ int s_last;
    __shared__ float s_mv[2][32];  // bounded-merge gathers, one per merging warp
    __shared__ int s_mi[2][32];

    // the next call's LM head may start now: it prefetches weights and waits for this grid
    // before it touches anything this kernel reads
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    const int r = blockIdx.x;
    const int b = r / a.T;
    const int t = r - b * a.T;
    const int anchor_b = t == 0 && threadIdx.x == 0 ? a.anchor[b] : 0;

    griddep_wait();
    if (a.status_mirror && r == 0 && threadIdx.x == 0)
        *a.status_mirror = *reinterpret_cast<const volatile uint32_t *>(a.status);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int k = a.k;

    // ---- 1. merge (warp 0: row r, warp 1: row r-1) while the other warps fetch the gate row
    if (warp < 2 && (warp == 0 || t > 0)) {
        const long long row_base = static_cast<long long>(warp == 0 ? r : r - 1) * a.n_split * KP;
        float av[KP];
        int ai[KP];
#pragma unroll
        for (int s = 0; s < KP; ++s) {
            av[s] = -INFINITY;
            ai[s] = INT_MAX;
        }
        // several lists per lane per round, all loads issued before the merges
        constexpr int kLists = KP <= 8 ? 5 : KP <= 16 ? 2 : 1;
        for (int list0 = lane; list0 < a.n_split; list0 += 32 * kLists) {
            float bv[kLists][KP];
            int bi[kLists][KP];
#pragma unroll
            for (int u = 0; u < kLists; ++u) {
                const int list = list0 + 32 * u;
                const bool have = list < a.n_split;
                const long long off = row_base + static_cast<long long>(have ? list : 0) * KP;
                const float4 *pv = reinterpret_cast<const float4 *>(a.pval + off);
                const int4 *pi = reinterpret_cast<const int4 *>(a.pid + off);
#pragma unroll
                for (int q = 0; q < KP / 4; ++q) {
                    const float4 v4 = __ldcg(pv + q);
                    const int4 i4 = __ldcg(pi + q);
                    bv[u][4 * q] = have ? v4.x : -INFINITY;
                    bv[u][4 * q + 1] = have ? v4.y : -INFINITY;
                    bv[u][4 * q + 2] = have ? v4.z : -INFINITY;
                    bv[u][4 * q + 3] = have ? v4.w : -INFINITY;
                    bi[u][4 * q] = have ? i4.x : INT_MAX;
                    bi[u][4 * q + 1] = have ? i4.y : INT_MAX;
                    bi[u][4 * q + 2] = have ? i4.z : INT_MAX;
                    bi[u][4 * q + 3] = have ? i4.w : INT_MAX;
                }
            }
#pragma unroll
            for (int u = 0; u < kLists; ++u)
                merge_top<KP>(av, ai, bv[u], bi[u]);
        }
        // the lanes' lists into the row's top-k: the bounded merge (measured on GB300 at 512
        // rows, k = 16: far fewer instructions than the butterfly), else the butterfly
        float mv;
        int mi;
        if (KP <= 16 && bounded_merge<KP>(av, ai, s_mv[warp], s_mi[warp], mv, mi)) {
            if (lane < k) {
                if (warp == 0) {
                    s_cand[lane] = clamp_id(mi, a.V);
                    s_unary[lane] = mv;
                } else {
                    s_prev[lane] = clamp_id(mi, a.V);
                }
            }
        } else {
            warp_merge_top<KP>(av, ai, 31);
            if (lane == 0) {
#pragma unroll
                for (int s = 0; s < KP; ++s) {
                    if (s < k) {
                        if (warp == 0) {
                            s_cand[s] = clamp_id(ai[s], a.V);
                            s_unary[s] = av[s];
                        } else {
                            s_prev[s] = clamp_id(ai[s], a.V);
                        }
                    }
                }
            }
        }
    } else if (warp >= 2) {
        load_gate_row(reinterpret_cast<float *>(smem), a.gate + static_cast<long long>(r) * a.D, a.D, 64,
                      blockDim.x - 64);
    }
    if (t == 0 && threadIdx.x == 0)
        s_prev[0] = clamp_id(anchor_b, a.V);
    __syncthreads();
    if (threadIdx.x < k) {
        const long long o = static_cast<long long>(r) * k + threadIdx.x;
        if (a.topk_ids)
            a.topk_ids[o] = s_cand[threadIdx.x];
        if (a.topk_vals)
            a.topk_vals[o] = s_unary[threadIdx.x];
    }

    // ---- 2. lattice row and the walk's choice from each predecessor row
    const long long width = k + static_cast<long long>(k) * k;
    lattice_row<KP>(k, a.D, t == 0 ? 1 : k, s_prev, s_cand, s_unary, a.pred_cb, a.succ_cb, smem,
                    a.lattice + r * width, a.best + static_cast<long long>(r) * k,
                    a.lattice_mirror ? a.lattice_mirror + r * width : nullptr);

    // ---- 3. the last CTA of the sequence walks it
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        s_last = atomicAdd(a.counters + b, 1u) == static_cast<unsigned>(a.T - 1);
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    const long long r0 = static_cast<long long>(b) * a.T;
    const int32_t *best = a.best + r0 * k;
    const float *rows = a.lattice + r0 * width;
    int32_t *draft = a.draft + r0;
    int32_t *draft_mirror = a.draft_mirror ? a.draft_mirror + r0 : nullptr;
    if (a.sample_walk) {
        // the confidence of each step needs the whole row the walk reads: one warp walks the
        // rows through L2, with the same device code as the stand-alone sampling walk
        if (warp == 0)
            walk_sample_rows<true>(a.T, k, width, rows, a.temperature, a.p_min, a.uniforms ? a.uniforms + r0 : nullptr,
                                   draft, draft_mirror, a.n_draft ? a.n_draft + b : nullptr,
                                   a.confidence ? a.confidence + r0 : nullptr);
    } else if (a.walk_in_smem) {
        int *sb = reinterpret_cast<int *>(smem);     // [T][k] choices
        int *sid = sb + a.T * k;                     // [T][k] candidate ids
        for (int i = threadIdx.x; i < a.T * k; i += blockDim.x) {
            const int tt = i / k, j = i - tt * k;
            sb[i] = __ldcg(best + i);
            sid[i] = static_cast<int>(__ldcg(rows + tt * width + j));
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int j = 0;
            for (int tt = 0; tt < a.T; ++tt) {
                j = sb[tt * k + j];
                draft[tt] = sid[tt * k + j];
                if (draft_mirror)
                    draft_mirror[tt] = sid[tt * k + j];
            }
        }
    } else if (threadIdx.x == 0) {
        int j = 0;
        for (int tt = 0; tt < a.T; ++tt) {
            j = __ldcg(best + static_cast<long long>(tt) * k + j);
            const int32_t id = static_cast<int32_t>(__ldcg(rows + tt * width + j));
            draft[tt] = id;
            if (draft_mirror)
                draft_mirror[tt] = id;
        }
    }
    if (threadIdx.x == 0)
        a.counters[b] = 0u;
}

constexpr size_t kWalkSmemCap = 64 * 1024;

template <int KP>
cudaError_t launch_kp(FinishArgs a, int B, cudaStream_t stream)
{
    const size_t walk_bytes = 2 * sizeof(int) * static_cast<size_t>(a.T) * a.k;
    a.walk_in_smem = walk_bytes <= kWalkSmemCap;
    size_t smem = lattice_smem_bytes(a.k, a.D);
    if (a.walk_in_smem && walk_bytes > smem)
        smem = walk_bytes;
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(finish_kernel<KP>), static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B * a.T));
    cfg.blockDim = dim3(kFinishThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, finish_kernel<KP>, a);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_finish(int B, int T, int k, int V, int D, int KP, int n_split, const float *pval,
                          const int32_t *pid, const float *gate, const uint16_t *pred_cb, const uint16_t *succ_cb,
                          const int32_t *anchor, float *lattice, int32_t *draft_ids, int32_t *topk_ids,
                          float *topk_vals, int32_t *best, unsigned *counters, const HostMirrors &mirrors,
                          const WalkOpts &walk, cudaStream_t stream)
{
    FinishArgs a{};
    a.sample_walk = walk.sample ? 1 : 0;
    a.temperature = walk.temperature;
    a.p_min = walk.p_min;
    a.uniforms = walk.uniforms;
    a.n_draft = walk.n_draft;
    a.confidence = walk.confidence;
    a.lattice_mirror = mirrors.lattice;
    a.draft_mirror = mirrors.draft;
    a.status = mirrors.status_dev;
    a.status_mirror = mirrors.status;
    a.T = T;
    a.k = k;
    a.V = V;
    a.D = D;
    a.n_split = n_split;
    a.pval = pval;
    a.pid = pid;
    a.gate = gate;
    a.pred_cb = pred_cb;
    a.succ_cb = succ_cb;
    a.anchor = anchor;
    a.lattice = lattice;
    a.draft = draft_ids;
    a.topk_ids = topk_ids;
    a.topk_vals = topk_vals;
    a.best = best;
    a.counters = counters;
    switch (KP) {
    case 4: return launch_kp<4>(a, B, stream);
    case 8: return launch_kp<8>(a, B, stream);
    case 16: return launch_kp<16>(a, B, stream);
    case 32: return launch_kp<32>(a, B, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace df2
