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

// One warp merges the n_split partial lists of row `row` into the row's top-k: each lane merges
// whole lists (several per lane per round, all loads issued before the merges); the lanes' lists
// then go through the bounded merge (measured on GB300 at 512 rows, k = 16: far fewer
// instructions than the butterfly), or the warp butterfly when more than 32 entries qualify.
// Writes the ids to s_ids[0..k) and, if s_vals is not null, the values to s_vals.
template <int KP>
__device__ __forceinline__ void merge_row_lists(const FinishArgs &a, long long row, int *s_ids, float *s_vals,
                                                float *s_mv, int *s_mi)
{
    const int lane = threadIdx.x & 31;
    const int k = a.k;
    const long long row_base = row * a.n_split * KP;
    float av[KP];
    int ai[KP];
#pragma unroll
    for (int s = 0; s < KP; ++s) {
        av[s] = -INFINITY;
        ai[s] = INT_MAX;
    }
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
    float mv;
    int mi;
    if (KP <= 16 && bounded_merge<KP>(av, ai, s_mv, s_mi, mv, mi)) {
        if (lane < k) {
            s_ids[lane] = clamp_id(mi, a.V);
            if (s_vals)
                s_vals[lane] = mv;
        }
    } else {
        warp_merge_top<KP>(av, ai, 31);
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < KP; ++s) {
                if (s < k) {
                    s_ids[s] = clamp_id(ai[s], a.V);
                    if (s_vals)
                        s_vals[s] = av[s];
                }
            }
        }
    }
}

// The last CTA of sequence b walks it (all threads of the CTA call this; it returns at once in
// the other CTAs): the greedy walk over the stored choices, or the confidence / p_min /
// sampling walk over the rows (walk_sample_rows).  The sequence's counter returns to zero.
// `smem` is the CTA's dynamic shared memory, free again by now.
__device__ __forceinline__ void walk_if_last(const FinishArgs &a, int b, long long width, uint8_t *smem, int *s_last)
{
    const int warp = threadIdx.x >> 5;
    const int k = a.k;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        *s_last = atomicAdd(a.counters + b, 1u) == static_cast<unsigned>(a.T - 1);
    __syncthreads();
    if (!*s_last)
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

// The merge and the walk are written out here rather than through the device functions
// above, which the small-CTA kernel uses: the same code through them ran 1.1-1.5 us slower at
// 16 and 64 rows in a same-box A/B (identical outputs).
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

// ---------------------------------------------------------------- 9 to 16 candidates: small CTAs

// With 9 to 16 candidates the scores come from warp-level tf32 tensor-core tiles, and a position
// needs only two warps: one merges its row's lists, the other the previous row's (the gate row
// arrives by cp.async meanwhile).  The codebook rows are staged in passes of at most kTilePass
// elements of D, so a CTA holds under 20 KB of shared memory and under 7k registers: at 1024
// positions on 152 SMs every CTA is resident at once (the 128-thread kernel above needs 1.35
// waves there), and the gathers of all positions go to DRAM together.
constexpr int kTileThreads = 64;
constexpr int kTilePass = 256;

__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(
                     smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// Dynamic shared memory of the small-CTA kernel: the gate row [D] float, then 2k staged codebook
// rows of min(D, kTilePass) + 8 elements.
__host__ __device__ constexpr int tile_row_stride(int D) { return (D < kTilePass ? D : kTilePass) + 8; }
__host__ __device__ constexpr size_t tile_smem_bytes(int k, int D)
{
    return sizeof(float) * static_cast<size_t>(D) + sizeof(uint16_t) * 2 * static_cast<size_t>(k) * tile_row_stride(D);
}

template <int KP>
__global__ void __launch_bounds__(kTileThreads) finish_tile_kernel(const FinishArgs a)
{
    static_assert(KP == 16, "the small-CTA kernel serves 9 to 16 candidates");
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_cand[32];
    __shared__ int s_prev[32];
    __shared__ float s_unary[32];
    __shared__ int s_last;
    __shared__ int s_anchor;
    __shared__ float s_mv[2][32];
    __shared__ int s_mi[2][32];
    __shared__ float s_part[2][16][17];  // each warp's partial 16 x 16 score tile

    if (threadIdx.x == 0)
        griddep_launch_dependents();
    const int r = blockIdx.x;
    const int b = r / a.T;
    const int t = r - b * a.T;
    if (t == 0 && threadIdx.x == 0)
        s_anchor = clamp_id(a.anchor[b], a.V);  // no earlier kernel of the call writes it

    griddep_wait();
    if (a.status_mirror && r == 0 && threadIdx.x == 0)
        *a.status_mirror = *reinterpret_cast<const volatile uint32_t *>(a.status);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int k = a.k;
    const int D = a.D;
    float *sg = reinterpret_cast<float *>(smem);                           // [D] gate
    uint16_t *rows = reinterpret_cast<uint16_t *>(smem + sizeof(float) * D);  // [2k][ld]
    const int ld = tile_row_stride(D);

    // ---- 1. gate row by cp.async; merges: warp 0 row r, warp 1 row r-1 (at t = 0 every
    // predecessor row is the anchor's, so the k score rows come out equal)
    const float *grow = a.gate + static_cast<long long>(r) * D;
    for (int i = threadIdx.x; i < D / 4; i += kTileThreads)
        cp_async_16(sg + 4 * i, grow + 4 * i);
    if (warp == 0 || t > 0)
        merge_row_lists<KP>(a, warp == 0 ? r : r - 1, warp == 0 ? s_cand : s_prev, warp == 0 ? s_unary : nullptr,
                            s_mv[warp], s_mi[warp]);
    __syncthreads();
    if (t == 0 && threadIdx.x < k)
        s_prev[threadIdx.x] = s_anchor;
    if (threadIdx.x < k) {
        const long long o = static_cast<long long>(r) * k + threadIdx.x;
        if (a.topk_ids)
            a.topk_ids[o] = s_cand[threadIdx.x];
        if (a.topk_vals)
            a.topk_vals[o] = s_unary[threadIdx.x];
    }
    cp_async_wait_all();  // the gate row
    __syncthreads();

    // ---- 2. scores S[i][j] - U[j] = <A(prev_i) (.) g, B(cand_j)> as one 16 x 16 tile per warp,
    // the D axis in passes of kTilePass staged rows (rows 0..k-1: A(prev_i), k..2k-1: B(cand_j)),
    // each warp taking every other 8-wide step of a pass.  A (.) g is split into tf32 high and low
    // parts and B is bf16 (exact in tf32), so the two products keep float32 accuracy; fragment
    // columns c and c + 4 take d = k0 + 2c and k0 + 2c + 1, one 32-bit word of each row.
    const int gq = lane >> 2, cq = lane & 3;
    const bool va0 = gq < k, va1 = gq + 8 < k;
    float acc[2][2][4] = {};  // [high / low part][candidate tile][fragment]
    for (int p0 = 0; p0 < D; p0 += kTilePass) {
        const int dp = D - p0 < kTilePass ? D - p0 : kTilePass;
        const int chunks = dp / 8;  // 16-byte chunks of a staged row
        for (int idx = threadIdx.x; idx < 2 * k * chunks; idx += kTileThreads) {
            const int row = idx / chunks;
            const int c8 = idx - row * chunks;
            const uint16_t *src = row < k ? a.pred_cb + static_cast<long long>(s_prev[row]) * D
                                          : a.succ_cb + static_cast<long long>(s_cand[row - k]) * D;
            cp_async_16(rows + row * ld + 8 * c8, src + p0 + 8 * c8);
        }
        cp_async_wait_all();
        __syncthreads();
        const uint32_t *rw = reinterpret_cast<const uint32_t *>(rows);
        const int ld2 = ld / 2;
        const uint32_t *pa0 = rw + (va0 ? gq : 0) * ld2;
        const uint32_t *pa1 = rw + (va1 ? gq + 8 : 0) * ld2;
        const uint32_t *pb0 = rw + (k + (va0 ? gq : 0)) * ld2;
        const uint32_t *pb1 = rw + (k + (va1 ? gq + 8 : 0)) * ld2;
        const float2 *g2 = reinterpret_cast<const float2 *>(sg + p0);
        for (int k0 = warp * 8; k0 < dp; k0 += 2 * 8) {
            const int w = k0 / 2 + cq;
            const float2 gg = g2[w];
            const uint32_t x0 = va0 ? pa0[w] : 0u, x1 = va1 ? pa1[w] : 0u;
            float p[4];
            p[0] = bf16_lo(x0) * gg.x;
            p[1] = bf16_lo(x1) * gg.x;
            p[2] = bf16_hi(x0) * gg.y;
            p[3] = bf16_hi(x1) * gg.y;
            uint32_t ahi[4], alo[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                ahi[q] = to_tf32(p[q]);
                alo[q] = to_tf32(p[q] - __uint_as_float(ahi[q]));
            }
            const uint32_t y0 = va0 ? pb0[w] : 0u, y1 = va1 ? pb1[w] : 0u;
            const uint32_t b00 = y0 << 16, b01 = y0 & 0xFFFF0000u;
            const uint32_t b10 = y1 << 16, b11 = y1 & 0xFFFF0000u;
            mma_tf32_16x8x8(acc[0][0], ahi, b00, b01);
            mma_tf32_16x8x8(acc[0][1], ahi, b10, b11);
            mma_tf32_16x8x8(acc[1][0], alo, b00, b01);
            mma_tf32_16x8x8(acc[1][1], alo, b10, b11);
        }
        __syncthreads();  // the next pass overwrites the staged rows
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int col = nt * 8 + 2 * cq;
        s_part[warp][gq][col] = acc[0][nt][0] + acc[1][nt][0];
        s_part[warp][gq][col + 1] = acc[0][nt][1] + acc[1][nt][1];
        s_part[warp][gq + 8][col] = acc[0][nt][2] + acc[1][nt][2];
        s_part[warp][gq + 8][col + 1] = acc[0][nt][3] + acc[1][nt][3];
    }
    __syncthreads();

    // ---- 3. the packed row and each predecessor row's argmax: two predecessor rows per warp
    // step, one per half-warp (lane j of a half holds candidate j)
    const long long width = k + static_cast<long long>(k) * k;
    float *out = a.lattice + r * width;
    float *mirror = a.lattice_mirror ? a.lattice_mirror + r * width : nullptr;
    int32_t *best = a.best + static_cast<long long>(r) * k;
    const int half = lane >> 4, j = lane & 15;
    for (int i0 = 2 * warp; i0 < k; i0 += 4) {
        const int i = i0 + half;
        const bool valid = i < k && j < k;
        const float sc = valid ? s_unary[j] + (s_part[0][i][j] + s_part[1][i][j]) : -INFINITY;
        if (valid) {
            out[k + i * k + j] = sc;
            if (mirror)
                mirror[k + i * k + j] = sc;
        }
        float x = sc;
        int jj = j < k ? j : 0x7fffffff;
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {
            const float ox = __shfl_xor_sync(kFullMask, x, off);
            const int oj = __shfl_xor_sync(kFullMask, jj, off);
            const bool take = ranks_before(ox, oj, x, jj);
            x = take ? ox : x;
            jj = take ? oj : jj;
        }
        if (j == 0 && i < k)
            best[i] = jj;
    }
    if (threadIdx.x < k) {
        out[threadIdx.x] = static_cast<float>(s_cand[threadIdx.x]);
        if (mirror)
            mirror[threadIdx.x] = static_cast<float>(s_cand[threadIdx.x]);
    }

    // ---- 4. the last CTA of the sequence walks it
    walk_if_last(a, b, width, smem, &s_last);
}

constexpr size_t kWalkSmemCap = 64 * 1024;
// Fair-share sizing of the small-CTA kernel's shared memory (GB300: 228 KB per SM with the
// largest carveout, 1 KB reserved per CTA, the kernel's static arrays; the CTAs per SM its
// registers and shared memory allow anyway).
constexpr size_t kSmemPerSm = 228 * 1024;
constexpr size_t kSmemReservePerCta = 1024;
constexpr size_t kTileStaticSmem = 3200;
constexpr size_t kFairSmemCap = 200 * 1024;
constexpr long long kTileCtasPerSm = 9;

template <int KP>
cudaError_t launch_kp(FinishArgs a, int B, cudaStream_t stream)
{
    // 9 to 16 candidates: the small-CTA kernel (tensor-core tiles on staged rows)
    const bool tile = KP == 16 && a.k > 8;
    auto kern = tile ? finish_tile_kernel<16> : finish_kernel<KP>;
    const size_t walk_bytes = 2 * sizeof(int) * static_cast<size_t>(a.T) * a.k;
    a.walk_in_smem = walk_bytes <= kWalkSmemCap;
    size_t smem = tile ? tile_smem_bytes(a.k, a.D) : lattice_smem_bytes(a.k, a.D);
    if (a.walk_in_smem && walk_bytes > smem)
        smem = walk_bytes;
    // Launched as a programmatic dependent, the CTAs become resident on the SMs the LM head frees
    // first and wait there for its grid: up to nine small CTAs on one SM, so at 512 positions
    // they would crowd onto some 57 SMs.  Shared memory sized to an SM's fair share of the
    // positions keeps any SM from taking more than ceil(R / SMs) of them.  Measured on GB300
    // (same-box A/Bs, interleaved): from the LM head to the end of the step 23.3 -> 15.7 us at 512
    // rows (18.9 with the 128-thread kernel).  The same sizing did nothing for the 128-thread
    // kernel at 16 and 64 rows (14.19 against 14.17 us for the kernel alone), so it keeps its own.
    if (tile) {
        const long long R = static_cast<long long>(B) * a.T;
        const long long sms = device_sm_count();
        const long long share = (R + sms - 1) / sms;
        if (share < kTileCtasPerSm) {
            size_t want = kSmemPerSm / static_cast<size_t>(share) - kSmemReservePerCta - kTileStaticSmem;
            if (want > kFairSmemCap)
                want = kFairSmemCap;
            if (want > smem)
                smem = want;
        }
    }
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    if (tile) {
        // as much shared memory as the SM has (the fair-share sizing above counts on it)
        thread_local int carveout_set_for = -1;
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess)
            return e;
        if (carveout_set_for != dev) {
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                          cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
                return e;
            carveout_set_for = dev;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(B * a.T));
    cfg.blockDim = dim3(tile ? kTileThreads : kFinishThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
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
