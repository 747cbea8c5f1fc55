// topk_kernels.cu -- top-k of materialised float32 logits, and the merge of partial lists.
//
// "DFlash2 Lands in llama.cpp", section "What llama.cpp Actually Builds for the
// Selector": candidates = top_k(logits); the unary scores are the gathered logits.
// Order: value descending, then token id ascending.
#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace df2 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Order-preserving map of a float to an unsigned key (larger float, larger key); every key
// of a float is above 0, which marks an empty bound slot.
__device__ __forceinline__ uint32_t bound_key(float x)
{
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float bound_value(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// One CTA per (row, column slice), 8 warps.  Each warp keeps one warp-wide sorted list
// (lane j holds entry j) over a contiguous part of the slice: lanes load 16-byte groups
// (8 in flight per lane); a group of 128 values is offered to the list only when one of
// them beats the list's k-th entry, which after the first few groups is rare, and then only
// the lanes holding such values insert (a per-thread list would diverge: some lane of the
// warp would insert on almost every step).  A bitonic butterfly then merges the 8 warp
// lists into the slice's partial list.
// The warps share a lower bound: warp w keeps its best S/8 entries in shared-memory slots
// (S = max(KP, 8), as order-preserving keys), so the slots hold values of S distinct
// columns and their minimum is a lower bound on the slice's KP-th best value.  A value
// below it is outranked by KP others and cannot reach the row's top-k, so each warp skips
// it: the warps warm up together instead of each on its own eighth of the slice.
template <int KP, bool kVec4>
__global__ void __launch_bounds__(kThreads) logits_topk_partial_kernel(const float *__restrict__ logits, int V,
                                                                       int n_split, float *__restrict__ pval,
                                                                       int32_t *__restrict__ pid)
{
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    griddep_wait();  // launched as a programmatic dependent
    const int r = blockIdx.x;
    const int s = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const float *row = logits + static_cast<long long>(r) * V;
    WarpList wl;
    wl.init();
    constexpr int kSlots = KP > kWarps ? KP : kWarps;
    constexpr int kPerWarp = kSlots / kWarps;
    __shared__ uint32_t s_slot[kSlots];
    if (threadIdx.x < kSlots)
        s_slot[threadIdx.x] = 0u;  // empty: no bound yet
    __syncthreads();
    if constexpr (kVec4) {
        const int groups = V / 4;
        const int g0 = static_cast<int>(static_cast<long long>(s) * groups / n_split);
        const int g1 = static_cast<int>(static_cast<long long>(s + 1) * groups / n_split);
        const int w0 = g0 + static_cast<int>(static_cast<long long>(warp) * (g1 - g0) / kWarps);
        const int w1 = g0 + static_cast<int>(static_cast<long long>(warp + 1) * (g1 - g0) / kWarps);
        const float4 *row4 = reinterpret_cast<const float4 *>(row);
        constexpr int kU = 8;  // 16-byte loads in flight per lane
        float thr = -INFINITY;  // the list's KP-th entry (warp-uniform)
        int thr_i = INT_MAX;
        for (int g = w0 + lane; g < w1 + lane; g += 32 * kU) {
            // the shared bound: values below it are skipped, values equal to it still pass
            const uint32_t key = lane < kSlots ? reinterpret_cast<volatile uint32_t *>(s_slot)[lane] : 0xffffffffu;
            const uint32_t kmin = __reduce_min_sync(kFullMask, key);
            const float bound = kmin == 0u ? -INFINITY : bound_value(kmin);
            float4 x[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int gi = g + 32 * u;
                x[u] = gi < w1 ? __ldcs(row4 + gi) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                // Every id of this 128-value group is above every id already in the list, so
                // a value equal to the KP-th entry ranks after it: only a strictly larger
                // value can enter, and most groups have none.
                const float m = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
                if (__any_sync(kFullMask, m > thr && m >= bound)) {
                    // ids of the group: 4 * (base + lane) + component, base warp-uniform
                    const int base = g - lane + 32 * u;
                    const float xc[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        // >= keeps every value that may enter; ranks_before decides exactly
                        unsigned cand = __ballot_sync(kFullMask, xc[c] >= thr && xc[c] >= bound);
                        while (cand) {
                            const int src = __ffs(cand) - 1;
                            cand &= cand - 1u;
                            const float cv = __shfl_sync(kFullMask, xc[c], src);
                            const int ci = 4 * (base + src) + c;
                            if (ranks_before(cv, ci, thr, thr_i)) {
                                wl.insert(cv, ci);
                                thr = __shfl_sync(kFullMask, wl.v, KP - 1);
                                thr_i = __shfl_sync(kFullMask, wl.i, KP - 1);
                                if (lane < kPerWarp)  // this warp's best entries, in its own slots
                                    reinterpret_cast<volatile uint32_t *>(s_slot)[warp * kPerWarp + lane] =
                                        bound_key(wl.v);
                            }
                        }
                    }
                }
            }
        }
    } else {
        const int e0 = static_cast<int>(static_cast<long long>(s) * V / n_split);
        const int e1 = static_cast<int>(static_cast<long long>(s + 1) * V / n_split);
        const int w0 = e0 + static_cast<int>(static_cast<long long>(warp) * (e1 - e0) / kWarps);
        const int w1 = e0 + static_cast<int>(static_cast<long long>(warp + 1) * (e1 - e0) / kWarps);
        for (int e = w0 + lane; e < w1 + lane; e += 32) {
            const float x = e < w1 ? __ldcs(row + e) : -INFINITY;
            wl.offer(x, e, KP);
        }
    }

    // merge the 8 warp lists: lane l of warp 0 takes warp l's list, bitonic butterfly
    __shared__ float sv[kWarps][32];
    __shared__ int si[kWarps][32];
    sv[warp][lane] = wl.v;
    si[warp][lane] = wl.i;
    __syncthreads();
    if (warp == 0) {
        float av[KP];
        int ai[KP];
        const int w = lane & (kWarps - 1);
#pragma unroll
        for (int j = 0; j < KP; ++j) {
            av[j] = sv[w][j];
            ai[j] = si[w][j];
        }
        warp_merge_top<KP>(av, ai, kWarps - 1);
        if (lane == 0) {
            const long long base = (static_cast<long long>(r) * n_split + s) * KP;
#pragma unroll
            for (int j = 0; j < KP; ++j) {
                pval[base + j] = av[j];
                pid[base + j] = ai[j];
            }
        }
    }
}

// Merges the n_split sorted lists of KP of row r (pval/pid, written by other CTAs: read
// through L2) into the row's top-k, one warp.  Lane l merges whole lists l, l + 32, ... into
// its own sorted top-KP; the lanes' lists are then combined by gathering the entries at or
// above a bound on the row's KP-th best (bounded_merge), or, when more than 32 are, by the warp
// butterfly.  (Offering every entry to one warp-wide list cost 12.7 us at 16 rows x 38 lists of
// 8 and 30.5 us at 16 x 64 lists of 16, measured on GB300: each insertion is a chain of
// dependent shuffles.)  s_mv / s_mi: 32 entries of shared memory for this warp.
template <int KP>
__device__ __forceinline__ void merge_row_lists(const float *pval, const int32_t *pid, int r, int n_split, int k,
                                                int32_t *ids, float *vals, float *s_mv, int *s_mi)
{
    const int lane = threadIdx.x & 31;
    if (n_split == 1) {
        // one slice covered the whole row: its sorted list is the row's top-KP (the lane
        // butterfly below would merge it with 31 lanes of empty entries)
        if (lane < k) {
            const long long o = static_cast<long long>(r) * KP + lane;
            ids[static_cast<long long>(r) * k + lane] = __ldcg(pid + o);
            vals[static_cast<long long>(r) * k + lane] = __ldcg(pval + o);
        }
        return;
    }
    float av[KP];
    int ai[KP];
#pragma unroll
    for (int j = 0; j < KP; ++j) {
        av[j] = -INFINITY;
        ai[j] = INT_MAX;
    }
    const long long row_base = static_cast<long long>(r) * n_split * KP;
    for (int list = lane; list < n_split; list += 32) {
        const float4 *pv = reinterpret_cast<const float4 *>(pval + row_base + static_cast<long long>(list) * KP);
        const int4 *pi = reinterpret_cast<const int4 *>(pid + row_base + static_cast<long long>(list) * KP);
        float bv[KP];
        int bi[KP];
#pragma unroll
        for (int q = 0; q < KP / 4; ++q) {
            const float4 v4 = __ldcg(pv + q);
            const int4 i4 = __ldcg(pi + q);
            bv[4 * q] = v4.x;
            bv[4 * q + 1] = v4.y;
            bv[4 * q + 2] = v4.z;
            bv[4 * q + 3] = v4.w;
            bi[4 * q] = i4.x;
            bi[4 * q + 1] = i4.y;
            bi[4 * q + 2] = i4.z;
            bi[4 * q + 3] = i4.w;
        }
        if (list == lane) {
            // the lane's first list is sorted in the merge's order already: it is the running
            // list (measured on GB300 by CUDA-graph replay, identical outputs: 8.04 -> 7.36 us per
            // call at 16 x 151936 with k = 8, where every lane takes one list of the 30)
#pragma unroll
            for (int j = 0; j < KP; ++j) {
                av[j] = bv[j];
                ai[j] = bi[j];
            }
        } else {
            merge_top<KP>(av, ai, bv, bi);
        }
    }
    float mv;
    int mi;
    if (!(KP <= 16 && bounded_merge<KP>(av, ai, s_mv, s_mi, mv, mi))) {
        warp_merge_top<KP>(av, ai, 31);  // every lane now holds the row's top-KP
        mv = -INFINITY;
        mi = INT_MAX;
#pragma unroll
        for (int j = 0; j < KP; ++j)
            if (j == lane) {
                mv = av[j];
                mi = ai[j];
            }
    }
    if (lane < k) {
        ids[static_cast<long long>(r) * k + lane] = mi;
        vals[static_cast<long long>(r) * k + lane] = mv;
    }
}

// Few rows (a grid of about one wave): one CTA per (row, balanced slice of at most 5120 columns),
// a thread holding 20 values in registers.  The per-warp list of the kernel above spends most of
// its time in the chain of insertions while a list fills, which at 16 rows is the whole
// kernel; here no list is filled value by value.  Warp w takes tau_w, the ceil(KP / 8)-th
// largest of its lanes' maxima: at least ceil(KP / 8) values of distinct columns are at or
// above it, so over the 8 warps at least KP values are at or above tau = min_w tau_w, which
// therefore bounds the slice's KP-th best from below.  The values at or above tau (typically
// a few dozen) are gathered in shared memory and warp 0 sorts them 32 at a time into the
// slice's top-KP.  The gather holds every value of the slice, so no count can overflow it.
// With row_done (one counter per row, zero before the launch and zero again after it) the
// kernel also finishes the rows: the CTA that completes a row's last slice, found by an atomic
// counter (nothing waits), merges the row's slice lists into ids / vals, so no merge launch
// follows.  Measured on GB300 by CUDA-graph replay, identical outputs, at 16 rows x 151936
// (k = 8): as fast as a separate merge launch, which the programmatic dependent launch already
// overlapped (13.0 against 12.98 us with the earlier slicing); the balanced slices below took it
// to 8.0 us.
constexpr int kSmallPerThread = 20;                          // values per thread (5120 columns per CTA)
constexpr int kSmallCols = kThreads * kSmallPerThread;       // columns per CTA

template <int KP>
__global__ void __launch_bounds__(kThreads) logits_topk_small_kernel(const float *__restrict__ logits, int V,
                                                                     int n_split, float *__restrict__ pval,
                                                                     int32_t *__restrict__ pid,
                                                                     unsigned *__restrict__ row_done, int k,
                                                                     int32_t *__restrict__ ids,
                                                                     float *__restrict__ vals)
{
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    griddep_wait();  // launched as a programmatic dependent
    __shared__ float s_v[kSmallCols];
    __shared__ int s_i[kSmallCols];
    __shared__ float s_tau[kWarps];
    __shared__ int s_count;
    const int r = blockIdx.x;
    const int s = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Balanced slices: the row's V / 4 groups of four columns split evenly (at most
    // ceil(V / 4 / n_split) <= kSmallCols / 4 groups each; V is a multiple of 4).  Slices of
    // kSmallCols with a short remainder left the last one a few hundred columns, most of its
    // warps empty, their bound -inf and every value a survivor: each row then waited for that
    // CTA's sorts.  Measured on GB300 by CUDA-graph replay, identical outputs: 13.0 -> 9.2 us per
    // call at 16 x 151936 with balanced slices of 4096 columns at most, 8.0 with 5120 (30 slices
    // instead of 38); 12.98 -> 12.37 us at 16 x 262144.
    const int groups = V / 4;
    const int c0 = static_cast<int>(static_cast<long long>(s) * groups / n_split) * 4;
    const int c1 = static_cast<int>(static_cast<long long>(s + 1) * groups / n_split) * 4;
    const float4 *row4 = reinterpret_cast<const float4 *>(logits + static_cast<long long>(r) * V);
    if (threadIdx.x == 0)
        s_count = 0;
    // group q of this thread: columns 4 * g .. 4 * g + 3, g = c0 / 4 + q * kThreads + tid
    float x[kSmallPerThread];
#pragma unroll
    for (int q = 0; q < kSmallPerThread / 4; ++q) {
        const int g = c0 / 4 + q * kThreads + threadIdx.x;
        const float4 v = 4 * g < c1 ? __ldcs(row4 + g) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        x[4 * q] = v.x;
        x[4 * q + 1] = v.y;
        x[4 * q + 2] = v.z;
        x[4 * q + 3] = v.w;
    }
    bool any = false;  // this thread holds a column of the slice
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < kSmallPerThread / 4; ++q) {
        const int g = c0 / 4 + q * kThreads + threadIdx.x;
        if (4 * g < c1) {
            any = true;
            m = fmaxf(m, fmaxf(fmaxf(x[4 * q], x[4 * q + 1]), fmaxf(x[4 * q + 2], x[4 * q + 3])));
        }
    }
    // tau_w: the ceil(KP / 8)-th largest lane maximum of the warp (-inf when fewer lanes hold
    // columns, which makes every value of the slice a survivor)
    float mv = any ? m : -INFINITY;
    int mi = any ? lane : INT_MAX;
    warp_sort_desc(mv, mi);
    constexpr int kJ = (KP + kWarps - 1) / kWarps;
    const float tw = __shfl_sync(kFullMask, mv, kJ - 1);
    const int tiw = __shfl_sync(kFullMask, mi, kJ - 1);
    if (lane == 0)
        s_tau[warp] = tiw == INT_MAX ? -INFINITY : tw;
    __syncthreads();
    float tau = s_tau[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w)
        tau = fminf(tau, s_tau[w]);
    // gather the survivors: values at or above tau of columns inside the slice
#pragma unroll
    for (int q = 0; q < kSmallPerThread / 4; ++q) {
        const int g = c0 / 4 + q * kThreads + threadIdx.x;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (4 * g + c < c1 && x[4 * q + c] >= tau) {
                const int slot = atomicAdd(&s_count, 1);
                s_v[slot] = x[4 * q + c];
                s_i[slot] = 4 * g + c;
            }
        }
    }
    __syncthreads();
    if (warp != 0)
        return;
    // warp 0: the top 32 of the survivors, 32 at a time (each batch sorted, then merged into
    // the running list with one bitonic clean); lane j ends with the j-th best
    const int count = s_count;
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int b0 = 0; b0 < count; b0 += 32) {
        float v = b0 + lane < count ? s_v[b0 + lane] : -INFINITY;
        int i = b0 + lane < count ? s_i[b0 + lane] : INT_MAX;
        warp_sort_desc(v, i);
        if (b0 == 0) {
            bv = v;
            bi = i;
            continue;
        }
        // best (descending) against the batch reversed: the better of each pair holds the top
        // 32 of both as a bitonic sequence
        const float rv = __shfl_sync(kFullMask, v, 31 - lane);
        const int ri = __shfl_sync(kFullMask, i, 31 - lane);
        if (ranks_before(rv, ri, bv, bi)) {
            bv = rv;
            bi = ri;
        }
#pragma unroll
        for (int stride = 16; stride > 0; stride >>= 1) {
            const float ov = __shfl_xor_sync(kFullMask, bv, stride);
            const int oi = __shfl_xor_sync(kFullMask, bi, stride);
            const bool lower = (lane & stride) == 0;
            if (lower == ranks_before(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
    }
    if (lane < KP) {
        const long long o = (static_cast<long long>(r) * n_split + s) * KP + lane;
        pval[o] = bv;
        pid[o] = bi;
    }
    if (!row_done)
        return;
    // the CTA that completes the row merges it: the count is an acquire-release atomic, so the
    // warp's list (ordered before it by the warp barrier) is visible to whoever counts last, and
    // the lists counted before are visible to it (measured on GB300 at 16 x 151936: 13.3 us per
    // call with a full fence on each side, 13.0 with the ordered atomic)
    __syncwarp();
    unsigned last = 0;
    if (lane == 0) {
        unsigned old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(row_done + r) : "memory");
        last = old == static_cast<unsigned>(n_split - 1);
    }
    if (!__shfl_sync(kFullMask, last, 0))
        return;
    __syncwarp();
    merge_row_lists<KP>(pval, pid, r, n_split, k, ids, vals, reinterpret_cast<float *>(s_v),
                        reinterpret_cast<int *>(s_i));
    if (lane == 0)
        row_done[r] = 0u;
}

// One warp per row: merge n_split sorted lists of KP into the row's top-k (merge_row_lists).
template <int KP>
__global__ void __launch_bounds__(kThreads) topk_merge_kernel(const float *__restrict__ pval,
                                                              const int32_t *__restrict__ pid, int R, int n_split,
                                                              int k, int32_t *__restrict__ ids,
                                                              float *__restrict__ vals)
{
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    griddep_wait();  // launched as a programmatic dependent
    __shared__ float s_mv[kWarps][32];
    __shared__ int s_mi[kWarps][32];
    const int warp = threadIdx.x >> 5;
    const int r = blockIdx.x * kWarps + warp;
    if (r >= R)
        return;
    merge_row_lists<KP>(pval, pid, r, n_split, k, ids, vals, s_mv[warp], s_mi[warp]);
}

template <int KP>
cudaError_t launch_partial(const float *logits, int R, int V, float *pval, int32_t *pid, int *n_split_out,
                           const TopkFinish &fin, bool *merged, cudaStream_t stream)
{
    *merged = false;
    // about one CTA per SM in total (one per row beyond), slices of at least 2048 columns.  Every
    // warp pays a warm-up of ~k (1 + ln(n / k)) list insertions over its n values, so long slices
    // win once the CTAs cover the SMs (measured on GB300: 78 us at 512 rows x 151936 with one
    // slice per row, 95 us with two, 139 us with four).
    const bool vec4 = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0);
    const int sms = device_sm_count();
    // Few rows: slices of at most 5120 columns without per-warp lists, while the grid is small
    // (measured on GB300 with 4096-column slices, same ids and values: 28.3 -> 26.3 us per call
    // at 16 x 151936, 40.6 -> 35.6 at 16 x 262144; 32.4 -> 38.6 at 64 x 152064, 2432 CTAs, so
    // larger grids keep the lists)
    const int small_split = (V + kSmallCols - 1) / kSmallCols;
    if (vec4 && static_cast<long long>(R) * small_split <= 8ll * sms && small_split <= max_splits_for(R)) {
        *n_split_out = small_split;
        *merged = fin.row_done != nullptr;
        return launch_dependent(logits_topk_small_kernel<KP>, dim3(static_cast<unsigned>(R), small_split),
                                dim3(kThreads), 0, stream, logits, V, small_split, pval, pid, fin.row_done, fin.k,
                                fin.ids, fin.vals);
    }
    int n_split = std::max(1, (sms + R - 1) / R);
    n_split = std::min({n_split, max_splits_for(R), std::max(1, V / 2048)});
    *n_split_out = n_split;
    const dim3 grid(static_cast<unsigned>(R), static_cast<unsigned>(n_split));
    if (vec4)
        return launch_dependent(logits_topk_partial_kernel<KP, true>, grid, dim3(kThreads), 0, stream, logits, V,
                                n_split, pval, pid);
    return launch_dependent(logits_topk_partial_kernel<KP, false>, grid, dim3(kThreads), 0, stream, logits, V, n_split,
                            pval, pid);
}

}  // namespace

cudaError_t launch_logits_topk_partial(const float *logits, int R, int V, int KP, float *pval, int32_t *pid,
                                       int *n_split_out, cudaStream_t stream, const TopkFinish &fin, bool *merged)
{
    bool m = false;
    cudaError_t e;
    switch (KP) {
    case 4: e = launch_partial<4>(logits, R, V, pval, pid, n_split_out, fin, &m, stream); break;
    case 8: e = launch_partial<8>(logits, R, V, pval, pid, n_split_out, fin, &m, stream); break;
    case 16: e = launch_partial<16>(logits, R, V, pval, pid, n_split_out, fin, &m, stream); break;
    case 32: e = launch_partial<32>(logits, R, V, pval, pid, n_split_out, fin, &m, stream); break;
    default: e = cudaErrorInvalidValue;
    }
    if (merged)
        *merged = m;
    return e;
}

cudaError_t launch_topk_merge(const float *pval, const int32_t *pid, int R, int n_split, int KP, int k,
                              int32_t *topk_ids, float *topk_vals, cudaStream_t stream)
{
    const dim3 grid(static_cast<unsigned>((R + kWarps - 1) / kWarps));
    switch (KP) {
    case 4:
        return launch_dependent(topk_merge_kernel<4>, grid, dim3(kThreads), 0, stream, pval, pid, R, n_split, k,
                                topk_ids, topk_vals);
    case 8:
        return launch_dependent(topk_merge_kernel<8>, grid, dim3(kThreads), 0, stream, pval, pid, R, n_split, k,
                                topk_ids, topk_vals);
    case 16:
        return launch_dependent(topk_merge_kernel<16>, grid, dim3(kThreads), 0, stream, pval, pid, R, n_split, k,
                                topk_ids, topk_vals);
    case 32:
        return launch_dependent(topk_merge_kernel<32>, grid, dim3(kThreads), 0, stream, pval, pid, R, n_split, k,
                                topk_ids, topk_vals);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace df2
