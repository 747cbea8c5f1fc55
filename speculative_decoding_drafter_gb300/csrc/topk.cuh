// topk.cuh -- top-k selection primitives under the total order (value desc, id asc).
//
// "DFlash2 Lands in llama.cpp", section "What llama.cpp Actually Builds for the
// Selector": candidates = top_k(logits), and the unary score of a candidate is its
// logit.  Equal logits are ordered by the lower token id, so every merge order
// gives the same list.
#pragma once

#include <climits>
#include <cstdint>

namespace df2 {

constexpr unsigned kFullMask = 0xffffffffu;

// Branch-free (no short-circuit): the sorting networks below evaluate it thousands of
// times per warp, and a branch per comparison costs more than the comparison.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib)
{
    return (va > vb) | ((va == vb) & (ia < ib));
}

// Sorted per-thread list of KP (value, id) pairs held in registers.
template <int KP>
struct ThreadTopK {
    float v[KP];
    int i[KP];

    __device__ __forceinline__ void init()
    {
#pragma unroll
        for (int s = 0; s < KP; ++s) {
            v[s] = -INFINITY;
            i[s] = INT_MAX;
        }
    }

    __device__ __forceinline__ float threshold() const { return v[KP - 1]; }

    // Insert when ids arrive in increasing order: an equal value never displaces an
    // entry (the entry has the lower id), so the strict '>' implements the tie-break.
    // Branch-free: every slot takes its upper neighbour (x ranks above it), x (x lands
    // here) or itself; slots are visited bottom-up so each reads its neighbour's old value.
    __device__ __forceinline__ void push_increasing_id(float x, int id)
    {
        if (!(x > v[KP - 1]))
            return;
#pragma unroll
        for (int s = KP - 1; s > 0; --s) {
            const bool above = x > v[s - 1];
            const bool here = x > v[s];
            const float nv = here ? x : v[s];
            const int ni = here ? id : i[s];
            v[s] = above ? v[s - 1] : nv;
            i[s] = above ? i[s - 1] : ni;
        }
        const bool first = x > v[0];
        v[0] = first ? x : v[0];
        i[0] = first ? id : i[0];
    }

    // Insert under the full order (value desc, id asc), ids in any order.
    __device__ __forceinline__ void push(float x, int id)
    {
        if (!ranks_before(x, id, v[KP - 1], i[KP - 1]))
            return;
#pragma unroll
        for (int s = KP - 1; s > 0; --s) {
            if (ranks_before(x, id, v[s - 1], i[s - 1])) {
                v[s] = v[s - 1];
                i[s] = i[s - 1];
            } else if (ranks_before(x, id, v[s], i[s])) {
                v[s] = x;
                i[s] = id;
            }
        }
        if (ranks_before(x, id, v[0], i[0])) {
            v[0] = x;
            i[0] = id;
        }
    }
};

// Top-KP of two lists sorted by (value desc, id asc), kept in a: the elementwise better
// of a[i] and b[KP-1-i] is a bitonic sequence holding exactly the KP best of the union,
// and a bitonic merge network sorts it again.  Fixed cost, no data-dependent branches.
template <int KP>
__device__ __forceinline__ void merge_top(float (&av)[KP], int (&ai)[KP], const float (&bv)[KP], const int (&bi)[KP])
{
#pragma unroll
    for (int s = 0; s < KP; ++s) {
        const bool take = ranks_before(bv[KP - 1 - s], bi[KP - 1 - s], av[s], ai[s]);
        av[s] = take ? bv[KP - 1 - s] : av[s];
        ai[s] = take ? bi[KP - 1 - s] : ai[s];
    }
#pragma unroll
    for (int stride = KP / 2; stride > 0; stride >>= 1) {
#pragma unroll
        for (int s = 0; s < KP; ++s) {
            if ((s & stride) == 0) {
                const int t = s + stride;
                const bool sw = ranks_before(av[t], ai[t], av[s], ai[s]);
                const float tv = av[s];
                const int ti = ai[s];
                av[s] = sw ? av[t] : av[s];
                ai[s] = sw ? ai[t] : ai[s];
                av[t] = sw ? tv : av[t];
                ai[t] = sw ? ti : ai[t];
            }
        }
    }
}

// Bitonic sort of one (value, id) pair per lane across the warp: lane j ends with the j-th
// pair in (value desc, id asc) order.
__device__ __forceinline__ void warp_sort_desc(float &v, int &i)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const float ov = __shfl_xor_sync(kFullMask, v, stride);
            const int oi = __shfl_xor_sync(kFullMask, i, stride);
            // the lower lane of a pair keeps the better pair where this block runs descending
            const bool keep_better = ((lane & stride) == 0) == ((lane & size) == 0);
            if (keep_better == ranks_before(ov, oi, v, i)) {
                v = ov;
                i = oi;
            }
        }
    }
}

// The row's top-KP from the lanes' sorted local lists (av, ai) without the warp butterfly.
// The KP-th best of the 32 lane heads, tau, is outranked or matched by at least KP entries,
// so every entry of the row's top-KP ranks at or before it; when more than 32 entries do, a
// second try takes the tightest of the bounds from list positions 1 and 3 as well.  When at
// most 32 entries rank at or before tau they are gathered in shared memory (`sv`, `si`: 32
// slots) and sorted across the warp, and lane j receives the j-th best.  Returns false
// (nothing changed) when more than 32 still do; the caller then merges with the butterfly.
// Warp-uniform.
template <int KP>
__device__ __forceinline__ bool bounded_merge(const float (&av)[KP], const int (&ai)[KP], float *sv, int *si,
                                              float &out_v, int &out_i)
{
    const int lane = threadIdx.x & 31;
    // tau_p: the m-th best of the lanes' entries at position p, m = ceil(KP / (p + 1)); m lanes
    // hold p + 1 entries each at or before it, so at least KP entries do
    auto bound_at = [&](int p, float &tv, int &ti) {
        float hv = av[0];
        int hi = ai[0];
#pragma unroll
        for (int j = 1; j < KP; ++j)
            if (j == p) {
                hv = av[j];
                hi = ai[j];
            }
        warp_sort_desc(hv, hi);
        const int m = (KP + p) / (p + 1);
        tv = __shfl_sync(kFullMask, hv, m - 1);
        ti = __shfl_sync(kFullMask, hi, m - 1);
    };
    // entries of this lane's list at or before tau (a prefix: the list is sorted), and their
    // inclusive prefix sum over the lanes
    auto count = [&](float tv, int ti, int &n, int &incl) {
        n = 0;
#pragma unroll
        for (int j = 0; j < KP; ++j)
            n += ranks_before(tv, ti, av[j], ai[j]) ? 0 : 1;
        incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int up = __shfl_up_sync(kFullMask, incl, o);
            if (lane >= o)
                incl += up;
        }
    };
    float tv;
    int ti, n, incl;
    bound_at(0, tv, ti);
    count(tv, ti, n, incl);
    if (__shfl_sync(kFullMask, incl, 31) > 32) {
        // few lists (one per lane or fewer): the heads bound it loosely; the best-ranked of the
        // bounds from positions 1 and 3 is tighter (measured on the 1024-row workload with 19
        // lists per row: the rows past 32 survivors fall from about 47% to under 1%)
#pragma unroll
        for (int p = 1; p < KP && p <= 3; p += 2) {
            float pv;
            int pi;
            bound_at(p, pv, pi);
            if (ranks_before(pv, pi, tv, ti)) {
                tv = pv;
                ti = pi;
            }
        }
        count(tv, ti, n, incl);
    }
    const int total = __shfl_sync(kFullMask, incl, 31);
    if (total > 32)
        return false;
    const int off = incl - n;
#pragma unroll
    for (int j = 0; j < KP; ++j) {
        if (j < n) {
            sv[off + j] = av[j];
            si[off + j] = ai[j];
        }
    }
    __syncwarp();
    out_v = lane < total ? sv[lane] : -INFINITY;
    out_i = lane < total ? si[lane] : INT_MAX;
    __syncwarp();
    warp_sort_desc(out_v, out_i);
    return true;
}

// Butterfly over the lanes whose index differs in the bits of `lane_mask` (a power of two
// minus one): afterwards each lane holds the top-KP of the lists of its group.
template <int KP>
__device__ __forceinline__ void warp_merge_top(float (&av)[KP], int (&ai)[KP], int lane_mask)
{
    for (int stride = 1; stride <= lane_mask; stride <<= 1) {
        float bv[KP];
        int bi[KP];
#pragma unroll
        for (int s = 0; s < KP; ++s) {
            bv[s] = __shfl_xor_sync(kFullMask, av[s], stride);
            bi[s] = __shfl_xor_sync(kFullMask, ai[s], stride);
        }
        merge_top<KP>(av, ai, bv, bi);
    }
}

// Warp-wide sorted list: lane j holds entry j (32 slots, only the first k are used by
// the callers; the rest are valid lower-ranked entries or sentinels).
struct WarpList {
    float v;
    int i;

    __device__ __forceinline__ void init()
    {
        v = -INFINITY;
        i = INT_MAX;
    }

    // Entry `slot` (warp-uniform) of the list, broadcast to all lanes.
    __device__ __forceinline__ void entry(int slot, float &ev, int &ei) const
    {
        ev = __shfl_sync(kFullMask, v, slot);
        ei = __shfl_sync(kFullMask, i, slot);
    }

    // Insert one candidate (warp-uniform value); entries it ranks before shift one lane down.
    __device__ __forceinline__ void insert(float cv, int ci)
    {
        const int lane = threadIdx.x & 31;
        const unsigned m = __ballot_sync(kFullMask, ranks_before(cv, ci, v, i));
        const float uv = __shfl_up_sync(kFullMask, v, 1);
        const int ui = __shfl_up_sync(kFullMask, i, 1);
        if (m) {
            const int pos = __ffs(m) - 1;
            if (lane > pos) {
                v = uv;
                i = ui;
            } else if (lane == pos) {
                v = cv;
                i = ci;
            }
        }
    }

    // Offer 32 candidates (one per lane); those ranking before entry k-1 are inserted.
    __device__ __forceinline__ void offer(float cv, int ci, int k)
    {
        float tv;
        int ti;
        entry(k - 1, tv, ti);
        unsigned m = __ballot_sync(kFullMask, ranks_before(cv, ci, tv, ti));
        while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1;
            const float xv = __shfl_sync(kFullMask, cv, src);
            const int xi = __shfl_sync(kFullMask, ci, src);
            entry(k - 1, tv, ti);
            if (ranks_before(xv, xi, tv, ti))
                insert(xv, xi);
        }
    }
};

}  // namespace df2
