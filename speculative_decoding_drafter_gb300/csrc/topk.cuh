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
