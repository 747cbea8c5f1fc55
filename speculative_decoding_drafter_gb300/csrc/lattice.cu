// lattice.cu -- the k x k transition lattice and the greedy walk.
//
// "DFlash 2: Keep Drafting Parallel", section "A Lightweight Path Selector":
//   S_t(a, b) = U_t(b) + < A(a) (.) H(h_t), B(b) >
// with a among the previous position's candidates (the last verified token at the
// first position) and b among the current ones; greedy follows the best successor
// from the last verified token.  "DFlash2 Lands in llama.cpp", sections "The Central
// Insight" (edge = unary + pairwise) and "What llama.cpp Actually Builds for the
// Selector" (codebook gathers, rows packed as candidate ids followed by transition
// scores, walk with predecessor = anchor).
#include <cstdint>

#include "internal.h"
#include "topk.cuh"

namespace df2 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ int clamp_id(int id, int V) { return static_cast<unsigned>(id) < static_cast<unsigned>(V) ? id : 0; }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One CTA per draft position r = b*T + t.
//  1. gather the predecessor rows A(prev_i) (one row, the anchor's, at t = 0) and the
//     successor rows B(cand_j) with 16-byte loads; scale A rows by the gate g_r;
//  2. each warp takes predecessor rows; its lanes stride over d and keep k partial
//     dot products, reduced across the warp with shuffles;
//  3. write [cand ids | U_j + pairwise(i, j)], copying the single t = 0 row k times.
template <int KP>
__global__ void __launch_bounds__(kThreads) lattice_kernel(int T, int k, int V, int D,
                                                           const int32_t *__restrict__ topk_ids,
                                                           const float *__restrict__ topk_vals,
                                                           const float *__restrict__ gate,
                                                           const uint16_t *__restrict__ pred_cb,
                                                           const uint16_t *__restrict__ succ_cb,
                                                           const int32_t *__restrict__ anchor,
                                                           float *__restrict__ lattice)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int r = blockIdx.x;
    const int b = r / T;
    const int t = r - b * T;
    const int n_prev = (t == 0) ? 1 : k;
    float *ghat = reinterpret_cast<float *>(smem);                              // [n_prev][D]  A(prev) * g
    uint16_t *succ = reinterpret_cast<uint16_t *>(smem + sizeof(float) * k * D);  // [k][D]       B(cand), bf16
    __shared__ int s_cand[32];
    __shared__ int s_prev[32];
    __shared__ float s_unary[32];

    if (threadIdx.x < k) {
        const long long o = static_cast<long long>(r) * k + threadIdx.x;
        s_cand[threadIdx.x] = clamp_id(topk_ids[o], V);
        s_unary[threadIdx.x] = topk_vals[o];
        s_prev[threadIdx.x] = (t == 0) ? clamp_id(anchor[b], V) : clamp_id(topk_ids[o - k], V);
    }
    __syncthreads();

    const float *g = gate + static_cast<long long>(r) * D;
    const int chunks = D / 8;  // 16-byte chunks of bf16 per codebook row
    for (int idx = threadIdx.x; idx < (n_prev + k) * chunks; idx += kThreads) {
        const int row = idx / chunks;
        const int c8 = idx - row * chunks;
        if (row < n_prev) {
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(pred_cb + static_cast<long long>(s_prev[row]) * D) + c8);
            const float4 g0 = __ldg(reinterpret_cast<const float4 *>(g) + 2 * c8);
            const float4 g1 = __ldg(reinterpret_cast<const float4 *>(g) + 2 * c8 + 1);
            float4 *dst = reinterpret_cast<float4 *>(ghat + row * D) + 2 * c8;
            dst[0] = make_float4(bf16_lo(w.x) * g0.x, bf16_hi(w.x) * g0.y, bf16_lo(w.y) * g0.z, bf16_hi(w.y) * g0.w);
            dst[1] = make_float4(bf16_lo(w.z) * g1.x, bf16_hi(w.z) * g1.y, bf16_lo(w.w) * g1.z, bf16_hi(w.w) * g1.w);
        } else {
            const int j = row - n_prev;
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(succ_cb + static_cast<long long>(s_cand[j]) * D) + c8);
            reinterpret_cast<uint4 *>(succ + j * D)[c8] = w;
        }
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long width = k + static_cast<long long>(k) * k;
    float *out = lattice + static_cast<long long>(r) * width;
    for (int i = warp; i < n_prev; i += kWarps) {
        float acc[KP];
#pragma unroll
        for (int j = 0; j < KP; ++j)
            acc[j] = 0.f;
        const float *a = ghat + i * D;
        for (int d = lane; d < D; d += 32) {
            const float ad = a[d];
#pragma unroll
            for (int j = 0; j < KP; ++j)
                if (j < k)
                    acc[j] = fmaf(ad, __uint_as_float(static_cast<uint32_t>(succ[j * D + d]) << 16), acc[j]);
        }
        float mine = 0.f;
#pragma unroll
        for (int j = 0; j < KP; ++j) {
            float x = acc[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                x += __shfl_xor_sync(kFullMask, x, off);
            if (lane == j)
                mine = x;
        }
        if (lane < k) {
            const float s = s_unary[lane] + mine;
            if (t == 0) {
                for (int ii = 0; ii < k; ++ii)
                    out[k + ii * k + lane] = s;
            } else {
                out[k + i * k + lane] = s;
            }
        }
    }
    if (threadIdx.x < k)
        out[threadIdx.x] = static_cast<float>(s_cand[threadIdx.x]);
}

// One warp per sequence: j_0 = argmax of row 0 at t = 0, then j_t = argmax of row
// j_(t-1); ties go to the lowest candidate index.
__global__ void __launch_bounds__(kThreads) walk_kernel(int B, int T, int k, const float *__restrict__ lattice,
                                                        int32_t *__restrict__ draft)
{
    const int b = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= B)
        return;
    const long long width = k + static_cast<long long>(k) * k;
    int jp = 0;
    for (int t = 0; t < T; ++t) {
        const float *row = lattice + (static_cast<long long>(b) * T + t) * width;
        float x = lane < k ? row[k + jp * k + lane] : -INFINITY;
        int j = lane < k ? lane : 0x7fffffff;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ox = __shfl_xor_sync(kFullMask, x, off);
            const int oj = __shfl_xor_sync(kFullMask, j, off);
            if (ox > x || (ox == x && oj < j)) {
                x = ox;
                j = oj;
            }
        }
        jp = j;
        if (lane == 0)
            draft[static_cast<long long>(b) * T + t] = static_cast<int32_t>(row[jp]);
    }
}

template <int KP>
cudaError_t launch_lattice_kp(int B, int T, int k, int V, int D, const int32_t *ids, const float *vals,
                              const float *gate, const uint16_t *pred, const uint16_t *succ, const int32_t *anchor,
                              float *lattice, cudaStream_t stream)
{
    // dynamic part only; the kernel's static arrays come on top, so the opt-in is always set
    const size_t smem = sizeof(float) * k * D + sizeof(uint16_t) * k * D;
    const cudaError_t e = cudaFuncSetAttribute(lattice_kernel<KP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    lattice_kernel<KP><<<static_cast<unsigned>(B * T), kThreads, smem, stream>>>(T, k, V, D, ids, vals, gate, pred,
                                                                                 succ, anchor, lattice);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lattice(int B, int T, int k, int V, int D, const int32_t *topk_ids, const float *topk_vals,
                           const float *gate, const uint16_t *pred_cb, const uint16_t *succ_cb,
                           const int32_t *anchor, float *lattice, cudaStream_t stream)
{
    switch (kp_for(k)) {
    case 4: return launch_lattice_kp<4>(B, T, k, V, D, topk_ids, topk_vals, gate, pred_cb, succ_cb, anchor, lattice, stream);
    case 8: return launch_lattice_kp<8>(B, T, k, V, D, topk_ids, topk_vals, gate, pred_cb, succ_cb, anchor, lattice, stream);
    case 16: return launch_lattice_kp<16>(B, T, k, V, D, topk_ids, topk_vals, gate, pred_cb, succ_cb, anchor, lattice, stream);
    default: return launch_lattice_kp<32>(B, T, k, V, D, topk_ids, topk_vals, gate, pred_cb, succ_cb, anchor, lattice, stream);
    }
}

cudaError_t launch_walk(int B, int T, int k, const float *lattice, int32_t *draft_ids, cudaStream_t stream)
{
    walk_kernel<<<static_cast<unsigned>((B + kWarps - 1) / kWarps), kThreads, 0, stream>>>(B, T, k, lattice, draft_ids);
    return cudaGetLastError();
}

}  // namespace df2
