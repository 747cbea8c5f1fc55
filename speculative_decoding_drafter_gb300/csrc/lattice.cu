// lattice.cu -- stage kernels: the lattice alone and the walk alone (the fused path
// runs the same device steps inside the finish kernel).
#include <cstdint>

#include "internal.h"
#include "lattice.cuh"
#include "ptx.cuh"

namespace df2 {
namespace {

constexpr int kWarps = kLatticeThreads / 32;

// One CTA per draft position r = b*T + t, from given candidates, unary scores and gate.
template <int KP>
__global__ void __launch_bounds__(kLatticeThreads) lattice_kernel(int T, int k, int V, int D,
                                                                  const int32_t *__restrict__ topk_ids,
                                                                  const float *__restrict__ topk_vals,
                                                                  const float *__restrict__ gate,
                                                                  const uint16_t *__restrict__ pred_cb,
                                                                  const uint16_t *__restrict__ succ_cb,
                                                                  const int32_t *__restrict__ anchor,
                                                                  float *__restrict__ lattice)
{
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_cand[32];
    __shared__ int s_prev[32];
    __shared__ float s_unary[32];
    const int r = blockIdx.x;
    const int b = r / T;
    const int t = r - b * T;
    if (threadIdx.x < k) {
        const long long o = static_cast<long long>(r) * k + threadIdx.x;
        s_cand[threadIdx.x] = clamp_id(topk_ids[o], V);
        s_unary[threadIdx.x] = topk_vals[o];
        s_prev[threadIdx.x] = (t == 0) ? clamp_id(anchor[b], V) : clamp_id(topk_ids[o - k], V);
    }
    load_gate_row(reinterpret_cast<float *>(smem), gate + static_cast<long long>(r) * D, D, 0, blockDim.x);
    const long long width = k + static_cast<long long>(k) * k;
    lattice_row<KP>(k, D, t == 0 ? 1 : k, s_prev, s_cand, s_unary, pred_cb, succ_cb, smem, lattice + r * width);
}

// One warp per sequence.
__global__ void __launch_bounds__(kLatticeThreads) walk_kernel(int B, int T, int k, const float *__restrict__ lattice,
                                                               int32_t *__restrict__ draft)
{
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    griddep_wait();  // launched as a programmatic dependent
    const int b = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (b >= B)
        return;
    const long long width = k + static_cast<long long>(k) * k;
    walk_rows<true>(T, k, width, lattice + static_cast<long long>(b) * T * width, draft + static_cast<long long>(b) * T);
}

// One warp per sequence: the walk with confidence, p_min stop and optional sampling
// (walk_sample_rows), over a lattice a previous launch wrote.
__global__ void __launch_bounds__(kLatticeThreads)
    walk_sample_kernel(int B, int T, int k, const float *__restrict__ lattice, float temperature, float p_min,
                       const float *__restrict__ uniforms, int32_t *__restrict__ draft, int32_t *__restrict__ n_draft,
                       float *__restrict__ confidence)
{
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    griddep_wait();  // launched as a programmatic dependent
    const int b = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (b >= B)
        return;
    const long long width = k + static_cast<long long>(k) * k;
    const long long r0 = static_cast<long long>(b) * T;
    walk_sample_rows<false>(T, k, width, lattice + r0 * width, temperature, p_min, uniforms ? uniforms + r0 : nullptr,
                            draft + r0, nullptr, n_draft ? n_draft + b : nullptr,
                            confidence ? confidence + r0 : nullptr);
}

template <int KP>
cudaError_t launch_lattice_kp(int B, int T, int k, int V, int D, const int32_t *ids, const float *vals,
                              const float *gate, const uint16_t *pred, const uint16_t *succ, const int32_t *anchor,
                              float *lattice, cudaStream_t stream)
{
    // dynamic part only; the kernel's static arrays come on top, so the opt-in is always set
    const size_t smem = lattice_smem_bytes(k, D);
    const cudaError_t e = cudaFuncSetAttribute(lattice_kernel<KP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    lattice_kernel<KP><<<static_cast<unsigned>(B * T), kLatticeThreads, smem, stream>>>(T, k, V, D, ids, vals, gate,
                                                                                         pred, succ, anchor, lattice);
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
    return launch_dependent(walk_kernel, dim3(static_cast<unsigned>((B + kWarps - 1) / kWarps)), dim3(kLatticeThreads),
                            0, stream, B, T, k, lattice, draft_ids);
}

}  // namespace df2

namespace df2 {

cudaError_t launch_walk_sample(int B, int T, int k, const float *lattice, float temperature, float p_min,
                               const float *uniforms, int32_t *draft_ids, int32_t *n_draft, float *confidence,
                               cudaStream_t stream)
{
    return launch_dependent(walk_sample_kernel, dim3(static_cast<unsigned>((B + kWarps - 1) / kWarps)),
                            dim3(kLatticeThreads), 0, stream, B, T, k, lattice, temperature, p_min, uniforms,
                            draft_ids, n_draft, confidence);
}

}  // namespace df2
