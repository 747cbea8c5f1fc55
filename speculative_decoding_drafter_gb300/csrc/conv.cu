// conv.cu -- grouped two-tap dynamic depthwise convolution of a draft block.
//
// "DFlash 2: Keep Drafting Parallel", section "A Lightweight Local Convolution":
//   Conv_k(x)_t = k_{t,0} (.) x_t + k_{t,1} (.) x_{t-1}
// each coefficient a learned per-channel base plus a correction computed from the
// current hidden state and shared by every group of channels; the first position reads
// the last verified token.  "DFlash2 Lands in llama.cpp", section "Dynamic Local
// Convolution": static weight + dynamic weight per group, block-local shift.
// The dynamic corrections arrive already projected (dyn [B*T, 2, C/G], float); the
// optional RMS normalisation of the conv input (gamma) is fused in.
//
// A CTA takes up to 8 consecutive rows of one block, one warp per row.  It stages those
// rows and the row before the first (the block's previous row, or the last verified
// token, or zeros) in shared memory with one batch of cp.async copies, so each row is
// read from DRAM once and a row's predecessor is the neighbouring warp's slot.  Each warp
// reduces its own row's sum of squares (shuffles) and publishes it; after one CTA barrier
// every warp has both RMS values and writes its bf16 output.  HBM-bound: per row 2C
// bytes read, 2C written, C/G*8 bytes of corrections (read through L1).
#include <cuda_bf16.h>

#include <cstdint>

#include "internal.h"

namespace df2 {
namespace {

constexpr int kRowsPerCta = 8;
constexpr int kThreads = 32 * kRowsPerCta;

struct ConvArgs {
    int T, C, G;
    int tiles;  // CTAs per block: ceil(T / kRowsPerCta)
    const uint16_t *x;
    const uint16_t *x_prev;
    const uint16_t *base;
    const float *dyn;
    const uint16_t *gamma;
    float eps;
    uint16_t *y;
};

__device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    f[0] = lo(v.x); f[1] = hi(v.x); f[2] = lo(v.y); f[3] = hi(v.y);
    f[4] = lo(v.z); f[5] = hi(v.z); f[6] = lo(v.w); f[7] = hi(v.w);
}

__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(
                     smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit_and_wait_all()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ float inv_rms(float sumsq, int C, float eps)
{
    // an all-zero row normalises to zero (even with eps = 0)
    return (sumsq > 0.f || eps > 0.f) ? 1.f / sqrtf(sumsq / static_cast<float>(C) + eps) : 0.f;
}

__global__ void __launch_bounds__(kThreads) dynamic_conv_kernel(const ConvArgs a)
{
    extern __shared__ __align__(16) uint4 rows[];  // slot 0: predecessor of the first row; slot 1+w: row t0+w
    __shared__ float s_sumsq[kRowsPerCta + 1];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x / a.tiles;
    const int t0 = (blockIdx.x - b * a.tiles) * kRowsPerCta;
    const int n = min(kRowsPerCta, a.T - t0);
    const int C = a.C;
    const int chunks = C / 8;
    const long long row0 = static_cast<long long>(b) * a.T + t0;  // global index of row t0

    // ---- stage rows t0-1 .. t0+n-1: warp w copies its own row into slot w+1, warp 0 also
    // the predecessor of row t0 into slot 0 (the block's previous row, the last verified
    // token, or zeros).  A warp reads another warp's slot only after the CTA barrier below.
    const uint4 *xs = reinterpret_cast<const uint4 *>(a.x);
    auto stage = [&](int s) {
        uint4 *dst = rows + static_cast<size_t>(s) * chunks;
        const uint4 *src = nullptr;
        if (s > 0)
            src = xs + (row0 + s - 1) * chunks;
        else if (t0 > 0)
            src = xs + (row0 - 1) * chunks;
        else if (a.x_prev)
            src = reinterpret_cast<const uint4 *>(a.x_prev) + static_cast<long long>(b) * chunks;
        for (int i = lane; i < chunks; i += 32) {
            if (src)
                cp_async16(dst + i, src + i);
            else
                dst[i] = make_uint4(0, 0, 0, 0);
        }
    };
    if (warp < n)
        stage(warp + 1);
    if (warp == 0)
        stage(0);
    cp_async_commit_and_wait_all();
    __syncwarp();

    // ---- sums of squares of the warp's own slots (for the RMS normalisation)
    auto slot_sumsq = [&](int s) {
        float sq = 0.f;
        const uint4 *v = rows + static_cast<size_t>(s) * chunks;
        for (int i = lane; i < chunks; i += 32) {
            float f[8];
            unpack8(v[i], f);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                sq = fmaf(f[e], f[e], sq);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            sq += __shfl_xor_sync(0xffffffffu, sq, off);
        if (lane == 0)
            s_sumsq[s] = sq;
    };
    if (a.gamma) {
        if (warp < n)
            slot_sumsq(warp + 1);
        if (warp == 0)
            slot_sumsq(0);
    }
    __syncthreads();
    if (warp >= n)
        return;

    // ---- output of row t0 + warp
    const long long r = row0 + warp;
    const uint4 *cur = rows + static_cast<size_t>(warp + 1) * chunks;
    const uint4 *prv = rows + static_cast<size_t>(warp) * chunks;
    const float ic = a.gamma ? inv_rms(s_sumsq[warp + 1], C, a.eps) : 1.f;
    const float ip = a.gamma ? inv_rms(s_sumsq[warp], C, a.eps) : 1.f;
    const int groups = C / a.G;
    const int chunks_per_group = a.G / 8;  // G is a multiple of 8: a chunk never straddles groups
    const float *d0 = a.dyn + r * 2 * groups;
    const float *d1 = d0 + groups;
    const uint4 *b0p = reinterpret_cast<const uint4 *>(a.base);
    const uint4 *b1p = b0p + chunks;
    const uint4 *gp = reinterpret_cast<const uint4 *>(a.gamma);
    uint4 *out = reinterpret_cast<uint4 *>(a.y) + r * chunks;
    for (int i = lane; i < chunks; i += 32) {
        const int g = i / chunks_per_group;
        const float k0d = __ldg(d0 + g), k1d = __ldg(d1 + g);
        float fc[8], fp[8], w0[8], w1[8];
        unpack8(cur[i], fc);
        unpack8(prv[i], fp);
        unpack8(__ldg(b0p + i), w0);
        unpack8(__ldg(b1p + i), w1);
        float yv[8];
        if (a.gamma) {
            float gg[8];
            unpack8(__ldg(gp + i), gg);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                yv[e] = fmaf((w1[e] + k1d) * ip, fp[e] * gg[e], ((w0[e] + k0d) * ic) * (fc[e] * gg[e]));
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                yv[e] = fmaf(w1[e] + k1d, fp[e], (w0[e] + k0d) * fc[e]);
        }
        __stcs(out + i, make_uint4(pack2(yv[0], yv[1]), pack2(yv[2], yv[3]), pack2(yv[4], yv[5]), pack2(yv[6], yv[7])));
    }
}

}  // namespace

cudaError_t launch_dynamic_conv(int B, int T, int C, int G, const uint16_t *x, const uint16_t *x_prev,
                                const uint16_t *base, const float *dyn, const uint16_t *gamma, float eps, uint16_t *y,
                                cudaStream_t stream)
{
    ConvArgs a{T, C, G, (T + kRowsPerCta - 1) / kRowsPerCta, x, x_prev, base, dyn, gamma, eps, y};
    const size_t smem = static_cast<size_t>(kRowsPerCta + 1) * C * 2;
    cudaError_t e = cudaFuncSetAttribute(dynamic_conv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    dynamic_conv_kernel<<<static_cast<unsigned>(B * a.tiles), kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace df2
