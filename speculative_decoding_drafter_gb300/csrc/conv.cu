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
// A CTA takes up to 8 consecutive rows of one block.  It stages those rows and the row
// before the first (the block's previous row, or the last verified token, or zeros) in
// shared memory with one batch of cp.async copies, so each row is read from DRAM once.
// Each thread then owns 16-byte channel chunks across all of the CTA's rows: the static
// taps and gamma of a chunk are unpacked once and serve every row, and a row's normalised
// input, kept in registers, is the next row's predecessor term.  The RMS of each staged
// row comes from a CTA-wide reduction.  HBM-bound: per row 2C bytes read, 2C written,
// C/G*8 bytes of corrections (read through L1).
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

constexpr int kSlots = kRowsPerCta + 1;

__global__ void __launch_bounds__(kThreads, 3) dynamic_conv_kernel(const ConvArgs a)
{
    extern __shared__ __align__(16) uint4 rows[];  // slot 0: predecessor of the first row; slot 1+s: row t0+s
    __shared__ float s_part[kThreads / 32][16];    // per-warp partial sums of squares, by slot
    __shared__ float s_scale[kSlots];              // 1/RMS of each slot (1 without normalisation)
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int b = blockIdx.x / a.tiles;
    const int t0 = (blockIdx.x - b * a.tiles) * kRowsPerCta;
    const int n = min(kRowsPerCta, a.T - t0);
    const int C = a.C;
    const int chunks = C / 8;
    const long long row0 = static_cast<long long>(b) * a.T + t0;  // global index of row t0

    // ---- stage slots 0..n: rows t0-1 .. t0+n-1, consecutive in x except the predecessor
    // of t0 = 0, which is the last verified token (x_prev) or zeros
    const uint4 *xs = reinterpret_cast<const uint4 *>(a.x);
    const uint4 *src0 = t0 > 0 ? xs + (row0 - 1) * chunks
                               : (a.x_prev ? reinterpret_cast<const uint4 *>(a.x_prev) + static_cast<long long>(b) * chunks
                                           : nullptr);
    for (int i = tid; i < chunks; i += kThreads) {
        if (src0)
            cp_async16(rows + i, src0 + i);
        else
            rows[i] = make_uint4(0, 0, 0, 0);
    }
    const uint4 *src1 = xs + row0 * chunks;
    for (int i = tid; i < n * chunks; i += kThreads)
        cp_async16(rows + chunks + i, src1 + i);
    cp_async_commit_and_wait_all();
    __syncthreads();

    // ---- 1/RMS of every slot (for the normalisation of the conv input)
    if (a.gamma) {
        float sq[kSlots];
#pragma unroll
        for (int s = 0; s < kSlots; ++s)
            sq[s] = 0.f;
        for (int i = tid; i < chunks; i += kThreads) {
#pragma unroll
            for (int s = 0; s < kSlots; ++s) {
                if (s <= n) {
                    float f[8];
                    unpack8(rows[s * chunks + i], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        sq[s] = fmaf(f[e], f[e], sq[s]);
                }
            }
        }
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                sq[s] += __shfl_xor_sync(0xffffffffu, sq[s], off);
        }
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < kSlots; ++s)
                s_part[warp][s] = sq[s];
        }
        __syncthreads();
        if (tid <= n) {
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w)
                tot += s_part[w][tid];
            s_scale[tid] = inv_rms(tot, C, a.eps);
        }
        __syncthreads();
    }

    // ---- outputs: y_t = (base0 + dyn0_t) * u_t + (base1 + dyn1_t) * u_{t-1}, u = gamma * x / RMS(x)
    const int groups = C / a.G;
    const int chunks_per_group = a.G / 8;  // G is a multiple of 8: a chunk never straddles groups
    const uint4 *b0p = reinterpret_cast<const uint4 *>(a.base);
    const uint4 *b1p = b0p + chunks;
    const uint4 *gp = reinterpret_cast<const uint4 *>(a.gamma);
    uint4 *out = reinterpret_cast<uint4 *>(a.y) + row0 * chunks;
    const float *dyn = a.dyn + row0 * 2 * groups;
    for (int i = tid; i < chunks; i += kThreads) {
        const int g = i / chunks_per_group;
        // every row's corrections first: one memory latency per chunk, not one per row
        float k0d[kRowsPerCta], k1d[kRowsPerCta];
#pragma unroll
        for (int s = 0; s < kRowsPerCta; ++s) {
            k0d[s] = s < n ? __ldg(dyn + (2 * s) * groups + g) : 0.f;
            k1d[s] = s < n ? __ldg(dyn + (2 * s + 1) * groups + g) : 0.f;
        }
        float w0[8], w1[8], gg[8], up[8];
        unpack8(__ldg(b0p + i), w0);
        unpack8(__ldg(b1p + i), w1);
        unpack8(rows[i], up);
        if (a.gamma) {
            unpack8(__ldg(gp + i), gg);
            const float sc = s_scale[0];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                up[e] = up[e] * gg[e] * sc;
        }
#pragma unroll
        for (int s = 0; s < kRowsPerCta; ++s) {
            if (s >= n)
                break;
            float u[8];
            unpack8(rows[(s + 1) * chunks + i], u);
            if (a.gamma) {
                const float sc = s_scale[s + 1];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    u[e] = u[e] * gg[e] * sc;
            }
            float yv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                yv[e] = fmaf(w1[e] + k1d[s], up[e], (w0[e] + k0d[s]) * u[e]);
                up[e] = u[e];
            }
            __stcs(out + s * chunks + i,
                   make_uint4(pack2(yv[0], yv[1]), pack2(yv[2], yv[3]), pack2(yv[4], yv[5]), pack2(yv[6], yv[7])));
        }
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
