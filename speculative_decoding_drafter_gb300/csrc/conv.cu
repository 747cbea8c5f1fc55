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
// Work is cut into tiles of up to kRows consecutive rows of one block, one tile per CTA.
// A CTA stages its rows, the row before the first (the block's previous row, the last
// verified token, or zeros) and its corrections in shared memory with one batch of
// cp.async copies, so each row is read from DRAM once; several CTAs per SM keep copies
// in flight while others compute.  (On GB300 this beat a persistent CTA that
// double-buffers its tiles, and a variant that keeps the rows in registers.)  Each thread owns
// 16-byte channel chunks across the tile's rows: the static taps and gamma of a chunk are
// unpacked once and serve every row, and a row's normalised input, kept in registers, is
// the next row's predecessor term.  The RMS of each staged row comes from a CTA-wide
// reduction.  HBM-bound: per row 2C bytes read, 2C written, C/G*8 bytes of corrections.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace df2 {
namespace {

constexpr int kThreads = 256;

struct ConvArgs {
    int B, T, C, G;
    int tiles_per_block;  // ceil(T / kRows)
    int n_tiles;          // B * tiles_per_block
    const uint16_t *x;
    const uint16_t *x_prev;
    const uint16_t *base;
    const float *dyn;
    const uint16_t *gamma;
    float eps;
    uint16_t *y;
    int dyn_vec4;  // corrections staged with 16-byte copies (aligned, even C/G)
};

__device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Pairs of fp32 in one 64-bit register for the packed f32x2 arithmetic of sm_100-class
// SMs: each lane is rounded exactly like the scalar instruction, at half the issue cost.
__device__ __forceinline__ uint64_t f2(float lo, float hi)
{
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}

__device__ __forceinline__ float2 f2_split(uint64_t v)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Eight bf16 (one 16-byte chunk) widened exactly to four fp32 pairs, in channel order.
__device__ __forceinline__ void unpack8x2(const uint4 &v, uint64_t (&p)[4])
{
    p[0] = f2(lo(v.x), hi(v.x));
    p[1] = f2(lo(v.y), hi(v.y));
    p[2] = f2(lo(v.z), hi(v.z));
    p[3] = f2(lo(v.w), hi(v.w));
}

__device__ __forceinline__ uint32_t pack2x(uint64_t v)
{
    const float2 f = f2_split(v);
    return pack2(f.x, f.y);
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(
                     smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gmem_src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(
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


__host__ __device__ constexpr size_t round16(size_t x) { return (x + 15) / 16 * 16; }

// One buffer: (kRows + 1) staged rows of C bf16, then kRows rows of 2 * C/G corrections.
template <int kRows>
__host__ __device__ constexpr size_t rows_bytes(int C)
{
    return round16(static_cast<size_t>(kRows + 1) * C * 2);
}

template <int kRows>
__host__ __device__ constexpr size_t buffer_bytes(int C, int G)
{
    return rows_bytes<kRows>(C) + round16(static_cast<size_t>(kRows) * 2 * (C / G) * sizeof(float));
}

struct TileRange {
    long long row0;  // global index of the tile's first row
    int t0, n, b;
};

template <int kRows>
__device__ __forceinline__ TileRange tile_range(const ConvArgs &a, int tile)
{
    TileRange r;
    r.b = tile / a.tiles_per_block;
    r.t0 = (tile - r.b * a.tiles_per_block) * kRows;
    r.n = min(kRows, a.T - r.t0);
    r.row0 = static_cast<long long>(r.b) * a.T + r.t0;
    return r;
}

// Enqueues this thread's share of the copies of `tile` into `buf` (one cp.async group is
// committed by the caller); slot 0 of a block's first tile without x_prev is zero-filled.
template <int kRows>
__device__ __forceinline__ void stage_tile(const ConvArgs &a, int tile, uint8_t *buf)
{
    const TileRange tr = tile_range<kRows>(a, tile);
    const int chunks = a.C / 8;
    const int groups = a.C / a.G;
    uint4 *rows = reinterpret_cast<uint4 *>(buf);
    float *dyn_s = reinterpret_cast<float *>(buf + rows_bytes<kRows>(a.C));
    const uint4 *xs = reinterpret_cast<const uint4 *>(a.x);
    const uint4 *src0 = tr.t0 > 0 ? xs + (tr.row0 - 1) * chunks
                                  : (a.x_prev ? reinterpret_cast<const uint4 *>(a.x_prev) +
                                                    static_cast<long long>(tr.b) * chunks
                                              : nullptr);
    for (int i = threadIdx.x; i < chunks; i += kThreads) {
        if (src0)
            cp_async16(rows + i, src0 + i);
        else
            rows[i] = make_uint4(0, 0, 0, 0);
    }
    const uint4 *src1 = xs + tr.row0 * chunks;
    for (int i = threadIdx.x; i < tr.n * chunks; i += kThreads)
        cp_async16(rows + chunks + i, src1 + i);
    const float *dsrc = a.dyn + tr.row0 * 2 * groups;
    if (a.dyn_vec4) {
        for (int i = threadIdx.x; i < tr.n * groups / 2; i += kThreads)
            cp_async16(reinterpret_cast<uint4 *>(dyn_s) + i, reinterpret_cast<const uint4 *>(dsrc) + i);
    } else {
        for (int i = threadIdx.x; i < tr.n * 2 * groups; i += kThreads)
            cp_async4(dyn_s + i, dsrc + i);
    }
}

// Computes and stores the rows of `tile` from `buf`.  All CTA threads call it.
template <int kRows>
__device__ __forceinline__ void compute_tile(const ConvArgs &a, int tile, const uint8_t *buf,
                                             float (*s_part)[kRows + 1], float *s_scale)
{
    constexpr int kSlots = kRows + 1;
    const TileRange tr = tile_range<kRows>(a, tile);
    const int n = tr.n;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int C = a.C;
    const int chunks = C / 8;
    const int groups = C / a.G;
    const uint4 *rows = reinterpret_cast<const uint4 *>(buf);
    const float *dyn_s = reinterpret_cast<const float *>(buf + rows_bytes<kRows>(C));

    // ---- 1/RMS of every slot (for the normalisation of the conv input)
    if (a.gamma) {
        uint64_t acc[kSlots];
#pragma unroll
        for (int s = 0; s < kSlots; ++s)
            acc[s] = 0ull;  // (+0, +0)
        for (int i = tid; i < chunks; i += kThreads) {
#pragma unroll
            for (int s = 0; s < kSlots; ++s) {
                if (s <= n) {
                    uint64_t f[4];
                    unpack8x2(rows[s * chunks + i], f);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        acc[s] = fma2(f[e], f[e], acc[s]);
                }
            }
        }
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
            const float2 h = f2_split(acc[s]);
            float sq = h.x + h.y;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
            if (lane == 0)
                s_part[warp][s] = sq;
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
    const int chunks_per_group = a.G / 8;  // G is a multiple of 8: a chunk never straddles groups
    const uint4 *b0p = reinterpret_cast<const uint4 *>(a.base);
    const uint4 *b1p = b0p + chunks;
    const uint4 *gp = reinterpret_cast<const uint4 *>(a.gamma);
    uint4 *out = reinterpret_cast<uint4 *>(a.y) + tr.row0 * chunks;
    for (int i = tid; i < chunks; i += kThreads) {
        const int g = i / chunks_per_group;
        uint64_t w0[4], w1[4], gg[4], up[4];
        unpack8x2(__ldg(b0p + i), w0);
        unpack8x2(__ldg(b1p + i), w1);
        unpack8x2(rows[i], up);
        if (a.gamma) {
            unpack8x2(__ldg(gp + i), gg);
            const uint64_t sc = f2(s_scale[0], s_scale[0]);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                up[e] = mul2(mul2(up[e], gg[e]), sc);
        }
#pragma unroll
        for (int s = 0; s < kRows; ++s) {
            if (s >= n)
                break;
            uint64_t u[4];
            unpack8x2(rows[(s + 1) * chunks + i], u);
            if (a.gamma) {
                const uint64_t sc = f2(s_scale[s + 1], s_scale[s + 1]);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    u[e] = mul2(mul2(u[e], gg[e]), sc);
            }
            const float k0d = dyn_s[(2 * s) * groups + g];
            const float k1d = dyn_s[(2 * s + 1) * groups + g];
            const uint64_t c0 = f2(k0d, k0d), c1 = f2(k1d, k1d);
            uint32_t yv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                yv[e] = pack2x(fma2(add2(w1[e], c1), up[e], mul2(add2(w0[e], c0), u[e])));
                up[e] = u[e];
            }
            __stcs(out + s * chunks + i, make_uint4(yv[0], yv[1], yv[2], yv[3]));
        }
    }
}

template <int kRows>
__global__ void __launch_bounds__(kThreads) dynamic_conv_kernel(const ConvArgs a)
{
    extern __shared__ __align__(16) uint8_t smem[];  // one tile buffer
    __shared__ float s_part[kThreads / 32][kRows + 1];
    __shared__ float s_scale[kRows + 1];
    // Launched as a programmatic dependent: the next launch's CTAs may take the slots this
    // grid's last wave frees, and each waits for the grid before it before reading inputs or
    // writing the output (a back-to-back call writes the same rows).
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    griddep_wait();
    stage_tile<kRows>(a, blockIdx.x, smem);
    cp_async_commit_and_wait_all();
    __syncthreads();  // every thread's copies are visible
    compute_tile<kRows>(a, blockIdx.x, smem, s_part, s_scale);
}

template <int kRows>
bool conv_fits(int C, int G)
{
    return buffer_bytes<kRows>(C, G) <= 200 * 1024;
}

template <int kRows>
cudaError_t launch_rows(ConvArgs a, cudaStream_t stream)
{
    a.tiles_per_block = (a.T + kRows - 1) / kRows;
    a.n_tiles = a.B * a.tiles_per_block;
    const size_t smem = buffer_bytes<kRows>(a.C, a.G);
    const cudaError_t e = cudaFuncSetAttribute(dynamic_conv_kernel<kRows>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.n_tiles));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, dynamic_conv_kernel<kRows>, a);
    if (le != cudaSuccess)
        return le;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dynamic_conv(int B, int T, int C, int G, const uint16_t *x, const uint16_t *x_prev,
                                const uint16_t *base, const float *dyn, const uint16_t *gamma, float eps, uint16_t *y,
                                cudaStream_t stream)
{
    const int groups = C / G;
    const int vec4 = (reinterpret_cast<uintptr_t>(dyn) % 16 == 0) && (groups % 2 == 0);
    ConvArgs a{B, T, C, G, 0, 0, x, x_prev, base, dyn, gamma, eps, y, vec4};
    if (conv_fits<4>(C, G))
        return launch_rows<4>(a, stream);
    return launch_rows<2>(a, stream);
}

}  // namespace df2
