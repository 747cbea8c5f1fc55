// lattice.cuh -- device steps shared by the fused finish kernel and the stage kernels:
// one draft position's row of the k x k transition lattice, and the greedy walk.
//
// "DFlash 2: Keep Drafting Parallel", section "A Lightweight Path Selector":
//   S_t(a, b) = U_t(b) + < A(a) (.) H(h_t), B(b) >
// with a among the previous position's candidates (the last verified token at the
// first position) and b among the current ones; greedy follows the best successor from
// the last verified token.  "DFlash2 Lands in llama.cpp", sections "The Central
// Insight" (edge = unary + pairwise) and "What llama.cpp Actually Builds for the
// Selector" (codebook gathers, rows packed as candidate ids followed by transition
// scores, walk with predecessor = anchor).
#pragma once

#include <cstdint>

#include "topk.cuh"

namespace df2 {

constexpr int kLatticeThreads = 256;

__device__ __forceinline__ int clamp_id(int id, int V)
{
    return static_cast<unsigned>(id) < static_cast<unsigned>(V) ? id : 0;
}

// Elements between consecutive gathered codebook rows in shared memory: D plus 16 bytes, so
// that the eight rows one tensor-core fragment load touches start in eight different groups of
// four banks (with a stride of D alone every row starts in bank 0 whenever D is a multiple of 64).
__host__ __device__ constexpr int lattice_row_stride(int D)
{
    return D + 8;
}

// Dynamic shared memory of one lattice row: the gate row as float [D], then the gathered
// codebook rows as bf16: up to k predecessor rows A(prev_i) followed by k rows B(cand_j), each
// lattice_row_stride(D) elements apart.
__host__ __device__ constexpr size_t lattice_smem_bytes(int k, int D)
{
    return sizeof(float) * static_cast<size_t>(D) +
           sizeof(uint16_t) * 2 * static_cast<size_t>(k) * lattice_row_stride(D);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// float32 -> tf32 (round to nearest, ties away), as the bit pattern an mma operand takes.
__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// D (16 x 8, float32) += A (16 x 8, tf32, row-major) . B (8 x 8, tf32, column-major), one warp.
// Fragments (g = lane / 4, c = lane % 4): a = A[g][c], A[g+8][c], A[g][c+4], A[g+8][c+4];
// b = B[c][g], B[c+4][g]; d = D[g][2c], D[g][2c+1], D[g+8][2c], D[g+8][2c+1].
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Rows of the lattice whose scores come from warp-level tensor-core tiles: 9 to 16
// predecessors and candidates (one 16 x 16 tile), with room in the gathered-row buffer for
// four 16 x 17 float partial tiles once the products are done.  Measured on GB300: 24.5 ->
// 23.0 us after the LM head at 512 rows (k = 16); at k = 8 the scalar path's latency is as
// low (12.6 vs 13.1 us at batch 1), so smaller k keep it.
__host__ __device__ constexpr bool lattice_uses_mma(int k, int n_prev, int D)
{
    return k > 8 && k <= 16 && n_prev == k && 2 * k * D * 2 >= 4 * 16 * 17 * 4;
}

// Copies the gate row g[0..D) into shared memory (threads [first, first + count) of the CTA).
__device__ __forceinline__ void load_gate_row(float *sg, const float *__restrict__ g, int D, int first, int count)
{
    for (int i = threadIdx.x - first; i >= 0 && i < D / 4; i += count)
        reinterpret_cast<float4 *>(sg)[i] = reinterpret_cast<const float4 *>(g)[i];
}

// Sum of v[j] over the 32 lanes, left in lane j for j < KP (KP a power of two <= 32):
// a reduce-scatter butterfly, KP - 1 + log2(32 / KP) shuffles instead of 5 * KP.
template <int KP>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[KP])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int h = KP / 2; h >= 1; h >>= 1) {
        const bool upper = (lane & h) != 0;
#pragma unroll
        for (int q = 0; q < h; ++q) {
            const float send = upper ? v[q] : v[q + h];
            const float keep = upper ? v[q + h] : v[q];
            v[q] = keep + __shfl_xor_sync(kFullMask, send, h);
        }
    }
    float x = v[0];
#pragma unroll
    for (int o = KP; o < 32; o <<= 1)
        x += __shfl_xor_sync(kFullMask, x, o);
    return x;  // lane l holds the total of index l & (KP - 1)
}

// Writes packed row r of the lattice: [cand ids | unary_j + <A(prev_i) (.) g, B(cand_j)>].
// prev[0..n_prev) are the predecessor tokens (n_prev = 1 at t = 0: the anchor, whose
// scores are copied to all k predecessor rows), cand/unary the current candidates, and
// sg the gate row, already in shared memory at the start of `smem`.
// If `best` is not null, best[i] receives the walk's choice from predecessor row i:
// the index of the row's maximum, lowest index on ties.  If `mirror` is not null the row is
// written there too (a row of a caller's page-locked host buffer).
// All CTA threads call it; it starts and ends with __syncthreads().
template <int KP>
__device__ void lattice_row(int k, int D, int n_prev, const int *s_prev, const int *s_cand, const float *s_unary,
                            const uint16_t *__restrict__ pred_cb, const uint16_t *__restrict__ succ_cb,
                            uint8_t *smem, float *__restrict__ out, int32_t *__restrict__ best = nullptr,
                            float *__restrict__ mirror = nullptr)
{
    constexpr int kBatch = 8;  // 16-byte gathers in flight per thread
    const float *sg = reinterpret_cast<const float *>(smem);                  // [D] gate
    uint16_t *rows = reinterpret_cast<uint16_t *>(smem + sizeof(float) * D);  // [n_prev + k][ld]
    const int ld = lattice_row_stride(D);
    __syncthreads();
    const int chunks = D / 8;  // 16-byte chunks of bf16 per codebook row
    const int total = (n_prev + k) * chunks;
    for (int base = threadIdx.x; base < total; base += blockDim.x * kBatch) {
        uint4 w[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int idx = base + q * blockDim.x;
            if (idx < total) {
                const int row = idx / chunks;
                const int c8 = idx - row * chunks;
                const uint16_t *src = row < n_prev ? pred_cb + static_cast<long long>(s_prev[row]) * D
                                                   : succ_cb + static_cast<long long>(s_cand[row - n_prev]) * D;
                w[q] = __ldg(reinterpret_cast<const uint4 *>(src) + c8);
            }
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int idx = base + q * blockDim.x;
            if (idx < total) {
                const int row = idx / chunks;
                reinterpret_cast<uint4 *>(rows + row * ld)[idx - row * chunks] = w[q];
            }
        }
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_warps = blockDim.x >> 5;
    // writes score row i (lane j: unary_j + tot) and, if asked, the walk's choice from it
    auto emit_row = [&](int i, float tot) {
        const float s = lane < k ? s_unary[lane] + tot : -INFINITY;
        if (lane < k) {
            if (n_prev == 1) {
                for (int ii = 0; ii < k; ++ii) {
                    out[k + ii * k + lane] = s;
                    if (mirror)
                        mirror[k + ii * k + lane] = s;
                }
            } else {
                out[k + i * k + lane] = s;
                if (mirror)
                    mirror[k + i * k + lane] = s;
            }
        }
        if (best) {
            float x = s;
            int j = lane < k ? lane : 0x7fffffff;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ox = __shfl_xor_sync(kFullMask, x, off);
                const int oj = __shfl_xor_sync(kFullMask, j, off);
                const bool take = ranks_before(ox, oj, x, j);
                x = take ? ox : x;
                j = take ? oj : j;
            }
            if (lane == 0)
                best[i] = j;
        }
    };

    if (KP > 8 && KP <= 16 && lattice_uses_mma(k, n_prev, D)) {  // k <= KP: no tile below KP = 16
        // Scores as one 16 x 16 tile of warp-level tf32 tensor-core products, the K = D axis
        // split over up to 4 warps: A = A(prev) (.) g is split into tf32 high and low parts
        // and B(cand) is bf16 (exact in tf32), so the two products keep float32 accuracy.
        // The order of the K axis inside an 8-wide step is free as long as A and B agree:
        // fragment columns c and c + 4 take d = k0 + 2c and k0 + 2c + 1, the two halves of one
        // 32-bit word of each row, so a thread reads one word per row and step.
        const int mw = n_warps < 4 ? n_warps : 4;
        const int gq = lane >> 2, cq = lane & 3;
        const int ld2 = ld / 2;
        float acc[2][2][4] = {};  // [high / low part][candidate tile][fragment]
        if (warp < mw) {
            const bool va0 = gq < n_prev, va1 = gq + 8 < n_prev;
            const bool vb0 = gq < k, vb1 = gq + 8 < k;
            const uint32_t *rw = reinterpret_cast<const uint32_t *>(rows);
            const uint32_t *pa0 = rw + (va0 ? gq : 0) * ld2;
            const uint32_t *pa1 = rw + (va1 ? gq + 8 : 0) * ld2;
            const uint32_t *pb0 = rw + (n_prev + (vb0 ? gq : 0)) * ld2;
            const uint32_t *pb1 = rw + (n_prev + (vb1 ? gq + 8 : 0)) * ld2;
            const float2 *g2 = reinterpret_cast<const float2 *>(sg);
            for (int k0 = warp * 8; k0 < D; k0 += mw * 8) {
                const int w = k0 / 2 + cq;
                const float2 gg = g2[w];
                const uint32_t a0 = va0 ? pa0[w] : 0u, a1 = va1 ? pa1[w] : 0u;
                float p[4];
                p[0] = bf16_lo(a0) * gg.x;
                p[1] = bf16_lo(a1) * gg.x;
                p[2] = bf16_hi(a0) * gg.y;
                p[3] = bf16_hi(a1) * gg.y;
                uint32_t ahi[4], alo[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    ahi[q] = to_tf32(p[q]);
                    alo[q] = to_tf32(p[q] - __uint_as_float(ahi[q]));
                }
                const uint32_t b0 = vb0 ? pb0[w] : 0u, b1 = vb1 ? pb1[w] : 0u;
                const uint32_t b00 = b0 << 16, b01 = b0 & 0xFFFF0000u;
                const uint32_t b10 = b1 << 16, b11 = b1 & 0xFFFF0000u;
                mma_tf32_16x8x8(acc[0][0], ahi, b00, b01);
                mma_tf32_16x8x8(acc[0][1], ahi, b10, b11);
                mma_tf32_16x8x8(acc[1][0], alo, b00, b01);
                mma_tf32_16x8x8(acc[1][1], alo, b10, b11);
            }
        }
        __syncthreads();  // every warp is done with the gathered rows: reuse them for the partial tiles
        float(*part)[16][17] = reinterpret_cast<float(*)[16][17]>(rows);
        if (warp < mw) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int col = nt * 8 + 2 * cq;
                part[warp][gq][col] = acc[0][nt][0] + acc[1][nt][0];
                part[warp][gq][col + 1] = acc[0][nt][1] + acc[1][nt][1];
                part[warp][gq + 8][col] = acc[0][nt][2] + acc[1][nt][2];
                part[warp][gq + 8][col + 1] = acc[0][nt][3] + acc[1][nt][3];
            }
        }
        __syncthreads();
        for (int i = warp; i < n_prev; i += n_warps) {
            float tot = 0.f;
            if (lane < k)
                for (int w = 0; w < mw; ++w)
                    tot += part[w][i][lane];
            emit_row(i, tot);
        }
    } else {
        // Each warp takes two predecessor rows at a time; lanes stride over pairs of d.
        const uint32_t *succ2 = reinterpret_cast<const uint32_t *>(rows + n_prev * ld);  // [k][ld/2]
        const float2 *g2 = reinterpret_cast<const float2 *>(sg);
        const int D2 = D / 2, ld2 = ld / 2;
        for (int i0 = 2 * warp; i0 < n_prev; i0 += 2 * n_warps) {
            const bool two = i0 + 1 < n_prev;
            const uint32_t *a0 = reinterpret_cast<const uint32_t *>(rows + i0 * ld);
            const uint32_t *a1 = two ? a0 + ld2 : a0;
            float acc0[KP], acc1[KP];
#pragma unroll
            for (int j = 0; j < KP; ++j) {
                acc0[j] = 0.f;
                acc1[j] = 0.f;
            }
            for (int d2 = lane; d2 < D2; d2 += 32) {
                const float2 gg = g2[d2];
                const uint32_t p0 = a0[d2], p1 = a1[d2];
                const float x0 = bf16_lo(p0) * gg.x, y0 = bf16_hi(p0) * gg.y;  // A(prev) (.) g
                const float x1 = bf16_lo(p1) * gg.x, y1 = bf16_hi(p1) * gg.y;
#pragma unroll
                for (int j = 0; j < KP; ++j) {
                    if (j < k) {
                        const uint32_t sb = succ2[j * ld2 + d2];
                        const float sl = bf16_lo(sb), sh = bf16_hi(sb);
                        acc0[j] = fmaf(y0, sh, fmaf(x0, sl, acc0[j]));
                        acc1[j] = fmaf(y1, sh, fmaf(x1, sl, acc1[j]));
                    }
                }
            }
            const float tot0 = warp_reduce_scatter<KP>(acc0);
            const float tot1 = warp_reduce_scatter<KP>(acc1);
            emit_row(i0, tot0);
            if (two)
                emit_row(i0 + 1, tot1);
        }
    }
    if (threadIdx.x < k) {
        out[threadIdx.x] = static_cast<float>(s_cand[threadIdx.x]);
        if (mirror)
            mirror[threadIdx.x] = static_cast<float>(s_cand[threadIdx.x]);
    }
    __syncthreads();
}

// Greedy walk of one sequence by one warp over its T packed rows (row stride `width`
// floats): j_0 = argmax of predecessor row 0 at t = 0, then j_t = argmax of row
// j_(t-1); ties go to the lowest candidate index.  kGlobal reads through L2 (rows
// written by other CTAs of the same grid); otherwise `rows` is in shared memory.
template <bool kGlobal>
__device__ __forceinline__ void walk_rows(int T, int k, long long width, const float *rows, int32_t *draft)
{
    const int lane = threadIdx.x & 31;
    int jp = 0;
    for (int t = 0; t < T; ++t) {
        const float *row = rows + static_cast<long long>(t) * width;
        const float *p = row + k + jp * k + lane;
        float x = -INFINITY;
        if (lane < k)
            x = kGlobal ? __ldcg(p) : *p;
        int j = lane < k ? lane : 0x7fffffff;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ox = __shfl_xor_sync(kFullMask, x, off);
            const int oj = __shfl_xor_sync(kFullMask, j, off);
            const bool take = ranks_before(ox, oj, x, j);
            x = take ? ox : x;
            j = take ? oj : j;
        }
        jp = j;
        if (lane == 0)
            draft[t] = static_cast<int32_t>(kGlobal ? __ldcg(row + jp) : row[jp]);
    }
}

// One sequence's walk with the chosen transition's softmax confidence, the p_min early stop
// and, when `uniforms` is given, inverse-CDF sampling from the same scores; one warp.
// "DFlash2 Lands in llama.cpp", section "p_min Means Something Different Under DFlash2": the
// confidence is the softmax of the current transition row at the chosen candidate, and the
// walk stops when it falls below p_min.  "DFlash 2: Keep Drafting Parallel", section "A
// Lightweight Path Selector": sampling draws from the same scores.
// rows: the sequence's T packed rows (stride `width` floats); uniforms, draft, confidence:
// its T entries (uniforms and confidence may be null); n_draft: its count (may be null);
// draft_mirror: a second copy of the draft (may be null).  kGlobal reads the rows through L2
// (rows written by other CTAs of the same grid).
template <bool kGlobal>
__device__ __forceinline__ void walk_sample_rows(int T, int k, long long width, const float *rows, float temperature,
                                                 float p_min, const float *uniforms, int32_t *draft,
                                                 int32_t *draft_mirror, int32_t *n_draft, float *confidence)
{
    const int lane = threadIdx.x & 31;
    int jp = 0;
    int n = T;
    bool stopped = false;
    for (int t = 0; t < T; ++t) {
        if (stopped) {
            if (lane == 0) {
                draft[t] = -1;
                if (draft_mirror)
                    draft_mirror[t] = -1;
                if (confidence)
                    confidence[t] = 0.f;
            }
            continue;
        }
        const float *row = rows + static_cast<long long>(t) * width;
        const float *px = row + k + jp * k + lane;
        const float x = lane < k ? (kGlobal ? __ldcg(px) : *px) : -INFINITY;
        // argmax (first maximum) and maximum
        float mx = x;
        int jm = lane < k ? lane : 0x7fffffff;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ox = __shfl_xor_sync(kFullMask, mx, off);
            const int oj = __shfl_xor_sync(kFullMask, jm, off);
            const bool take = ranks_before(ox, oj, mx, jm);
            mx = take ? ox : mx;
            jm = take ? oj : jm;
        }
        const float e = lane < k ? expf((x - mx) / temperature) : 0.f;
        float pre = e;  // inclusive prefix sum over lanes
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(kFullMask, pre, off);
            if (lane >= off)
                pre += o;
        }
        const float z = __shfl_sync(kFullMask, pre, 31);
        int pick = jm;
        if (uniforms) {
            const float target = uniforms[t] * z;
            const unsigned over = __ballot_sync(kFullMask, lane < k && pre > target);
            const unsigned live = __ballot_sync(kFullMask, e > 0.f);
            pick = over ? __ffs(over) - 1 : 31 - __clz(live);
        }
        const float p = __shfl_sync(kFullMask, e, pick) / z;
        if (lane == 0 && confidence)
            confidence[t] = p;
        if (p < p_min) {
            stopped = true;
            n = t;
            if (lane == 0) {
                draft[t] = -1;
                if (draft_mirror)
                    draft_mirror[t] = -1;
            }
        } else {
            jp = pick;
            if (lane == 0) {
                const int32_t id = static_cast<int32_t>(kGlobal ? __ldcg(row + pick) : row[pick]);
                draft[t] = id;
                if (draft_mirror)
                    draft_mirror[t] = id;
            }
        }
    }
    if (lane == 0 && n_draft)
        *n_draft = n;
}

}  // namespace df2
