// gemm_tc.cu -- the selector head's LM head (and gate) on tcgen05 tensor cores.
//
// C[R, N] = A[R, K] . B[N, K]^T with A = hidden states (bf16, K = H) and B = the
// LM-head rows W_vocab (N = V) or the selector projection W_sel (N = D).
// "DFlash 2: Keep Drafting Parallel", section "A Lightweight Path Selector": the
// unary score of a candidate is the drafter's own logit; the gate H(h_t) is a
// projection of the same hidden state.
//
// Design (one CTA per SM, 192 threads, warp-specialised):
//   warp 0      TMA producer: 128-row tiles of A and up-to-256-row tiles of B,
//               64 K-elements (128 bytes, 128-byte swizzle) per stage, 4 stages.
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma (M=128, N<=256,
//               K=16 per instruction) into one of two 256-column accumulators.
//   warps 2-5   epilogue: tcgen05.ld the accumulator (thread = one row of C),
//               then either keep a per-row top-KP list in registers (the LM head:
//               full logits never reach global memory) or store float32 (gate).
// Work split: CTA (m, s) owns row tile m and a contiguous slice of C's columns
// (multiples of 16), walked in chunks of 256.  CTAs sharing a slice are launched
// next to each other, so W_vocab is read from HBM about once and re-read from L2.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace df2 {
namespace {

constexpr int BM = 128;                        // rows of C per tile = TMEM lanes
constexpr int BN = 256;                        // columns of C per chunk (MMA N, max)
constexpr int BK = 64;                         // K elements per stage: one 128-byte swizzle row
constexpr int UNIT = 16;                       // column granularity of slices and of MMA N
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;           // 16 KB
constexpr int B_BYTES = BN * BK * 2;           // 32 KB
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int STASH_STRIDE = 33;               // floats per epilogue thread (32 + 1 pad)
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = 1024 + STAGES * (A_BYTES + B_BYTES) + BAR_BYTES + BM * STASH_STRIDE * 4;

struct GemmArgs {
    int R, K, N;
    int row_tiles, n_split;
    float *pval;     // top-k mode: [R, n_split, KP]
    int32_t *pid;
    float *out;      // store mode: out[r * ldo + n]
    long long ldo;
    uint32_t *status;
};

// Waits without looking at the abort flag; used only to drain in-flight work after an abort.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity)
{
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kWaitTimeoutNs / 10)
            return;
}

template <int KP, bool kStore>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b_wide,
                   const __grid_constant__ CUtensorMap map_b_narrow, const GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + STAGES * B_BYTES);
    // bars: full[STAGES] | empty[STAGES] | tfull[2] | tempty[2] | drain
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *stash = reinterpret_cast<float *>(sB + STAGES * B_BYTES + BAR_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m_tile = blockIdx.x % args.row_tiles;
    const int split = blockIdx.x / args.row_tiles;
    const int units = (args.N + UNIT - 1) / UNIT;
    const int u0 = static_cast<int>(static_cast<long long>(split) * units / args.n_split);
    const int u1 = static_cast<int>(static_cast<long long>(split + 1) * units / args.n_split);
    const int col_begin = u0 * UNIT;
    const int col_end = min(u1 * UNIT, args.N);
    const int n_chunks = col_end > col_begin ? (col_end - col_begin + BN - 1) / BN : 0;
    const int kblocks = (args.K + BK - 1) / BK;

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4 * 32);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&map_a);
        prefetch_tmap(&map_b_wide);
        prefetch_tmap(&map_b_narrow);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int c = 0; c < n_chunks && ok; ++c) {
                const int c0 = col_begin + c * BN;
                const int nc = min(BN, col_end - c0);
                const int nmma = (nc + UNIT - 1) / UNIT * UNIT;
                const uint32_t tx = static_cast<uint32_t>(A_BYTES + nmma * BK * 2);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(stage), tx);
                    tma_load_2d(smem_u32(sA + stage * A_BYTES), &map_a, full_bar(stage), kb * BK, m_tile * BM);
                    const uint32_t b_dst = smem_u32(sB + stage * B_BYTES);
                    if (nmma == BN) {
                        tma_load_2d(b_dst, &map_b_wide, full_bar(stage), kb * BK, c0);
                    } else {
                        for (int q = 0; q < nmma / UNIT; ++q)
                            tma_load_2d(b_dst + q * UNIT * BK * 2, &map_b_narrow, full_bar(stage), kb * BK,
                                        c0 + q * UNIT);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA leaves
                const long long first = issued > STAGES ? issued - STAGES : 0;
                for (long long n = first; n < issued; ++n)
                    drain_wait(full_bar(static_cast<int>(n % STAGES)), static_cast<uint32_t>((n / STAGES) & 1));
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int c = 0; c < n_chunks && ok; ++c) {
                const int buf = c & 1;
                const uint32_t use = static_cast<uint32_t>(c >> 1);
                const int c0 = col_begin + c * BN;
                const int nc = min(BN, col_end - c0);
                const int nmma = (nc + UNIT - 1) / UNIT * UNIT;
                const uint32_t idesc = idesc_bf16_f32(BM, nmma);
                if (!mbar_wait(tempty_bar(buf), (use & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * A_BYTES);
                    const uint32_t b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16(d_tmem, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(b0 + kk * 32), idesc,
                                  (kb | kk) != 0 ? 1u : 0u);
                    umma_commit(empty_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok)
                    umma_commit(tfull_bar(buf));
            }
            if (!ok) {
                // every MMA issued so far must finish before TMEM is released
                umma_commit(drain_bar);
                drain_wait(drain_bar, 0);
            }
        }
    } else {
        // ---------------- epilogue: thread = one row of the 128-row tile
        const int q = warp & 3;  // TMEM lane quarter this warp may read
        const int row = m_tile * BM + q * 32 + lane;
        const bool row_ok = row < args.R;
        float *my_stash = stash + (q * 32 + lane) * STASH_STRIDE;
        ThreadTopK<KP> top;
        top.init();
        for (int c = 0; c < n_chunks; ++c) {
            const int buf = c & 1;
            const uint32_t use = static_cast<uint32_t>(c >> 1);
            const int c0 = col_begin + c * BN;
            const int nc = min(BN, col_end - c0);
            const bool ready = mbar_wait(tfull_bar(buf), use & 1u, abort_flag);
            if (!__all_sync(kFullMask, ready))
                break;
            tc_fence_after();
            for (int cb = 0; cb < (nc + 31) / 32; ++cb) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(buf * BN + cb * 32),
                                   r);
                tmem_wait_ld(r);
                const int base_col = c0 + cb * 32;
                const int valid = min(32, col_end - base_col);
                if constexpr (kStore) {
                    if (row_ok) {
                        float *dst = args.out + static_cast<long long>(row) * args.ldo + base_col;
                        if (valid == 32 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
                            for (int j = 0; j < 32; j += 4)
                                *reinterpret_cast<float4 *>(dst + j) =
                                    make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                                __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j < valid)
                                    dst[j] = __uint_as_float(r[j]);
                        }
                    }
                } else {
                    if (row_ok) {
                        const float thr = top.threshold();
                        uint32_t mask = 0;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            mask |= static_cast<uint32_t>(__uint_as_float(r[j]) > thr) << j;
                        if (valid < 32)
                            mask &= (1u << valid) - 1u;
                        if (mask) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                my_stash[j] = __uint_as_float(r[j]);
                            while (mask) {
                                const int j = __ffs(mask) - 1;
                                mask &= mask - 1u;
                                top.push_increasing_id(my_stash[j], base_col + j);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(tempty_bar(buf));
        }
        if constexpr (!kStore) {
            if (row_ok) {
                const long long base = (static_cast<long long>(row) * args.n_split + split) * KP;
#pragma unroll
                for (int s = 0; s < KP; ++s) {
                    args.pval[base + s] = top.v[s];
                    args.pid[base + s] = top.i[s];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag)
        atomicOr(args.status, kStatusTimeoutGemm);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Row-major bf16 [rows, K] tensor, boxes of 64 K-elements x box_rows rows, 128-byte swizzle.
cudaError_t make_map(CUtensorMap *map, const void *ptr, int K, int rows, int box_rows)
{
    auto encode = tensor_map_encoder();
    if (!encode)
        return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int KP, bool kStore>
cudaError_t launch(const void *A, const void *B, int R, int K, int N, GemmArgs args, int *n_split_out,
                   cudaStream_t stream)
{
    CUtensorMap ma, mbw, mbn;
    cudaError_t e;
    if ((e = make_map(&ma, A, K, R, BM)) != cudaSuccess)
        return e;
    if ((e = make_map(&mbw, B, K, N, BN)) != cudaSuccess)
        return e;
    if ((e = make_map(&mbn, B, K, N, UNIT)) != cudaSuccess)
        return e;
    auto kern = gemm_tc_kernel<KP, kStore>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES)) != cudaSuccess)
        return e;
    const int sms = device_sm_count();
    const int units = (N + UNIT - 1) / UNIT;
    args.R = R;
    args.K = K;
    args.N = N;
    args.row_tiles = (R + BM - 1) / BM;
    args.n_split = std::max(1, std::min({kMaxSplits, units, std::max(1, sms / args.row_tiles)}));
    if (n_split_out)
        *n_split_out = args.n_split;
    const dim3 grid(static_cast<unsigned>(args.row_tiles * args.n_split));
    gemm_tc_kernel<KP, kStore><<<grid, THREADS, SMEM_BYTES, stream>>>(ma, mbw, mbn, args);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_topk(const void *A, const void *B, int R, int K, int N, int KP, float *pval, int32_t *pid,
                             int *n_split_out, uint32_t *status, cudaStream_t stream)
{
    GemmArgs a{};
    a.pval = pval;
    a.pid = pid;
    a.status = status;
    switch (KP) {
    case 4: return launch<4, false>(A, B, R, K, N, a, n_split_out, stream);
    case 8: return launch<8, false>(A, B, R, K, N, a, n_split_out, stream);
    case 16: return launch<16, false>(A, B, R, K, N, a, n_split_out, stream);
    case 32: return launch<32, false>(A, B, R, K, N, a, n_split_out, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemm_store(const void *A, const void *B, int R, int K, int N, float *out, long long ldo,
                              uint32_t *status, cudaStream_t stream)
{
    GemmArgs a{};
    a.out = out;
    a.ldo = ldo;
    a.status = status;
    return launch<4, true>(A, B, R, K, N, a, nullptr, stream);
}

}  // namespace df2
