// gemm_tc.cu -- the selector head's LM head and gate on tcgen05 tensor cores.
//
// C[R, n] = A[R, K] . B[n, K]^T with A = hidden states (bf16, K = H).  One launch covers
// two column segments of C:
//   top-k segment  B = W_vocab (n = V): "DFlash 2: Keep Drafting Parallel", section "A
//                  Lightweight Path Selector" -- the unary score of a candidate is the
//                  drafter's own logit; only a per-row top-k of these columns is kept;
//   store segment  B = W_sel (n = D): the context gate H(h_t), a projection of the same
//                  hidden state, stored as float32.
// Either segment may be empty (the stage entry points use the store segment alone).
//
// Design (one CTA per SM, 64 + 128 * mt threads, warp-specialised; mt = row tiles per CTA):
//   warp 0      TMA producer: per stage, kbs consecutive K-blocks of 64 elements (128
//               bytes, 128-byte swizzle) of mt A boxes of the live rows (<= 128 each) and
//               of a chunk of bn (128 or 256) rows of B.  Up to 64 rows: bn = 128, kbs = 2
//               (each W row read in 256-byte runs); beyond: bn = 256, kbs = 1.
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma (M=128, N<=bn, K=16 per
//               instruction), one per row tile, into bn-column accumulators: two buffers
//               per tile when they fit (mt = 1), one when two tiles fill TMEM (mt = 2).
//   warps 2..   epilogue, four warps per row tile: tcgen05.ld the accumulator (thread =
//               one row of C), then keep a per-row top-KP list in registers (full logits
//               never reach global memory) or store float32.
// Two row tiles per CTA (beyond 128 rows) halve what an SM takes in per MMA flop: 64 KB of
// A and B per 2 x 128x256x64 block instead of 48 KB per 128x256x64, which is what limits
// the tensor pipe when all SMs stream.
// CTA pairs (129 to 1024 rows): the two row tiles go to a cluster of two CTAs on two SMs
// instead.  The even CTA issues tcgen05.mma.cta_group::2 (M = 256); each CTA loads its
// 128-row A tile and a 128-row box of B at its half of the chunk, both completing on the
// even CTA's barriers, and the commits arrive on both CTAs' barriers.  An SM then takes in
// the same bytes per flop as with two tiles in one CTA, but holds one 256-column
// accumulator per buffer, so the epilogue runs under the next chunk's MMAs.  A stage
// carries two K-blocks, each operand as one box of a 3-D view of the matrix (64 elements
// of K x rows x K-block): the feed is bound by the number of TMA operations, and one
// K-block per stage (four operations per 128x256x64 instead of two) was slower than two
// tiles in one CTA.
// Work split: CTA (g, s) owns row group g (mt consecutive row tiles) and a contiguous
// slice of the columns of both segments (multiples of 16), walked in chunks of <= 256
// that never straddle the segment boundary.  CTAs sharing a slice are launched next to
// each other, so W_vocab is read from HBM about once and re-read from L2 by the other
// row groups.
// Shared bound (two-tile mode, where the MMA waits for the epilogue): each row has KP
// slots; after each chunk CTA s raises slot s mod KP to the best logit its slice has
// given so far (atomicMax on an order-preserving key).  The KP slots then hold logits of
// KP distinct columns, so their minimum is a lower bound on the row's KP-th best logit,
// and every CTA's epilogue skips values below it.  A value below the bound is outranked
// by at least KP others and cannot reach the row's top-k; every value of the top-k still
// reaches its slice's list, so the merged top-k is exactly the same.  The last CTA of each
// row group returns its rows' slots to zero.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cfloat>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace df2 {
namespace {

constexpr int BM = 128;                        // rows of C per tile = TMEM lanes
constexpr int BN = 256;                        // columns of C per chunk (MMA N, max)
constexpr int BK = 64;                         // K elements per K-block: one 128-byte swizzle row
constexpr int UNIT = 16;                       // column granularity of slices and of MMA N
constexpr int MAX_STAGES = 8;
constexpr int A_TILE_BYTES = BM * BK * 2;      // what one MMA reads of A: 16 KB
constexpr int TMEM_COLS = 2 * BN;
constexpr int STASH_STRIDE = 33;               // floats per epilogue thread (32 + 1 pad)
constexpr int BAR_BYTES = 256;
constexpr int STASH_TILE_BYTES = BM * STASH_STRIDE * 4;
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr int kWarmStages = 16;                // stages of W brought into L2 before a dependent launch waits

struct GemmArgs {
    int R, K;
    int n_topk;       // columns of the top-k segment
    int n_topk_pad;   // rounded up to UNIT: start of the store segment in the column space
    int n_store;      // columns of the store segment
    int row_tiles, n_split;
    int mt;           // row tiles per CTA (1 or 2)
    int pair;         // CTA pairs (clusters of two): one row tile per CTA, M = 256 per pair
    int row_groups;   // ceil(row_tiles / mt); pairs: row_tiles rounded up to even
    int n_bufs;       // accumulator buffers per row tile (2, or 1 when mt tiles fill TMEM)
    int stages;       // pipeline depth
    int bn;           // columns per chunk (128 or 256)
    int kbs;          // K-blocks per stage
    int a_bytes;      // bytes of one A box (live rows x 128), a multiple of 1024
    float *pval;      // top-k lists [R, n_split, KP]
    int32_t *pid;
    float *out;       // store segment: out[r * ldo + n]
    long long ldo;
    uint32_t *bound;        // [R, KP] slot keys of the shared bound (null: each CTA alone)
    unsigned *group_done;   // [row_groups] CTAs finished per row group
    uint32_t *status;
    int dependent;    // launched as a programmatic dependent of the grid before it
};

// Order-preserving map of a float to an unsigned key (larger float, larger key); every key
// of a float is above 0, which marks an empty slot.
__device__ __forceinline__ uint32_t order_key(float x)
{
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// The shared bound of one row as a filter threshold: below the minimum slot by at least
// one float32 step (values equal to the bound must still pass), or -inf while a slot is empty.
template <int KP>
__device__ __forceinline__ float shared_threshold(const uint32_t *slots)
{
    uint32_t m = 0xffffffffu;
#pragma unroll
    for (int q = 0; q < KP / 4; ++q) {
        const uint4 k4 = __ldcg(reinterpret_cast<const uint4 *>(slots) + q);
        m = min(m, min(min(k4.x, k4.y), min(k4.z, k4.w)));
    }
    if (m == 0u)
        return -INFINITY;
    const float t = key_value(m);
    return t - (fabsf(t) * 0x1p-22f + FLT_MIN);
}

// One chunk of a CTA's column slice.
struct Chunk {
    int c0;       // first column in the joint column space
    int n;        // columns (a multiple of UNIT, <= BN)
    bool store;   // store segment?
    int b_row;    // first row of the segment's B matrix
    int valid;    // columns of the chunk that exist in the segment (<= n)
};

struct Slice {
    int a0, a1;   // top-k segment part [a0, a1)
    int b0, b1;   // store segment part [b0, b1)
    int n0, n1;   // chunks in each part
};

__device__ __forceinline__ Slice slice_of(const GemmArgs &g, int split)
{
    const int total_units = (g.n_topk_pad + g.n_store + UNIT - 1) / UNIT;
    const int u0 = static_cast<int>(static_cast<long long>(split) * total_units / g.n_split);
    const int u1 = static_cast<int>(static_cast<long long>(split + 1) * total_units / g.n_split);
    Slice s;
    const int c_begin = u0 * UNIT, c_end = u1 * UNIT;
    s.a0 = c_begin;
    s.a1 = min(c_end, g.n_topk_pad);
    s.b0 = max(c_begin, g.n_topk_pad);
    s.b1 = c_end;
    s.n0 = s.a1 > s.a0 ? (s.a1 - s.a0 + g.bn - 1) / g.bn : 0;
    s.n1 = s.b1 > s.b0 ? (s.b1 - s.b0 + g.bn - 1) / g.bn : 0;
    return s;
}

__device__ __forceinline__ Chunk chunk_of(const GemmArgs &g, const Slice &s, int c)
{
    Chunk ch;
    if (c < s.n0) {
        ch.c0 = s.a0 + c * g.bn;
        ch.n = min(g.bn, s.a1 - ch.c0);
        ch.store = false;
        ch.b_row = ch.c0;
        ch.valid = max(0, min(ch.n, g.n_topk - ch.c0));
    } else {
        ch.c0 = s.b0 + (c - s.n0) * g.bn;
        ch.n = min(g.bn, s.b1 - ch.c0);
        ch.store = true;
        ch.b_row = ch.c0 - g.n_topk_pad;
        ch.valid = max(0, min(ch.n, g.n_store - ch.b_row));
    }
    return ch;
}

// Waits without looking at the abort flag; used only to drain in-flight work after an abort.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity)
{
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kWaitTimeoutNs / 10)
            return;
}

// MT (row tiles per CTA) is a template parameter: with one tile the per-tile loops must
// vanish at compile time (a loop of one run-time iteration around the TMA and MMA issue cost
// 3% at 16 rows, measured on GB300).
template <int KP, int MT, bool PAIR>
__global__ void __launch_bounds__(64 + MT * BM, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_t_wide,
                   const __grid_constant__ CUtensorMap map_t_narrow, const __grid_constant__ CUtensorMap map_s_wide,
                   const __grid_constant__ CUtensorMap map_s_narrow, const GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stages = args.stages;
    const int kbs = args.kbs;
    constexpr int mt = MT;
    constexpr int n_bufs = 2 * MT * BN <= TMEM_COLS ? 2 : 1;  // bn = 256 whenever MT = 2
    // bytes of one B K-block of a full chunk (of this CTA's half of it in a pair)
    const int b_sub = (PAIR ? args.bn / 2 : args.bn) * BK * 2;
    // stage layout: kbs x mt A K-blocks (K-block major), then kbs B K-blocks (every part
    // 1024-byte aligned)
    const int stage_bytes = kbs * (mt * args.a_bytes + b_sub);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + stages * stage_bytes);
    // bars: full[MAX_STAGES] | empty[MAX_STAGES] | tfull[2] | tempty[2] | drain
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * MAX_STAGES + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *stash = reinterpret_cast<float *>(smem + stages * stage_bytes + BAR_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // in a pair, rank 0 issues the MMAs and owns the barriers both CTAs' loads and
    // accumulator releases complete on
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool issuer = rank == 0u;
    const int group = blockIdx.x % args.row_groups;
    const int tile0 = group * mt;
    const int split = blockIdx.x / args.row_groups;
    const int tiles = MT == 1 ? 1 : min(MT, args.row_tiles - tile0);  // row tiles this CTA computes
    const Slice slice = slice_of(args, split);
    const int n_chunks = slice.n0 + slice.n1;
    const int kstages = (args.K + BK * kbs - 1) / (BK * kbs);  // stages per chunk

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (MAX_STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * MAX_STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * MAX_STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * MAX_STAGES + 4);

    if (threadIdx.x == 0) {
        griddep_launch_dependents();
        for (int s = 0; s < stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), PAIR ? 2 * BM : tiles * BM);  // a pair: both CTAs' rows
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&map_a);
        if (slice.n0) {
            prefetch_tmap(&map_t_wide);
            prefetch_tmap(&map_t_narrow);
        }
        if (slice.n1) {
            prefetch_tmap(&map_s_wide);
            prefetch_tmap(&map_s_narrow);
        }
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR)
        cluster_sync();  // the issuer's barriers are initialised before either CTA signals them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            const uint64_t stream_policy = l2_policy_evict_first();
            if (args.dependent) {
                // The weights do not depend on the grid before this one: bring the first
                // stages' W boxes into L2 while it finishes (one tile per CTA only: a pair's
                // feed is bound by TMA operations), then wait for it before any load of A (the
                // hidden states may be its output).
                const int warm = PAIR ? 0 : min(kWarmStages, n_chunks * kstages);
                for (int n = 0; n < warm; ++n) {
                    const Chunk wch = chunk_of(args, slice, n / kstages);
                    const CUtensorMap *wmap = wch.store ? &map_s_wide : &map_t_wide;
                    for (int q = 0; q < kbs; ++q)
                        tma_prefetch_l2_2d(wmap, ((n % kstages) * kbs + q) * BK, wch.b_row);
                }
                griddep_wait();
            }
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int c = 0; c < n_chunks && ok; ++c) {
                const Chunk ch = chunk_of(args, slice, c);
                const CUtensorMap *wide = ch.store ? &map_s_wide : &map_t_wide;
                const CUtensorMap *narrow = ch.store ? &map_s_narrow : &map_t_narrow;
                // with two tiles one 256-row box brings both A tiles (rows past R read zeros)
                // With two tiles (bound by TMA operations, not bytes) a narrow chunk's B rows come
                // in one full-width box too: the rows past the chunk are W's next rows or zeros
                // past its end, and the MMA reads only the chunk's n.
                const int b_rows = MT == 2 ? args.bn : ch.n;
                // a pair: each CTA loads its A tile and a 128-row box of B ending at the end of
                // its half of the chunk, all onto the issuer's barrier.  A narrow chunk's box
                // then starts (bn - n) / 2 rows early (a multiple of 8: whole swizzle atoms) in
                // rows this slice has just streamed, which L2 still holds; a box starting at the
                // half would run into the next slice's first rows, fetched from HBM a second time
                // (measured on GB300 at 512 rows: 1.011 -> 1.005 x the algorithmic DRAM bytes,
                // same time).  Rows before the matrix read zeros.
                const uint32_t tx = PAIR ? static_cast<uint32_t>(2 * kbs * (args.a_bytes + b_sub))
                                         : static_cast<uint32_t>(kbs * ((MT == 2 ? 2 : tiles) * args.a_bytes +
                                                                        b_rows * BK * 2));
                const int b_shift = PAIR ? (args.bn - ch.n) / 2 : 0;
                const int b_row = PAIR ? ch.b_row + static_cast<int>(rank) * (ch.n / 2) - b_shift : ch.b_row;
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = smem + stage * stage_bytes;
                    const uint32_t fb = PAIR ? mapa_shared(full_bar(stage), 0u) : full_bar(stage);
                    if (!PAIR || issuer)
                        mbar_arrive_expect_tx(full_bar(stage), tx);
                    for (int q = 0; q < kbs; ++q) {
                        const int x = (ks * kbs + q) * BK;  // past K the boxes read zeros
                        // the group's tiles are adjacent rows of A and adjacent in shared memory: one box
                        const uint32_t a_dst = smem_u32(st + q * mt * args.a_bytes);
                        const uint32_t b_dst = smem_u32(st + kbs * mt * args.a_bytes + q * b_sub);
                        if constexpr (PAIR) {
                            // 3-D maps: one box brings the stage's kbs K-blocks (one TMA operation
                            // each for A and B, as many as a 256-row box takes in one CTA)
                            if (q == 0) {
                                tma_load_3d_pair(a_dst, &map_a, fb, 0, tile0 * BM, ks * kbs);
                                tma_load_3d_pair_policy(b_dst, wide, fb, 0, b_row, ks * kbs, stream_policy);
                            }
                            continue;
                        }
                        tma_load_2d(a_dst, &map_a, full_bar(stage), x, tile0 * BM);
                        // the weights stream through once: evict-first in L2 (measured on GB300:
                        // 197.3 vs 198.0 us at 16 rows, 248.3 vs 250.0 at 64, 449.9 vs 455.1 at 512)
                        if (ch.n == args.bn || MT == 2) {
                            tma_load_2d_policy(b_dst, wide, full_bar(stage), x, ch.b_row, stream_policy);
                        } else {
                            for (int u = 0; u < ch.n / UNIT; ++u)
                                tma_load_2d_policy(b_dst + u * UNIT * BK * 2, narrow, full_bar(stage), x,
                                                   ch.b_row + u * UNIT, stream_policy);
                        }
                    }
                    ++issued;
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA leaves (a pair's second CTA
                // cannot wait on the issuer's barriers: it gives them a fixed 100 us)
                if (PAIR && !issuer) {
                    const unsigned long long t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < 100000ull) {
                    }
                } else {
                    const long long first = issued > stages ? issued - stages : 0;
                    for (long long n = first; n < issued; ++n)
                        drain_wait(full_bar(static_cast<int>(n % stages)), static_cast<uint32_t>((n / stages) & 1));
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && (!PAIR || issuer)) {
            // ---------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int c = 0; c < n_chunks && ok; ++c) {
                const int buf = c % n_bufs;
                const uint32_t use = static_cast<uint32_t>(c / n_bufs);
                const Chunk ch = chunk_of(args, slice, c);
                const uint32_t idesc = idesc_bf16_f32(PAIR ? 2 * BM : BM, ch.n);
                // a pair's B rows sit at the end of each CTA's box (see the producer)
                const uint32_t b_skip = PAIR ? static_cast<uint32_t>((args.bn - ch.n) / 2 * BK * 2) : 0u;
                if (!mbar_wait(tempty_bar(buf), (use & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * mt * args.bn);
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_u32(smem + stage * stage_bytes);
                    for (int q = 0; q < kbs; ++q) {
                        const uint32_t b0 = st + static_cast<uint32_t>(kbs * mt * args.a_bytes + q * b_sub) + b_skip;
                        for (int t = 0; t < tiles; ++t) {
                            const uint32_t a0 = st + static_cast<uint32_t>((q * mt + t) * args.a_bytes);
                            const uint32_t d = d_tmem + static_cast<uint32_t>(t * args.bn);
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk) {
                                const uint64_t ad = sw128_kmajor_desc(a0 + kk * 32);
                                const uint64_t bd = sw128_kmajor_desc(b0 + kk * 32);
                                const uint32_t acc = (ks | q | kk) != 0 ? 1u : 0u;
                                if constexpr (PAIR)
                                    umma_bf16_pair(d, ad, bd, idesc, acc);
                                else
                                    umma_bf16(d, ad, bd, idesc, acc);
                            }
                        }
                    }
                    if constexpr (PAIR)
                        umma_commit_pair_both(empty_bar(stage));  // both CTAs' producers reuse the stage
                    else
                        umma_commit(empty_bar(stage));
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) {
                    if constexpr (PAIR)
                        umma_commit_pair_both(tfull_bar(buf));
                    else
                        umma_commit(tfull_bar(buf));
                }
            }
            if (!ok) {
                // every MMA issued so far must finish before TMEM is released
                if constexpr (PAIR)
                    umma_commit_pair(drain_bar);
                else
                    umma_commit(drain_bar);
                drain_wait(drain_bar, 0);
            }
        }
    } else if ((warp - 2) / 4 < tiles) {
        // ---------------- epilogue: thread = one row of row tile t
        const int t = (warp - 2) / 4;
        const int q = warp & 3;  // TMEM lane quarter this warp may read
        const int row = (tile0 + t) * BM + q * 32 + lane;
        const bool row_ok = row < args.R;
        float *my_stash = stash + (threadIdx.x - 64) * STASH_STRIDE;
        const uint32_t acc_col = static_cast<uint32_t>(t * args.bn);
        if (args.dependent)
            griddep_wait();  // the grid before may still read what the epilogue writes
        uint32_t *slots = args.bound && row_ok ? args.bound + static_cast<long long>(row) * KP : nullptr;
        float published = -INFINITY;
        ThreadTopK<KP> top;
        top.init();
        // values waiting for insertion, newest first (column ids increase with age reversed)
        constexpr int kQueue = 4;
        float queue_v[kQueue];
        int queue_i[kQueue];
        int n_queued = 0;
        auto drain_queue = [&]() {
#pragma unroll
            for (int e = kQueue - 1; e >= 0; --e)
                if (e < n_queued)
                    top.push_increasing_id(queue_v[e], queue_i[e]);
            n_queued = 0;
        };
        for (int c = 0; c < n_chunks; ++c) {
            const int buf = c % n_bufs;
            const uint32_t use = static_cast<uint32_t>(c / n_bufs);
            const Chunk ch = chunk_of(args, slice, c);
            // read before the accumulator is ready: the load's latency hides under the wait
            const float ext = slots && !ch.store && c > 0 ? shared_threshold<KP>(slots) : -INFINITY;
            const bool ready = mbar_wait(tfull_bar(buf), use & 1u, abort_flag);
            if (!__all_sync(kFullMask, ready))
                break;
            tc_fence_after();
            for (int cb = 0; cb < ch.n / 32 + ((ch.n & 31) ? 1 : 0); ++cb) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(buf * mt * args.bn + cb * 32) + acc_col,
                                   r);
                tmem_wait_ld(r);
                const int valid = min(32, ch.valid - cb * 32);
                if (ch.store) {
                    if (row_ok && valid > 0) {
                        float *dst = args.out + static_cast<long long>(row) * args.ldo + (ch.b_row + cb * 32);
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
                } else if (row_ok && valid > 0) {
                    const float thr = fmaxf(top.threshold(), ext);
                    // most blocks hold no value above the threshold: test their maximum first
                    float m[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        m[j] = fmaxf(fmaxf(__uint_as_float(r[j]), __uint_as_float(r[j + 8])),
                                     fmaxf(__uint_as_float(r[j + 16]), __uint_as_float(r[j + 24])));
                    const float block_max = fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])),
                                                  fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
                    if (block_max > thr) {
                        uint32_t mask = 0;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            mask |= static_cast<uint32_t>(__uint_as_float(r[j]) > thr) << j;
                        if (valid < 32)
                            mask &= (1u << valid) - 1u;
                        const int base_col = ch.c0 + cb * 32;
                        if (valid == 32 && __popc(mask) == 1 && n_queued < kQueue && block_max != 0.0f) {
                            // a single value passes, so it is the block's maximum: queue it
                            // and insert it once the accumulator is released (a zero goes the
                            // exact way below, where its sign is the accumulator's)
#pragma unroll
                            for (int e = kQueue - 1; e > 0; --e) {
                                queue_v[e] = queue_v[e - 1];
                                queue_i[e] = queue_i[e - 1];
                            }
                            queue_v[0] = block_max;
                            queue_i[0] = base_col + __ffs(mask) - 1;
                            ++n_queued;
                        } else if (mask) {
                            drain_queue();  // ids must reach the list in increasing order
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
            if (PAIR && !issuer)
                mbar_arrive_cluster(mapa_shared(tempty_bar(buf), 0u));
            else
                mbar_arrive(tempty_bar(buf));
            drain_queue();  // overlaps the next chunk's MMAs
            if (slots && !ch.store && top.v[0] > published) {
                atomicMax(slots + split % KP, order_key(top.v[0]));
                published = top.v[0];
            }
        }
        if (slots)
            __threadfence();  // the slot updates land before this CTA counts itself done
        if (row_ok && args.n_topk > 0) {
            const long long base = (static_cast<long long>(row) * args.n_split + split) * KP;
#pragma unroll
            for (int s = 0; s < KP; ++s) {
                args.pval[base + s] = top.v[s];
                args.pid[base + s] = top.i[s];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR)
        cluster_sync();  // neither CTA leaves while the other may still signal or read it
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag)
        atomicOr(args.status, kStatusTimeoutGemm);
    if (args.bound) {
        // the last CTA of the row group returns the group's slots (and its counter) to zero
        __shared__ int s_last;
        if (threadIdx.x == 0)
            s_last = atomicAdd(args.group_done + group, 1u) == static_cast<unsigned>(args.n_split - 1);
        __syncthreads();
        if (s_last) {
            __threadfence();
            const long long k0 = static_cast<long long>(tile0) * BM * KP;
            const long long k1 = static_cast<long long>(min(args.R, (tile0 + tiles) * BM)) * KP;
            for (long long i = k0 + threadIdx.x; i < k1; i += blockDim.x)
                args.bound[i] = 0u;
            if (threadIdx.x == 0)
                args.group_done[group] = 0u;
        }
    }
}

// The driver's encoder, looked up on first use (again after a failed lookup); safe to call from
// several host threads.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 fn = cached.load(std::memory_order_acquire);
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
            cached.store(fn, std::memory_order_release);
        }
    }
    return fn;
}

// CTAs of a pair kernel resident at once on the current device (clusters of two need two SMs
// of one GPC), cached per device and KP instantiation (kp_slot); safe to call from several
// host threads.
int resident_pair_ctas(const void *kern, int kp_slot, int smem_bytes, int sms)
{
    static std::mutex mu;
    static int cache[64][4] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return std::max(2, sms / 2 * 2);
    }
    std::lock_guard<std::mutex> lock(mu);
    int &cached = cache[dev][kp_slot];
    if (cached == 0) {
        cudaLaunchConfig_t qc = {};
        qc.gridDim = dim3(static_cast<unsigned>(2 * sms));
        qc.blockDim = dim3(64 + BM);
        qc.dynamicSmemBytes = smem_bytes;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = 2;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        qc.attrs = qa;
        qc.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &qc) != cudaSuccess || clusters < 1) {
            (void)cudaGetLastError();
            clusters = sms / 2;
        }
        cached = std::min(sms, 2 * clusters);
    }
    return cached;
}

// Row-major bf16 [rows, K] tensor, boxes of 64 K-elements x box_rows rows, 128-byte swizzle.
cudaError_t encode_map(CUtensorMap *map, const void *ptr, int K, int rows, int box_rows)
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

// The same matrix as a 3-D view (x = 64 elements of K, y = row, z = K-block; K a multiple of
// 64): a box of 64 x box_rows x kb lands as kb consecutive 128-byte-swizzled K-major tiles.
cudaError_t encode_map3(CUtensorMap *map, const void *ptr, int K, int rows, int box_rows, int kb)
{
    auto encode = tensor_map_encoder();
    if (!encode || K % BK != 0)
        return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(BK), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(K / BK)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(BK) * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows),
                               static_cast<cuuint32_t>(kb)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A map is a pure function of its encode parameters, so a drafting loop that calls with the
// same buffers every step reuses the encodings (a small per-thread cache, oldest entry out).
cudaError_t make_map(CUtensorMap *map, const void *ptr, int K, int rows, int box_rows, int kb = 0)
{
    struct Entry {
        const void *ptr;
        int K, rows, box_rows, kb;  // kb = 0: the 2-D map
        CUtensorMap map;
    };
    constexpr int kEntries = 16;
    thread_local Entry cache[kEntries];
    thread_local int used = 0, next = 0;
    for (int i = 0; i < used; ++i) {
        const Entry &e = cache[i];
        if (e.ptr == ptr && e.K == K && e.rows == rows && e.box_rows == box_rows && e.kb == kb) {
            *map = e.map;
            return cudaSuccess;
        }
    }
    const cudaError_t err = kb ? encode_map3(map, ptr, K, rows, box_rows, kb) : encode_map(map, ptr, K, rows, box_rows);
    if (err != cudaSuccess)
        return err;
    cache[next] = Entry{ptr, K, rows, box_rows, kb, *map};
    next = (next + 1) % kEntries;
    used = used < kEntries ? used + 1 : kEntries;
    return cudaSuccess;
}

cudaError_t make_map3(CUtensorMap *map, const void *ptr, int K, int rows, int box_rows, int kb)
{
    return make_map(map, ptr, K, rows, box_rows, kb);
}

template <int KP>
cudaError_t launch(const void *A, int R, int K, const void *Bt, int n_topk, const void *Bs, int n_store,
                   GemmArgs args, int *n_split_out, cudaStream_t stream)
{
    // A box: the live rows of a tile, rounded to 8 (one swizzle atom); the MMA still reads
    // 128 rows, the rows past the box hold stale shared memory and only feed unused rows of C.
    const int a_rows = std::min(BM, (std::max(R, 1) + 7) / 8 * 8);
    args.a_bytes = a_rows * BK * 2;
    // Up to 64 rows the stream of W sets the time: 128-column chunks with 2 K-blocks per
    // stage read each W row in 256-byte runs (measured on GB300: 193.5 vs 199.8 us for the
    // 8B-class head at 16 rows).  Beyond, 256-column chunks with 1 K-block per stage feed
    // the tensor cores best (438.5 vs 480.3 us at 512 rows).
    args.bn = R <= 64 ? 128 : BN;
    args.kbs = R <= 64 ? 2 : 1;
    args.row_tiles = (R + BM - 1) / BM;
    // Beyond 128 rows two row tiles share each chunk of B.  As a CTA pair each SM holds one
    // tile and half of B, so an accumulator takes 256 TMEM columns and the epilogue runs under
    // the next chunk's MMAs (two buffers); in one CTA (mt = 2) the two tiles' accumulators
    // fill TMEM (one buffer) and the MMA waits for the epilogue.  Both take 64 KB of operands
    // per stage in two TMA operations (three stages).  Measured on GB300 (same bits): pairs
    // 464.4 -> 429.6 us per call at 512 rows; at 1024 rows, in one process with the two
    // kernels' calls interleaved in blocks of ten (20 rounds), 1686.9 -> 1613.9 us per LM head.
    // In one CTA the MMA warp waited 6.9% of its cycles for the epilogue and 8.0% for TMA
    // (cycle counters in an instrumented copy); as pairs, 0.2% and 14.6%.  Beyond 1024 rows
    // (not measured) two tiles stay in one CTA.
    const bool two_tiles = args.bn == BN && args.row_tiles >= 2;
    // pairs read A and B through 3-D views whose K-blocks must not straddle rows
    args.pair = two_tiles && args.row_tiles <= 8 && K % BK == 0 ? 1 : 0;
    if (args.pair)
        args.kbs = 2;
    args.mt = two_tiles && !args.pair ? 2 : 1;
    args.n_bufs = 2 * args.mt * args.bn <= TMEM_COLS ? 2 : 1;
    args.row_groups = args.pair ? (args.row_tiles + 1) / 2 * 2 : (args.row_tiles + args.mt - 1) / args.mt;
    const int b_box = args.pair ? args.bn / 2 : args.bn;  // rows of the wide B box
    const int stash_bytes = args.mt * STASH_TILE_BYTES;
    const int stage_bytes = args.kbs * (args.mt * args.a_bytes + b_box * BK * 2);
    args.stages = std::min(MAX_STAGES, (SMEM_LIMIT - 1024 - BAR_BYTES - stash_bytes) / stage_bytes);
    if (args.stages < 2 || args.a_bytes + args.bn * BK * 2 < A_TILE_BYTES)
        return cudaErrorInvalidConfiguration;
    const int smem_bytes = 1024 + args.stages * stage_bytes + BAR_BYTES + stash_bytes;

    CUtensorMap ma, mtw, mtn, msw, msn;
    cudaError_t e;
    // two row tiles per CTA: one box covers both (256 rows, the largest TMA box)
    const int a_box = args.mt == 2 ? 2 * a_rows : a_rows;
    if ((e = args.pair ? make_map3(&ma, A, K, R, a_box, args.kbs) : make_map(&ma, A, K, R, a_box)) != cudaSuccess)
        return e;
    // an empty segment gets the other segment's maps (never read)
    const void *tb = n_topk > 0 ? Bt : Bs;
    const int tn = n_topk > 0 ? n_topk : n_store;
    const void *sb = n_store > 0 ? Bs : Bt;
    const int sn = n_store > 0 ? n_store : n_topk;
    if ((e = args.pair ? make_map3(&mtw, tb, K, tn, b_box, args.kbs) : make_map(&mtw, tb, K, tn, b_box)) !=
            cudaSuccess ||
        (e = make_map(&mtn, tb, K, tn, UNIT)) != cudaSuccess ||
        (e = args.pair ? make_map3(&msw, sb, K, sn, b_box, args.kbs) : make_map(&msw, sb, K, sn, b_box)) !=
            cudaSuccess ||
        (e = make_map(&msn, sb, K, sn, UNIT)) != cudaSuccess)
        return e;
    auto kern = args.pair ? gemm_tc_kernel<KP, 1, true>
                          : (args.mt == 1 ? gemm_tc_kernel<KP, 1, false> : gemm_tc_kernel<KP, 2, false>);
    if ((e = ensure_dynamic_smem(reinterpret_cast<const void *>(kern), smem_bytes)) != cudaSuccess)
        return e;
    const int sms = device_sm_count();
    args.R = R;
    args.K = K;
    args.n_topk = n_topk;
    args.n_topk_pad = (n_topk + UNIT - 1) / UNIT * UNIT;
    args.n_store = n_store;
    const int units = (args.n_topk_pad + n_store + UNIT - 1) / UNIT;
    // Starting under the grid before and warming L2 with W pays where the W stream sets the
    // time (one tile per CTA; measured on GB300: 205.6 -> 201.1 us per back-to-back call at
    // 16 rows).  CTA pairs start under it too, with no warm-up (their setup and the launch
    // itself leave the step; measured on GB300, same-box interleaved A/B of 60 rounds, identical
    // outputs: 420.4 -> 417.1 us per step at 512 rows, the same median at 1024).  Two tiles in
    // one CTA stay plain: the prefetch cost 1739 -> 1797 us at 1024 rows and the bare dependent
    // launch 1757 -> 1830.
    if (args.mt != 1 && !args.pair)
        args.dependent = 0;
    // the shared bound pays where the MMA waits for the epilogue (one accumulator buffer; with
    // pairs, measured on GB300, it cost 7 us at 512 rows)
    if (args.n_bufs != 1 || n_topk == 0) {
        args.bound = nullptr;
        args.group_done = nullptr;
    }
    int ctas = sms;  // CTAs resident at once: one per SM
    if (args.pair)  // pairs need two SMs of one GPC: size the grid by the pairs that fit at once
        ctas = resident_pair_ctas(reinterpret_cast<const void *>(kern), KP == 4 ? 0 : KP == 8 ? 1 : KP == 16 ? 2 : 3,
                                  smem_bytes, sms);
    args.n_split = std::max(1, std::min({max_splits_for(R), units, std::max(1, ctas / args.row_groups)}));
    if (n_split_out)
        *n_split_out = args.n_split;
    const dim3 grid(static_cast<unsigned>(args.row_groups * args.n_split));
    if (!args.dependent && !args.pair) {
        kern<<<grid, 64 + args.mt * BM, smem_bytes, stream>>>(ma, mtw, mtn, msw, msn, args);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(64 + args.mt * BM);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n_attr = 0;
    if (args.pair) {
        // CTAs 2i and 2i + 1 (row tiles 2j and 2j + 1 of one slice: row_groups is even)
        attr[n_attr].id = cudaLaunchAttributeClusterDimension;
        attr[n_attr].val.clusterDim.x = 2;
        attr[n_attr].val.clusterDim.y = 1;
        attr[n_attr].val.clusterDim.z = 1;
        ++n_attr;
    }
    if (args.dependent) {
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
        ++n_attr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    if ((e = cudaLaunchKernelEx(&cfg, kern, ma, mtw, mtn, msw, msn, args)) != cudaSuccess)
        return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lm_head(const void *hidden, int R, int K, const void *W_vocab, int V, int KP, float *pval,
                           int32_t *pid, int *n_split_out, const void *W_store, int n_store, float *out,
                           long long ldo, uint32_t *bound, unsigned *group_done, uint32_t *status,
                           bool dependent, cudaStream_t stream)
{
    GemmArgs a{};
    a.dependent = dependent ? 1 : 0;  // one-tile and pair launches only, decided in launch()
    a.pval = pval;
    a.pid = pid;
    a.out = out;
    a.ldo = ldo;
    a.bound = bound;
    a.group_done = group_done;
    a.status = status;
    switch (KP) {
    case 4: return launch<4>(hidden, R, K, W_vocab, V, W_store, n_store, a, n_split_out, stream);
    case 8: return launch<8>(hidden, R, K, W_vocab, V, W_store, n_store, a, n_split_out, stream);
    case 16: return launch<16>(hidden, R, K, W_vocab, V, W_store, n_store, a, n_split_out, stream);
    case 32: return launch<32>(hidden, R, K, W_vocab, V, W_store, n_store, a, n_split_out, stream);
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
    return launch<4>(A, R, K, nullptr, 0, B, N, a, nullptr, stream);
}

}  // namespace df2
