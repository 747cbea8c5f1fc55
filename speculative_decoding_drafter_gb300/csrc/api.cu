// api.cu -- the C ABI declared in include/dflash2.h: argument checks, workspace
// carving and the launch sequence of the selector head.  No allocation, no sync
// (except dflash2_check_device_status and dflash2_select_host).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "dflash2.h"
#include "internal.h"

namespace df2 {

// NVTX range around an entry point: the calls show up by name in a profiler's timeline, and
// `ncu --nvtx --nvtx-include "dflash2_select/"` captures the kernels of one call.  Without a
// profiler attached the push and pop return at once (header-only NVTX, no library linked).
struct TraceRange {
    explicit TraceRange(const char *name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};

int device_sm_count()
{
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

cudaError_t ensure_dynamic_smem(const void *kernel, int bytes)
{
    struct Entry {
        const void *kernel;
        int dev, bytes;
    };
    constexpr int kEntries = 32;
    thread_local Entry seen[kEntries];
    thread_local int used = 0, next = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    for (int i = 0; i < used; ++i)
        if (seen[i].kernel == kernel && seen[i].dev == dev && seen[i].bytes >= bytes)
            return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess)
        return e;
    seen[next] = Entry{kernel, dev, bytes};
    next = (next + 1) % kEntries;
    used = used < kEntries ? used + 1 : kEntries;
    return cudaSuccess;
}

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

df2_status check_dims(const df2_dims *d)
{
    if (!d)
        return DF2_ERR_INVALID_ARG;
    if (d->B < 1 || d->T < 1 || d->H < 1 || d->V < 1 || d->k < 1 || d->D < 1)
        return DF2_ERR_INVALID_ARG;
    if (d->k > d->V)
        return DF2_ERR_INVALID_ARG;
    if (d->k > 32 || d->V >= (1 << 24) || d->H < 8 || d->H % 8 != 0 || d->D < 8 || d->D % 8 != 0 ||
        d->D > 1024 || static_cast<long long>(d->B) * d->T > (1LL << 20))
        return DF2_ERR_UNSUPPORTED;
    return DF2_OK;
}

struct Workspace {
    uint32_t *status;
    unsigned *counters;
    unsigned *group_done;  // LM head: CTAs finished per row group
    uint32_t *bound;       // LM head: [R, KP] shared lower-bound keys
    float *pval;
    int32_t *pid;
    int32_t *best;
    float *gate;
    size_t bytes;
};

// Control block (zeroed by dflash2_workspace_init, left zeroed by every call): status word,
// per-sequence counters, the LM head's per-row-group counters and per-row bound keys.
size_t control_bytes(const df2_dims &d)
{
    const size_t R = static_cast<size_t>(d.B) * d.T;
    return kAlign + round_up(sizeof(unsigned) * static_cast<size_t>(d.B)) +
           round_up(sizeof(unsigned) * static_cast<size_t>(lm_head_max_groups(static_cast<long long>(R)))) +
           round_up(sizeof(uint32_t) * R * static_cast<size_t>(kp_for(d.k)));
}

// Layout (each part 256-byte aligned): status word | sequence counters | row-group counters |
// bound keys | partial values | partial ids | walk choices | gate.
Workspace carve(const df2_dims &d, void *base)
{
    const size_t R = static_cast<size_t>(d.B) * d.T;
    const size_t kp = static_cast<size_t>(kp_for(d.k));
    uint8_t *p = static_cast<uint8_t *>(base);
    Workspace w{};
    size_t off = 0;
    w.status = reinterpret_cast<uint32_t *>(p ? p + off : nullptr);
    off += kAlign;
    w.counters = reinterpret_cast<unsigned *>(p ? p + off : nullptr);
    off += round_up(sizeof(unsigned) * static_cast<size_t>(d.B));
    w.group_done = reinterpret_cast<unsigned *>(p ? p + off : nullptr);
    off += round_up(sizeof(unsigned) * static_cast<size_t>(lm_head_max_groups(static_cast<long long>(R))));
    w.bound = reinterpret_cast<uint32_t *>(p ? p + off : nullptr);
    off += round_up(sizeof(uint32_t) * R * kp);
    w.pval = reinterpret_cast<float *>(p ? p + off : nullptr);
    const size_t splits = static_cast<size_t>(max_splits_for(static_cast<long long>(R)));
    off += round_up(R * splits * kp * sizeof(float));
    w.pid = reinterpret_cast<int32_t *>(p ? p + off : nullptr);
    off += round_up(R * splits * kp * sizeof(int32_t));
    w.best = reinterpret_cast<int32_t *>(p ? p + off : nullptr);
    off += round_up(R * d.k * sizeof(int32_t));
    w.gate = reinterpret_cast<float *>(p ? p + off : nullptr);
    off += round_up(R * d.D * sizeof(float));
    w.bytes = off;
    return w;
}

// Device staging of dflash2_select_host, placed after the select workspace (each part
// 256-byte aligned): hidden [R, H] bf16 | anchor [B] | lattice [R, k + k*k] | draft [R].
struct Staging {
    uint16_t *hidden;
    int32_t *anchor;
    float *lattice;
    int32_t *draft;
    size_t bytes;  // select workspace + staging
};

Staging carve_staging(const df2_dims &d, void *base)
{
    const size_t R = static_cast<size_t>(d.B) * d.T;
    const size_t width = static_cast<size_t>(d.k) + static_cast<size_t>(d.k) * d.k;
    uint8_t *p = static_cast<uint8_t *>(base);
    Staging s{};
    size_t off = carve(d, nullptr).bytes;
    s.hidden = reinterpret_cast<uint16_t *>(p ? p + off : nullptr);
    off += round_up(R * d.H * sizeof(uint16_t));
    s.anchor = reinterpret_cast<int32_t *>(p ? p + off : nullptr);
    off += round_up(static_cast<size_t>(d.B) * sizeof(int32_t));
    s.lattice = reinterpret_cast<float *>(p ? p + off : nullptr);
    off += round_up(R * width * sizeof(float));
    s.draft = reinterpret_cast<int32_t *>(p ? p + off : nullptr);
    off += round_up(R * sizeof(int32_t));
    s.bytes = off;
    return s;
}

df2_status check_workspace(const df2_dims &d, void *ws, size_t bytes)
{
    if (!ws || !aligned(ws, kAlign))
        return DF2_ERR_WORKSPACE;
    if (bytes < carve(d, nullptr).bytes)
        return DF2_ERR_WORKSPACE;
    return DF2_OK;
}

df2_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DF2_OK : DF2_ERR_CUDA; }

// Events recorded around the top-k producing launch (dflash2_profile_events).
thread_local cudaEvent_t t_profile_begin = nullptr;
thread_local cudaEvent_t t_profile_end = nullptr;

cudaError_t profile_mark(cudaEvent_t ev, cudaStream_t st) { return ev ? cudaEventRecord(ev, st) : cudaSuccess; }

#define DF2_TRY(expr)                        \
    do {                                     \
        const df2_status _s = (expr);        \
        if (_s != DF2_OK)                    \
            return _s;                       \
    } while (0)

#define DF2_CUDA(expr) DF2_TRY(from_cuda(expr))

// Shared tail of both select paths: merge, lattice and walk in one launch.
df2_status finish(const df2_dims &d, const Workspace &w, int n_split, const float *gate, const void *pred_cb,
                  const void *succ_cb, const int32_t *anchor, float *lattice, int32_t *draft_ids, int32_t *topk_ids,
                  float *topk_vals, cudaStream_t st, const HostMirrors &mirrors = HostMirrors{},
                  const WalkOpts &walk = WalkOpts{})
{
    DF2_CUDA(launch_finish(d.B, d.T, d.k, d.V, d.D, kp_for(d.k), n_split, w.pval, w.pid, gate,
                           static_cast<const uint16_t *>(pred_cb), static_cast<const uint16_t *>(succ_cb), anchor,
                           lattice, draft_ids, topk_ids, topk_vals, w.best, w.counters, mirrors, walk, st));
    return DF2_OK;
}

// The fused path after argument checks: LM head (top-k, gate) and the finish launch.
df2_status select_checked(const df2_dims &d, const void *hidden, const void *W_vocab, const void *W_sel,
                          const void *pred_cb, const void *succ_cb, const int32_t *anchor, float *lattice,
                          int32_t *draft_ids, int32_t *topk_ids, float *topk_logits, float *gate, void *workspace,
                          cudaStream_t st, const HostMirrors &mirrors = HostMirrors{},
                          const WalkOpts &walk = WalkOpts{})
{
    const Workspace w = carve(d, workspace);
    const int R = d.B * d.T;
    const int kp = kp_for(d.k);
    float *g = gate ? gate : w.gate;
    int n_split = 0;
    DF2_CUDA(profile_mark(t_profile_begin, st));
    DF2_CUDA(launch_lm_head(hidden, R, d.H, W_vocab, d.V, kp, w.pval, w.pid, &n_split, W_sel, d.D, g, d.D, w.bound,
                            w.group_done, w.status, true, st));
    DF2_CUDA(profile_mark(t_profile_end, st));
    HostMirrors m = mirrors;
    m.status_dev = w.status;
    return finish(d, w, n_split, g, pred_cb, succ_cb, anchor, lattice, draft_ids, topk_ids, topk_logits, st, m, walk);
}

// Checks the walk options of dflash2_select_walk and turns them into the finish kernel's.
df2_status walk_opts_of(const df2_walk_opts *o, WalkOpts *out)
{
    *out = WalkOpts{};
    if (!o)
        return DF2_OK;
    if (!(o->temperature > 0.f) || !std::isfinite(o->temperature) || std::isnan(o->p_min))
        return DF2_ERR_INVALID_ARG;
    if ((o->uniforms && !aligned(o->uniforms, 4)) || (o->n_draft && !aligned(o->n_draft, 4)) ||
        (o->confidence && !aligned(o->confidence, 4)))
        return DF2_ERR_INVALID_ARG;
    out->sample = true;
    out->temperature = o->temperature;
    out->p_min = o->p_min;
    out->uniforms = o->uniforms;
    out->n_draft = o->n_draft;
    out->confidence = o->confidence;
    return DF2_OK;
}

// Device-visible address of a caller's host buffer if it is page-locked memory mapped into
// this device's address space (the finish kernel may then write it directly), else null.
template <typename Ptr>
Ptr *device_view(Ptr *host)
{
    if (!host)
        return nullptr;
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, host) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    int dev = -1;
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer || cudaGetDevice(&dev) != cudaSuccess ||
        attr.device != dev)
        return nullptr;
    return static_cast<Ptr *>(attr.devicePointer);
}

df2_status check_tail_pointers(const void *W_sel, const void *pred_cb, const void *succ_cb, const int32_t *anchor,
                               const float *lattice, const int32_t *draft_ids, const int32_t *topk_ids,
                               const float *topk_logits, const float *gate)
{
    if (!W_sel || !pred_cb || !succ_cb || !anchor || !lattice || !draft_ids)
        return DF2_ERR_INVALID_ARG;
    if (!aligned(W_sel, 16) || !aligned(pred_cb, 16) || !aligned(succ_cb, 16) || !aligned(anchor, 4) ||
        !aligned(lattice, 4) || !aligned(draft_ids, 4))
        return DF2_ERR_INVALID_ARG;
    if ((topk_ids && !aligned(topk_ids, 4)) || (topk_logits && !aligned(topk_logits, 4)) ||
        (gate && !aligned(gate, 16)))
        return DF2_ERR_INVALID_ARG;
    return DF2_OK;
}

}  // namespace
}  // namespace df2

using namespace df2;

extern "C" {

size_t dflash2_workspace_bytes(const df2_dims *dims)
{
    if (check_dims(dims) != DF2_OK)
        return 0;
    return carve(*dims, nullptr).bytes;
}

df2_status dflash2_workspace_init(const df2_dims *dims, void *workspace, size_t workspace_bytes, void *stream)
{
    DF2_TRY(check_dims(dims));
    DF2_TRY(check_workspace(*dims, workspace, workspace_bytes));
    return from_cuda(
        cudaMemsetAsync(workspace, 0, control_bytes(*dims), static_cast<cudaStream_t>(stream)));
}

df2_status dflash2_select(const df2_dims *dims, const void *hidden, const void *W_vocab, const void *W_sel,
                          const void *pred_cb, const void *succ_cb, const int32_t *anchor, float *lattice,
                          int32_t *draft_ids, int32_t *topk_ids, float *topk_logits, float *gate,
                          void *workspace, size_t workspace_bytes, void *stream)
{
    const TraceRange range("dflash2_select");
    DF2_TRY(check_dims(dims));
    const df2_dims d = *dims;
    if (!hidden || !W_vocab || !aligned(hidden, 16) || !aligned(W_vocab, 16))
        return DF2_ERR_INVALID_ARG;
    DF2_TRY(check_tail_pointers(W_sel, pred_cb, succ_cb, anchor, lattice, draft_ids, topk_ids, topk_logits, gate));
    DF2_TRY(check_workspace(d, workspace, workspace_bytes));
    cudaGetLastError();  // clear a stale error so the status reflects this call
    return select_checked(d, hidden, W_vocab, W_sel, pred_cb, succ_cb, anchor, lattice, draft_ids, topk_ids,
                          topk_logits, gate, workspace, static_cast<cudaStream_t>(stream));
}

df2_status dflash2_select_walk(const df2_dims *dims, const df2_walk_opts *walk, const void *hidden,
                               const void *W_vocab, const void *W_sel, const void *pred_cb, const void *succ_cb,
                               const int32_t *anchor, float *lattice, int32_t *draft_ids, int32_t *topk_ids,
                               float *topk_logits, float *gate, void *workspace, size_t workspace_bytes, void *stream)
{
    const TraceRange range("dflash2_select_walk");
    DF2_TRY(check_dims(dims));
    const df2_dims d = *dims;
    WalkOpts opts;
    DF2_TRY(walk_opts_of(walk, &opts));
    if (!hidden || !W_vocab || !aligned(hidden, 16) || !aligned(W_vocab, 16))
        return DF2_ERR_INVALID_ARG;
    DF2_TRY(check_tail_pointers(W_sel, pred_cb, succ_cb, anchor, lattice, draft_ids, topk_ids, topk_logits, gate));
    DF2_TRY(check_workspace(d, workspace, workspace_bytes));
    cudaGetLastError();
    return select_checked(d, hidden, W_vocab, W_sel, pred_cb, succ_cb, anchor, lattice, draft_ids, topk_ids,
                          topk_logits, gate, workspace, static_cast<cudaStream_t>(stream), HostMirrors{}, opts);
}

size_t dflash2_select_host_workspace_bytes(const df2_dims *dims)
{
    if (check_dims(dims) != DF2_OK)
        return 0;
    return carve_staging(*dims, nullptr).bytes;
}

df2_status dflash2_select_host(const df2_dims *dims, const void *hidden_host, const void *W_vocab, const void *W_sel,
                               const void *pred_cb, const void *succ_cb, const int32_t *anchor_host,
                               float *lattice_host, int32_t *draft_ids_host, uint32_t *status_host, void *workspace,
                               size_t workspace_bytes, void *stream)
{
    const TraceRange range("dflash2_select_host");
    DF2_TRY(check_dims(dims));
    const df2_dims d = *dims;
    if (!hidden_host || !anchor_host || !draft_ids_host || !W_vocab || !aligned(W_vocab, 16))
        return DF2_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < carve_staging(d, nullptr).bytes)
        return DF2_ERR_WORKSPACE;
    const Staging s = carve_staging(d, workspace);
    // every check dflash2_select makes, before anything is enqueued
    DF2_TRY(check_tail_pointers(W_sel, pred_cb, succ_cb, s.anchor, s.lattice, s.draft, nullptr, nullptr, nullptr));
    const size_t R = static_cast<size_t>(d.B) * d.T;
    const size_t width = static_cast<size_t>(d.k) + static_cast<size_t>(d.k) * d.k;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaGetLastError();
    // once work is enqueued, a failure still waits for the stream: no copy from or to the
    // caller's host buffers may be in flight when the call returns
    auto fail = [&](df2_status e) {
        cudaStreamSynchronize(st);
        return e;
    };
    if (cudaMemcpyAsync(s.hidden, hidden_host, R * d.H * sizeof(uint16_t), cudaMemcpyHostToDevice, st) !=
        cudaSuccess)
        return fail(DF2_ERR_CUDA);
    // Page-locked host buffers mapped into this device's address space are read and written
    // by the finish kernel itself: every copy on the stream costs about 3 us whatever its size
    // (measured on GB300), and this takes four of the five off the step.  Other buffers go
    // through copies.  The lookups run while the hidden states upload.
    const int32_t *anchor_dv = device_view(anchor_host);
    int32_t *draft_dv = device_view(draft_ids_host);
    float *lattice_dv = device_view(lattice_host);
    uint32_t *status_dv = device_view(status_host);
    const bool direct = anchor_dv && draft_dv && status_dv && (!lattice_host || lattice_dv) && aligned(anchor_dv, 4) &&
                        aligned(draft_dv, 4) && aligned(status_dv, 4) && (!lattice_dv || aligned(lattice_dv, 4));
    HostMirrors mirrors;
    if (direct) {
        mirrors.lattice = lattice_dv;
        mirrors.draft = draft_dv;
        mirrors.status = status_dv;
    } else if (cudaMemcpyAsync(s.anchor, anchor_host, d.B * sizeof(int32_t), cudaMemcpyHostToDevice, st) !=
               cudaSuccess) {
        return fail(DF2_ERR_CUDA);
    }
    const df2_status e = select_checked(d, s.hidden, W_vocab, W_sel, pred_cb, succ_cb, direct ? anchor_dv : s.anchor,
                                        s.lattice, s.draft, nullptr, nullptr, nullptr, workspace, st, mirrors);
    if (e != DF2_OK)
        return fail(e);
    uint32_t word = 0;
    uint32_t *dst = status_host ? status_host : &word;
    if (!direct) {
        if (cudaMemcpyAsync(draft_ids_host, s.draft, R * sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
            (lattice_host &&
             cudaMemcpyAsync(lattice_host, s.lattice, R * width * sizeof(float), cudaMemcpyDeviceToHost, st) !=
                 cudaSuccess))
            return fail(DF2_ERR_CUDA);
        // The status word comes back behind the results, into the caller's page-locked word or a
        // stack word (pageable memory, for which the copy returns only once it is complete).
        if (cudaMemcpyAsync(dst, workspace, sizeof word, cudaMemcpyDeviceToHost, st) != cudaSuccess)
            return fail(DF2_ERR_CUDA);
    }
    DF2_CUDA(cudaStreamSynchronize(st));
    word = *static_cast<volatile uint32_t *>(dst);
    return word == 0 ? DF2_OK : DF2_ERR_TIMEOUT;
}

df2_status dflash2_select_from_logits(const df2_dims *dims, const float *logits, const void *hidden,
                                      const void *W_sel, const void *pred_cb, const void *succ_cb,
                                      const int32_t *anchor, float *lattice, int32_t *draft_ids,
                                      int32_t *topk_ids, float *topk_logits, float *gate, void *workspace,
                                      size_t workspace_bytes, void *stream)
{
    const TraceRange range("dflash2_select_from_logits");
    DF2_TRY(check_dims(dims));
    const df2_dims d = *dims;
    if (!logits || !hidden || !aligned(logits, 16) || !aligned(hidden, 16))
        return DF2_ERR_INVALID_ARG;
    DF2_TRY(check_tail_pointers(W_sel, pred_cb, succ_cb, anchor, lattice, draft_ids, topk_ids, topk_logits, gate));
    DF2_TRY(check_workspace(d, workspace, workspace_bytes));
    cudaGetLastError();
    const Workspace w = carve(d, workspace);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int R = d.B * d.T;
    const int kp = kp_for(d.k);
    float *g = gate ? gate : w.gate;
    int n_split = 0;
    DF2_CUDA(profile_mark(t_profile_begin, st));
    DF2_CUDA(launch_logits_topk_partial(logits, R, d.V, kp, w.pval, w.pid, &n_split, st));
    DF2_CUDA(profile_mark(t_profile_end, st));
    DF2_CUDA(launch_gemm_store(hidden, W_sel, R, d.H, d.D, g, d.D, w.status, st));
    return finish(d, w, n_split, g, pred_cb, succ_cb, anchor, lattice, draft_ids, topk_ids, topk_logits, st);
}

df2_status dflash2_lm_head_logits(const df2_dims *dims, const void *hidden, const void *W_vocab, float *logits,
                                  void *workspace, size_t workspace_bytes, void *stream)
{
    const TraceRange range("dflash2_lm_head_logits");
    DF2_TRY(check_dims(dims));
    const df2_dims d = *dims;
    if (!hidden || !W_vocab || !logits || !aligned(hidden, 16) || !aligned(W_vocab, 16) || !aligned(logits, 4))
        return DF2_ERR_INVALID_ARG;
    DF2_TRY(check_workspace(d, workspace, workspace_bytes));
    cudaGetLastError();
    const Workspace w = carve(d, workspace);
    DF2_CUDA(launch_gemm_store(hidden, W_vocab, d.B * d.T, d.H, d.V, logits, d.V, w.status,
                               static_cast<cudaStream_t>(stream)));
    return DF2_OK;
}

df2_status dflash2_topk(const df2_dims *dims, const float *logits, int32_t *topk_ids, float *topk_logits,
                        void *workspace, size_t workspace_bytes, void *stream)
{
    const TraceRange range("dflash2_topk");
    DF2_TRY(check_dims(dims));
    const df2_dims d = *dims;
    if (!logits || !topk_ids || !topk_logits || !aligned(logits, 16) || !aligned(topk_ids, 4) ||
        !aligned(topk_logits, 4))
        return DF2_ERR_INVALID_ARG;
    DF2_TRY(check_workspace(d, workspace, workspace_bytes));
    cudaGetLastError();
    const Workspace w = carve(d, workspace);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int R = d.B * d.T;
    const int kp = kp_for(d.k);
    int n_split = 0;
    // the bound slots (zero between calls, unused without the LM head) count each row's slices
    TopkFinish fin;
    fin.row_done = w.bound;
    fin.k = d.k;
    fin.ids = topk_ids;
    fin.vals = topk_logits;
    bool merged = false;
    DF2_CUDA(launch_logits_topk_partial(logits, R, d.V, kp, w.pval, w.pid, &n_split, st, fin, &merged));
    if (!merged)
        DF2_CUDA(launch_topk_merge(w.pval, w.pid, R, n_split, kp, d.k, topk_ids, topk_logits, st));
    return DF2_OK;
}

df2_status dflash2_gate(const df2_dims *dims, const void *hidden, const void *W_sel, float *gate, void *workspace,
                        size_t workspace_bytes, void *stream)
{
    const TraceRange range("dflash2_gate");
    DF2_TRY(check_dims(dims));
    const df2_dims d = *dims;
    if (!hidden || !W_sel || !gate || !aligned(hidden, 16) || !aligned(W_sel, 16) || !aligned(gate, 16))
        return DF2_ERR_INVALID_ARG;
    DF2_TRY(check_workspace(d, workspace, workspace_bytes));
    cudaGetLastError();
    const Workspace w = carve(d, workspace);
    DF2_CUDA(launch_gemm_store(hidden, W_sel, d.B * d.T, d.H, d.D, gate, d.D, w.status,
                               static_cast<cudaStream_t>(stream)));
    return DF2_OK;
}

df2_status dflash2_lattice(const df2_dims *dims, const int32_t *topk_ids, const float *topk_logits,
                           const float *gate, const void *pred_cb, const void *succ_cb, const int32_t *anchor,
                           float *lattice, void *stream)
{
    const TraceRange range("dflash2_lattice");
    DF2_TRY(check_dims(dims));
    const df2_dims d = *dims;
    if (!topk_ids || !topk_logits || !gate || !pred_cb || !succ_cb || !anchor || !lattice)
        return DF2_ERR_INVALID_ARG;
    if (!aligned(topk_ids, 4) || !aligned(topk_logits, 4) || !aligned(gate, 16) || !aligned(pred_cb, 16) ||
        !aligned(succ_cb, 16) || !aligned(anchor, 4) || !aligned(lattice, 4))
        return DF2_ERR_INVALID_ARG;
    cudaGetLastError();
    DF2_CUDA(launch_lattice(d.B, d.T, d.k, d.V, d.D, topk_ids, topk_logits, gate,
                            static_cast<const uint16_t *>(pred_cb), static_cast<const uint16_t *>(succ_cb), anchor,
                            lattice, static_cast<cudaStream_t>(stream)));
    return DF2_OK;
}

df2_status dflash2_walk(const df2_dims *dims, const float *lattice, int32_t *draft_ids, void *stream)
{
    const TraceRange range("dflash2_walk");
    DF2_TRY(check_dims(dims));
    const df2_dims d = *dims;
    if (!lattice || !draft_ids || !aligned(lattice, 4) || !aligned(draft_ids, 4))
        return DF2_ERR_INVALID_ARG;
    cudaGetLastError();
    DF2_CUDA(launch_walk(d.B, d.T, d.k, lattice, draft_ids, static_cast<cudaStream_t>(stream)));
    return DF2_OK;
}

df2_status dflash2_walk_sample(const df2_dims *dims, const float *lattice, float temperature, float p_min,
                               const float *uniforms, int32_t *draft_ids, int32_t *n_draft, float *confidence,
                               void *stream)
{
    const TraceRange range("dflash2_walk_sample");
    DF2_TRY(check_dims(dims));
    const df2_dims d = *dims;
    if (!lattice || !draft_ids || !aligned(lattice, 4) || !aligned(draft_ids, 4) ||
        (uniforms && !aligned(uniforms, 4)) || (n_draft && !aligned(n_draft, 4)) ||
        (confidence && !aligned(confidence, 4)))
        return DF2_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || !std::isfinite(temperature) || std::isnan(p_min))
        return DF2_ERR_INVALID_ARG;
    cudaGetLastError();
    DF2_CUDA(launch_walk_sample(d.B, d.T, d.k, lattice, temperature, p_min, uniforms, draft_ids, n_draft, confidence,
                                static_cast<cudaStream_t>(stream)));
    return DF2_OK;
}

df2_status dflash2_dynamic_conv(const df2_conv_dims *dims, const void *x, const void *x_prev, const void *base,
                                const float *dyn, const void *gamma, float eps, void *y, void *stream)
{
    const TraceRange range("dflash2_dynamic_conv");
    if (!dims)
        return DF2_ERR_INVALID_ARG;
    const df2_conv_dims d = *dims;
    if (d.B < 1 || d.T < 1 || d.C < 1 || d.G < 1 || d.C % d.G != 0 || !(eps >= 0.f) || !std::isfinite(eps))
        return DF2_ERR_INVALID_ARG;
    if (d.G % 8 != 0 || d.C < 8 || d.C > 8192 || static_cast<long long>(d.B) * d.T > (1LL << 24))
        return DF2_ERR_UNSUPPORTED;
    if (!x || !base || !dyn || !y || !aligned(x, 16) || !aligned(base, 16) || !aligned(y, 16) || !aligned(dyn, 4) ||
        (x_prev && !aligned(x_prev, 16)) || (gamma && !aligned(gamma, 16)))
        return DF2_ERR_INVALID_ARG;
    cudaGetLastError();
    DF2_CUDA(launch_dynamic_conv(d.B, d.T, d.C, d.G, static_cast<const uint16_t *>(x),
                                 static_cast<const uint16_t *>(x_prev), static_cast<const uint16_t *>(base), dyn,
                                 static_cast<const uint16_t *>(gamma), eps, static_cast<uint16_t *>(y),
                                 static_cast<cudaStream_t>(stream)));
    return DF2_OK;
}

df2_status dflash2_check_device_status(void *workspace, size_t workspace_bytes, void *stream)
{
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < kAlign)
        return DF2_ERR_WORKSPACE;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    DF2_CUDA(cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, st));
    DF2_CUDA(cudaStreamSynchronize(st));
    if (word != 0) {
        DF2_CUDA(cudaMemsetAsync(workspace, 0, sizeof word, st));
        DF2_CUDA(cudaStreamSynchronize(st));
        return DF2_ERR_TIMEOUT;
    }
    return DF2_OK;
}

df2_status dflash2_selftest_wait_timeout(uint32_t limit_us, void *workspace, size_t workspace_bytes, void *stream)
{
    if (limit_us == 0 || limit_us > 1000000u)
        return DF2_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < kAlign)
        return DF2_ERR_WORKSPACE;
    cudaGetLastError();
    DF2_CUDA(launch_wait_selftest(static_cast<uint32_t *>(workspace), 1000ull * limit_us,
                                  static_cast<cudaStream_t>(stream)));
    return DF2_OK;
}

df2_status dflash2_profile_events(void *begin, void *end)
{
    if ((begin == nullptr) != (end == nullptr))
        return DF2_ERR_INVALID_ARG;
    t_profile_begin = static_cast<cudaEvent_t>(begin);
    t_profile_end = static_cast<cudaEvent_t>(end);
    return DF2_OK;
}

const char *dflash2_status_string(df2_status status)
{
    switch (status) {
    case DF2_OK: return "ok";
    case DF2_ERR_INVALID_ARG: return "invalid argument (null pointer, bad dimension or misaligned tensor)";
    case DF2_ERR_UNSUPPORTED: return "unsupported dimensions (outside the implemented limits)";
    case DF2_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DF2_ERR_CUDA: return "CUDA runtime or launch error";
    case DF2_ERR_TIMEOUT: return "a device-side pipeline wait timed out; outputs are invalid";
    default: return "unknown status";
    }
}

int32_t dflash2_version(void) { return 300; }

}  // extern "C"
