// noalloc.cu -- dflash2_topk_noalloc: the top-k entry point for callers that cannot
// allocate device memory.
//
// dflash2_topk needs a caller-provided workspace for its per-slice partial lists.
// Some hosts cannot provide one: an inference engine that plans every byte of device
// memory up front and hands plugins no allocator, or a latency-critical decode loop
// where cudaMalloc's implicit device synchronisation is not acceptable.  This variant
// keeps those partial lists in a fixed array that lives in the library's own device
// image, so a call needs only its inputs and outputs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "dflash2.h"
#include "internal.h"

namespace df2 {
namespace {

// Partial (value, id) lists of the top-k of given logits: at most R * kMaxSplits * KP
// entries of 8 bytes.  Every GPU that loads the library holds these 8 MiB until exit.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_topk_scratch[kNoAllocScratchBytes];

// Device address of g_topk_scratch, looked up once per device and CUDA context, with that
// device current.  (In host code the symbol name is only a host-side stand-in, never a
// device address.)  Keying by the context as well as the device keeps a caller that switches
// contexts on one device from getting another context's address.  A device reset
// (cudaDeviceReset) may recreate the primary context under the same handle, so the library
// must not be used across a reset.
std::mutex g_mu;
struct ScratchEntry {
    int dev;
    CUcontext ctx;
    void *ptr;
};
constexpr int kScratchEntries = 64;
ScratchEntry g_scratch[kScratchEntries];
int g_scratch_used = 0;

CUcontext current_context()
{
    using GetCurrent = CUresult (*)(CUcontext *);
    // looked up on first use (again after a failed lookup); safe from several host threads
    static std::atomic<GetCurrent> cached{nullptr};
    GetCurrent fn = cached.load(std::memory_order_acquire);
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<GetCurrent>(p);
            cached.store(fn, std::memory_order_release);
        }
    }
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS)
        return nullptr;
    return ctx;
}

cudaError_t scratch_for_current_device(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    // (null before the first runtime call on this thread: the lookup below then makes the
    // device's primary context current, and the context is read again)
    CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_scratch_used; ++i)
        if (g_scratch[i].dev == dev && g_scratch[i].ctx == ctx && ctx != nullptr) {
            *out = g_scratch[i].ptr;
            return cudaSuccess;
        }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess)
        return e;
    if (ctx == nullptr)
        ctx = current_context();
    if (ctx != nullptr) {
        const int slot = g_scratch_used < kScratchEntries ? g_scratch_used++ : (dev % kScratchEntries);
        g_scratch[slot] = ScratchEntry{dev, ctx, p};
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace df2

using namespace df2;

extern "C" df2_status dflash2_topk_noalloc(const df2_dims *dims, const float *logits, int32_t *topk_ids,
                                           float *topk_logits, void *stream)
{
    if (!dims)
        return DF2_ERR_INVALID_ARG;
    const df2_dims d = *dims;
    if (d.B < 1 || d.T < 1 || d.V < 1 || d.k < 1 || d.k > d.V)
        return DF2_ERR_INVALID_ARG;
    if (d.k > 32 || d.V >= (1 << 24) || static_cast<long long>(d.B) * d.T > (1LL << 20))
        return DF2_ERR_UNSUPPORTED;
    if (!logits || !topk_ids || !topk_logits || (reinterpret_cast<uintptr_t>(logits) & 15u) ||
        (reinterpret_cast<uintptr_t>(topk_ids) & 3u) || (reinterpret_cast<uintptr_t>(topk_logits) & 3u))
        return DF2_ERR_INVALID_ARG;
    const int R = d.B * d.T;
    const int kp = kp_for(d.k);
    const size_t list_entries = static_cast<size_t>(R) * kMaxSplits * kp;
    if (list_entries * (sizeof(float) + sizeof(int32_t)) > kNoAllocScratchBytes)
        return DF2_ERR_UNSUPPORTED;  // B*T*KP above 4096 (KP = k rounded up to 4, 8, 16 or 32)
    void *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess)
        return DF2_ERR_CUDA;
    cudaGetLastError();
    float *pval = static_cast<float *>(scratch);
    int32_t *pid = reinterpret_cast<int32_t *>(static_cast<unsigned char *>(scratch) + list_entries * sizeof(float));
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    int n_split = 0;
    if (launch_logits_topk_partial(logits, R, d.V, kp, pval, pid, &n_split, st) != cudaSuccess)
        return DF2_ERR_CUDA;
    if (launch_topk_merge(pval, pid, R, n_split, kp, d.k, topk_ids, topk_logits, st) != cudaSuccess)
        return DF2_ERR_CUDA;
    return DF2_OK;
}
