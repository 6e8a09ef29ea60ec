// noalloc.cu -- ring attention forward that allocates nothing.
//
// Some callers cannot call cudaMalloc, or cannot hand this library a
// workspace:
//   * code inside a custom device allocator's own callbacks: a cudaMalloc there
//     re-enters the allocator it is serving (or waits on its lock);
//   * runtimes that reserve all device memory at start-up and forbid allocation
//     afterwards, so that memory use and latency stay fixed;
//   * processes whose device memory pool belongs to another framework: memory
//     taken outside that pool escapes its accounting and can push it out of
//     memory;
//   * code recorded under stream capture in the global mode, where cudaMalloc
//     is refused.
// For them cp_ring_attention_fwd_noalloc runs the same ring as
// cp_ring_attention_fwd (zero-copy owner rotation, no prefetch) with its
// scratch -- the per-step partial output and lse, and the fp32 accumulator for
// a bf16 output -- taken from one file-scope device array of fixed size.
//
// The array occupies kNoallocScratchBytes of device memory in every CUDA
// context that loads this library's module, until the context goes away.  In
// host code its name is only a host-side stand-in, so its device address is
// looked up with cudaGetSymbolAddress in the context current at the call.
// The address belongs to that context's copy of the module: it is cached per
// context (keyed by the driver's context id, which is never reused within a
// process), so a call made after cudaDeviceReset, or under another context
// the caller made current on the same device, looks the address up afresh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "cp_internal.h"

namespace cpattn {
namespace {

constexpr size_t kNoallocScratchBytes = CP_NOALLOC_SCRATCH_BYTES;

// Shared by every call of cp_ring_attention_fwd_noalloc in a context.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct DriverFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const DriverFns &driver_fns() {
    static DriverFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    return fns;
}

// A few recently used contexts and the array's address in each.
constexpr int kCacheSlots = 16;
struct Slot {
    unsigned long long ctx_id = 0;  // 0: empty (driver ids start at 1)
    void *addr = nullptr;
};
std::mutex g_scratch_mu;
Slot g_slots[kCacheSlots];
int g_next_slot = 0;

// Device address of the scratch array in the current context.
cp_status scratch_address(void **out) {
    void *p = nullptr;
    unsigned long long id = 0;
    const DriverFns &fns = driver_fns();
    CUcontext ctx = nullptr;
    if (fns.get_current && fns.get_id && fns.get_current(&ctx) == CUDA_SUCCESS && ctx &&
        fns.get_id(ctx, &id) == CUDA_SUCCESS && id != 0) {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        for (const Slot &s : g_slots)
            if (s.ctx_id == id) {
                *out = s.addr;
                return CP_OK;
            }
    } else {
        id = 0;  // no usable context id: look the address up on every call
    }
    // also makes the runtime's primary context current on this thread if none
    // is, and loads the module
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_status(e);
    if (!p) return CP_ERR_CUDA;
    if (id == 0) {
        // the lookup above made the runtime's context current: key it now
        if (fns.get_current && fns.get_id && fns.get_current(&ctx) == CUDA_SUCCESS && ctx &&
            fns.get_id(ctx, &id) != CUDA_SUCCESS)
            id = 0;
    }
    if (id != 0) {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        g_slots[g_next_slot].ctx_id = id;
        g_slots[g_next_slot].addr = p;
        g_next_slot = (g_next_slot + 1) % kCacheSlots;
    }
    *out = p;
    return CP_OK;
}

}  // namespace
}  // namespace cpattn

extern "C" cp_status cp_ring_attention_fwd_noalloc(const void *q_sh, const void *k_sh, const void *v_sh,
                                                   const int32_t *pos, int64_t B, int64_t S, int64_t N,
                                                   int64_t Nkv, int64_t D, int C, float scale, cp_layout layout,
                                                   void *o_sh, cp_dtype o_dtype, float *lse_sh,
                                                   cudaStream_t stream) {
    // the ring's own argument checks first, so a bad pointer or shape is
    // reported as such whatever the size
    cp_status st = cpattn::ring_check_args(q_sh, k_sh, v_sh, pos, B, S, N, Nkv, D, C, scale, layout, 0, o_sh,
                                           o_dtype, lse_sh);
    if (st != CP_OK) return st;
    size_t need = 0;
    st = cp_ring_workspace_size(B, S, N, Nkv, D, C, 0, o_dtype, &need);
    if (st != CP_OK) return st;
    if (need > cpattn::kNoallocScratchBytes) return CP_ERR_WORKSPACE;
    void *scratch = nullptr;
    st = cpattn::scratch_address(&scratch);
    if (st != CP_OK) return st;
    // Every scratch byte this ring reads is written earlier in the same call
    // (step 0 writes the accumulator, each later step writes the partial it
    // merges), so nothing left by a previous call needs clearing.
    return cp_ring_attention_fwd(q_sh, k_sh, v_sh, pos, B, S, N, Nkv, D, C, scale, layout, 0, o_sh, o_dtype, lse_sh,
                                 scratch, cpattn::kNoallocScratchBytes, stream);
}
