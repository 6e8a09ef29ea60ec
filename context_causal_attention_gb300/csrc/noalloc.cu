// noalloc.cu -- ring attention forward that allocates nothing.
//
// Some callers cannot call cudaMalloc: code that runs where the device
// allocator is off limits (inside a custom allocator's own callbacks, in a
// runtime that forbids allocation after start-up, or in a process whose
// memory pool is owned by another framework), or that cannot hand this library
// a workspace.  For them cp_ring_attention_fwd_noalloc runs the same ring as
// cp_ring_attention_fwd (zero-copy owner rotation, no prefetch) with its
// scratch -- the per-step partial output and lse, and the fp32 accumulator for
// a bf16 output -- taken from one file-scope device array of fixed size.
//
// The array occupies kNoallocScratchBytes of device memory on every GPU on
// which this library's module is loaded, until the process exits.  In host
// code its name is only a host-side stand-in, so its device address is looked
// up with cudaGetSymbolAddress once per device (with that device current) on
// the first call made on that device, and cached.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "cp_internal.h"

namespace cpattn {
namespace {

constexpr size_t kNoallocScratchBytes = CP_NOALLOC_SCRATCH_BYTES;

// Shared by every call of cp_ring_attention_fwd_noalloc on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.
cp_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return CP_ERR_ARGUMENT;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        if (!p) return CP_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return CP_OK;
}

}  // namespace
}  // namespace cpattn

extern "C" cp_status cp_ring_attention_fwd_noalloc(const void *q_sh, const void *k_sh, const void *v_sh,
                                                   const int32_t *pos, int64_t B, int64_t S, int64_t N,
                                                   int64_t Nkv, int64_t D, int C, float scale, cp_layout layout,
                                                   void *o_sh, cp_dtype o_dtype, float *lse_sh,
                                                   cudaStream_t stream) {
    size_t need = 0;
    cp_status st = cp_ring_workspace_size(B, S, N, Nkv, D, C, 0, o_dtype, &need);
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
