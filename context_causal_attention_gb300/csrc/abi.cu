// abi.cu -- status strings and version of the libcpattn C ABI.
#include <cuda_runtime.h>

#include "cp_internal.h"

extern "C" const char *cp_status_string(cp_status status) {
    switch (status) {
        case CP_OK: return "CP_OK";
        case CP_ERR_NULL: return "CP_ERR_NULL: a required pointer is NULL";
        case CP_ERR_SHAPE: return "CP_ERR_SHAPE: a size is out of the supported range";
        case CP_ERR_DIVISIBILITY: return "CP_ERR_DIVISIBILITY: S, N or Nkv not divisible as required";
        case CP_ERR_DTYPE: return "CP_ERR_DTYPE: unknown dtype";
        case CP_ERR_ALIGNMENT: return "CP_ERR_ALIGNMENT: pointer or row not 16-byte aligned";
        case CP_ERR_WORKSPACE: return "CP_ERR_WORKSPACE: workspace missing or too small";
        case CP_ERR_UNSUPPORTED: return "CP_ERR_UNSUPPORTED: unsupported configuration (head dim must be 64 or 128)";
        case CP_ERR_CUDA: return "CP_ERR_CUDA: a CUDA call or kernel launch failed";
        case CP_ERR_DEVICE_TIMEOUT: return "CP_ERR_DEVICE_TIMEOUT: a kernel gave up a bounded device wait";
        case CP_ERR_ARGUMENT: return "CP_ERR_ARGUMENT: invalid argument";
    }
    return "unknown cp_status";
}

extern "C" const char *cp_version(void) { return "0.1.0"; }

namespace cpattn {
namespace {
thread_local cudaError_t t_last_error = cudaSuccess;
}
void note_cuda_error(cudaError_t e) { t_last_error = e; }
}  // namespace cpattn

extern "C" const char *cp_last_cuda_error(void) {
    return cpattn::t_last_error == cudaSuccess ? "no error" : cudaGetErrorString(cpattn::t_last_error);
}
