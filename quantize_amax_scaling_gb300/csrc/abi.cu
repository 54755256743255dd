// abi.cu -- libfp8q's error reporting and status strings.

#include "fp8q_common.cuh"

namespace fp8q_detail {

thread_local char g_last_error[256] = "";

fp8q_status cuda_fail(cudaError_t e, const char* where) {
    std::snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where, cudaGetErrorName(e),
                  cudaGetErrorString(e));
    // The failing runtime call also left e as the thread's last CUDA error.
    // Consume it here, where it is reported, so that the caller's own next
    // check (cudaGetLastError) does not report it a second time.  A sticky
    // error (a lost context) stays set whatever is done here.
    (void)cudaGetLastError();
    return FP8Q_ERR_CUDA;
}

}  // namespace fp8q_detail

using namespace fp8q_detail;

extern "C" {

const char* fp8q_status_string(fp8q_status status) {
    switch (status) {
        case FP8Q_OK: return "FP8Q_OK";
        case FP8Q_ERR_INVALID_ARG: return "FP8Q_ERR_INVALID_ARG";
        case FP8Q_ERR_UNSUPPORTED: return "FP8Q_ERR_UNSUPPORTED";
        case FP8Q_ERR_CUDA: return "FP8Q_ERR_CUDA";
        case FP8Q_ERR_TOO_MANY_TENSORS: return "FP8Q_ERR_TOO_MANY_TENSORS";
    }
    return "FP8Q_ERR_UNKNOWN";
}

const char* fp8q_last_cuda_error(void) { return g_last_error; }

}  // extern "C"
