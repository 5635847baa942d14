// iha_decode.cu -- the C-ABI of incremental decoding: one new token per sequence against a
// cache of pseudo-keys and pseudo-values (kernels in k_decode.cu).
#include <cuda_runtime.h>

#include "iha.h"
#include "iha_internal.h"

using namespace iha;

extern "C" {

size_t iha_decode_workspace_bytes(int B, int H, int d, int P) {
    if (B <= 0 || H <= 0 || P <= 0 || !decode_supported(H, d, P)) return 0;
    return decode_workspace_bytes(B, H, d, P);
}

int iha_decode_step(const void *x, const void *W_Q, const void *W_K, const void *W_V, const float *alpha_Q,
                    const float *alpha_K, const float *alpha_V, const float *R, int B, int H, int d, int P,
                    int mask_mode, int window, void *K_cache, void *V_cache, int cache_tokens, int t, void *out,
                    int dtype, void *stream, void *workspace, size_t workspace_bytes) {
    // the shape checks of iha_forward_ex with N = t + 1 tokens of history
    int rc = check_forward_args(x, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, t + 1, H, d, P, mask_mode, window,
                                out, dtype);
    if (rc != IHA_OK) return rc;
    if (!K_cache || !V_cache || t < 0 || t >= cache_tokens || mask_mode == IHA_MASK_NONE) return IHA_ERR_INVALID_ARG;
    // cache rows are written 16 bytes at a time and read by TMA; W rows are read by bulk copies
    if ((reinterpret_cast<uintptr_t>(K_cache) & 15) || (reinterpret_cast<uintptr_t>(V_cache) & 15) ||
        (reinterpret_cast<uintptr_t>(W_Q) & 15) || (reinterpret_cast<uintptr_t>(W_K) & 15) ||
        (reinterpret_cast<uintptr_t>(W_V) & 15))
        return IHA_ERR_INVALID_ARG;
    if (dtype != IHA_DTYPE_BF16 || !decode_supported(H, d, P)) return IHA_ERR_UNSUPPORTED;
    const size_t need = decode_workspace_bytes(B, H, d, P);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool own = false;
    if (!workspace) {
        if (cudaMallocAsync(&workspace, need, st) != cudaSuccess) return IHA_ERR_CUDA;
        own = true;
    } else if (workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255)) {
        return IHA_ERR_WORKSPACE;
    }
    cudaError_t e = launch_decode(x, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, H, d, P, mask_mode, window,
                                  K_cache, V_cache, cache_tokens, t, out, workspace, st, status_word_ptr());
    if (own) {
        const cudaError_t e2 = cudaFreeAsync(workspace, st);
        if (e == cudaSuccess) e = e2;
    }
    return status_from_cuda(e);
}

}  // extern "C"
