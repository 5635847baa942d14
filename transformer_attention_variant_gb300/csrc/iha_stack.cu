// iha_stack.cu -- a stack of IHA layers, the setting of "Interleaved Head Attention"
// appendix C (the hybrid local/global schedule: four sliding-window IHA layers with window
// N/(2P^2) tokens, then one global layer).  Layer l maps its input [B][N][H*d] to its
// output with its own weights, P, mask and window; layer 0 reads X and layer l+1 reads
// layer l's output.  Algorithm 1 defines the attention layer alone, so nothing else
// (residual, normalisation, MLP) runs between layers.
//
// Each layer is the launch sequence of iha_forward_ex in a slice of one workspace:
//   [activation 0][activation 1][the largest single-layer workspace]   (256-byte aligned)
// Layers alternate between the two activation buffers; the last one writes `out`.
#include <cuda_runtime.h>

#include "iha.h"
#include "iha_internal.h"

namespace iha {

static size_t align256_s(size_t x) { return (x + 255) & ~size_t(255); }

static size_t stack_act_bytes(int B, int N, int H, int d, int dtype) {
    return align256_s((size_t)B * N * H * d * (dtype == IHA_DTYPE_BF16 ? 2 : 4));
}

// Largest single-layer workspace (0 when a layer's shape is invalid).
static size_t stack_layer_ws(int num_layers, const int *P, int B, int N, int H, int d, int dtype) {
    size_t m = 0;
    for (int l = 0; l < num_layers; ++l) {
        const size_t w = iha_workspace_bytes(B, N, H, d, P[l], dtype);
        if (w == 0) return 0;
        if (w > m) m = w;
    }
    return m;
}

}  // namespace iha

using namespace iha;

extern "C" {

size_t iha_stack_workspace_bytes(int num_layers, const int *P, int B, int N, int H, int d, int dtype) {
    if (num_layers <= 0 || !P) return 0;
    const size_t lw = stack_layer_ws(num_layers, P, B, N, H, d, dtype);
    if (lw == 0) return 0;
    return 2 * stack_act_bytes(B, N, H, d, dtype) + lw;
}

int iha_forward_stack(const void *X, int num_layers, const void *const *W_Q, const void *const *W_K,
                      const void *const *W_V, const float *const *alpha_Q, const float *const *alpha_K,
                      const float *const *alpha_V, const float *const *R, const int *P, const int *mask_mode,
                      const int *window, int B, int N, int H, int d, int dtype, void *out, void *stream,
                      void *workspace, size_t workspace_bytes) {
    if (num_layers <= 0 || !W_Q || !W_K || !W_V || !alpha_Q || !alpha_K || !alpha_V || !R || !P || !mask_mode ||
        !window)
        return IHA_ERR_INVALID_ARG;
    // every layer's arguments are checked before anything is launched
    for (int l = 0; l < num_layers; ++l) {
        const int rc = check_forward_args(X, W_Q[l], W_K[l], W_V[l], alpha_Q[l], alpha_K[l], alpha_V[l], R[l], B, N,
                                          H, d, P[l], mask_mode[l], window[l], out, dtype);
        if (rc != IHA_OK) return rc;
    }
    const size_t act = stack_act_bytes(B, N, H, d, dtype);
    const size_t lw = stack_layer_ws(num_layers, P, B, N, H, d, dtype);
    const size_t total = 2 * act + lw;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool own = false;
    if (!workspace) {
        if (cudaMallocAsync(&workspace, total, st) != cudaSuccess) return IHA_ERR_CUDA;
        own = true;
    } else if (workspace_bytes < total || (reinterpret_cast<uintptr_t>(workspace) & 255)) {
        return IHA_ERR_WORKSPACE;
    }
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *buf[2] = {ws, ws + act};
    int rc = IHA_OK;
    for (int l = 0; l < num_layers && rc == IHA_OK; ++l) {
        const void *in = l == 0 ? X : buf[(l - 1) & 1];
        void *dst = l == num_layers - 1 ? out : buf[l & 1];
        rc = forward_in_workspace(in, W_Q[l], W_K[l], W_V[l], alpha_Q[l], alpha_K[l], alpha_V[l], R[l],
                                  Shape{B, N, H, d, P[l]}, mask_mode[l], window[l], dst, dtype, st, ws + 2 * act,
                                  lw);
    }
    if (own) {
        const cudaError_t e = cudaFreeAsync(workspace, st);
        if (rc == IHA_OK && e != cudaSuccess) rc = IHA_ERR_CUDA;
    }
    return rc;
}

}  // extern "C"
