// iha_noalloc.cu -- iha_forward_noalloc: the forward pass for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocator): a process whose device memory is
// already reserved in full by another framework's pool, or code on a path where an
// allocation may not happen at all (it could fail, block on the driver, or synchronise the
// device).  For them the workspace of the four steps lives in a fixed array compiled into
// this library, so a call needs nothing but the caller's inputs and output.
#include <cuda_runtime.h>

#include <mutex>

#include "iha.h"
#include "iha_internal.h"

namespace iha {

// The scratch array: every GPU on which the library is loaded holds one copy until the
// process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[IHA_NOALLOC_SCRATCH_BYTES];

static constexpr int kMaxNoallocDevices = 64;
static void *g_scratch_addr[kMaxNoallocDevices];
static std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on the current device.  On the host the array's name
// only stands in for it, so the address is looked up once per device (with that device
// current) and cached; a lookup failure is returned as NULL.
static void *scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoallocDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace iha

extern "C" int iha_forward_noalloc(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                                   const float *alpha_Q, const float *alpha_K, const float *alpha_V,
                                   const float *R, int B, int N, int H, int d, int P, int mask_mode, int window,
                                   void *out, int dtype, void *stream) {
    const int rc = iha::check_forward_args(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P,
                                           mask_mode, window, out, dtype);
    if (rc != IHA_OK) return rc;
    // problems whose workspace does not fit the fixed array are refused
    if (iha_workspace_bytes(B, N, H, d, P, dtype) > (size_t)IHA_NOALLOC_SCRATCH_BYTES) return IHA_ERR_WORKSPACE;
    void *scratch = iha::scratch_address();
    if (!scratch) return IHA_ERR_CUDA;
    return iha::forward_in_workspace(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, iha::Shape{B, N, H, d, P},
                                     mask_mode, window, out, dtype, static_cast<cudaStream_t>(stream), scratch,
                                     (size_t)IHA_NOALLOC_SCRATCH_BYTES);
}
