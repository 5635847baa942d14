// iha_api.cu -- the C ABI declared in include/iha.h: argument validation, workspace
// layout, the per-device status word, and the launch sequence (slice -> project+mix, or
// fold -> project) -> attention -> contract of "Interleaved Head Attention" Algorithm 1.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "iha.h"
#include "iha_internal.h"

namespace iha {

// Per-device word that kernels set (first writer wins) when a bounded wait expires.
static __device__ int g_status_word;

static constexpr int kMaxDevices = 64;
static int *g_status_ptr[kMaxDevices];
static std::mutex g_mu;

static int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

// Device address of g_status_word on the current device (looked up once per device;
// the host-side name of the variable is only a stand-in for it).
static int *status_ptr() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

int *status_word_ptr() { return status_ptr(); }

int device_sm_count() {
    static int counts[kMaxDevices];
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 1;
    if (!counts[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        counts[dev] = n > 0 ? n : 1;
    }
    return counts[dev];
}

static size_t elem_size(int dtype) { return dtype == IHA_DTYPE_BF16 ? 2 : 4; }
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static int validate_shape(int B, int N, int H, int d, int P, int dtype) {
    if (B <= 0 || N <= 0 || H <= 0 || d <= 0 || P <= 0) return IHA_ERR_INVALID_ARG;
    if (dtype != IHA_DTYPE_F32 && dtype != IHA_DTYPE_BF16) return IHA_ERR_INVALID_ARG;
    const long long L = (long long)N * P, D = (long long)H * d;
    // index ranges the kernels use: int for rows/columns, grid dims < 2^31 / 65536
    if (L > (1LL << 24) || D > (1LL << 20) || (long long)B * N > INT_MAX / 2 || (long long)B * H > INT_MAX / 2 ||
        3LL * H * P * d > INT_MAX / 2)
        return IHA_ERR_UNSUPPORTED;
    // attention grids: one CTA per (b, h, 256 stacked rows) (bf16), one warp per row (fp32)
    if ((long long)B * H * ((L + 255) / 256) > INT_MAX || (long long)B * H * L > (1LL << 34)) return IHA_ERR_UNSUPPORTED;
    if (dtype == IHA_DTYPE_BF16 && d != 64 && d != 128) return IHA_ERR_UNSUPPORTED;
    if (H > 64) return IHA_ERR_UNSUPPORTED;   // the weight fold keeps one W column per head in registers
    if (dtype == IHA_DTYPE_F32 && d > 256) return IHA_ERR_UNSUPPORTED;
    return IHA_OK;
}

static int validate_mask(int mask_mode, int window) {
    if (mask_mode < IHA_MASK_NONE || mask_mode > IHA_MASK_WINDOW) return IHA_ERR_INVALID_ARG;
    if (mask_mode == IHA_MASK_WINDOW && window < 1) return IHA_ERR_INVALID_ARG;
    return IHA_OK;
}

struct WsLayout {
    size_t wt, qkv, pbar, ctr, total;
};

static WsLayout ws_layout(const Shape &sh, int dtype) {
    const size_t es = elem_size(dtype);
    WsLayout w;
    w.wt = 0;   // folded weights Wt, or the slice-major weights Wp on the unfolded route
    const size_t first = unfolded_route(sh, dtype) ? sliced_weights_bytes(sh) : (size_t)sh.wt_rows() * (size_t)sh.D() * es;
    w.qkv = align256(first);
    w.pbar = w.qkv + align256(3 * (size_t)sh.qkv_elems() * es);
    w.ctr = w.pbar + align256((size_t)sh.B * sh.N * sh.H * sh.P * sh.d * es);
    w.total = w.ctr + kCtrlBytes;   // the call's own attention work counter
    return w;
}

static int cuda_status(cudaError_t e) { return status_from_cuda(e); }

static int run_forward(const void *X, const void *WQ, const void *WK, const void *WV, const float *aQ,
                       const float *aK, const float *aV, const float *R, const Shape &sh, int mask_mode, int window,
                       void *out, int dtype, cudaStream_t st, void *workspace, size_t workspace_bytes) {
    const WsLayout lay = ws_layout(sh, dtype);
    bool own = false;
    if (!workspace) {
        if (cudaMallocAsync(&workspace, lay.total, st) != cudaSuccess) return IHA_ERR_CUDA;
        own = true;
    } else if (workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255)) {
        return IHA_ERR_WORKSPACE;
    }
    int *status = status_ptr();
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *Wt = ws + lay.wt, *QKV = ws + lay.qkv, *Pbar = ws + lay.pbar;
    unsigned int *ticket = reinterpret_cast<unsigned int *>(ws + lay.ctr);
    cudaError_t e;
    if (unfolded_route(sh, dtype)) {
        e = launch_slice_weights(WQ, WK, WV, sh, Wt, st);
        if (e == cudaSuccess)
            e = launch_project_mix(X, Wt, aQ, aK, aV, sh, 0, (long long)sh.B * sh.N, QKV, nullptr, st, status);
    } else {
        e = launch_fold(WQ, WK, WV, aQ, aK, aV, sh, dtype, Wt, st);
        if (e == cudaSuccess) e = launch_project(X, Wt, sh, dtype, QKV, st, status);
    }
    if (e == cudaSuccess) e = launch_attention(QKV, sh, mask_mode, window, dtype, Pbar, st, status, ticket);
    if (e == cudaSuccess) e = launch_contract(Pbar, R, sh, dtype, out, st, status);
    if (own) {
        const cudaError_t e2 = cudaFreeAsync(workspace, st);
        if (e == cudaSuccess) e = e2;
    }
    return cuda_status(e);
}

// Two non-blocking streams per device for host<->device copies: one takes every upload and
// the other every download, so the two directions overlap (about 207 GB/s up and 191 GB/s
// down; a second stream in the same direction did not add to that).
static cudaStream_t *copy_streams() {
    static std::mutex mu;
    static cudaStream_t streams[64][2];
    static bool made[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!made[dev]) {
        if (cudaStreamCreateWithFlags(&streams[dev][0], cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        if (cudaStreamCreateWithFlags(&streams[dev][1], cudaStreamNonBlocking) != cudaSuccess) {
            cudaStreamDestroy(streams[dev][0]);
            return nullptr;
        }
        made[dev] = true;
    }
    return streams[dev];
}

// iha_forward_host on the unfolded bf16 route with the copies overlapped with the work.  All
// uploads go on copy stream 0 in the order the work needs them (W, alpha, R, then X in token
// chunks) and all downloads on copy stream 1: copies queued on two streams in the same
// direction did not share the host link but ran one stream after the other.  The projection
// and mixing of a chunk start as soon as it has landed.  With several batch elements the
// chunks are whole batch elements: each chunk's attention and contraction follow its
// projection, and its output goes down while the next chunk is computed (window 1024, B=4,
// N=4096: 1.26 against 1.43 ms end to end).  With one batch element the attention runs once
// after the last projection and the contraction runs in token chunks: chunking the attention by
// ranges of query blocks (the keys a causal query reads all come earlier) was slower, because
// each range's work items are alike and every launch ends on a long tail of them (causal P=4
// N=8192: 3.80 against 3.55 ms).  `st` waits for both copy streams at the end, so the call
// completes on `st` as the plain sequence does.
constexpr int FH_CHUNKS = 4;
static int forward_host_overlapped(const void *X, const void *WQ, const void *WK, const void *WV, const float *aQ,
                                   const float *aK, const float *aV, const float *R, const Shape &sh, int mask_mode,
                                   int window, void *out, void *dX, void *dWQ, void *dWK, void *dWV, float *daQ,
                                   float *daK, float *daV, float *dR, void *dOut, void *ws, cudaStream_t st) {
    cudaStream_t *cs = copy_streams();
    if (!cs) return IHA_ERR_CUDA;
    const long long T = (long long)sh.B * sh.N, D = sh.D();
    const size_t wb = (size_t)D * D * 2, ab = (size_t)sh.H * sh.H * sh.P * sizeof(float);
    const size_t row_x = (size_t)D * 2, row_p = (size_t)sh.H * sh.P * sh.d * 2;
    const WsLayout lay = ws_layout(sh, IHA_DTYPE_BF16);
    uint8_t *w8 = static_cast<uint8_t *>(ws);
    uint8_t *Wp = w8 + lay.wt, *QKV = w8 + lay.qkv, *Pbar = w8 + lay.pbar;
    unsigned int *ticket = reinterpret_cast<unsigned int *>(w8 + lay.ctr);
    int *status = status_ptr();
    // token chunks [tk[c], tk[c+1]) and, when the attention runs per chunk (whole batch
    // elements), its head ranges
    long long tk[FH_CHUNKS + 1];
    AttnRange rg[FH_CHUNKS];
    int nc = FH_CHUNKS;
    bool per_chunk = false;
    const int nqb = (int)((sh.L() + kAttnRowsPerBlock - 1) / kAttnRowsPerBlock);
    if (sh.B > 1) {   // whole batch elements
        nc = sh.B < FH_CHUNKS ? sh.B : FH_CHUNKS;
        per_chunk = true;
        for (int c = 0; c <= nc; ++c) tk[c] = (long long)(sh.B * c / nc) * sh.N;
        for (int c = 0; c < nc; ++c)
            rg[c] = AttnRange{(int)(tk[c] / sh.N) * sh.H, (int)((tk[c + 1] - tk[c]) / sh.N) * sh.H, 0, nqb};
    } else {
        for (int c = 0; c <= nc; ++c) tk[c] = T * c / nc;
    }
    // events: 0 start, 1 W ready, 2.. X chunks, then contraction chunks, then the two copy
    // streams' last copies
    constexpr int NEV = 2 + 2 * FH_CHUNKS + 2;
    cudaEvent_t ev[NEV] = {};
    cudaError_t e = cudaSuccess;
    int made = 0;
    while (made < NEV && (e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming)) == cudaSuccess) ++made;
    const uint8_t *Xh = static_cast<const uint8_t *>(X);
    uint8_t *outh = static_cast<uint8_t *>(out);
    if (e == cudaSuccess) e = cudaEventRecord(ev[0], st);   // after earlier work on st
    for (int c = 0; c < 2 && e == cudaSuccess; ++c) e = cudaStreamWaitEvent(cs[c], ev[0], 0);
    // uploads, in the order the work needs them, on copy stream 0
    const cudaStream_t up = cs[0], down = cs[1];
    if (e == cudaSuccess) e = cudaMemcpyAsync(dWQ, WQ, wb, cudaMemcpyHostToDevice, up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dWK, WK, wb, cudaMemcpyHostToDevice, up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dWV, WV, wb, cudaMemcpyHostToDevice, up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(daQ, aQ, ab, cudaMemcpyHostToDevice, up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(daK, aK, ab, cudaMemcpyHostToDevice, up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(daV, aV, ab, cudaMemcpyHostToDevice, up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dR, R, ab, cudaMemcpyHostToDevice, up);
    if (e == cudaSuccess) e = cudaEventRecord(ev[1], up);
    for (int c = 0; c < nc && e == cudaSuccess; ++c) {
        if (tk[c + 1] > tk[c])
            e = cudaMemcpyAsync(static_cast<uint8_t *>(dX) + tk[c] * row_x, Xh + tk[c] * row_x,
                                (tk[c + 1] - tk[c]) * row_x, cudaMemcpyHostToDevice, up);
        if (e == cudaSuccess) e = cudaEventRecord(ev[2 + c], up);
    }
    // contraction of tokens [r0, r1) and its download
    int ncon = 0;
    auto contract_down = [&](long long r0, long long r1) {
        if (r1 > r0)
            e = launch_contract_tc(Pbar + r0 * row_p, dR, Shape{1, (int)(r1 - r0), sh.H, sh.d, sh.P},
                                   static_cast<uint8_t *>(dOut) + r0 * row_x, st, status);
        const int k = 2 + FH_CHUNKS + ncon++;
        if (e == cudaSuccess) e = cudaEventRecord(ev[k], st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(down, ev[k], 0);
        if (e == cudaSuccess && r1 > r0)
            e = cudaMemcpyAsync(outh + r0 * row_x, static_cast<uint8_t *>(dOut) + r0 * row_x, (r1 - r0) * row_x,
                                cudaMemcpyDeviceToHost, down);
    };
    // projection and mixing chunk by chunk, straight into the stacked layout
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev[1], 0);
    if (e == cudaSuccess) e = launch_slice_weights(dWQ, dWK, dWV, sh, Wp, st);
    for (int c = 0; c < nc && e == cudaSuccess; ++c) {
        e = cudaStreamWaitEvent(st, ev[2 + c], 0);
        if (e == cudaSuccess && tk[c + 1] > tk[c])
            e = launch_project_mix(dX, Wp, daQ, daK, daV, sh, tk[c], tk[c + 1] - tk[c], QKV, nullptr, st, status);
        if (per_chunk && e == cudaSuccess) {
            // the chunk's batch elements: their queries read keys of their own only
            e = launch_attention_range(QKV, sh, mask_mode, window, Pbar, rg[c], st, status, ticket);
            if (e == cudaSuccess) contract_down(tk[c], tk[c + 1]);
        }
    }
    if (!per_chunk) {
        if (e == cudaSuccess)
            e = launch_attention(QKV, sh, mask_mode, window, IHA_DTYPE_BF16, Pbar, st, status, ticket);
        for (int c = 0; c < nc && e == cudaSuccess; ++c) contract_down(tk[c], tk[c + 1]);
    }
    // The call completes on st: st waits for everything queued on the copy streams -- also
    // after an error, so that no copy still runs when the caller reuses its buffers (without
    // the events, the host waits for the copy streams instead).
    for (int c = 0; c < 2; ++c) {
        const int k = 2 + 2 * FH_CHUNKS + c;
        cudaError_t e2 = k < made ? cudaEventRecord(ev[k], cs[c]) : cudaErrorInvalidValue;
        if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st, ev[k], 0);
        if (e2 != cudaSuccess) {
            const cudaError_t e3 = cudaStreamSynchronize(cs[c]);
            if (e == cudaSuccess) e = e3 != cudaSuccess ? e3 : e2;
        }
    }
    for (int k = 0; k < made; ++k) cudaEventDestroy(ev[k]);   // released once their work is done
    return cuda_status(e);
}

// Entry points outside this file reuse the checks and the launch sequence of
// iha_forward_ex through these two functions.
int check_forward_args(const void *X, const void *WQ, const void *WK, const void *WV, const float *aQ,
                       const float *aK, const float *aV, const float *R, int B, int N, int H, int d, int P,
                       int mask_mode, int window, const void *out, int dtype) {
    if (!X || !WQ || !WK || !WV || !aQ || !aK || !aV || !R || !out) return IHA_ERR_INVALID_ARG;
    int rc = validate_shape(B, N, H, d, P, dtype);
    if (rc == IHA_OK) rc = validate_mask(mask_mode, window);
    return rc;
}

int forward_in_workspace(const void *X, const void *WQ, const void *WK, const void *WV, const float *aQ,
                         const float *aK, const float *aV, const float *R, const Shape &sh, int mask_mode,
                         int window, void *out, int dtype, cudaStream_t st, void *workspace,
                         size_t workspace_bytes) {
    if (!workspace) return IHA_ERR_WORKSPACE;
    return run_forward(X, WQ, WK, WV, aQ, aK, aV, R, sh, mask_mode, window, out, dtype, st, workspace,
                       workspace_bytes);
}

}  // namespace iha

using namespace iha;

extern "C" {

const char *iha_error_string(int status) {
    switch (status) {
        case IHA_OK: return "ok";
        case IHA_ERR_INVALID_ARG: return "invalid argument";
        case IHA_ERR_UNSUPPORTED: return "unsupported configuration";
        case IHA_ERR_WORKSPACE: return "workspace too small or misaligned";
        case IHA_ERR_CUDA: return "CUDA error";
        case IHA_ERR_TIMEOUT: return "device wait timed out";
        case IHA_ERR_BUILD: return "library build does not match this device or a kernel's register contract: rebuild";
        default: return "unknown status";
    }
}

size_t iha_workspace_bytes(int B, int N, int H, int d, int P, int dtype) {
    if (validate_shape(B, N, H, d, P, dtype) != IHA_OK) return 0;
    return ws_layout(Shape{B, N, H, d, P}, dtype).total;
}

int iha_forward_ex(const void *X, const void *W_Q, const void *W_K, const void *W_V, const float *alpha_Q,
                   const float *alpha_K, const float *alpha_V, const float *R, int B, int N, int H, int d, int P,
                   int mask_mode, int window, void *out, int dtype, void *stream, void *workspace,
                   size_t workspace_bytes) {
    if (!X || !W_Q || !W_K || !W_V || !alpha_Q || !alpha_K || !alpha_V || !R || !out) return IHA_ERR_INVALID_ARG;
    int rc = validate_shape(B, N, H, d, P, dtype);
    if (rc == IHA_OK) rc = validate_mask(mask_mode, window);
    if (rc != IHA_OK) return rc;
    return run_forward(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, Shape{B, N, H, d, P}, mask_mode, window, out,
                       dtype, static_cast<cudaStream_t>(stream), workspace, workspace_bytes);
}

int iha_prefill(const void *X, const void *W_Q, const void *W_K, const void *W_V, const float *alpha_Q,
                const float *alpha_K, const float *alpha_V, const float *R, int B, int N, int H, int d, int P,
                int mask_mode, int window, void *out, void *K_cache, void *V_cache, int cache_tokens, int dtype,
                void *stream, void *workspace, size_t workspace_bytes) {
    int rc = check_forward_args(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window,
                                out, dtype);
    if (rc != IHA_OK) return rc;
    if (!K_cache || !V_cache || cache_tokens < N || mask_mode == IHA_MASK_NONE) return IHA_ERR_INVALID_ARG;
    if (dtype != IHA_DTYPE_BF16 || !decode_supported(H, d, P)) return IHA_ERR_UNSUPPORTED;
    const Shape sh{B, N, H, d, P};
    const WsLayout lay = ws_layout(sh, dtype);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool own = false;
    if (!workspace) {
        if (cudaMallocAsync(&workspace, lay.total, st) != cudaSuccess) return IHA_ERR_CUDA;
        own = true;
        workspace_bytes = lay.total;
    }
    rc = run_forward(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, sh, mask_mode, window, out, dtype, st, workspace,
                     workspace_bytes);
    if (rc == IHA_OK) {
        // Kbar, Vbar [B][H][N*P][d] -> the caches [B][H][cache_tokens*P][d]
        const uint8_t *qkv = static_cast<const uint8_t *>(workspace) + lay.qkv;
        const size_t blk = (size_t)N * P * d * 2, cap = (size_t)cache_tokens * P * d * 2;
        const size_t third = (size_t)sh.qkv_elems() * 2;
        cudaError_t e = cudaMemcpy2DAsync(K_cache, cap, qkv + third, blk, blk, (size_t)B * H, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(V_cache, cap, qkv + 2 * third, blk, blk, (size_t)B * H, cudaMemcpyDeviceToDevice, st);
        rc = cuda_status(e);
    }
    if (own) {
        const cudaError_t e = cudaFreeAsync(workspace, st);
        if (rc == IHA_OK && e != cudaSuccess) rc = IHA_ERR_CUDA;
    }
    return rc;
}

int iha_forward(const void *X, const void *W_Q, const void *W_K, const void *W_V, const float *alpha_Q,
                const float *alpha_K, const float *alpha_V, const float *R, int B, int N, int H, int d, int P,
                int mask_mode, int window, void *out) {
    return iha_forward_ex(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, out,
                          IHA_DTYPE_BF16, nullptr, nullptr, 0);
}

int iha_check_device_status(void *stream, int *code_out) {
    if (code_out) *code_out = 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return IHA_ERR_CUDA;
    int *p = status_ptr();
    if (!p) return IHA_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return IHA_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return IHA_ERR_CUDA;
    }
    if (code_out) *code_out = word;
    return word ? IHA_ERR_TIMEOUT : IHA_OK;
}

size_t iha_host_buffer_bytes(int B, int N, int H, int d, int P, int dtype) {
    if (validate_shape(B, N, H, d, P, dtype) != IHA_OK) return 0;
    const Shape sh{B, N, H, d, P};
    const size_t es = elem_size(dtype);
    const size_t x = (size_t)B * N * sh.D() * es, w = (size_t)sh.D() * sh.D() * es;
    const size_t a = (size_t)H * H * P * sizeof(float), r = (size_t)H * H * P * sizeof(float);
    return align256(x) + 3 * align256(w) + 3 * align256(a) + align256(r) + align256(x) + ws_layout(sh, dtype).total;
}

int iha_forward_host(const void *X, const void *W_Q, const void *W_K, const void *W_V, const float *alpha_Q,
                     const float *alpha_K, const float *alpha_V, const float *R, int B, int N, int H, int d, int P,
                     int mask_mode, int window, void *out, int dtype, void *stream, void *device_buffer,
                     size_t device_buffer_bytes) {
    if (!X || !W_Q || !W_K || !W_V || !alpha_Q || !alpha_K || !alpha_V || !R || !out) return IHA_ERR_INVALID_ARG;
    int rc = validate_shape(B, N, H, d, P, dtype);
    if (rc == IHA_OK) rc = validate_mask(mask_mode, window);
    if (rc != IHA_OK) return rc;
    const Shape sh{B, N, H, d, P};
    const size_t need = iha_host_buffer_bytes(B, N, H, d, P, dtype);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool own = false;
    if (!device_buffer) {
        if (cudaMallocAsync(&device_buffer, need, st) != cudaSuccess) return IHA_ERR_CUDA;
        own = true;
    } else if (device_buffer_bytes < need || (reinterpret_cast<uintptr_t>(device_buffer) & 255)) {
        return IHA_ERR_WORKSPACE;
    }
    const size_t es = elem_size(dtype);
    const size_t xb = (size_t)B * N * sh.D() * es, wb = (size_t)sh.D() * sh.D() * es;
    const size_t ab = (size_t)H * H * P * sizeof(float), rb = ab;
    uint8_t *p = static_cast<uint8_t *>(device_buffer);
    auto take = [&](size_t bytes) {
        uint8_t *q = p;
        p += align256(bytes);
        return q;
    };
    void *dX = take(xb), *dWQ = take(wb), *dWK = take(wb), *dWV = take(wb);
    float *daQ = (float *)take(ab), *daK = (float *)take(ab), *daV = (float *)take(ab), *dR = (float *)take(rb);
    void *dOut = take(xb);
    void *ws = p;
    if (unfolded_route(sh, dtype) && contract_tc_fits(sh)) {
        rc = forward_host_overlapped(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, sh, mask_mode, window, out,
                                     dX, dWQ, dWK, dWV, daQ, daK, daV, dR, dOut, ws, st);
        if (own && cudaFreeAsync(device_buffer, st) != cudaSuccess && rc == IHA_OK) rc = IHA_ERR_CUDA;
        const int rc2 = iha_check_device_status(stream, nullptr);
        return rc != IHA_OK ? rc : rc2;
    }
    cudaError_t e = cudaSuccess;
    const void *srcs[8] = {X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R};
    void *dsts[8] = {dX, dWQ, dWK, dWV, daQ, daK, daV, dR};
    const size_t sizes[8] = {xb, wb, wb, wb, ab, ab, ab, rb};
    for (int i = 0; i < 8 && e == cudaSuccess; ++i)
        e = cudaMemcpyAsync(dsts[i], srcs[i], sizes[i], cudaMemcpyHostToDevice, st);
    rc = e == cudaSuccess ? IHA_OK : IHA_ERR_CUDA;
    if (rc == IHA_OK)
        rc = run_forward(dX, dWQ, dWK, dWV, daQ, daK, daV, dR, sh, mask_mode, window, dOut, dtype, st, ws,
                         ws_layout(sh, dtype).total);
    if (rc == IHA_OK && cudaMemcpyAsync(out, dOut, xb, cudaMemcpyDeviceToHost, st) != cudaSuccess) rc = IHA_ERR_CUDA;
    if (own && cudaFreeAsync(device_buffer, st) != cudaSuccess && rc == IHA_OK) rc = IHA_ERR_CUDA;
    const int rc2 = iha_check_device_status(stream, nullptr);
    return rc != IHA_OK ? rc : rc2;
}

int iha_selftest_wait_timeout(void *stream, int limit_ms) {
    if (limit_ms < 1 || limit_ms > 10000) return IHA_ERR_INVALID_ARG;
    int *status = status_ptr();
    if (!status) return IHA_ERR_CUDA;
    return cuda_status(
        launch_wait_selftest(status, (unsigned long long)limit_ms * 1000000ull, static_cast<cudaStream_t>(stream)));
}

int iha_fold_weights(const void *W_Q, const void *W_K, const void *W_V, const float *alpha_Q, const float *alpha_K,
                     const float *alpha_V, int H, int d, int P, int dtype, void *Wt, void *stream) {
    if (!W_Q || !W_K || !W_V || !alpha_Q || !alpha_K || !alpha_V || !Wt) return IHA_ERR_INVALID_ARG;
    const int rc = validate_shape(1, 1, H, d, P, dtype);
    if (rc != IHA_OK) return rc;
    return cuda_status(launch_fold(W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, Shape{1, 1, H, d, P}, dtype, Wt,
                                   static_cast<cudaStream_t>(stream)));
}

int iha_project(const void *X, const void *Wt, int B, int N, int H, int d, int P, int dtype, void *QKV,
                void *stream) {
    if (!X || !Wt || !QKV) return IHA_ERR_INVALID_ARG;
    const int rc = validate_shape(B, N, H, d, P, dtype);
    if (rc != IHA_OK) return rc;
    return cuda_status(
        launch_project(X, Wt, Shape{B, N, H, d, P}, dtype, QKV, static_cast<cudaStream_t>(stream), status_ptr()));
}

int iha_projection_route(int H, int d, int P, int dtype) {
    if (validate_shape(1, 1, H, d, P, dtype) != IHA_OK) return -1;
    return unfolded_route(Shape{1, 1, H, d, P}, dtype) ? 1 : 0;
}

int iha_project_heads(const void *X, const void *W_Q, const void *W_K, const void *W_V, int B, int N, int H, int d,
                      int dtype, void *Y, void *stream) {
    if (!X || !W_Q || !W_K || !W_V || !Y) return IHA_ERR_INVALID_ARG;
    const int rc = validate_shape(B, N, H, d, 1, dtype);
    if (rc != IHA_OK) return rc;
    if (dtype != IHA_DTYPE_BF16) return IHA_ERR_UNSUPPORTED;
    return cuda_status(launch_project_heads(X, W_Q, W_K, W_V, Shape{B, N, H, d, 1}, Y,
                                            static_cast<cudaStream_t>(stream), status_ptr()));
}

size_t iha_sliced_weights_bytes(int H, int d, int dtype) {
    if (validate_shape(1, 1, H, d, 1, dtype) != IHA_OK || dtype != IHA_DTYPE_BF16) return 0;
    const Shape sh{1, 1, H, d, 1};
    return project_mix_supported(sh) ? sliced_weights_bytes(sh) : 0;
}

int iha_slice_weights(const void *W_Q, const void *W_K, const void *W_V, int H, int d, int dtype, void *Wp,
                      void *stream) {
    if (!W_Q || !W_K || !W_V || !Wp) return IHA_ERR_INVALID_ARG;
    if (iha_sliced_weights_bytes(H, d, dtype) == 0) return IHA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(W_Q) | reinterpret_cast<uintptr_t>(W_K) | reinterpret_cast<uintptr_t>(W_V) |
         reinterpret_cast<uintptr_t>(Wp)) & 15)
        return IHA_ERR_INVALID_ARG;
    return cuda_status(launch_slice_weights(W_Q, W_K, W_V, Shape{1, 1, H, d, 1}, Wp, static_cast<cudaStream_t>(stream)));
}

int iha_project_mix(const void *X, const void *Wp, const float *alpha_Q, const float *alpha_K, const float *alpha_V,
                    int B, int N, int H, int d, int P, int dtype, void *QKV, void *stream) {
    if (!X || !Wp || !alpha_Q || !alpha_K || !alpha_V || !QKV) return IHA_ERR_INVALID_ARG;
    const int rc = validate_shape(B, N, H, d, P, dtype);
    if (rc != IHA_OK) return rc;
    const Shape sh{B, N, H, d, P};
    if (dtype != IHA_DTYPE_BF16 || !project_mix_supported(sh)) return IHA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(QKV) & 31) || (reinterpret_cast<uintptr_t>(Wp) & 15)) return IHA_ERR_INVALID_ARG;
    return cuda_status(launch_project_mix(X, Wp, alpha_Q, alpha_K, alpha_V, sh, 0, (long long)B * N, QKV, nullptr,
                                          static_cast<cudaStream_t>(stream), status_ptr()));
}

int iha_mix_heads(const void *Y, const float *alpha_Q, const float *alpha_K, const float *alpha_V, int B, int N, int H,
                  int d, int P, int dtype, void *QKV, void *stream) {
    if (!Y || !alpha_Q || !alpha_K || !alpha_V || !QKV) return IHA_ERR_INVALID_ARG;
    const int rc = validate_shape(B, N, H, d, P, dtype);
    if (rc != IHA_OK) return rc;
    if (dtype != IHA_DTYPE_BF16 || H > 16 || H * P > 128) return IHA_ERR_UNSUPPORTED;
    if (((reinterpret_cast<uintptr_t>(Y) | reinterpret_cast<uintptr_t>(QKV)) & 15) != 0) return IHA_ERR_INVALID_ARG;
    return cuda_status(launch_mix(Y, alpha_Q, alpha_K, alpha_V, Shape{B, N, H, d, P}, QKV,
                                  static_cast<cudaStream_t>(stream), status_ptr()));
}

int iha_attention(const void *QKV, int B, int N, int H, int d, int P, int mask_mode, int window, int dtype,
                  void *Pbar, void *stream) {
    if (!QKV || !Pbar) return IHA_ERR_INVALID_ARG;
    if (((reinterpret_cast<uintptr_t>(QKV) | reinterpret_cast<uintptr_t>(Pbar)) & 15) != 0) return IHA_ERR_INVALID_ARG;
    int rc = validate_shape(B, N, H, d, P, dtype);
    if (rc == IHA_OK) rc = validate_mask(mask_mode, window);
    if (rc != IHA_OK) return rc;
    return cuda_status(launch_attention(QKV, Shape{B, N, H, d, P}, mask_mode, window, dtype, Pbar,
                                        static_cast<cudaStream_t>(stream), status_ptr()));
}

int iha_contract(const void *Pbar, const float *R, int B, int N, int H, int d, int P, int dtype, void *out,
                 void *stream) {
    if (!Pbar || !R || !out) return IHA_ERR_INVALID_ARG;
    const int rc = validate_shape(B, N, H, d, P, dtype);
    if (rc != IHA_OK) return rc;
    return cuda_status(
        launch_contract(Pbar, R, Shape{B, N, H, d, P}, dtype, out, static_cast<cudaStream_t>(stream), status_ptr()));
}

}  // extern "C"
