// iha_backward.cu -- the C-ABI of the backward pass of one IHA layer (kernels in
// k_backward.cu, k_backward_tc.cu and the forward kernels it reuses): iha_backward (forward
// pieces recomputed), and the training pair iha_forward_train (the forward, leaving its
// pieces in the backward workspace) + iha_backward_saved (the gradients from them).
//
// Step order (one stream, bf16 tensors, fp32 arithmetic):
//   forward pieces:  Y = X [W_Q|W_K|W_V] and Q~K~V~ = mix(Y) (one kernel: the mixing runs in
//                    the projection GEMM's epilogue);  Pbar, lse = attention(Q~, K~, V~)
//   dPbar  = the mixing of dO with R in alpha's place (stacked; dPbar_{h',j} = sum_h R[h,h'P+j] dO_h)
//   dR     = sum over tokens and columns of dO_h Pbar_k                 (gram_tc)
//   D      = rowdot(dPbar, Pbar)                                       (rowdot)
//   dq~, dk~, dv~ from the attention rule, on the tensor cores           (bwd_attn_tc)
//   dalpha_s = sum over tokens and columns of Y_s,m dS~_s,hj           (gram_tc)
//   dY_s   = the contraction of dS~_s with alpha_s in R's place        (contract_tc)
//   dX     = sum_s dY_s W_s^T,  dW_s = X^T dY_s                        (bwd_gemm_tc)
// The attention gradients need Vbar in bf16 (its products with dPbar pair two bf16
// operands); the forward's copy is f16, so the mixing runs once more for V in bf16.
#include <cuda_runtime.h>

#include "iha.h"
#include "iha_internal.h"

namespace iha {
cudaError_t launch_bwd_rowdot(const void *dPst, const void *Pbar, const Shape &sh, long long ld, float *Dv,
                              cudaStream_t st);
int bwd_ld_stride(long long L);
cudaError_t launch_bwd_attention_tc(const void *Q, const void *K, const void *Vb, const void *dPst, const float *lse,
                                    const float *Dv, const Shape &sh, int mask_mode, int window, void *dQ, void *dK,
                                    void *dV, cudaStream_t st, int *status);
size_t bwd_gram_part_floats(long long ntok, int NA, int NB);
cudaError_t launch_bwd_gram(const void *U, long long us, int NA, const void *V, long long vs, int NB, int d,
                            long long ntok, float *part, float *out, cudaStream_t st, int *status);
cudaError_t launch_bwd_dx_tc(const void *const dY[3], const void *const W[3], long long T, int D, void *dX,
                             cudaStream_t st, int *status);
cudaError_t launch_bwd_dw_tc(const void *X, const void *const dY[3], long long T, int D, void *const dW[3],
                             cudaStream_t st, int *status);

struct BwdLayout {
    size_t y, wp, qkv, vb, pbar, lse, dpst, dv, ds, dy, part, ctr, total;
    size_t ld_bytes;   // lse and D: [B*H][bwd_ld_stride(L)] floats each
};

static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

static BwdLayout bwd_layout(const Shape &sh) {
    const size_t T = (size_t)sh.B * sh.N, D = (size_t)sh.D(), HP = (size_t)sh.H * sh.P, L = (size_t)sh.L();
    const size_t BHL = (size_t)sh.B * sh.H * L;
    const size_t BHLp = (size_t)sh.B * sh.H * bwd_ld_stride((long long)L);
    BwdLayout l{};
    size_t o = 0;
    l.y = o;    o += al256(3 * T * D * 2);
    l.wp = o;   o += al256(sliced_weights_bytes(sh));
    l.qkv = o;  o += al256(3 * (size_t)sh.qkv_elems() * 2);
    l.vb = o;   o += al256((size_t)sh.qkv_elems() * 2);
    l.pbar = o; o += al256(T * HP * sh.d * 2);
    l.ld_bytes = BHLp * 4;
    l.lse = o;  o += al256(BHLp * 4);
    l.dpst = o; o += al256(BHL * sh.d * 2);
    l.dv = o;   o += al256(BHLp * 4);
    l.ds = o;   o += al256(3 * T * HP * sh.d * 2);
    l.dy = o;   o += al256(3 * T * D * 2);
    l.part = o; o += al256(bwd_gram_part_floats((long long)T, sh.H, (int)HP) * 4);
    l.ctr = o;  o += kCtrlBytes;   // the forward attention's work counter
    l.total = o;
    return l;
}

static bool bwd_supported(const Shape &sh, int dtype) {
    return dtype == IHA_DTYPE_BF16 && (sh.d == 64 || sh.d == 128) && sh.H <= 16 && sh.H * sh.P <= 128;
}

}  // namespace iha

using namespace iha;

extern "C" {

size_t iha_backward_workspace_bytes(int B, int N, int H, int d, int P, int dtype) {
    if (iha_workspace_bytes(B, N, H, d, P, dtype) == 0) return 0;   // the forward's shape checks
    const Shape sh{B, N, H, d, P};
    if (!bwd_supported(sh, dtype)) return 0;
    return bwd_layout(sh).total;
}

}  // extern "C"

namespace iha {

// The forward pieces the gradients need, written into the workspace regions: Y, Q~ K~ V~ (V~
// f16), Pbar and lse (the forward attention), V~ again in bf16; and the layer output when
// `out` is given (the contraction of Pbar with R).
static cudaError_t bwd_forward_pieces(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                                      const float *alpha_Q, const float *alpha_K, const float *alpha_V,
                                      const float *R, const Shape &sh, int mask_mode, int window, void *out,
                                      const BwdLayout &lay, uint8_t *ws, cudaStream_t st, int *status) {
    uint8_t *Y = ws + lay.y, *QKV = ws + lay.qkv, *Vb = ws + lay.vb, *Pbar = ws + lay.pbar;
    float *lse = reinterpret_cast<float *>(ws + lay.lse), *Dv = reinterpret_cast<float *>(ws + lay.dv);
    const long long D = sh.D();
    // lse and D rows are padded so that every 64-row block of them starts 256 bytes into a
    // 256-aligned row; the padding reads as 0 (its pairs are masked)
    const int ld = bwd_ld_stride(sh.L());
    cudaError_t e = cudaMemsetAsync(lse, 0, lay.ld_bytes, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(Dv, 0, lay.ld_bytes, st);
    // Q~ K~ V~ as the forward computes them, and the head projections Y for dalpha
    if (e == cudaSuccess) e = launch_slice_weights(W_Q, W_K, W_V, sh, ws + lay.wp, st);
    if (e == cudaSuccess)
        e = launch_project_mix(X, ws + lay.wp, alpha_Q, alpha_K, alpha_V, sh, 0, (long long)sh.B * sh.N, QKV, Y, st,
                               status);
    if (e == cudaSuccess)
        e = launch_attention_lse(QKV, sh, mask_mode, window, IHA_DTYPE_BF16, Pbar, lse, ld, st, status,
                                 reinterpret_cast<unsigned int *>(ws + lay.ctr));
    // Vbar again, in bf16: the V third of Y mixed with alpha_V
    if (e == cudaSuccess)
        e = launch_mix_sets(Y + (size_t)2 * D * 2, alpha_V, alpha_V, alpha_V, sh, 1, Vb, st, status, 3, -1);
    if (e == cudaSuccess && out) e = launch_contract_tc(Pbar, R, sh, out, st, status);
    return e;
}

// Everything after the forward pieces: the gradients of every input.
static cudaError_t bwd_gradients(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                                 const float *alpha_Q, const float *alpha_K, const float *alpha_V, const float *R,
                                 const Shape &sh, int mask_mode, int window, const void *dO, void *dX, void *dW_Q,
                                 void *dW_K, void *dW_V, float *dalpha_Q, float *dalpha_K, float *dalpha_V, float *dR,
                                 const BwdLayout &lay, uint8_t *ws, cudaStream_t st, int *status) {
    const int H = sh.H, d = sh.d;
    const long long T = (long long)sh.B * sh.N, D = sh.D(), HP = (long long)H * sh.P;
    uint8_t *Y = ws + lay.y, *QKV = ws + lay.qkv, *Vb = ws + lay.vb, *Pbar = ws + lay.pbar, *dPst = ws + lay.dpst,
            *dS = ws + lay.ds, *dY = ws + lay.dy;
    float *lse = reinterpret_cast<float *>(ws + lay.lse), *Dv = reinterpret_cast<float *>(ws + lay.dv);
    float *part = reinterpret_cast<float *>(ws + lay.part);
    const size_t ds_bytes = (size_t)T * HP * d * 2, dy_bytes = (size_t)T * D * 2;
    const size_t third = (size_t)sh.qkv_elems() * 2;
    const int ld = bwd_ld_stride(sh.L());
    const void *W[3] = {W_Q, W_K, W_V};
    const float *alpha[3] = {alpha_Q, alpha_K, alpha_V};
    float *dalpha[3] = {dalpha_Q, dalpha_K, dalpha_V};
    void *dW[3] = {dW_Q, dW_K, dW_V};
    const void *dYs[3] = {dY, dY + dy_bytes, dY + 2 * dy_bytes};

    // dPbar (stacked) = dO mixed with R in alpha's place
    cudaError_t e = launch_mix_sets(dO, R, R, R, sh, 1, dPst, st, status);
    if (e == cudaSuccess) e = launch_bwd_gram(dO, D, H, Pbar, HP * d, (int)HP, d, T, part, dR, st, status);
    if (e == cudaSuccess) e = launch_bwd_rowdot(dPst, Pbar, sh, ld, Dv, st);
    if (e == cudaSuccess)
        e = launch_bwd_attention_tc(QKV, QKV + third, Vb, dPst, lse, Dv, sh, mask_mode, window, dS, dS + ds_bytes,
                                    dS + 2 * ds_bytes, st, status);
    for (int s = 0; s < 3 && e == cudaSuccess; ++s) {
        const uint8_t *dSs = dS + s * ds_bytes;
        // dalpha_s[m][h*P + j] = sum_t,c Y_s[t][m][c] dS~_s[t][h*P + j][c]
        e = launch_bwd_gram(Y + (size_t)s * D * 2, 3 * D, H, dSs, HP * d, (int)HP, d, T, part, dalpha[s], st, status);
        // dY_s[t][m][c] = sum_hj alpha_s[m][hj] dS~_s[t][hj][c]
        if (e == cudaSuccess) e = launch_contract_tc(dSs, alpha[s], sh, dY + s * dy_bytes, st, status);
    }
    if (e == cudaSuccess) e = launch_bwd_dx_tc(dYs, W, T, (int)D, dX, st, status);
    if (e == cudaSuccess) e = launch_bwd_dw_tc(X, dYs, T, (int)D, dW, st, status);
    return e;
}

// The checks shared by the three entry points; the workspace (caller's, or allocated).
static int bwd_begin(const void *X, const void *W_Q, const void *W_K, const void *W_V, const float *alpha_Q,
                     const float *alpha_K, const float *alpha_V, const float *R, int B, int N, int H, int d, int P,
                     int mask_mode, int window, const void *o_or_dO, int dtype, cudaStream_t st, void *&workspace,
                     size_t workspace_bytes, bool &own, bool may_allocate) {
    int rc = check_forward_args(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window,
                                o_or_dO, dtype);
    if (rc != IHA_OK) return rc;
    const Shape sh{B, N, H, d, P};
    if (!bwd_supported(sh, dtype)) return IHA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(o_or_dO) & 15) != 0) return IHA_ERR_INVALID_ARG;   // read or written by TMA
    const BwdLayout lay = bwd_layout(sh);
    own = false;
    if (!workspace) {
        if (!may_allocate) return IHA_ERR_WORKSPACE;
        if (cudaMallocAsync(&workspace, lay.total, st) != cudaSuccess) return IHA_ERR_CUDA;
        own = true;
    } else if (workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255)) {
        return IHA_ERR_WORKSPACE;
    }
    return IHA_OK;
}

static bool grads_aligned(const void *a, const void *b, const void *c, const void *d) {
    return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) | reinterpret_cast<uintptr_t>(c) |
             reinterpret_cast<uintptr_t>(d)) &
            15) == 0;
}

static int bwd_end(cudaError_t e, bool own, void *workspace, cudaStream_t st) {
    if (own) {
        const cudaError_t e2 = cudaFreeAsync(workspace, st);
        if (e == cudaSuccess) e = e2;
    }
    return status_from_cuda(e);
}

}  // namespace iha

extern "C" {

int iha_backward(const void *X, const void *W_Q, const void *W_K, const void *W_V, const float *alpha_Q,
                 const float *alpha_K, const float *alpha_V, const float *R, int B, int N, int H, int d, int P,
                 int mask_mode, int window, const void *dO, void *dX, void *dW_Q, void *dW_K, void *dW_V,
                 float *dalpha_Q, float *dalpha_K, float *dalpha_V, float *dR, int dtype, void *stream,
                 void *workspace, size_t workspace_bytes) {
    if (!dX || !dW_Q || !dW_K || !dW_V || !dalpha_Q || !dalpha_K || !dalpha_V || !dR) return IHA_ERR_INVALID_ARG;
    if (!grads_aligned(dX, dW_Q, dW_K, dW_V)) return IHA_ERR_INVALID_ARG;   // written by TMA stores
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool own = false;
    int rc = bwd_begin(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, dO, dtype,
                       st, workspace, workspace_bytes, own, true);
    if (rc != IHA_OK) return rc;
    const Shape sh{B, N, H, d, P};
    const BwdLayout lay = bwd_layout(sh);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int *status = status_word_ptr();
    cudaError_t e = bwd_forward_pieces(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, sh, mask_mode, window, nullptr,
                                       lay, ws, st, status);
    if (e == cudaSuccess)
        e = bwd_gradients(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, sh, mask_mode, window, dO, dX, dW_Q, dW_K,
                          dW_V, dalpha_Q, dalpha_K, dalpha_V, dR, lay, ws, st, status);
    return bwd_end(e, own, workspace, st);
}

int iha_forward_train(const void *X, const void *W_Q, const void *W_K, const void *W_V, const float *alpha_Q,
                      const float *alpha_K, const float *alpha_V, const float *R, int B, int N, int H, int d, int P,
                      int mask_mode, int window, void *out, int dtype, void *stream, void *workspace,
                      size_t workspace_bytes) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool own = false;
    int rc = bwd_begin(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, out, dtype,
                       st, workspace, workspace_bytes, own, false);
    if (rc != IHA_OK) return rc;
    const Shape sh{B, N, H, d, P};
    return bwd_end(bwd_forward_pieces(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, sh, mask_mode, window, out,
                                      bwd_layout(sh), static_cast<uint8_t *>(workspace), st, status_word_ptr()),
                   own, workspace, st);
}

int iha_backward_saved(const void *X, const void *W_Q, const void *W_K, const void *W_V, const float *alpha_Q,
                       const float *alpha_K, const float *alpha_V, const float *R, int B, int N, int H, int d, int P,
                       int mask_mode, int window, const void *dO, void *dX, void *dW_Q, void *dW_K, void *dW_V,
                       float *dalpha_Q, float *dalpha_K, float *dalpha_V, float *dR, int dtype, void *stream,
                       void *workspace, size_t workspace_bytes) {
    if (!dX || !dW_Q || !dW_K || !dW_V || !dalpha_Q || !dalpha_K || !dalpha_V || !dR) return IHA_ERR_INVALID_ARG;
    if (!grads_aligned(dX, dW_Q, dW_K, dW_V)) return IHA_ERR_INVALID_ARG;   // written by TMA stores
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool own = false;
    int rc = bwd_begin(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, B, N, H, d, P, mask_mode, window, dO, dtype,
                       st, workspace, workspace_bytes, own, false);
    if (rc != IHA_OK) return rc;
    const Shape sh{B, N, H, d, P};
    return bwd_end(bwd_gradients(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, sh, mask_mode, window, dO, dX, dW_Q,
                                 dW_K, dW_V, dalpha_Q, dalpha_K, dalpha_V, dR, bwd_layout(sh),
                                 static_cast<uint8_t *>(workspace), st, status_word_ptr()),
                   own, workspace, st);
}

}  // extern "C"
