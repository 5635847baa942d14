// iha_internal.h -- launchers shared by the C-ABI translation unit and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "iha.h"

namespace iha {

// A CUDA error as an IHA status: kernel images that do not match the device or their
// register contract (see check_register_contract) are IHA_ERR_BUILD, anything else
// IHA_ERR_CUDA.
inline int status_from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return IHA_OK;
    if (e == cudaErrorInvalidKernelImage || e == cudaErrorNoKernelImageForDevice) return IHA_ERR_BUILD;
    return IHA_ERR_CUDA;
}

// Warp-specialised kernels that move registers between warpgroups (setmaxnreg) assume
// they were compiled to exactly `regs` registers per thread: a warpgroup asking for more
// than the launch provided would wait forever.  The build checks this from the ptxas
// report; this guard turns a library built any other way into an error before launch.
template <typename Kernel>
inline cudaError_t check_register_contract(Kernel kern, int regs) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    return fa.numRegs == regs ? cudaSuccess : cudaErrorInvalidKernelImage;
}

// Wait-site codes written to the status word (low 12 bits) when a bounded wait expires.
enum WaitSite {
    kSiteProjProducer = 1,
    kSiteProjMma = 2,
    kSiteProjEpilogue = 3,
    kSiteProjMmaAcc = 4,
    kSiteProjStore = 5,
    kSiteAttnProducer = 16,
    kSiteAttnMmaQ = 17,
    kSiteAttnMmaK = 18,
    kSiteAttnMmaP = 19,
    kSiteAttnMmaV = 20,
    kSiteAttnSoftmax = 21,
    kSiteAttnEpilogue = 22,
    kSiteAttnMmaO = 23,
    kSiteAttnProducerQ = 24,
    kSiteAttnItem = 25,
    kSiteRowMix = 30,
    kSiteMixProducer = 31,
    kSiteMixMma = 32,
    kSiteMixEpilogue = 33,
    kSiteContractProducer = 34,
    kSiteContractMma = 35,
    kSiteContractEpilogue = 36,
    kSiteDecodeProducer = 37,
    kSiteDecodeConsumer = 38,
    kSiteBwdProducer = 40,
    kSiteBwdMma = 41,
    kSiteBwdSoftmax = 42,
    kSiteBwdEpilogue = 43,
    kSiteBwdGemmProducer = 44,
    kSiteBwdGemmMma = 45,
    kSiteBwdGemmEpilogue = 46,
    kSiteGramProducer = 47,
    kSiteGramMma = 48,
    kSiteGramEpilogue = 49,
    kSiteDecodeTcProducer = 50,
    kSiteDecodeTcMma = 51,
    kSiteDecodeTc = 52,
    kSiteDecodeProj = 53,
    kSiteSelfTest = 99,
};

struct Shape {
    int B, N, H, d, P;
    long long D() const { return (long long)H * d; }
    long long L() const { return (long long)N * P; }                     // stacked length
    long long qkv_elems() const { return (long long)B * H * N * P * d; }  // one of Qbar/Kbar/Vbar
    long long wt_rows() const { return 3LL * H * P * d; }
};

// Step 1+2 weights: Wt[(s,h,j,c)][k] = sum_m alpha_s[m,h,j] W_s[k][m*d + c].
cudaError_t launch_fold(const void *WQ, const void *WK, const void *WV, const float *aQ, const float *aK,
                        const float *aV, const Shape &sh, int dtype, void *Wt, cudaStream_t st);

// Steps 1+2 + stacking: QKV = X Wt^T in the stacked [s][B][H][N*P][d] layout.
cudaError_t launch_project(const void *X, const void *Wt, const Shape &sh, int dtype, void *QKV,
                           cudaStream_t st, int *status);

// Steps 1+2 without the fold (bf16): Y = X [W_Q | W_K | W_V], Y [B*N][3][H*d] row-major.
cudaError_t launch_project_heads(const void *X, const void *WQ, const void *WK, const void *WV, const Shape &sh,
                                 void *Y, cudaStream_t st, int *status);

// Steps 1+2 fused (bf16; project_mix_supported): the head projections on the tensor cores
// with the pseudo-head mixing in the GEMM epilogue.  launch_slice_weights first writes
// W_Q, W_K, W_V slice-major into Wp (sliced_weights_bytes(sh) bytes, 16-byte aligned);
// launch_project_mix then maps token rows [tok0, tok0 + ntok) of X [B*N][D] into the stacked
// QKV [3][B][H][N*P][d] (bf16 Qbar/Kbar, f16 Vbar; 32-byte aligned) and, when Y is not NULL,
// writes the head projections Y [B*N][3][H*d] bf16 too.
bool project_mix_supported(const Shape &sh);
size_t sliced_weights_bytes(const Shape &sh);
cudaError_t launch_slice_weights(const void *WQ, const void *WK, const void *WV, const Shape &sh, void *Wp,
                                 cudaStream_t st);
cudaError_t launch_project_mix(const void *X, const void *Wp, const float *aQ, const float *aK, const float *aV,
                               const Shape &sh, long long tok0, long long ntok, void *QKV, void *Y, cudaStream_t st,
                               int *status);

// The pseudo-head mixing of Y into the stacked QKV layout (bf16 Qbar/Kbar, f16 Vbar).
cudaError_t launch_mix(const void *Y, const float *aQ, const float *aK, const float *aV, const Shape &sh, void *QKV,
                       cudaStream_t st, int *status);

// Which way the library computes steps 1+2: true = the head projections with the mixing in
// the GEMM epilogue (bf16, H <= 16, H*P <= 128: 1/P of the folded GEMM's work; at P = 1 the
// same GEMM, without the fold's pass over the weights), false = fold alpha into W, then one
// GEMM.
inline bool unfolded_route(const Shape &sh, int dtype) {
    return dtype == 1 && sh.H <= 16 && sh.H * sh.P <= 128;
}

// The mixing kernel for nsets projections: Y [t][y_sets][H][d] (the first nsets of each
// token's y_sets blocks are mixed) -> QKV [nsets][B][H][N*P][d]; set f16_set is written as
// f16 (2: Vbar for the forward's P V product; -1: every set bf16).
cudaError_t launch_mix_sets(const void *Y, const float *aQ, const float *aK, const float *aV, const Shape &sh,
                            int nsets, void *QKV, cudaStream_t st, int *status, int y_sets = -1, int f16_set = 2);

// Attention that also writes each stacked row's log2 softmax normaliser (bf16 only) into
// lse[b*H + h][lse_stride] (lse_stride >= N*P).
cudaError_t launch_attention_lse(const void *QKV, const Shape &sh, int mask_mode, int window, int dtype,
                                 void *Pbar, float *lse, int lse_stride, cudaStream_t st, int *status,
                                 unsigned int *ticket = nullptr);

// Step 3: masked softmax attention per head over the stacked sequence -> Pbar [B][N][H][P][d].
// ticket: the launch's work counter (one unsigned int of the caller's workspace, zeroed on
// `st` before the kernel), or NULL to take the next one of a ring of library-owned counters.
cudaError_t launch_attention(const void *QKV, const Shape &sh, int mask_mode, int window, int dtype,
                             void *Pbar, cudaStream_t st, int *status, unsigned int *ticket = nullptr);

// The attention of part of a layer (bf16): stacked-query blocks of 256 rows
// [qb_begin, qb_begin + qb_count) of heads b*H + h in [bh_begin, bh_begin + bh_count).  Each
// row's result is the one the whole-layer launch gives it (the same work items).
struct AttnRange {
    int bh_begin, bh_count, qb_begin, qb_count;
};
constexpr int kAttnRowsPerBlock = 256;
cudaError_t launch_attention_range(const void *QKV, const Shape &sh, int mask_mode, int window, void *Pbar,
                                   const AttnRange &range, cudaStream_t st, int *status, unsigned int *ticket);

// Bytes of the control slot every workspace ends with (the attention's work counter).
constexpr size_t kCtrlBytes = 256;

// Step 4: out[b][t][h][:] = sum_i R[h][i] Pbar[b][t][i][:], i = h'*P + j.
cudaError_t launch_contract(const void *Pbar, const float *R, const Shape &sh, int dtype, void *out,
                            cudaStream_t st, int *status);

// The bf16 contraction on tensor cores (d in {64, 128}, H <= 16, H*P <= 128); else the
// TMA-fed row mixing when its 3-stage ring fits in shared memory; otherwise, and for fp32,
// a SIMT kernel.
bool contract_tc_fits(const Shape &sh);
cudaError_t launch_contract_tc(const void *Pbar, const float *R, const Shape &sh, void *out, cudaStream_t st,
                               int *status);
bool contract_rowmix_fits(const Shape &sh);
cudaError_t launch_contract_rowmix(const void *Pbar, const float *R, const Shape &sh, void *out, cudaStream_t st,
                                   int *status);

// A kernel whose only wait can never be satisfied: it must give up after limit_ns and
// record kSiteSelfTest in the status word (exercises the failure path of every wait).
cudaError_t launch_wait_selftest(int *status, unsigned long long limit_ns, cudaStream_t st);

// The argument checks of iha_forward_ex (IHA_OK or the status it would return).
int check_forward_args(const void *X, const void *WQ, const void *WK, const void *WV, const float *aQ,
                       const float *aK, const float *aV, const float *R, int B, int N, int H, int d, int P,
                       int mask_mode, int window, const void *out, int dtype);

// The launch sequence of iha_forward_ex in a caller-given device workspace (never NULL;
// nothing is allocated).
int forward_in_workspace(const void *X, const void *WQ, const void *WK, const void *WV, const float *aQ,
                         const float *aK, const float *aV, const float *R, const Shape &sh, int mask_mode,
                         int window, void *out, int dtype, cudaStream_t st, void *workspace,
                         size_t workspace_bytes);

// One decoding step over a pseudo-token cache (bf16; d = 64 with P <= 8, d = 128 with P <= 4).
bool decode_supported(int H, int d, int P);
size_t decode_workspace_bytes(int B, int H, int d, int P);
cudaError_t launch_decode(const void *x, const void *WQ, const void *WK, const void *WV, const float *aQ,
                          const float *aK, const float *aV, const float *R, int B, int H, int d, int P, int mask_mode,
                          int window, void *Kc, void *Vc, long long cache_tokens, long long t, void *out, void *ws,
                          cudaStream_t st, int *status);

// The status word of the current device (bounded device waits record timeouts there).
int *status_word_ptr();

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace iha
