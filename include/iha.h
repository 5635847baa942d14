/*
 * iha.h -- C ABI of the GB300 (sm_103a) Interleaved Head Attention forward pass.
 *
 * The operation is Algorithm 1 of "Interleaved Head Attention" (Duvvuri et al.,
 * arXiv 2602.21371; summary page "交錯頭注意力機制", section 4):
 *   1. per-head projections      X W_s^(m),              s in {Q, K, V}, m = 1..H
 *   2. pseudo-head mixing        S~_{h,j} = sum_m alpha_s[m,h,j] X W_s^(m),  j = 1..P
 *   3. stacking to length P*N and per-head softmax attention
 *                                Pbar_h = softmax(Qbar_h Kbar_h^T / sqrt(d)) Vbar_h
 *   4. unstacking and contraction O_h[t] = sum_{h',j} R[h, h'P + j] P_{h',j}[t],
 *      heads concatenated to X~ [N, D].
 * The scores are masked by original token position ("注意力机制" eq. (5.12):
 * visibility by absolute position): pseudo-token (j, t) may read (j', t') iff
 *   IHA_MASK_NONE:   always;
 *   IHA_MASK_CAUSAL: t' <= t;
 *   IHA_MASK_WINDOW: t' <= t and t - t' < window  (window >= N behaves as causal).
 * Pseudo-tokens of one position see one another; every row has at least P
 * readable keys, so no row is ever empty.
 *
 * Conventions shared by every entry point
 *   - All arrays are dense, row-major, owned by the caller; the library never
 *     frees them and never keeps a pointer after a call returns.
 *   - D = H * d by contract (the signatures carry no D).
 *   - X [B][N][D]; W_Q, W_K, W_V [D][H*d], column block m (columns m*d..m*d+d-1)
 *     is W^(m) (the packed layout of "注意力机制" eq. (5.22)); note that torch's
 *     nn.Linear stores the transpose.
 *   - alpha_Q/K/V [H(m)][H(h)][P(j)] float32; R [H][H*P] float32, column h'*P + j.
 *   - out (X~) [B][N][D], D = H*d, head h at columns h*d..h*d+d-1.
 *   - dtype IHA_DTYPE_BF16: X, W, intermediates and out are bfloat16; products
 *     accumulate in float32 (tcgen05 tensor cores).  IHA_DTYPE_F32: everything
 *     float32 with exact fp32 FMA arithmetic (no TF32).  alpha and R are float32
 *     in both.
 *   - Device entry points take DEVICE pointers and run asynchronously on the
 *     given stream (NULL = the legacy default stream).  out must not alias an
 *     input.
 *   - Return value: IHA_OK or an IHA_ERR_* code; nothing is thrown across the ABI.
 *     Argument errors are detected on the host before anything is launched.
 *     A device-side bounded wait that expires (IHA_ERR_TIMEOUT) is recorded in a
 *     per-device status word and reported by iha_check_device_status().
 *   - The library looks up the device addresses of its per-device state (the
 *     status word, the attention work-counter ring, the array behind
 *     iha_forward_noalloc) and creates the two copy streams of iha_forward_host on
 *     first use on each device, and keeps them for the life of the process.  cudaDeviceReset() invalidates them: no call may
 *     follow a device reset in the same process.
 */
#ifndef IHA_H
#define IHA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* exported from libiha.so (everything else in the library is hidden) */
#if defined(__GNUC__)
#define IHA_API __attribute__((visibility("default")))
#else
#define IHA_API
#endif

#define IHA_OK 0
#define IHA_ERR_INVALID_ARG 1   /* null pointer, non-positive size, bad mode/dtype/window */
#define IHA_ERR_UNSUPPORTED 2   /* valid but not supported here (e.g. bf16 with d not 64/128) */
#define IHA_ERR_WORKSPACE 3     /* caller workspace smaller than iha_workspace_bytes() */
#define IHA_ERR_CUDA 4          /* a CUDA call or launch failed */
#define IHA_ERR_TIMEOUT 5       /* a device-side bounded wait expired */
#define IHA_ERR_BUILD 6         /* the library's kernels do not match this device, or a
                                   warp-specialised kernel was compiled to another register
                                   count than its register split needs: rebuild */

#define IHA_DTYPE_F32 0
#define IHA_DTYPE_BF16 1

#define IHA_MASK_NONE 0
#define IHA_MASK_CAUSAL 1
#define IHA_MASK_WINDOW 2

/*
 * iha_forward -- the whole forward pass (steps 1-4) in bfloat16 on the legacy
 * default stream, with a workspace the library allocates stream-ordered
 * (cudaMallocAsync) and frees after the last launch.  Asynchronous.
 * Errors: IHA_ERR_INVALID_ARG, IHA_ERR_UNSUPPORTED (d not in {64, 128}),
 * IHA_ERR_CUDA (allocation or launch failure).
 */
IHA_API int iha_forward(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                const float *alpha_Q, const float *alpha_K, const float *alpha_V,
                const float *R, int B, int N, int H, int d, int P,
                int mask_mode, int window, void *out);

/*
 * iha_forward_ex -- iha_forward with the arithmetic type, the stream and the
 * workspace chosen by the caller.  workspace may be NULL (allocated and freed
 * stream-ordered by the library); otherwise it must be a device buffer of at
 * least iha_workspace_bytes(B, N, H, d, P, dtype) bytes, 256-byte aligned, not
 * used concurrently by another call.
 * Errors: as iha_forward, plus IHA_ERR_WORKSPACE.
 */
IHA_API int iha_forward_ex(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                   const float *alpha_Q, const float *alpha_K, const float *alpha_V,
                   const float *R, int B, int N, int H, int d, int P,
                   int mask_mode, int window, void *out,
                   int dtype, void *stream, void *workspace, size_t workspace_bytes);

/* Bytes of device workspace one call needs (0 if the sizes are invalid): the folded
 * weights (the slice-major weights on the unfolded route) + stacked Qbar, Kbar, Vbar
 * + Pbar, each 256-byte aligned, + a 256-byte control slot (the call's own attention work
 * counter, reset on the stream by every call). */
IHA_API size_t iha_workspace_bytes(int B, int N, int H, int d, int P, int dtype);

/* A static, human-readable name for a status code (never NULL). */
IHA_API const char *iha_error_string(int status);

/*
 * iha_check_device_status -- synchronise the stream, then read and clear the
 * current device's status word.  Returns IHA_OK, IHA_ERR_TIMEOUT (a kernel
 * gave up a bounded wait since the last check; its output is invalid) or
 * IHA_ERR_CUDA (the stream reported an error).  If code_out is not NULL it
 * receives the raw word (0, or the wait site that expired).
 */
IHA_API int iha_check_device_status(void *stream, int *code_out);

/*
 * iha_forward_host -- the forward pass on HOST buffers: copies X, W_*, alpha_*,
 * R host->device, runs iha_forward_ex, copies out device->host and synchronises
 * the stream before returning.  Host buffers should be pinned for full copy
 * bandwidth.  device_buffer may be NULL (allocated and freed by the call) or a
 * device buffer of at least iha_host_buffer_bytes(...) bytes.
 * Errors: as iha_forward_ex; IHA_ERR_TIMEOUT if a device wait expired.
 */
IHA_API int iha_forward_host(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                     const float *alpha_Q, const float *alpha_K, const float *alpha_V,
                     const float *R, int B, int N, int H, int d, int P,
                     int mask_mode, int window, void *out, int dtype, void *stream,
                     void *device_buffer, size_t device_buffer_bytes);

/* Device bytes iha_forward_host needs: inputs + out + workspace (0 if invalid). */
IHA_API size_t iha_host_buffer_bytes(int B, int N, int H, int d, int P, int dtype);

/*
 * iha_selftest_wait_timeout -- launch one tiny kernel whose only wait (on an
 * mbarrier nothing arrives at) must give up after limit_ms milliseconds
 * (1..10000), record its site in the status word and return normally.  It
 * exercises the device-side timeout path used by every pipeline wait; the next
 * iha_check_device_status() must report IHA_ERR_TIMEOUT.  No counterpart in the
 * method: it is a failure-detection check of this library.
 */
IHA_API int iha_selftest_wait_timeout(void *stream, int limit_ms);

/*
 * iha_forward_noalloc -- iha_forward_ex for callers that cannot allocate device
 * memory: processes whose device memory is already reserved in full by another
 * framework's pool, or code paths where an allocation may not happen (it could
 * fail, block, or synchronise).  The pass's workspace is a fixed array of
 * IHA_NOALLOC_SCRATCH_BYTES compiled into the library (every GPU that loads
 * the library holds one until exit); the call itself allocates nothing.  The
 * method has no counterpart to this entry point: it is about where the
 * workspace lives.
 *   - Arguments, layouts and dtypes as iha_forward_ex (device pointers, the
 *     caller's stream); same kernels, so the same results.
 *   - Problems with iha_workspace_bytes(...) > IHA_NOALLOC_SCRATCH_BYTES are
 *     refused with IHA_ERR_WORKSPACE before anything runs.
 *   - The first call on a device looks up the array's device address (with that
 *     device current) and caches it; make that first call before any stream
 *     capture.  A failed lookup returns IHA_ERR_CUDA.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind.  No part of it needs to start at zero (each step overwrites what
 *     the next reads), but calls that overlap on the GPU (other streams, other
 *     threads) race on it: serialise them.
 */
#define IHA_NOALLOC_SCRATCH_BYTES (64u << 20)
IHA_API int iha_forward_noalloc(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                                const float *alpha_Q, const float *alpha_K, const float *alpha_V,
                                const float *R, int B, int N, int H, int d, int P,
                                int mask_mode, int window, void *out, int dtype, void *stream);

/* ---------------------------------------------------------------------------
 * The four steps as separate entry points (same validation, same kernels as
 * iha_forward_ex; asynchronous on the stream).  Intermediate layouts:
 *   Wt   [3*H*P*d][D]   folded, transposed weights: row s*H*P*d + h*P*d + j*d + c
 *                       holds  sum_m alpha_s[m,h,j] W_s[:, m*d + c]   (s = Q, K, V)
 *   Qbar, Kbar, Vbar [B][H][N*P][d]   stacked pseudo-tokens of head h; row t*P + j
 *                       (for IHA_DTYPE_BF16: Qbar, Kbar bfloat16, Vbar float16 -- the
 *                       softmax weights and Vbar meet in an f16 x f16 product; for
 *                       IHA_DTYPE_F32 all three float32)
 *                       is pseudo-token (j, t) (t-major interleaving; with a mask
 *                       on t only this ordering gives the same output as the row
 *                       concatenation j*N + t, "注意力机制" eq. (5.41))
 *   Pbar [B][N][H][P][d] attention output of pseudo-token (j, t) of head h
 * ------------------------------------------------------------------------- */

/* Step 1+2 weights: fold alpha into the projection weights (linearity of the
 * mixing sum over m).  Wt as above, dtype-sized elements. */
IHA_API int iha_fold_weights(const void *W_Q, const void *W_K, const void *W_V,
                     const float *alpha_Q, const float *alpha_K, const float *alpha_V,
                     int H, int d, int P, int dtype, void *Wt, void *stream);

/* Steps 1+2 and the stacking: [Qbar|Kbar|Vbar] = X Wt^T written in the stacked
 * layout.  QKV points to 3 consecutive arrays of B*H*N*P*d elements. */
IHA_API int iha_project(const void *X, const void *Wt, int B, int N, int H, int d, int P,
                int dtype, void *QKV, void *stream);

/* Which way steps 1+2 run for this shape (what iha_forward_ex does):
 *   1 = unfolded: iha_slice_weights then iha_project_mix, the head projections with the
 *       mixing in the GEMM epilogue (bf16, H <= 16, H*P <= 128 -- the GEMM does 1/P of the
 *       folded GEMM's work, the head projections never reach memory, and at P = 1 the
 *       weights are only reordered, not folded);
 *   0 = folded:   iha_fold_weights then iha_project;
 *  -1 = invalid sizes or dtype. */
IHA_API int iha_projection_route(int H, int d, int P, int dtype);

/* Steps 1+2, first half, without the fold (bf16 only): the per-head projections of all
 * heads, Y = X [W_Q | W_K | W_V], Y [B*N][3][H*d] bfloat16 row-major (block s, column
 * m*d + c holds (X W_s^(m))[t][c]).  The weights are read as stored. */
IHA_API int iha_project_heads(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                              int B, int N, int H, int d, int dtype, void *Y, void *stream);

/* Steps 1+2 and the stacking in one kernel (bf16 only, H <= 16, H*P <= 128, d in {64, 128};
 * IHA_ERR_UNSUPPORTED otherwise): the head projections X W_s^(m) on the tensor cores with the
 * mixing S~_{h,j} = sum_m alpha_s[m,h,j] (X W_s^(m)) in fp32 in the GEMM epilogue, written into
 * QKV (layout as for iha_project; 32-byte aligned, IHA_ERR_INVALID_ARG otherwise).  It reads
 * the weights slice-major, as iha_slice_weights writes them:
 *   Wp [3][D][S]: for s = Q, K, V, column sl*C + m*CW + c of row k holds W_s[k][m*d + sl*CW + c],
 *   CW = the widest of 64, 32, 16 with H*CW <= 256 and CW <= d, C = H*CW rounded up to a
 *   multiple of 64 (padding columns zero), S = (d/CW)*C; iha_sliced_weights_bytes(H, d, dtype)
 *   bytes, 16-byte aligned.
 * iha_forward_ex runs iha_slice_weights then iha_project_mix when iha_projection_route() is 1. */
IHA_API size_t iha_sliced_weights_bytes(int H, int d, int dtype);
IHA_API int iha_slice_weights(const void *W_Q, const void *W_K, const void *W_V, int H, int d, int dtype,
                              void *Wp, void *stream);
IHA_API int iha_project_mix(const void *X, const void *Wp,
                            const float *alpha_Q, const float *alpha_K, const float *alpha_V,
                            int B, int N, int H, int d, int P, int dtype, void *QKV, void *stream);

/* Steps 1+2, second half, and the stacking (bf16 only, H <= 16, H*P <= 128): the mixing
 * S~_{h,j} = sum_m alpha_s[m,h,j] (X W_s^(m)) of Y into QKV (layout as for iha_project).
 * Y and QKV must be 16-byte aligned (IHA_ERR_INVALID_ARG otherwise). */
IHA_API int iha_mix_heads(const void *Y, const float *alpha_Q, const float *alpha_K, const float *alpha_V,
                          int B, int N, int H, int d, int P, int dtype, void *QKV, void *stream);

/* Step 3: masked softmax attention over each head's stacked sequence.
 * QKV as written by iha_project; Pbar [B][N][H][P][d]; both 16-byte aligned
 * (IHA_ERR_INVALID_ARG otherwise).  This entry point has no workspace,
 * so for bf16 each call takes the next of 1024 library-owned work counters (zeroed on
 * `stream` before the kernel): at most 1024 calls may be executing or queued on different
 * streams at once, and a CUDA graph that captured this call uses the same counter on every
 * replay, so replays of it must not overlap.  Calls on one stream are ordered and never
 * collide.  The whole-pass entry points keep their counter in their own workspace. */
IHA_API int iha_attention(const void *QKV, int B, int N, int H, int d, int P,
                  int mask_mode, int window, int dtype, void *Pbar, void *stream);

/* Step 4: unstack and contract with R, heads concatenated into out [B][N][H*d]. */
IHA_API int iha_contract(const void *Pbar, const float *R, int B, int N, int H, int d, int P,
                 int dtype, void *out, void *stream);

/* A stack of IHA layers ("Interleaved Head Attention" appendix C, the hybrid local/global
 * schedule, e.g. four sliding-window layers with window N/(2P^2) tokens and one global
 * layer).  Layer l maps its input [B][N][H*d] to its output with its own weights and its
 * own P[l], mask_mode[l], window[l]; layer 0 reads X, layer l+1 reads layer l's output and
 * `out` receives the last layer's.  Nothing runs between layers (Algorithm 1 defines the
 * attention layer alone: no residual, normalisation or MLP).
 *   W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R: HOST arrays of num_layers DEVICE pointers,
 *     each with the layout and dtype of the iha_forward_ex argument of that name;
 *   P, mask_mode, window: host arrays of num_layers ints;
 *   workspace: NULL (allocated and freed on `stream`) or at least
 *     iha_stack_workspace_bytes(num_layers, P, B, N, H, d, dtype) bytes, 256-byte aligned.
 * Every layer's arguments are checked (as by iha_forward_ex) before the first launch; the
 * first failing check's status is returned and nothing runs. */
IHA_API size_t iha_stack_workspace_bytes(int num_layers, const int *P, int B, int N, int H, int d, int dtype);
IHA_API int iha_forward_stack(const void *X, int num_layers,
                              const void *const *W_Q, const void *const *W_K, const void *const *W_V,
                              const float *const *alpha_Q, const float *const *alpha_K,
                              const float *const *alpha_V, const float *const *R,
                              const int *P, const int *mask_mode, const int *window,
                              int B, int N, int H, int d, int dtype, void *out, void *stream,
                              void *workspace, size_t workspace_bytes);

/* Incremental decoding over a cache of pseudo-keys and pseudo-values (Algorithm 1 evaluated
 * for the rows of one new token; the mask is by original position, so the P pseudo-queries
 * of token t read the cached pseudo-tokens of positions t' <= t, and t - t' < window).
 * bf16 only; d = 64 with P <= 8, or d = 128 with P <= 4, and H*d <= 2048 (IHA_ERR_UNSUPPORTED otherwise);
 * mask_mode 1 or 2 (mode 0 would read future tokens: IHA_ERR_INVALID_ARG).
 *   K_cache [B][H][cache_tokens*P][d] bfloat16, V_cache same shape float16: stacked row
 *     t*P + j holds pseudo-key/value j of token t (the layout of Kbar/Vbar in iha_project);
 *     both 16-byte aligned for iha_decode_step, as are W_Q, W_K, W_V (IHA_ERR_INVALID_ARG
 *     otherwise).  Rows of tokens not yet appended may hold any bits (the caches need no
 *     initialisation): they never reach an output.
 *
 * iha_prefill: iha_forward_ex over X [B][N][H*d] (the prompt) that also writes the prompt's
 *   pseudo-keys/values into rows 0 .. N*P-1 of the caches (cache_tokens >= N). */
IHA_API int iha_prefill(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                        const float *alpha_Q, const float *alpha_K, const float *alpha_V, const float *R,
                        int B, int N, int H, int d, int P, int mask_mode, int window, void *out,
                        void *K_cache, void *V_cache, int cache_tokens, int dtype, void *stream,
                        void *workspace, size_t workspace_bytes);

/* iha_decode_step: x [B][H*d] is token t of every sequence (t = the number of tokens
 *   already cached, 0 <= t < cache_tokens).  Appends its pseudo-keys/values at rows
 *   t*P .. t*P+P-1 of the caches and writes its output row out [B][H*d] (the row iha_forward
 *   would give token t of the whole sequence).  workspace: NULL (allocated and freed on
 *   `stream`) or iha_decode_workspace_bytes(B, H, d, P) bytes, 256-byte aligned. */
IHA_API size_t iha_decode_workspace_bytes(int B, int H, int d, int P);
IHA_API int iha_decode_step(const void *x, const void *W_Q, const void *W_K, const void *W_V,
                            const float *alpha_Q, const float *alpha_K, const float *alpha_V, const float *R,
                            int B, int H, int d, int P, int mask_mode, int window,
                            void *K_cache, void *V_cache, int cache_tokens, int t, void *out,
                            int dtype, void *stream, void *workspace, size_t workspace_bytes);

/* The backward pass of one IHA layer: given dO [B][N][H*d] (the gradient of a loss with
 * respect to iha_forward's output for the same inputs), the gradients with respect to every
 * input of Algorithm 1.  bf16 only, d in {64, 128}, H <= 16, H*P <= 128
 * (IHA_ERR_UNSUPPORTED otherwise); every mask mode.
 *   dX [B][N][H*d], dW_Q/dW_K/dW_V [H*d][H*d]: bfloat16, layouts of X and W, 16-byte
 *     aligned (IHA_ERR_INVALID_ARG otherwise; dO too);
 *   dalpha_Q/K/V [H][H][P] and dR [H][H*P]: float32, layouts of alpha and R.
 * The forward intermediates are recomputed inside the call.  workspace: NULL (allocated
 * and freed on `stream`) or iha_backward_workspace_bytes(...) bytes, 256-byte aligned. */
IHA_API size_t iha_backward_workspace_bytes(int B, int N, int H, int d, int P, int dtype);
IHA_API int iha_backward(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                         const float *alpha_Q, const float *alpha_K, const float *alpha_V, const float *R,
                         int B, int N, int H, int d, int P, int mask_mode, int window, const void *dO,
                         void *dX, void *dW_Q, void *dW_K, void *dW_V,
                         float *dalpha_Q, float *dalpha_K, float *dalpha_V, float *dR,
                         int dtype, void *stream, void *workspace, size_t workspace_bytes);

/* A training step without recomputation, on the shapes iha_backward takes:
 * iha_forward_train computes the layer output `out` [B][N][H*d] (bfloat16; bit-identical to
 *   iha_forward's: every shape it takes is on the unfolded route) and leaves the forward
 *   pieces the gradients need
 *   (head projections, stacked pseudo-queries/keys/values, the attention output and each
 *   row's softmax normaliser) in `workspace`, which is required here:
 *   iha_backward_workspace_bytes(...) bytes, 256-byte aligned.
 * iha_backward_saved then computes the same gradients as iha_backward (bit-identical) from
 *   that workspace: same inputs, same shape and mask, and the workspace untouched in between
 *   (stream-ordered after iha_forward_train).  NULL workspace: IHA_ERR_WORKSPACE. */
IHA_API int iha_forward_train(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                              const float *alpha_Q, const float *alpha_K, const float *alpha_V, const float *R,
                              int B, int N, int H, int d, int P, int mask_mode, int window, void *out,
                              int dtype, void *stream, void *workspace, size_t workspace_bytes);
IHA_API int iha_backward_saved(const void *X, const void *W_Q, const void *W_K, const void *W_V,
                               const float *alpha_Q, const float *alpha_K, const float *alpha_V, const float *R,
                               int B, int N, int H, int d, int P, int mask_mode, int window, const void *dO,
                               void *dX, void *dW_Q, void *dW_K, void *dW_V,
                               float *dalpha_Q, float *dalpha_K, float *dalpha_V, float *dR,
                               int dtype, void *stream, void *workspace, size_t workspace_bytes);

#ifdef __cplusplus
}
#endif

#endif /* IHA_H */
