// k_backward.cu -- the reductions of the backward pass of one IHA layer ("Interleaved Head
// Attention" section 4, Algorithm 1, differentiated step by step): the per-row term of the
// softmax gradient ("注意力机制" eqs. (5.24)-(5.31)),
//
//     D_r = sum_c dPbar_r[c] Pbar_r[c]      (r a stacked row t*P + j; dPbar the gradient
//                                            reaching the attention output)
//
// The token reductions that give the gradients of the small mixing matrices and the dense
// contractions (attention gradients, weight and input GEMMs) are in k_backward_tc.cu.
//
// Layouts: stacked [B][H][L][d] (L = N*P); token-major [B*N][H*P][d] (row h*P + j of token t,
// the layout of Pbar); D [B*H][ld] (rows padded to ld >= L).  Arithmetic in fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "iha_internal.h"

namespace iha {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------------------
// D_r = dPbar_r . Pbar_r  (one warp per stacked row)
// ---------------------------------------------------------------------------------------
__global__ void bwd_rowdot(const __nv_bfloat16 *__restrict__ dPst, const __nv_bfloat16 *__restrict__ Pbar_tm, int B,
                           int N, int H, int d, int P, long long ld, float *__restrict__ Dv) {
    const long long L = (long long)N * P;
    const long long row = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;   // (b*H + h)*L + r
    const int lane = threadIdx.x & 31;
    if (row >= (long long)B * H * L) return;   // whole warp
    const long long bh = row / L, r = row % L;
    const long long b = bh / H, h = bh % H, t = r / P, j = r % P;
    const __nv_bfloat16 *a = dPst + row * d;
    const __nv_bfloat16 *o = Pbar_tm + (((b * N + t) * H + h) * P + j) * d;
    float v = 0.f;
    for (int c = lane; c < d; c += 32) v += __bfloat162float(a[c]) * __bfloat162float(o[c]);
    v = warp_sum(v);
    if (lane == 0) Dv[bh * ld + r] = v;
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
cudaError_t launch_bwd_rowdot(const void *dPst, const void *Pbar, const Shape &sh, long long ld, float *Dv,
                              cudaStream_t st) {
    const long long rows = (long long)sh.B * sh.H * sh.L();
    bwd_rowdot<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>((const __nv_bfloat16 *)dPst, (const __nv_bfloat16 *)Pbar,
                                                           sh.B, sh.N, sh.H, sh.d, sh.P, ld, Dv);
    return cudaGetLastError();
}

}  // namespace iha
