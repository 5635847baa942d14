// k_backward.cu -- the reductions of the backward pass of one IHA layer ("Interleaved Head
// Attention" section 4, Algorithm 1, differentiated step by step): the per-row term of the
// softmax gradient ("注意力机制" eqs. (5.24)-(5.31)),
//
//     D_r = sum_c dPbar_r[c] Pbar_r[c]      (r a stacked row t*P + j; dPbar the gradient
//                                            reaching the attention output)
//
// and the token reductions that give the gradients of the small mixing matrices
// (token_gram: sum over tokens and columns of products of two head blocks).  The dense
// contractions (attention gradients, weight and input GEMMs) are in k_backward_tc.cu.
//
// Layouts: stacked [B][H][L][d] (L = N*P); token-major [B*N][H*P][d] (row h*P + j of token t,
// the layout of Pbar); D [B*H][L].  Arithmetic in fp32.
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
                           int N, int H, int d, int P, float *__restrict__ Dv) {
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
    if (lane == 0) Dv[row] = v;
}

// ---------------------------------------------------------------------------------------
// token_gram: part[blk][a][b] = sum over this block's tokens t, and c < d, of
//             U[t*us + a*d + c] * V[t*vs + b*d + c]      (a < NA, b < NB)
// ---------------------------------------------------------------------------------------
constexpr int TG_THREADS = 256, TG_PAIRS = 8;   // NA*NB <= TG_THREADS*TG_PAIRS
__global__ void __launch_bounds__(TG_THREADS)
bwd_token_gram(const __nv_bfloat16 *__restrict__ U, long long us, int NA, const __nv_bfloat16 *__restrict__ V,
               long long vs, int NB, int d, long long ntok, int tok_per_blk, float *__restrict__ part) {
    extern __shared__ __nv_bfloat16 tg[];
    const int ld = d + 2;   // padded rows: consecutive rows start one bank apart
    __nv_bfloat16 *us_ = tg, *vs_ = tg + (size_t)NA * ld;
    float acc[TG_PAIRS];
#pragma unroll
    for (int i = 0; i < TG_PAIRS; ++i) acc[i] = 0.f;
    const long long t0 = (long long)blockIdx.x * tok_per_blk;
    const long long t1 = min(ntok, t0 + tok_per_blk);
    for (long long t = t0; t < t1; ++t) {
        __syncthreads();
        for (int i = threadIdx.x; i < NA * d; i += blockDim.x) us_[(i / d) * ld + i % d] = U[t * us + i];
        for (int i = threadIdx.x; i < NB * d; i += blockDim.x) vs_[(i / d) * ld + i % d] = V[t * vs + i];
        __syncthreads();
#pragma unroll
        for (int i = 0; i < TG_PAIRS; ++i) {
            const int pr = threadIdx.x + i * TG_THREADS;
            if (pr >= NA * NB) break;
            const __nv_bfloat16 *ua = us_ + (pr / NB) * ld, *vb = vs_ + (pr % NB) * ld;
            float sacc = 0.f;
            for (int c = 0; c < d; ++c) sacc = fmaf(__bfloat162float(ua[c]), __bfloat162float(vb[c]), sacc);
            acc[i] += sacc;
        }
    }
#pragma unroll
    for (int i = 0; i < TG_PAIRS; ++i) {
        const int pr = threadIdx.x + i * TG_THREADS;
        if (pr < NA * NB) part[(size_t)blockIdx.x * NA * NB + pr] = acc[i];
    }
}

__global__ void bwd_sum_partials(const float *__restrict__ part, int nparts, int n, float *__restrict__ out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float v = 0.f;
    for (int p = 0; p < nparts; ++p) v += part[(size_t)p * n + i];
    out[i] = v;
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
cudaError_t launch_bwd_rowdot(const void *dPst, const void *Pbar, const Shape &sh, float *Dv, cudaStream_t st) {
    const long long rows = (long long)sh.B * sh.H * sh.L();
    bwd_rowdot<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>((const __nv_bfloat16 *)dPst, (const __nv_bfloat16 *)Pbar,
                                                           sh.B, sh.N, sh.H, sh.d, sh.P, Dv);
    return cudaGetLastError();
}

size_t bwd_gram_part_floats(long long ntok, int NA, int NB) {
    const long long nblk = ntok < 1024 ? ntok : 1024;
    return (size_t)nblk * NA * NB;
}

cudaError_t launch_bwd_gram(const void *U, long long us, int NA, const void *V, long long vs, int NB, int d,
                            long long ntok, float *part, float *out, cudaStream_t st) {
    if (NA * NB > TG_THREADS * TG_PAIRS) return cudaErrorInvalidValue;
    const long long nblk = ntok < 1024 ? ntok : 1024;
    const int tpb = (int)((ntok + nblk - 1) / nblk);
    const size_t smem = (size_t)(NA + NB) * (d + 2) * 2;
    cudaError_t e = cudaFuncSetAttribute(bwd_token_gram, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    bwd_token_gram<<<(unsigned)nblk, TG_THREADS, smem, st>>>((const __nv_bfloat16 *)U, us, NA,
                                                             (const __nv_bfloat16 *)V, vs, NB, d, ntok, tpb, part);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int n = NA * NB;
    bwd_sum_partials<<<(n + 255) / 256, 256, 0, st>>>(part, (int)nblk, n, out);
    return cudaGetLastError();
}

}  // namespace iha
