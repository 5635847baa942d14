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
// D_r = dPbar_r . Pbar_r: G = d/8 lanes per stacked row, one 16-byte load of each operand per
// lane, the G partial sums added by shuffles within the group
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float dot_bf16x8(const uint4 a, const uint4 b) {
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
    float v = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        v = fmaf(__uint_as_float(av[e] << 16), __uint_as_float(bv[e] << 16), v);
        v = fmaf(__uint_as_float(av[e] & 0xffff0000u), __uint_as_float(bv[e] & 0xffff0000u), v);
    }
    return v;
}

template <int G>
__global__ void bwd_rowdot(const __nv_bfloat16 *__restrict__ dPst, const __nv_bfloat16 *__restrict__ Pbar_tm, int B,
                           int N, int H, int P, long long ld, float *__restrict__ Dv) {
    constexpr int d = 8 * G;
    const long long L = (long long)N * P;
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / G;   // (b*H + h)*L + r
    const int sub = threadIdx.x % G;
    const bool in = row < (long long)B * H * L;
    float v = 0.f;
    long long bh = 0, r = 0;
    if (in) {
        bh = row / L;
        r = row % L;
        const long long b = bh / H, h = bh % H, t = r / P, j = r % P;
        const uint4 a = *reinterpret_cast<const uint4 *>(dPst + row * d + sub * 8);
        const uint4 o = *reinterpret_cast<const uint4 *>(Pbar_tm + (((b * N + t) * H + h) * P + j) * d + sub * 8);
        v = dot_bf16x8(a, o);
    }
#pragma unroll
    for (int off = G / 2; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);   // every lane takes part
    if (in && sub == 0) Dv[bh * ld + r] = v;
}

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
    const long long threads = rows * (sh.d / 8);
    const unsigned grid = (unsigned)((threads + 255) / 256);
    if (sh.d == 128)
        bwd_rowdot<16><<<grid, 256, 0, st>>>((const __nv_bfloat16 *)dPst, (const __nv_bfloat16 *)Pbar, sh.B, sh.N, sh.H,
                                             sh.P, ld, Dv);
    else if (sh.d == 64)
        bwd_rowdot<8><<<grid, 256, 0, st>>>((const __nv_bfloat16 *)dPst, (const __nv_bfloat16 *)Pbar, sh.B, sh.N, sh.H,
                                            sh.P, ld, Dv);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace iha
