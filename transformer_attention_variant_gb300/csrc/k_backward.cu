// k_backward.cu -- kernels of the backward pass of one IHA layer ("Interleaved Head
// Attention" section 4, Algorithm 1, differentiated step by step; the softmax part follows
// "注意力机制" eqs. (5.24)-(5.31)).  With the forward's stacked Q~, K~, V~ (rows r = t*P + j),
// its attention output Pbar, the per-row log2 normaliser lse (p = 2^(s*log2(e)/sqrt(d) - lse))
// and dPbar (the gradient reaching the attention output), per head:
//
//     D_r   = sum_c dPbar_r[c] Pbar_r[c]
//     p_rc  = 2^(q_r.k_c * log2(e)/sqrt(d) - lse_r),  dp_rc = dPbar_r . v_c
//     ds_rc = p_rc (dp_rc - D_r)
//     dq_r  = sum_c ds_rc k_c / sqrt(d),  dk_c = sum_r ds_rc q_r / sqrt(d),  dv_c = sum_r p_rc dPbar_r
//
// over the readable pairs (c in [lo(r), hi(r)] by original position).  The other steps are
// small contractions over the heads (done by the forward's mixing and contraction kernels
// with the roles of alpha and R exchanged) and reductions over tokens (token_gram) or GEMMs
// (gemm_strided) for the weight gradients.  All arithmetic is fp32; tensors are bf16.
//
// Layouts: stacked [B][H][L][d] (L = N*P); token-major [B*N][H*P][d] (row h*P + j of token t,
// the layout of Pbar); lse and D [B*H][L].
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "iha_internal.h"

namespace iha {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// readable stacked key rows of query row r (original positions: t' <= t, t - t' < w)
__device__ __forceinline__ void bwd_key_interval(int r, int P, int L, int mode, int w, int &lo, int &hi) {
    const int t = r / P;
    lo = 0;
    hi = L - 1;
    if (mode >= 1) hi = min(hi, (t + 1) * P - 1);
    if (mode == 2) lo = max(lo, (t - w + 1) * P);
}
// stacked query rows that can read key row c: [qlo, qhi]
__device__ __forceinline__ void bwd_query_interval(int c, int P, int L, int mode, int w, int &qlo, int &qhi) {
    const int t = c / P;
    qlo = 0;
    qhi = L - 1;
    if (mode >= 1) qlo = t * P;
    if (mode == 2) qhi = min(qhi, (t + w) * P - 1);
}

template <typename T>
__device__ __forceinline__ float ldf(const T *p);
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
template <>
__device__ __forceinline__ float ldf<__half>(const __half *p) { return __half2float(*p); }

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
// dq (one warp per query row; lanes over d)
// ---------------------------------------------------------------------------------------
template <int DPL>   // d / 32
__global__ void bwd_attn_dq(const __nv_bfloat16 *__restrict__ Qs, const __nv_bfloat16 *__restrict__ Ks,
                            const __half *__restrict__ Vs, const __nv_bfloat16 *__restrict__ dPst,
                            const float *__restrict__ lse, const float *__restrict__ Dv, int B, int N, int H, int P,
                            int mode, int window, float sl2, float scale, __nv_bfloat16 *__restrict__ dQtm) {
    constexpr int d = DPL * 32;
    const int L = N * P;
    const long long row = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= (long long)B * H * L) return;   // whole warp
    const long long bh = row / L;
    const int r = (int)(row % L);
    float q[DPL], g[DPL], acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
        q[e] = __bfloat162float(Qs[row * d + lane + 32 * e]);
        g[e] = __bfloat162float(dPst[row * d + lane + 32 * e]);
        acc[e] = 0.f;
    }
    const float l2 = lse[row], Dr = Dv[row];
    int lo, hi;
    bwd_key_interval(r, P, L, mode, window, lo, hi);
    for (int c = lo; c <= hi; ++c) {
        const long long kr = (bh * L + c) * d;
        float k[DPL], s = 0.f, dp = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            k[e] = __bfloat162float(Ks[kr + lane + 32 * e]);
            s = fmaf(q[e], k[e], s);
            dp = fmaf(g[e], __half2float(Vs[kr + lane + 32 * e]), dp);
        }
        s = warp_sum(s);
        dp = warp_sum(dp);
        const float pr = exp2f(s * sl2 - l2);
        const float ds = pr * (dp - Dr);
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[e] = fmaf(ds, k[e], acc[e]);
    }
    const long long b = bh / H, h = bh % H, t = r / P, j = r % P;
    __nv_bfloat16 *dst = dQtm + (((b * N + t) * H + h) * P + j) * d;
#pragma unroll
    for (int e = 0; e < DPL; ++e) dst[lane + 32 * e] = __float2bfloat16_rn(acc[e] * scale);
}

// ---------------------------------------------------------------------------------------
// dk, dv (one warp per key row; lanes over d)
// ---------------------------------------------------------------------------------------
template <int DPL>
__global__ void bwd_attn_dkdv(const __nv_bfloat16 *__restrict__ Qs, const __nv_bfloat16 *__restrict__ Ks,
                              const __half *__restrict__ Vs, const __nv_bfloat16 *__restrict__ dPst,
                              const float *__restrict__ lse, const float *__restrict__ Dv, int B, int N, int H, int P,
                              int mode, int window, float sl2, float scale, __nv_bfloat16 *__restrict__ dKtm,
                              __nv_bfloat16 *__restrict__ dVtm) {
    constexpr int d = DPL * 32;
    const int L = N * P;
    const long long row = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= (long long)B * H * L) return;   // whole warp
    const long long bh = row / L;
    const int c = (int)(row % L);
    float k[DPL], v[DPL], dk[DPL], dv[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
        k[e] = __bfloat162float(Ks[row * d + lane + 32 * e]);
        v[e] = __half2float(Vs[row * d + lane + 32 * e]);
        dk[e] = dv[e] = 0.f;
    }
    int qlo, qhi;
    bwd_query_interval(c, P, L, mode, window, qlo, qhi);
    for (int r = qlo; r <= qhi; ++r) {
        const long long qr = (bh * L + r) * d;
        float q[DPL], g[DPL], s = 0.f, dp = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            q[e] = __bfloat162float(Qs[qr + lane + 32 * e]);
            g[e] = __bfloat162float(dPst[qr + lane + 32 * e]);
            s = fmaf(q[e], k[e], s);
            dp = fmaf(g[e], v[e], dp);
        }
        s = warp_sum(s);
        dp = warp_sum(dp);
        const float pr = exp2f(s * sl2 - lse[bh * L + r]);
        const float ds = pr * (dp - Dv[bh * L + r]);
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            dv[e] = fmaf(pr, g[e], dv[e]);
            dk[e] = fmaf(ds, q[e], dk[e]);
        }
    }
    const long long b = bh / H, h = bh % H, t = c / P, j = c % P;
    const long long o = (((b * N + t) * H + h) * P + j) * d;
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
        dKtm[o + lane + 32 * e] = __float2bfloat16_rn(dk[e] * scale);
        dVtm[o + lane + 32 * e] = __float2bfloat16_rn(dv[e]);
    }
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
// gemm_strided: C[m][n] (+)= sum_k A(m, k) B(k, n); A(m, k) = A[m*am + k*ak], B(k, n) =
// B[k*bk + n*bn] (bf16); C fp32 row-major [M][N].  64x64 tiles, 16-deep k steps, 256 threads
// with a 4x4 register tile each.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
bwd_gemm_strided(const __nv_bfloat16 *__restrict__ A, long long am, long long ak, const __nv_bfloat16 *__restrict__ Bm,
                 long long bk, long long bn, int M, int N, int K, float *__restrict__ C, int accumulate) {
    __shared__ float As[16][64 + 1];
    __shared__ float Bs[16][64 + 1];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int i = threadIdx.x; i < 16 * 64; i += 256) {
            const int kk = i / 64, mm = i % 64;
            const int m = m0 + mm, k = k0 + kk;
            As[kk][mm] = (m < M && k < K) ? __bfloat162float(A[(long long)m * am + (long long)k * ak]) : 0.f;
            const int n = n0 + mm;
            Bs[kk][mm] = (n < N && k < K) ? __bfloat162float(Bm[(long long)k * bk + (long long)n * bn]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
            if (m < M && n < N) {
                float *c = C + (long long)m * N + n;
                *c = accumulate ? *c + acc[i][j] : acc[i][j];
            }
        }
}

__global__ void bwd_to_bf16(const float *__restrict__ in, long long n, __nv_bfloat16 *__restrict__ out) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = __float2bfloat16_rn(in[i]);
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

cudaError_t launch_bwd_attention(const void *QKV, const void *dPst, const float *lse, const float *Dv, const Shape &sh,
                                 int mask_mode, int window, void *dQtm, void *dKtm, void *dVtm, cudaStream_t st) {
    const long long rows = (long long)sh.B * sh.H * sh.L();
    const long long third = sh.qkv_elems();
    const __nv_bfloat16 *Qs = (const __nv_bfloat16 *)QKV, *Ks = Qs + third;
    const __half *Vs = (const __half *)(Ks + third);
    const float scale = 1.f / sqrtf((float)sh.d), sl2 = 1.4426950408889634f * scale;
    const unsigned grid = (unsigned)((rows + 7) / 8);
    if (sh.d == 128) {
        bwd_attn_dq<4><<<grid, 256, 0, st>>>(Qs, Ks, Vs, (const __nv_bfloat16 *)dPst, lse, Dv, sh.B, sh.N, sh.H, sh.P,
                                             mask_mode, window, sl2, scale, (__nv_bfloat16 *)dQtm);
        bwd_attn_dkdv<4><<<grid, 256, 0, st>>>(Qs, Ks, Vs, (const __nv_bfloat16 *)dPst, lse, Dv, sh.B, sh.N, sh.H,
                                               sh.P, mask_mode, window, sl2, scale, (__nv_bfloat16 *)dKtm,
                                               (__nv_bfloat16 *)dVtm);
    } else if (sh.d == 64) {
        bwd_attn_dq<2><<<grid, 256, 0, st>>>(Qs, Ks, Vs, (const __nv_bfloat16 *)dPst, lse, Dv, sh.B, sh.N, sh.H, sh.P,
                                             mask_mode, window, sl2, scale, (__nv_bfloat16 *)dQtm);
        bwd_attn_dkdv<2><<<grid, 256, 0, st>>>(Qs, Ks, Vs, (const __nv_bfloat16 *)dPst, lse, Dv, sh.B, sh.N, sh.H,
                                               sh.P, mask_mode, window, sl2, scale, (__nv_bfloat16 *)dKtm,
                                               (__nv_bfloat16 *)dVtm);
    } else {
        return cudaErrorInvalidValue;
    }
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

cudaError_t launch_bwd_gemm(const void *A, long long am, long long ak, const void *Bm, long long bk, long long bn, int M,
                            int N, int K, float *C, bool accumulate, cudaStream_t st) {
    const dim3 grid((N + 63) / 64, (M + 63) / 64);
    bwd_gemm_strided<<<grid, 256, 0, st>>>((const __nv_bfloat16 *)A, am, ak, (const __nv_bfloat16 *)Bm, bk, bn, M, N, K,
                                           C, accumulate ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_bwd_to_bf16(const float *in, long long n, void *out, cudaStream_t st) {
    bwd_to_bf16<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(in, n, (__nv_bfloat16 *)out);
    return cudaGetLastError();
}

}  // namespace iha
