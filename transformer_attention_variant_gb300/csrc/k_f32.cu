// k_f32.cu -- exact-fp32 SIMT kernels for the float32 arithmetic type (IHA_DTYPE_F32):
// the projection GEMM with the stacked store, and the masked online-softmax attention.
// Plain FFMA arithmetic (no TF32 tensor cores) so that results stay within a few fp32
// ulps of the exact forward pass.
#include <cuda_runtime.h>

#include "iha_internal.h"

namespace iha {

// ---------------------------------------------------------------------------------------
// Projection: C[m][n] = sum_k X[m][k] Wt[n][k], m = b*N + t, n = s*H*P*d + h*P*d + j*d + c,
// stored at QKV[s][b][h][t*P + j][c].  64x64 output tile, 16-wide K slices, 4x4 per thread.
// ---------------------------------------------------------------------------------------
constexpr int F32_TM = 64, F32_TN = 64, F32_TK = 16;

__global__ void __launch_bounds__(256)
proj_f32_kernel(const float *__restrict__ X, const float *__restrict__ Wt, float *__restrict__ qkv, long long M,
                long long Ncols, long long K, int N_tok, int H, int P, int d, long long s_stride) {
    __shared__ float As[F32_TK][F32_TM + 4];
    __shared__ float Bs[F32_TK][F32_TN + 4];
    const long long m0 = (long long)blockIdx.y * F32_TM, n0 = (long long)blockIdx.x * F32_TN;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (long long k0 = 0; k0 < K; k0 += F32_TK) {
        for (int i = threadIdx.x; i < F32_TK * F32_TM; i += 256) {
            const int kk = i % F32_TK, mm = i / F32_TK;
            const long long m = m0 + mm, k = k0 + kk;
            As[kk][mm] = (m < M && k < K) ? X[m * K + k] : 0.f;
            const long long n = n0 + mm;
            Bs[kk][mm] = (n < Ncols && k < K) ? Wt[n * K + k] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < F32_TK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int i = 0; i < 4; ++i) b[i] = Bs[kk][tx * 4 + i];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    const long long HPd = (long long)H * P * d, Pd = (long long)P * d;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const long long m = m0 + ty * 4 + i;
        if (m >= M) continue;
        const long long b = m / N_tok, t = m % N_tok;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const long long n = n0 + tx * 4 + j;
            if (n >= Ncols) continue;
            const long long s = n / HPd, rem = n % HPd, h = rem / Pd, jc = rem % Pd;
            qkv[s * s_stride + ((b * H + h) * N_tok + t) * Pd + jc] = acc[i][j];
        }
    }
}

// ---------------------------------------------------------------------------------------
// Attention: one warp per stacked query row r = t*P + j of head (b, h); the lanes split
// the head dimension.  Keys are visited in order over the row's readable interval
// [lo, hi] of stacked rows (t' <= t, and t - t' < w for the window), with an online
// softmax (running max, rescaled sum and accumulator).
// ---------------------------------------------------------------------------------------
constexpr int F32_MAXD = 256;

__global__ void __launch_bounds__(256)
attn_f32_kernel(const float *__restrict__ qkv, float *__restrict__ pbar, int B, int N, int H, int P, int d,
                int mask_mode, int window, float scale, long long s_stride) {
    const long long L = (long long)N * P;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    if (gw >= (long long)B * H * L) return;
    const long long bh = gw / L, r = gw % L;
    const long long t = r / P, j = r % P;
    const float *Qh = qkv + bh * L * d;
    const float *Kh = qkv + s_stride + bh * L * d;
    const float *Vh = qkv + 2 * s_stride + bh * L * d;
    constexpr int PER = F32_MAXD / 32;
    float q[PER], acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int c = lane + 32 * i;
        q[i] = c < d ? Qh[r * d + c] : 0.f;
        acc[i] = 0.f;
    }
    long long lo = 0, hi = L - 1;
    if (mask_mode >= 1) hi = (t + 1) * P - 1 < L - 1 ? (t + 1) * P - 1 : L - 1;
    if (mask_mode == 2) lo = t - window + 1 > 0 ? (t - window + 1) * P : 0;
    float m = -INFINITY, l = 0.f;
    for (long long kr = lo; kr <= hi; ++kr) {
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int c = lane + 32 * i;
            if (c < d) part = fmaf(q[i], Kh[kr * d + c], part);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        const float s = part * scale;
        const float m_new = fmaxf(m, s);
        const float corr = expf(m - m_new);   // m = -inf on the first key: exp(-inf) = 0
        const float pr = expf(s - m_new);
        l = l * corr + pr;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int c = lane + 32 * i;
            const float v = c < d ? Vh[kr * d + c] : 0.f;
            acc[i] = fmaf(pr, v, acc[i] * corr);
        }
        m = m_new;
    }
    const long long b = bh / H, h = bh % H;
    float *dst = pbar + (((b * N + t) * H + h) * P + j) * d;
    const float inv = 1.f / l;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int c = lane + 32 * i;
        if (c < d) dst[c] = acc[i] * inv;
    }
}

cudaError_t launch_project_f32(const void *X, const void *Wt, const Shape &sh, void *QKV, cudaStream_t st) {
    const long long M = (long long)sh.B * sh.N, Ncols = sh.wt_rows(), K = sh.D();
    dim3 grid((unsigned)((Ncols + F32_TN - 1) / F32_TN), (unsigned)((M + F32_TM - 1) / F32_TM));
    proj_f32_kernel<<<grid, 256, 0, st>>>((const float *)X, (const float *)Wt, (float *)QKV, M, Ncols, K, sh.N,
                                          sh.H, sh.P, sh.d, sh.qkv_elems());
    return cudaGetLastError();
}

cudaError_t launch_attention_f32(const void *QKV, const Shape &sh, int mask_mode, int window, void *Pbar,
                                 cudaStream_t st) {
    if (sh.d > F32_MAXD) return cudaErrorInvalidValue;
    const long long warps = (long long)sh.B * sh.H * sh.L();
    const long long threads = warps * 32;
    attn_f32_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
        (const float *)QKV, (float *)Pbar, sh.B, sh.N, sh.H, sh.P, sh.d, mask_mode, window,
        1.0f / sqrtf((float)sh.d), sh.qkv_elems());
    return cudaGetLastError();
}

}  // namespace iha
