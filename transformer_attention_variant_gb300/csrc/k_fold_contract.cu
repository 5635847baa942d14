// k_fold_contract.cu -- the two HBM-bound steps around the tensor-core kernels.
//
//  * fold: the pseudo-head mixing of "Interleaved Head Attention" section 4, Algorithm 1
//    ("偽頭混合"), S~_{h,j} = sum_m alpha_s[m,h,j] X W_s^(m), is linear in W, so it is
//    applied once to the weights:  W~_s[:, (h,j,c)] = sum_m alpha_s[m,h,j] W_s[:, m*d + c].
//    The result is stored transposed, Wt[(s,h,j,c)][k], so the projection GEMM reads
//    both operands K-major.
//  * contract: the unstack-and-contract step of Algorithm 1 ("反堆疊與收縮"),
//    O_h[t] = sum_{h'} sum_j R[h, h'P + j] P_{h',j}[t], heads concatenated.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "iha_internal.h"

namespace iha {

template <typename T>
__device__ __forceinline__ float ld_f(const T *p);
template <>
__device__ __forceinline__ float ld_f<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// ---------------------------------------------------------------------------------------
// fold: block = one s, FOLD_K consecutive k (the 32 lanes of a warp) and FOLD_C
// consecutive c.  The W slab W_s[k][m][c] of the block (all m) is staged in shared memory
// as [m][c][k] (padded); each warp owns FOLD_PP output pseudo-head pairs (h, j) at a time
// with their alpha_s[:, h, j] in registers, so one shared-memory read of W feeds FOLD_PP
// FMAs, and each output row segment (32 consecutive k) is one coalesced 64/128-byte store.
// ---------------------------------------------------------------------------------------
constexpr int FOLD_K = 32, FOLD_C = 32, FOLD_THREADS = 256, FOLD_WARPS = FOLD_THREADS / 32;

template <typename T, int MAXH, int FOLD_PP>
__global__ void __launch_bounds__(FOLD_THREADS)
fold_kernel(const T *__restrict__ WQ, const T *__restrict__ WK, const T *__restrict__ WV,
            const float *__restrict__ aQ, const float *__restrict__ aK, const float *__restrict__ aV,
            T *__restrict__ Wt, int H, int d, int P) {
    extern __shared__ float fsm[];
    const int s = blockIdx.z;
    const T *W = s == 0 ? WQ : (s == 1 ? WK : WV);
    const float *alpha = s == 0 ? aQ : (s == 1 ? aK : aV);
    const long long D = (long long)H * d;
    const int k0 = blockIdx.x * FOLD_K, c0 = blockIdx.y * FOLD_C;
    constexpr int KP = FOLD_K + 1;                            // padded row (no bank conflicts)
    float *Ws = fsm;                                          // [H][FOLD_C][KP]
    float *as = fsm + (size_t)H * FOLD_C * KP;                // [H][H][P]
    for (int idx = threadIdx.x; idx < H * FOLD_C * FOLD_K; idx += blockDim.x) {
        const int cc = idx % FOLD_C, rest = idx / FOLD_C, kk = rest % FOLD_K, m = rest / FOLD_K;
        const long long k = k0 + kk;
        const int c = c0 + cc;
        Ws[((size_t)m * FOLD_C + cc) * KP + kk] = (k < D && c < d) ? ld_f(W + k * D + (long long)m * d + c) : 0.f;
    }
    for (int idx = threadIdx.x; idx < H * H * P; idx += blockDim.x) as[idx] = alpha[idx];
    __syncthreads();
    const int kk = threadIdx.x % 32, warp = threadIdx.x / 32;
    const long long k = k0 + kk;
    const int HP = H * P;
    const int ccmax = d - c0 < FOLD_C ? d - c0 : FOLD_C;
    for (int p0 = warp * FOLD_PP; p0 < HP; p0 += FOLD_WARPS * FOLD_PP) {
        float a[FOLD_PP][MAXH];
#pragma unroll
        for (int q = 0; q < FOLD_PP; ++q)
#pragma unroll
            for (int m = 0; m < MAXH; ++m)
                a[q][m] = (m < H && p0 + q < HP) ? as[(size_t)m * HP + p0 + q] : 0.f;   // alpha[m][h][j], pair = h*P + j
        for (int cc = 0; cc < ccmax; ++cc) {
            float acc[FOLD_PP] = {};
#pragma unroll
            for (int m = 0; m < MAXH; ++m) {
                if (m < H) {
                    const float wv = Ws[((size_t)m * FOLD_C + cc) * KP + kk];
#pragma unroll
                    for (int q = 0; q < FOLD_PP; ++q) acc[q] = fmaf(a[q][m], wv, acc[q]);
                }
            }
            if (k < D) {
#pragma unroll
                for (int q = 0; q < FOLD_PP; ++q)
                    if (p0 + q < HP)   // row (s, h, j, c) = s*H*P*d + (h*P + j)*d + c
                        Wt[((long long)s * HP * d + (long long)(p0 + q) * d + c0 + cc) * D + k] = from_f<T>(acc[q]);
            }
        }
    }
}

template <typename T, int MAXH, int PP>
static cudaError_t launch_fold_t(const void *WQ, const void *WK, const void *WV, const float *aQ, const float *aK,
                                 const float *aV, const Shape &sh, void *Wt, cudaStream_t st) {
    const long long D = sh.D();
    dim3 grid((unsigned)((D + FOLD_K - 1) / FOLD_K), (unsigned)((sh.d + FOLD_C - 1) / FOLD_C), 3);
    const size_t smem = sizeof(float) * ((size_t)sh.H * FOLD_C * (FOLD_K + 1) + (size_t)sh.H * sh.H * sh.P);
    cudaError_t e =
        cudaFuncSetAttribute(fold_kernel<T, MAXH, PP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    fold_kernel<T, MAXH, PP><<<grid, FOLD_THREADS, smem, st>>>((const T *)WQ, (const T *)WK, (const T *)WV, aQ, aK,
                                                               aV, (T *)Wt, sh.H, sh.d, sh.P);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_fold_h(const void *WQ, const void *WK, const void *WV, const float *aQ, const float *aK,
                                 const float *aV, const Shape &sh, void *Wt, cudaStream_t st) {
    if (sh.H <= 8) return launch_fold_t<T, 8, 4>(WQ, WK, WV, aQ, aK, aV, sh, Wt, st);
    if (sh.H <= 16) return launch_fold_t<T, 16, 4>(WQ, WK, WV, aQ, aK, aV, sh, Wt, st);
    if (sh.H <= 32) return launch_fold_t<T, 32, 2>(WQ, WK, WV, aQ, aK, aV, sh, Wt, st);
    if (sh.H <= 64) return launch_fold_t<T, 64, 1>(WQ, WK, WV, aQ, aK, aV, sh, Wt, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_fold(const void *WQ, const void *WK, const void *WV, const float *aQ, const float *aK,
                        const float *aV, const Shape &sh, int dtype, void *Wt, cudaStream_t st) {
    if (dtype == 1) return launch_fold_h<__nv_bfloat16>(WQ, WK, WV, aQ, aK, aV, sh, Wt, st);
    return launch_fold_h<float>(WQ, WK, WV, aQ, aK, aV, sh, Wt, st);
}

// ---------------------------------------------------------------------------------------
// contract: thread = (token, group of CON_HG output heads, VEC-wide chunk of the head dim).
// For each pseudo-head row i it loads VEC values of Pbar[token][i][:] (the d/VEC threads
// of one (token, group) read one contiguous row) and adds R[h][i] times them into its
// CON_HG x VEC accumulators; R is in shared memory and read as a warp-wide broadcast.
// The CON_HG-fold re-reads of a row hit L1, so DRAM sees Pbar once.
// ---------------------------------------------------------------------------------------
constexpr int CON_HG = 4, CON_THREADS = 256;

template <typename T, int VEC>
struct VecLoad;
template <>
struct VecLoad<__nv_bfloat16, 8> {
    __device__ static void load(const __nv_bfloat16 *p, float (&v)[8]) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(b[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    __device__ static void store(__nv_bfloat16 *p, const float (&v)[8]) {
        uint4 u;
        __nv_bfloat162 *b = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) b[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        *reinterpret_cast<uint4 *>(p) = u;
    }
};
template <>
struct VecLoad<float, 4> {
    __device__ static void load(const float *p, float (&v)[4]) {
        const float4 u = __ldg(reinterpret_cast<const float4 *>(p));
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    }
    __device__ static void store(float *p, const float (&v)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <>
struct VecLoad<float, 1> {
    __device__ static void load(const float *p, float (&v)[1]) { v[0] = __ldg(p); }
    __device__ static void store(float *p, const float (&v)[1]) { *p = v[0]; }
};

template <typename T, int VEC>
__global__ void __launch_bounds__(CON_THREADS)
contract_kernel(const T *__restrict__ pbar, const float *__restrict__ R, T *__restrict__ out, long long BN, int H,
                int P, int d) {
    extern __shared__ float Rs[];   // [H][H*P]
    const int HP = H * P;
    for (int i = threadIdx.x; i < H * HP; i += blockDim.x) Rs[i] = R[i];
    __syncthreads();
    const int cpr = d / VEC;                         // chunks per row
    const int ngroups = (H + CON_HG - 1) / CON_HG;
    const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (item >= BN * ngroups * cpr) return;
    const int cc = (int)(item % cpr);
    const long long rest = item / cpr;
    const int hg = (int)(rest % ngroups) * CON_HG;
    const long long bt = rest / ngroups;
    const T *src = pbar + bt * HP * (long long)d + (long long)cc * VEC;
    T *dst = out + bt * (long long)H * d + (long long)cc * VEC;
    float acc[CON_HG][VEC];
#pragma unroll
    for (int a = 0; a < CON_HG; ++a)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[a][e] = 0.f;
    const float *Rg = Rs + (size_t)hg * HP;
#pragma unroll 4
    for (int i = 0; i < HP; ++i) {
        float v[VEC];
        VecLoad<T, VEC>::load(src + (long long)i * d, v);
#pragma unroll
        for (int a = 0; a < CON_HG; ++a) {
            const float r = (hg + a < H) ? Rg[a * HP + i] : 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[a][e] = fmaf(r, v[e], acc[a][e]);
        }
    }
#pragma unroll
    for (int a = 0; a < CON_HG; ++a)
        if (hg + a < H) VecLoad<T, VEC>::store(dst + (long long)(hg + a) * d, acc[a]);
}

template <typename T, int VEC>
static cudaError_t launch_contract_t(const void *Pbar, const float *R, const Shape &sh, void *out, cudaStream_t st) {
    const long long BN = (long long)sh.B * sh.N;
    const size_t smem = sizeof(float) * (size_t)sh.H * sh.H * sh.P;
    const long long items = BN * ((sh.H + CON_HG - 1) / CON_HG) * (sh.d / VEC);
    cudaError_t e = cudaFuncSetAttribute(contract_kernel<T, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    contract_kernel<T, VEC><<<(unsigned)((items + CON_THREADS - 1) / CON_THREADS), CON_THREADS, smem, st>>>(
        (const T *)Pbar, R, (T *)out, BN, sh.H, sh.P, sh.d);
    return cudaGetLastError();
}

cudaError_t launch_contract(const void *Pbar, const float *R, const Shape &sh, int dtype, void *out,
                            cudaStream_t st, int *status) {
    if (dtype == 1) {
        if (contract_tc_fits(sh) && (reinterpret_cast<uintptr_t>(out) & 15) == 0)
            return launch_contract_tc(Pbar, R, sh, out, st, status);
        if (contract_rowmix_fits(sh)) return launch_contract_rowmix(Pbar, R, sh, out, st, status);
        return launch_contract_t<__nv_bfloat16, 8>(Pbar, R, sh, out, st);
    }
    if (sh.d % 4 == 0) return launch_contract_t<float, 4>(Pbar, R, sh, out, st);
    return launch_contract_t<float, 1>(Pbar, R, sh, out, st);
}

}  // namespace iha
