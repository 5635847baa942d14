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
// fold: block = (32 k) x (16 c) tile of one s; loops over every (h, j).
// smem: Ws[m][kk][cc] (padded) and alpha_s.
// ---------------------------------------------------------------------------------------
constexpr int FOLD_TK = 32, FOLD_TC = 16, FOLD_THREADS = 256;

template <typename T>
__global__ void __launch_bounds__(FOLD_THREADS)
fold_kernel(const T *__restrict__ WQ, const T *__restrict__ WK, const T *__restrict__ WV,
            const float *__restrict__ aQ, const float *__restrict__ aK, const float *__restrict__ aV,
            T *__restrict__ Wt, int H, int d, int P) {
    extern __shared__ float fsm[];
    const int s = blockIdx.z;
    const T *W = s == 0 ? WQ : (s == 1 ? WK : WV);
    const float *alpha = s == 0 ? aQ : (s == 1 ? aK : aV);
    const long long D = (long long)H * d, Hd = D;
    const int k0 = blockIdx.x * FOLD_TK, c0 = blockIdx.y * FOLD_TC;
    float *Ws = fsm;                                   // [H][FOLD_TK][FOLD_TC + 1]
    float *as = fsm + (size_t)H * FOLD_TK * (FOLD_TC + 1);   // [H][H][P]
    const int tile = FOLD_TK * FOLD_TC;
    for (int idx = threadIdx.x; idx < H * tile; idx += blockDim.x) {
        const int m = idx / tile, rem = idx % tile, kk = rem / FOLD_TC, cc = rem % FOLD_TC;
        const long long k = k0 + kk;
        const int c = c0 + cc;
        Ws[((size_t)m * FOLD_TK + kk) * (FOLD_TC + 1) + cc] = (k < D && c < d) ? ld_f(W + k * Hd + (long long)m * d + c) : 0.f;
    }
    for (int idx = threadIdx.x; idx < H * H * P; idx += blockDim.x) as[idx] = alpha[idx];
    __syncthreads();
    const long long HPd = (long long)H * P * d, Pd = (long long)P * d;
    for (int pair = 0; pair < H * P; ++pair) {
        const int h = pair / P, j = pair % P;
        for (int e = threadIdx.x; e < tile; e += blockDim.x) {
            const int kk = e % FOLD_TK, cc = e / FOLD_TK;
            float acc = 0.f;
            for (int m = 0; m < H; ++m)
                acc = fmaf(as[((size_t)m * H + h) * P + j], Ws[((size_t)m * FOLD_TK + kk) * (FOLD_TC + 1) + cc], acc);
            const long long k = k0 + kk;
            const int c = c0 + cc;
            if (k < D && c < d) Wt[(s * HPd + h * Pd + (long long)j * d + c) * D + k] = from_f<T>(acc);
        }
    }
}

cudaError_t launch_fold(const void *WQ, const void *WK, const void *WV, const float *aQ, const float *aK,
                        const float *aV, const Shape &sh, int dtype, void *Wt, cudaStream_t st) {
    const long long D = sh.D();
    dim3 grid((unsigned)((D + FOLD_TK - 1) / FOLD_TK), (unsigned)((sh.d + FOLD_TC - 1) / FOLD_TC), 3);
    const size_t smem = sizeof(float) * ((size_t)sh.H * FOLD_TK * (FOLD_TC + 1) + (size_t)sh.H * sh.H * sh.P);
    cudaError_t e;
    if (dtype == 1) {
        e = cudaFuncSetAttribute(fold_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        fold_kernel<__nv_bfloat16><<<grid, FOLD_THREADS, smem, st>>>(
            (const __nv_bfloat16 *)WQ, (const __nv_bfloat16 *)WK, (const __nv_bfloat16 *)WV, aQ, aK, aV,
            (__nv_bfloat16 *)Wt, sh.H, sh.d, sh.P);
    } else {
        e = cudaFuncSetAttribute(fold_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        fold_kernel<float><<<grid, FOLD_THREADS, smem, st>>>((const float *)WQ, (const float *)WK,
                                                             (const float *)WV, aQ, aK, aV, (float *)Wt, sh.H,
                                                             sh.d, sh.P);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------
// contract: one thread = (token row bt, VEC-wide chunk of the head dim), all H output
// heads in groups of HB.  R lives in shared memory.  Reads of one pseudo-head row by the
// d/VEC threads of a token are contiguous.
// ---------------------------------------------------------------------------------------
constexpr int CON_HB = 16, CON_THREADS = 256;

template <typename T, int VEC>
struct VecLoad;
template <>
struct VecLoad<__nv_bfloat16, 8> {
    __device__ static void load(const __nv_bfloat16 *p, float (&v)[8]) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
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
        const float4 u = *reinterpret_cast<const float4 *>(p);
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    }
    __device__ static void store(float *p, const float (&v)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <>
struct VecLoad<float, 1> {
    __device__ static void load(const float *p, float (&v)[1]) { v[0] = *p; }
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
    const int cpr = d / VEC;   // chunks per row
    const long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (item >= BN * cpr) return;
    const long long bt = item / cpr;
    const int cc = (int)(item % cpr);
    const T *src = pbar + bt * HP * (long long)d + (long long)cc * VEC;
    T *dst = out + bt * (long long)H * d + (long long)cc * VEC;
    for (int hg = 0; hg < H; hg += CON_HB) {
        float acc[CON_HB][VEC];
#pragma unroll
        for (int a = 0; a < CON_HB; ++a)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[a][e] = 0.f;
        for (int i = 0; i < HP; ++i) {
            float v[VEC];
            VecLoad<T, VEC>::load(src + (long long)i * d, v);
#pragma unroll
            for (int a = 0; a < CON_HB; ++a) {
                const int h = hg + a;
                const float r = h < H ? Rs[h * HP + i] : 0.f;
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[a][e] = fmaf(r, v[e], acc[a][e]);
            }
        }
#pragma unroll
        for (int a = 0; a < CON_HB; ++a)
            if (hg + a < H) VecLoad<T, VEC>::store(dst + (long long)(hg + a) * d, acc[a]);
    }
}

cudaError_t launch_contract(const void *Pbar, const float *R, const Shape &sh, int dtype, void *out,
                            cudaStream_t st) {
    const long long BN = (long long)sh.B * sh.N;
    const size_t smem = sizeof(float) * (size_t)sh.H * sh.H * sh.P;
    cudaError_t e;
    if (dtype == 1) {
        const long long items = BN * (sh.d / 8);
        e = cudaFuncSetAttribute(contract_kernel<__nv_bfloat16, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        contract_kernel<__nv_bfloat16, 8><<<(unsigned)((items + CON_THREADS - 1) / CON_THREADS), CON_THREADS, smem, st>>>(
            (const __nv_bfloat16 *)Pbar, R, (__nv_bfloat16 *)out, BN, sh.H, sh.P, sh.d);
    } else if (sh.d % 4 == 0) {
        const long long items = BN * (sh.d / 4);
        e = cudaFuncSetAttribute(contract_kernel<float, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        contract_kernel<float, 4><<<(unsigned)((items + CON_THREADS - 1) / CON_THREADS), CON_THREADS, smem, st>>>(
            (const float *)Pbar, R, (float *)out, BN, sh.H, sh.P, sh.d);
    } else {
        const long long items = BN * sh.d;
        e = cudaFuncSetAttribute(contract_kernel<float, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        contract_kernel<float, 1><<<(unsigned)((items + CON_THREADS - 1) / CON_THREADS), CON_THREADS, smem, st>>>(
            (const float *)Pbar, R, (float *)out, BN, sh.H, sh.P, sh.d);
    }
    return cudaGetLastError();
}

}  // namespace iha
