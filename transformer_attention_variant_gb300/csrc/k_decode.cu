// k_decode.cu -- one decoding step of Interleaved Head Attention over a cache of pseudo-keys
// and pseudo-values ("Interleaved Head Attention" section 4, Algorithm 1, evaluated for the
// rows of one new token t; the mask is by original position, so the P pseudo-queries of
// token t read exactly the cached pseudo-tokens of positions t' <= t, and t - t' < w).
//
// Per step (bf16 storage, fp32 arithmetic):
//   1. decode_proj:    y_s[b] = x[b] W_s (s = Q, K, V) as a split-K GEMV; W is read once.
//   2. decode_mix:     q~/k~/v~_{h,j}[b] = sum_m alpha_s[m,h,j] y_s[b][m]; k~ and v~ go into
//                      the cache at stacked row t*P + j, q~ into the workspace.
//   3. decode_attn_tc (k_decode_tc.cu): split-KV attention on the tensor cores, a CTA per
//                      chunk of the readable cached rows of one (b, h); the chunk's (max, sum,
//                      unnormalised output) of every query go to the workspace.
//   4. decode_merge:   merge the chunks of every (b, h, j);
//      decode_contract: the R contraction out[b][h][c] = sum_{h',j} R[h][h'P + j] Pbar[b][h'][j][c].
// The step is HBM-bound: W (3 D^2 bf16) and the cached rows of K and V are the bytes.  The
// kernels are chained with programmatic dependent launch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "iha_internal.h"
#include "ptx.cuh"

namespace iha {

constexpr int DC_KS = 16;         // K splits of the projection GEMV
constexpr int DC_BMAX = 8;        // batch rows per pass of the GEMV (at most)
constexpr int DC_KROWS_MAX = 128; // rows per K split: D / DC_KS, D <= 2048
constexpr int DC_NCH_MAX = 64;    // KV chunks per (b, h)

// ---------------------------------------------------------------------------------------
// 1. projection GEMV: Yp[ks][b][s][n] = sum_{k in split ks} x[b][k] W_s[k][n]
// ---------------------------------------------------------------------------------------
// A CTA owns up to 256 columns of one W_s and one split of D / DC_KS rows (a 64 KB slab).
// Warp 0 moves the slab into shared memory with one bulk copy per row (no registers held,
// so three CTAs fit on an SM and the whole of W is in flight at once); then a lane owns 8
// columns and warp w the rows w, w+8, ..., and the 8 warps' sums are added in shared
// memory.  BM batch rows per pass.
constexpr int DP_SLAB = DC_KROWS_MAX * 256 * 2;   // 64 KB
template <int BM>
constexpr size_t dp_smem_bytes() {
    return DP_SLAB + (size_t)BM * DC_KROWS_MAX * 4 + (size_t)8 * BM * 256 * 4 + 16 + 128;
}
template <int BM>
__global__ void __launch_bounds__(256)
decode_proj(const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *__restrict__ WQ,
            const __nv_bfloat16 *__restrict__ WK, const __nv_bfloat16 *__restrict__ WV, int B, int D,
            float *__restrict__ Yp, int *status) {
    extern __shared__ uint8_t psm_raw[];
    uint8_t *psm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(psm_raw) + 127) & ~uintptr_t(127));
    pdl_trigger();   // the mixing kernel may launch; it waits for this grid before reading Yp
    const int nblk = (D + 255) / 256;
    const int s = blockIdx.x / nblk, n0 = (blockIdx.x % nblk) * 256;
    const int ks = blockIdx.y, krows = D / DC_KS, k0 = ks * krows;
    const int ncols = min(256, D - n0);
    const __nv_bfloat16 *W = s == 0 ? WQ : (s == 1 ? WK : WV);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *slab = psm;                                                    // [krows][256] bf16
    float *xs = reinterpret_cast<float *>(psm + DP_SLAB);                   // [BM][krows]
    float *red = xs + BM * DC_KROWS_MAX;                                    // [8 warps][BM][256]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + 8 * BM * 256);
    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(krows * ncols * 2));
        __syncwarp();
        for (int k = lane; k < krows; k += 32)
            bulk_load(slab + k * 512, W + (size_t)(k0 + k) * D + n0, (uint32_t)ncols * 2, full);
    }
    const int n = lane * 8;   // this lane's 8 columns of the slab
    for (int b0 = 0; b0 < B; b0 += BM) {
        const int nb = min(BM, B - b0);
        if (b0 > 0) __syncthreads();
        for (int i = threadIdx.x; i < nb * krows; i += blockDim.x)
            xs[i] = __bfloat162float(x[(size_t)(b0 + i / krows) * D + k0 + i % krows]);
        __syncthreads();
        // the slab has landed (a wait that gives up leaves zeros and records the timeout)
        const bool have = mbar_wait(full, 0, status, kSiteDecodeProj, nullptr, kWaitLimitNs);
        float acc[BM][8];
#pragma unroll
        for (int b = 0; b < BM; ++b)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[b][e] = 0.f;
        if (have && n < ncols) {
#pragma unroll 4
            for (int k = warp; k < krows; k += 8) {
                const uint4 wv = *reinterpret_cast<const uint4 *>(slab + k * 512 + n * 2);
                const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
                float wf[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    wf[2 * e] = __uint_as_float(w4[e] << 16);
                    wf[2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
                }
#pragma unroll
                for (int b = 0; b < BM; ++b) {
                    if (b < nb) {
                        const float xv = xs[b * krows + k];
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[b][e] = fmaf(xv, wf[e], acc[b][e]);
                    }
                }
            }
        }
        // reduce over the 8 warps
#pragma unroll
        for (int b = 0; b < BM; ++b)
            if (b < nb)
#pragma unroll
                for (int e = 0; e < 8; ++e) red[(warp * BM + b) * 256 + n + e] = acc[b][e];
        __syncthreads();
        for (int i = threadIdx.x; i < nb * 256; i += blockDim.x) {
            const int b = i / 256, c = i % 256;
            if (c >= ncols) continue;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) v += red[(w * BM + b) * 256 + c];
            Yp[(((size_t)ks * B + b0 + b) * 3 + s) * D + n0 + c] = v;
        }
    }
}

// ---------------------------------------------------------------------------------------
// 2. mixing + cache append, DM_GROUPS CTAs of DM_THREADS per (b, s): y_s[b] = the sum of the
//    K-split partials (every load of a thread in flight at once) and alpha_s go to shared
//    memory, then each thread makes 8 consecutive columns of one (h, j) output row of the
//    CTA's share: 8 FMAs per two 16-byte shared loads of y and one of alpha
// ---------------------------------------------------------------------------------------
constexpr int DM_THREADS = 1024, DM_GROUPS = 4;
__global__ void __launch_bounds__(DM_THREADS)
decode_mix(const float *__restrict__ Yp, const float *__restrict__ aQ, const float *__restrict__ aK,
           const float *__restrict__ aV, int B, int H, int d, int P, long long t, long long cache_rows,
           __nv_bfloat16 *__restrict__ qt, __nv_bfloat16 *__restrict__ Kc, __half *__restrict__ Vc) {
    extern __shared__ float msm[];
    pdl_trigger();
    const int b = blockIdx.x, s = blockIdx.y, g = blockIdx.z;
    const int D = H * d, HP = H * P;
    float *y = msm;              // [H][d]
    float *al = msm + D;         // alpha_s [H][H][P]
    const float *alg = s == 0 ? aQ : (s == 1 ? aK : aV);
    for (int i = threadIdx.x; i < H * HP; i += DM_THREADS) al[i] = alg[i];   // an input: no wait
    pdl_wait();   // the projection's partial sums
    constexpr int PER = 2;       // D <= PER * DM_THREADS
    {
        float v[PER][DC_KS];
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int i = threadIdx.x + u * DM_THREADS;
#pragma unroll
            for (int ks = 0; ks < DC_KS; ++ks) v[u][ks] = i < D ? Yp[(((size_t)ks * B + b) * 3 + s) * D + i] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int i = threadIdx.x + u * DM_THREADS;
            float acc = 0.f;
#pragma unroll
            for (int ks = 0; ks < DC_KS; ++ks) acc += v[u][ks];
            if (i < D) y[i] = acc;
        }
    }
    __syncthreads();
    // this CTA's rows (h, j): hj in [g*HP/G, (g+1)*HP/G); 8-column units of each row
    const int hj0 = (int)((long long)g * HP / DM_GROUPS), hj1 = (int)((long long)(g + 1) * HP / DM_GROUPS);
    const int upr = d / 8;   // units per row
    for (int i = threadIdx.x; i < (hj1 - hj0) * upr; i += DM_THREADS) {
        const int hj = hj0 + i / upr, c0 = (i % upr) * 8, h = hj / P, j = hj % P;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int m = 0; m < H; ++m) {
            const float a = al[(m * H + h) * P + j];   // alpha_s[m][h][j]
            const float4 y0 = *reinterpret_cast<const float4 *>(y + m * d + c0);
            const float4 y1 = *reinterpret_cast<const float4 *>(y + m * d + c0 + 4);
            acc[0] = fmaf(a, y0.x, acc[0]);
            acc[1] = fmaf(a, y0.y, acc[1]);
            acc[2] = fmaf(a, y0.z, acc[2]);
            acc[3] = fmaf(a, y0.w, acc[3]);
            acc[4] = fmaf(a, y1.x, acc[4]);
            acc[5] = fmaf(a, y1.y, acc[5]);
            acc[6] = fmaf(a, y1.z, acc[6]);
            acc[7] = fmaf(a, y1.w, acc[7]);
        }
        uint4 pk;
        if (s == 2) {
            pk = make_uint4(pack_f16x2(acc[0], acc[1]), pack_f16x2(acc[2], acc[3]), pack_f16x2(acc[4], acc[5]),
                            pack_f16x2(acc[6], acc[7]));
        } else {
            pk = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                            pack_bf16x2(acc[6], acc[7]));
        }
        if (s == 0) {
            *reinterpret_cast<uint4 *>(qt + (((size_t)b * H + h) * P + j) * d + c0) = pk;
        } else {
            const size_t row = ((size_t)b * H + h) * cache_rows + (size_t)t * P + j;   // stacked row t*P + j
            if (s == 1)
                *reinterpret_cast<uint4 *>(Kc + row * d + c0) = pk;
            else
                *reinterpret_cast<uint4 *>(Vc + row * d + c0) = pk;
        }
    }
}

// ---------------------------------------------------------------------------------------
// 4a. merge the chunks of one (b, h', j): Pbar[b][h'*P + j][c], one thread per column; the
//     chunks' partial results are read 16 at a time, all loads of a group in flight
// ---------------------------------------------------------------------------------------
constexpr int DM_CHUNK_GROUP = 16;
__global__ void decode_merge(const float *__restrict__ part_ml, const float *__restrict__ part_o, int H, int d, int P,
                             int nch, float *__restrict__ pbar) {
    pdl_trigger();
    pdl_wait();   // the attention's partial results
    const int bh = blockIdx.x, j = blockIdx.y, c = threadIdx.x;
    const size_t base = (size_t)bh * nch;
    float mt = -INFINITY, lt = 0.f, ot = 0.f;   // running merge (max, sum, output) in log2 units
    for (int c0 = 0; c0 < nch; c0 += DM_CHUNK_GROUP) {
        float m[DM_CHUNK_GROUP], l[DM_CHUNK_GROUP], o[DM_CHUNK_GROUP];
#pragma unroll
        for (int u = 0; u < DM_CHUNK_GROUP; ++u) {
            const bool in = c0 + u < nch;
            const size_t pidx = (base + c0 + u) * P + j;
            m[u] = in ? part_ml[pidx * 2] : -INFINITY;
            l[u] = in ? part_ml[pidx * 2 + 1] : 0.f;
            o[u] = in ? part_o[pidx * d + c] : 0.f;
        }
        float mg = mt;
#pragma unroll
        for (int u = 0; u < DM_CHUNK_GROUP; ++u) mg = fmaxf(mg, m[u]);
        if (mg == -INFINITY) continue;
        const float f = exp2f(mt - mg);   // mt = -inf -> 0
        lt *= f;
        ot *= f;
#pragma unroll
        for (int u = 0; u < DM_CHUNK_GROUP; ++u) {
            const float cw = m[u] == -INFINITY ? 0.f : exp2f(m[u] - mg);
            lt = fmaf(l[u], cw, lt);
            ot = fmaf(o[u], cw, ot);
        }
        mt = mg;
    }
    pbar[((size_t)bh * P + j) * d + c] = lt > 0.f ? ot / lt : 0.f;   // [b][h'][j][c] = [b][h'*P + j][c]
}

// ---------------------------------------------------------------------------------------
// 4b. R contraction: out[b][h][c] = sum_k R[h][k] Pbar[b][k][c], one CTA per (b, h); R[h][:]
//     goes to shared memory, and a thread's H*P loads are issued 64 at a time
// ---------------------------------------------------------------------------------------
constexpr int DK_GROUP = 64, DK_HPMAX = 256;
__global__ void decode_contract(const float *__restrict__ pbar, const float *__restrict__ R, int H, int d, int P,
                                __nv_bfloat16 *__restrict__ out) {
    pdl_trigger();
    const int b = blockIdx.x, h = blockIdx.y, c = threadIdx.x, HP = H * P;
    __shared__ float rs[DK_HPMAX];
    for (int i = threadIdx.x; i < HP; i += blockDim.x) rs[i] = R[(size_t)h * HP + i];   // an input: no wait
    __syncthreads();
    pdl_wait();   // the merged Pbar
    const float *pb = pbar + (size_t)b * HP * d;
    float v = 0.f;
    for (int k0 = 0; k0 < HP; k0 += DK_GROUP) {
        float xv[DK_GROUP];
#pragma unroll
        for (int u = 0; u < DK_GROUP; ++u) xv[u] = k0 + u < HP ? pb[(size_t)(k0 + u) * d + c] : 0.f;
#pragma unroll
        for (int u = 0; u < DK_GROUP; ++u)
            if (k0 + u < HP) v = fmaf(rs[k0 + u], xv[u], v);
    }
    out[((size_t)b * H + h) * d + c] = __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
bool decode_tc_supported(int d, int P, const void *Kc, const void *Vc);
int decode_tc_chunks(int B, int H, long long rows, int max_chunks, int &rows_per_chunk);
cudaError_t launch_decode_attn_tc(const void *qt, const void *Kc, const void *Vc, int B, int H, int d, int P,
                                  long long cache_rows, long long lo, long long hi, int nch, int rows_per_chunk,
                                  float *part_ml, float *part_o, cudaStream_t st, int *status);

// Launch with programmatic stream serialization: the kernel may start while its
// predecessor on the stream is still running (it calls pdl_wait() before reading that
// predecessor's results), so launch latency and prologue overlap the predecessor's tail.
template <typename Kern, typename... Act>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, Act... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

bool decode_supported(int H, int d, int P) {
    // H*d <= 2048: one K split of the projection GEMV is at most DC_KROWS_MAX rows
    return ((d == 64 && P <= 8) || (d == 128 && P <= 4)) && H * d <= DC_KS * DC_KROWS_MAX;
}

size_t decode_workspace_bytes(int B, int H, int d, int P) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    const size_t D = (size_t)H * d;
    return al((size_t)DC_KS * B * 3 * D * 4) + al((size_t)B * H * P * d * 2) +
           al((size_t)B * H * DC_NCH_MAX * P * 2 * 4) + al((size_t)B * H * DC_NCH_MAX * P * d * 4) +
           al((size_t)B * H * P * d * 4);
}

cudaError_t launch_decode(const void *x, const void *WQ, const void *WK, const void *WV, const float *aQ,
                          const float *aK, const float *aV, const float *R, int B, int H, int d, int P, int mask_mode,
                          int window, void *Kc, void *Vc, long long cache_tokens, long long t, void *out, void *ws,
                          cudaStream_t st, int *status) {
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    const int D = H * d;
    uint8_t *w = static_cast<uint8_t *>(ws);
    float *Yp = reinterpret_cast<float *>(w);
    w += al((size_t)DC_KS * B * 3 * D * 4);
    __nv_bfloat16 *qt = reinterpret_cast<__nv_bfloat16 *>(w);
    w += al((size_t)B * H * P * d * 2);
    float *part_ml = reinterpret_cast<float *>(w);
    w += al((size_t)B * H * DC_NCH_MAX * P * 2 * 4);
    float *part_o = reinterpret_cast<float *>(w);
    w += al((size_t)B * H * DC_NCH_MAX * P * d * 4);
    float *pbar = reinterpret_cast<float *>(w);
    const long long cache_rows = cache_tokens * P;

    // 1. projections
    const int krows = D / DC_KS;
    if (krows > DC_KROWS_MAX || D > 2 * DM_THREADS || H * P > DK_HPMAX) return cudaErrorInvalidValue;   // decode_supported
    cudaError_t e = cudaSuccess;
    {
        const int bm = B <= 1 ? 1 : (B <= 2 ? 2 : (B <= 4 ? 4 : 8));
        const dim3 g1(3 * ((D + 255) / 256), DC_KS);
        auto run = [&](auto kern, size_t smem1) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
            if (e == cudaSuccess)
                kern<<<g1, 256, smem1, st>>>((const __nv_bfloat16 *)x, (const __nv_bfloat16 *)WQ,
                                             (const __nv_bfloat16 *)WK, (const __nv_bfloat16 *)WV, B, D, Yp, status);
        };
        if (bm == 1) run(decode_proj<1>, dp_smem_bytes<1>());
        else if (bm == 2) run(decode_proj<2>, dp_smem_bytes<2>());
        else if (bm == 4) run(decode_proj<4>, dp_smem_bytes<4>());
        else run(decode_proj<8>, dp_smem_bytes<8>());
        if (e != cudaSuccess) return e;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // 2. mixing + append
    const size_t smem2 = ((size_t)D + (size_t)H * H * P) * 4;
    e = cudaFuncSetAttribute(decode_mix, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_mix, dim3(B, 3, DM_GROUPS), dim3(DM_THREADS), smem2, st, (const float *)Yp, aQ, aK, aV, B, H,
                   d, P, t, cache_rows, qt, (__nv_bfloat16 *)Kc, (__half *)Vc);
    if (e != cudaSuccess) return e;
    // 3. attention over the readable cached rows [lo, hi]
    const long long hi = (t + 1) * P - 1;
    long long lo = 0;
    if (mask_mode == 2) lo = (t - window + 1) * P > 0 ? (t - window + 1) * P : 0;
    const long long rows = hi - lo + 1;
    // 3. attention over the readable cached rows [lo, hi] on the tensor cores (k_decode_tc.cu),
    //    one wave of CTAs over the chunks of every (b, h)
    if (!decode_tc_supported(d, P, Kc, Vc)) return cudaErrorInvalidValue;   // checked by the entry point
    int rpc = 0;
    const int nch = decode_tc_chunks(B, H, rows, DC_NCH_MAX, rpc);
    e = launch_decode_attn_tc(qt, Kc, Vc, B, H, d, P, cache_rows, lo, hi, nch, rpc, part_ml, part_o, st, status);
    if (e != cudaSuccess) return e;
    // 4. merge the chunks, then the contraction
    e = launch_pdl(decode_merge, dim3(B * H, P), dim3(d), 0, st, (const float *)part_ml, (const float *)part_o, H, d,
                   P, nch, pbar);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_contract, dim3(B, H), dim3(d), 0, st, (const float *)pbar, R, H, d, P,
                      (__nv_bfloat16 *)out);
}

}  // namespace iha
