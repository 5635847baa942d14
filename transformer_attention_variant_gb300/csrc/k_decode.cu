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
//   4. decode_combine: merge the chunks of every (b, h', j) and apply the R contraction
//                      out[b][h][c] = sum_{h',j} R[h][h'P + j] Pbar[b][h'][j][c] in one pass.
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
// memory.  BM batch rows per pass.  ONE_PASS (B <= BM): the 8 warps' sums go into the slab's
// space once every warp is done with the slab, so a CTA holds about 66 KB and three fit on an
// SM for every BM (with a buffer of their own, 98 KB at BM = 4 allowed two per SM and the
// 384 CTAs ran in two waves: 17.5 against 8.5 us at B = 4).
constexpr int DP_SLAB = DC_KROWS_MAX * 256 * 2;   // 64 KB
static_assert((size_t)8 * DC_BMAX * 256 * 4 <= (size_t)DP_SLAB, "the warps' sums fit in the slab");
template <int BM, bool ONE_PASS>
constexpr size_t dp_smem_bytes() {
    return DP_SLAB + (size_t)BM * DC_KROWS_MAX * 4 + (ONE_PASS ? 0 : (size_t)8 * BM * 256 * 4) + 16 + 128;
}
template <int BM, bool ONE_PASS>
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
    float *red = ONE_PASS ? reinterpret_cast<float *>(slab) : xs + BM * DC_KROWS_MAX;   // [8 warps][BM][256]
    uint64_t *full = reinterpret_cast<uint64_t *>(ONE_PASS ? xs + BM * DC_KROWS_MAX : red + 8 * BM * 256);
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
        if (ONE_PASS) __syncthreads();   // every warp is done with the slab the sums overwrite
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
// 4. chunk merge and R contraction in one pass.  With w = 2^(m_ch - M) over the chunks of one
//    pseudo-query row k = (h', j) (M the largest chunk max) and L_k = sum_ch w l_ch,
//      out[b][h][c] = sum_k R[h][k] Pbar_k[c] = sum_{k, ch} (R[h][k] w / L_k) o_{k,ch}[c],
//    which is linear in the chunks' partial outputs.  A CTA per (b, h, 32 columns): R[h][:]
//    is an input, so it goes to shared memory before the wait for the attention; then one warp
//    per row k turns the (max, sum) pairs into those coefficients, each stored beside the index
//    of its partial-output row, and DCB_THREADS / 32 groups (warps) reduce those rows with
//    them, DCB_UNROLL loads of a thread in flight at once.
// ---------------------------------------------------------------------------------------
constexpr int DCB_THREADS = 1024, DCB_COLS = 32, DCB_UNROLL = 16, DK_HPMAX = 256;
constexpr size_t dcb_smem_bytes(int terms) { return ((size_t)2 * terms + DK_HPMAX + DCB_THREADS) * 4; }
__global__ void __launch_bounds__(DCB_THREADS)
decode_combine(const float *__restrict__ part_ml, const float *__restrict__ part_o, const float *__restrict__ R,
               int H, int d, int P, int nch, __nv_bfloat16 *__restrict__ out) {
    extern __shared__ float cb_sm[];
    pdl_trigger();
    const int b = blockIdx.x, h = blockIdx.y, c0 = blockIdx.z * DCB_COLS;
    const int HP = H * P, T = HP * nch;
    float *coef = cb_sm;                                           // [HP][nch]
    int *row = reinterpret_cast<int *>(cb_sm + T);                 // [HP][nch]: (b, h', ch, j) row of part_o
    float *rs = cb_sm + 2 * T;                                     // [DK_HPMAX]: R[h][:]
    float *red = rs + DK_HPMAX;                                    // [DCB_THREADS]
    for (int k = threadIdx.x; k < HP; k += DCB_THREADS) rs[k] = R[(size_t)h * HP + k];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();   // the attention's partial results
    constexpr int RPW = 4;   // rows of a warp whose (max, sum) loads are in flight at once
    for (int k0 = warp; k0 < HP; k0 += 32 * RPW) {
        float m[RPW][2], l[RPW][2];
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const int k = k0 + 32 * i, base = (b * H + k / P) * nch * P + k % P;   // + ch * P: (b, h', ch, j)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int ch = lane + 32 * u;   // nch <= 64
                const bool in = k < HP && ch < nch;
                m[i][u] = in ? part_ml[(size_t)(base + ch * P) * 2] : -INFINITY;
                l[i][u] = in ? part_ml[(size_t)(base + ch * P) * 2 + 1] : 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const int k = k0 + 32 * i;
            if (k >= HP) break;   // warp-uniform
            const int base = (b * H + k / P) * nch * P + k % P;
            float mg = fmaxf(m[i][0], m[i][1]);
#pragma unroll
            for (int o = 16; o; o >>= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, o));
            float w[2], L = 0.f;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                w[u] = m[i][u] == -INFINITY ? 0.f : exp2f(m[i][u] - mg);   // an empty chunk weighs nothing
                L = fmaf(l[i][u], w[u], L);
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
            const float r = L > 0.f ? rs[k] / L : 0.f;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int ch = lane + 32 * u;
                if (ch < nch) {
                    coef[k * nch + ch] = w[u] * r;
                    row[k * nch + ch] = base + ch * P;
                }
            }
        }
    }
    __syncthreads();
    constexpr int G = DCB_THREADS / DCB_COLS;
    const int g = threadIdx.x / DCB_COLS, c = c0 + threadIdx.x % DCB_COLS;   // c0 + 32 <= d
    float acc = 0.f;
    for (int t0 = g; t0 < T; t0 += G * DCB_UNROLL) {
        float xv[DCB_UNROLL];
#pragma unroll
        for (int u = 0; u < DCB_UNROLL; ++u) {
            const int t = t0 + u * G;
            xv[u] = t < T ? part_o[(size_t)row[t] * d + c] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < DCB_UNROLL; ++u)
            if (t0 + u * G < T) acc = fmaf(coef[t0 + u * G], xv[u], acc);
    }
    red[threadIdx.x] = acc;
    __syncthreads();
    if (threadIdx.x < DCB_COLS) {
        float v = 0.f;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) v += red[gg * DCB_COLS + threadIdx.x];
        out[((size_t)b * H + h) * d + c0 + threadIdx.x] = __float2bfloat16_rn(v);
    }
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
           al((size_t)B * H * DC_NCH_MAX * P * 2 * 4) + al((size_t)B * H * DC_NCH_MAX * P * d * 4);
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
        if (bm == 1) run(decode_proj<1, true>, dp_smem_bytes<1, true>());
        else if (bm == 2) run(decode_proj<2, true>, dp_smem_bytes<2, true>());
        else if (bm == 4) run(decode_proj<4, true>, dp_smem_bytes<4, true>());
        else if (B <= 8) run(decode_proj<8, true>, dp_smem_bytes<8, true>());
        else run(decode_proj<8, false>, dp_smem_bytes<8, false>());
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
    // 4. merge the chunks and contract with R
    if (d % DCB_COLS != 0 || (long long)B * H * nch * P >= (1LL << 31)) return cudaErrorInvalidValue;
    const size_t smem4 = dcb_smem_bytes(H * P * nch);
    e = cudaFuncSetAttribute(decode_combine, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem4);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_combine, dim3(B, H, d / DCB_COLS), dim3(DCB_THREADS), smem4, st,
                      (const float *)part_ml, (const float *)part_o, R, H, d, P, nch, (__nv_bfloat16 *)out);
}

}  // namespace iha
