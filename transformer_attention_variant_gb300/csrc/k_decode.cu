// k_decode.cu -- one decoding step of Interleaved Head Attention over a cache of pseudo-keys
// and pseudo-values ("Interleaved Head Attention" section 4, Algorithm 1, evaluated for the
// rows of one new token t; the mask is by original position, so the P pseudo-queries of
// token t read exactly the cached pseudo-tokens of positions t' <= t, and t - t' < w).
//
// Per step (bf16 storage, fp32 arithmetic):
//   1. decode_proj:    y_s[b] = x[b] W_s (s = Q, K, V) as a split-K GEMV; W is read once.
//   2. decode_mix:     q~/k~/v~_{h,j}[b] = sum_m alpha_s[m,h,j] y_s[b][m]; k~ and v~ go into
//                      the cache at stacked row t*P + j, q~ into the workspace.
//   3. decode_attn:    split-KV attention: a CTA takes a chunk of the cached rows of one
//                      (b, h); all P pseudo-queries share the chunk's K and V reads (eight
//                      lanes hold one key row, 16 bytes of K and V per lane per row); online
//                      softmax per query; the chunk's (max, sum, unnormalised output) go to
//                      the workspace.
//   4. decode_combine: merge the chunks of every (b, h, j), then the R contraction
//                      out[b][h][c] = sum_{h',j} R[h][h'P + j] Pbar[b][h'][j][c].
// All four are HBM-bound: W (3 D^2 bf16) and the cached rows of K and V are the bytes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "iha_internal.h"
#include "ptx.cuh"

namespace iha {

constexpr int DC_KS = 8;          // K splits of the projection GEMV
constexpr int DC_BMAX = 8;        // batch rows per pass of the GEMV
constexpr int DC_NCH_MAX = 64;    // KV chunks per (b, h)
constexpr int DC_ATT_THREADS = 128;

// ---------------------------------------------------------------------------------------
// 1. projection GEMV: Yp[ks][b][s][n] = sum_{k in split ks} x[b][k] W_s[k][n]
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
decode_proj(const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *__restrict__ WQ,
            const __nv_bfloat16 *__restrict__ WK, const __nv_bfloat16 *__restrict__ WV, int B, int D,
            float *__restrict__ Yp) {
    extern __shared__ float dsm[];
    const int nblk = (D + 255) / 256;
    const int s = blockIdx.x / nblk, n0 = (blockIdx.x % nblk) * 256;
    const int ks = blockIdx.y, krows = D / DC_KS, k0 = ks * krows;
    const __nv_bfloat16 *W = s == 0 ? WQ : (s == 1 ? WK : WV);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = n0 + lane * 8;                      // this lane's 8 columns
    float *xs = dsm;                                  // [DC_BMAX][krows]
    float *red = dsm + DC_BMAX * krows;               // [8 warps][DC_BMAX][256]
    for (int b0 = 0; b0 < B; b0 += DC_BMAX) {
        const int nb = min(DC_BMAX, B - b0);
        __syncthreads();
        for (int i = threadIdx.x; i < nb * krows; i += blockDim.x)
            xs[i] = __bfloat162float(x[(size_t)(b0 + i / krows) * D + k0 + i % krows]);
        __syncthreads();
        float acc[DC_BMAX][8];
#pragma unroll
        for (int b = 0; b < DC_BMAX; ++b)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[b][e] = 0.f;
        if (n < D) {
            for (int k = warp; k < krows; k += 8) {
                const uint4 wv = *reinterpret_cast<const uint4 *>(W + (size_t)(k0 + k) * D + n);
                const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
                float wf[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    wf[2 * e] = __uint_as_float(w4[e] << 16);
                    wf[2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
                }
#pragma unroll
                for (int b = 0; b < DC_BMAX; ++b) {
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
        for (int b = 0; b < DC_BMAX; ++b)
#pragma unroll
            for (int e = 0; e < 8; ++e) red[(warp * DC_BMAX + b) * 256 + lane * 8 + e] = acc[b][e];
        __syncthreads();
        for (int i = threadIdx.x; i < nb * 256; i += blockDim.x) {
            const int b = i / 256, c = i % 256;
            if (n0 + c >= D) continue;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) v += red[(w * DC_BMAX + b) * 256 + c];
            Yp[(((size_t)ks * B + b0 + b) * 3 + s) * D + n0 + c] = v;
        }
    }
}

// ---------------------------------------------------------------------------------------
// 2. mixing + cache append, one CTA per (b, s, h), one thread per column c
// ---------------------------------------------------------------------------------------
__global__ void decode_mix(const float *__restrict__ Yp, const float *__restrict__ aQ, const float *__restrict__ aK,
                           const float *__restrict__ aV, int B, int H, int d, int P, long long t, long long cache_rows,
                           __nv_bfloat16 *__restrict__ qt, __nv_bfloat16 *__restrict__ Kc, __half *__restrict__ Vc) {
    const int b = blockIdx.x, s = blockIdx.y, h = blockIdx.z, c = threadIdx.x;
    const int D = H * d;
    const float *al = s == 0 ? aQ : (s == 1 ? aK : aV);
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    for (int m = 0; m < H; ++m) {
        float y = 0.f;
#pragma unroll
        for (int ks = 0; ks < DC_KS; ++ks) y += Yp[(((size_t)ks * B + b) * 3 + s) * D + m * d + c];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (j < P) acc[j] = fmaf(al[((size_t)m * H + h) * P + j], y, acc[j]);   // alpha_s[m][h][j]
    }
    for (int j = 0; j < P; ++j) {
        if (s == 0) {
            qt[(((size_t)b * H + h) * P + j) * d + c] = __float2bfloat16_rn(acc[j]);
        } else {
            const size_t row = ((size_t)b * H + h) * cache_rows + (size_t)t * P + j;   // stacked row t*P + j
            if (s == 1)
                Kc[row * d + c] = __float2bfloat16_rn(acc[j]);
            else
                Vc[row * d + c] = __float2half_rn(acc[j]);
        }
    }
}

// ---------------------------------------------------------------------------------------
// 3. split-KV attention of the P pseudo-queries of token t
// ---------------------------------------------------------------------------------------
template <int DPL, int PMAX>   // DPL = d / 8 dims per lane; PMAX = largest P
__global__ void __launch_bounds__(DC_ATT_THREADS)
decode_attn(const __nv_bfloat16 *__restrict__ qt, const __nv_bfloat16 *__restrict__ Kc, const __half *__restrict__ Vc,
            int H, int P, long long cache_rows, long long lo, long long hi, int rows_per_chunk, float scale_log2,
            float *__restrict__ part_ml, float *__restrict__ part_o) {
    constexpr int d = DPL * 8;
    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z, nch = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane >> 3, gl = lane & 7;          // 4 groups of 8 lanes per warp
    const long long bh = (long long)b * H + h;
    const long long r_begin = lo + (long long)chunk * rows_per_chunk;
    const long long r_end = min(hi + 1, r_begin + rows_per_chunk);
    // this lane's DPL dims of every pseudo-query
    float q[PMAX][DPL];
#pragma unroll
    for (int j = 0; j < PMAX; ++j)
#pragma unroll
        for (int e = 0; e < DPL; ++e)
            q[j][e] = j < P ? __bfloat162float(qt[((bh * P) + j) * d + gl * DPL + e]) * scale_log2 : 0.f;
    float m[PMAX], l[PMAX], o[PMAX][DPL];
#pragma unroll
    for (int j = 0; j < PMAX; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[j][e] = 0.f;
    }
    // rows r_begin + 4*warp + grp, stepping by 16 (4 warps x 4 groups).  The loop runs the
    // same number of times on every lane of the warp (its shuffles name all 32 lanes); a
    // group whose row is past the chunk loads nothing and skips the update.
    for (long long base = r_begin + warp * 4; base < r_end; base += 16) {
        const long long r = base + grp;
        const bool valid = r < r_end;
        float kf[DPL], vf[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) kf[e] = vf[e] = 0.f;
        if (valid) {
            const __nv_bfloat16 *kr = Kc + (bh * cache_rows + r) * d + gl * DPL;
            const __half *vr = Vc + (bh * cache_rows + r) * d + gl * DPL;
#pragma unroll
            for (int e8 = 0; e8 < DPL; e8 += 8) {
                const uint4 ku = *reinterpret_cast<const uint4 *>(kr + e8);
                const uint4 vu = *reinterpret_cast<const uint4 *>(vr + e8);
                const uint32_t k4[4] = {ku.x, ku.y, ku.z, ku.w}, v4[4] = {vu.x, vu.y, vu.z, vu.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    kf[e8 + 2 * e] = __uint_as_float(k4[e] << 16);
                    kf[e8 + 2 * e + 1] = __uint_as_float(k4[e] & 0xffff0000u);
                    const __half2 vh = *reinterpret_cast<const __half2 *>(&v4[e]);
                    const float2 vv = __half22float2(vh);
                    vf[e8 + 2 * e] = vv.x;
                    vf[e8 + 2 * e + 1] = vv.y;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < PMAX; ++j) {
            if (j >= P) break;   // P is the same on every lane
            float sc = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) sc = fmaf(q[j][e], kf[e], sc);
            sc += __shfl_xor_sync(0xffffffffu, sc, 4);
            sc += __shfl_xor_sync(0xffffffffu, sc, 2);
            sc += __shfl_xor_sync(0xffffffffu, sc, 1);   // the group's score in log2 units
            if (valid) {                                 // uniform over the group
                if (sc > m[j]) {
                    const float corr = exp2f(m[j] - sc);     // m = -inf -> 0
                    l[j] *= corr;
#pragma unroll
                    for (int e = 0; e < DPL; ++e) o[j][e] *= corr;
                    m[j] = sc;
                }
                const float pr = exp2f(sc - m[j]);
                l[j] += pr;
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[j][e] = fmaf(pr, vf[e], o[j][e]);
            }
        }
    }
    // merge the 4 groups of the warp (lanes gl, gl+8, gl+16, gl+24 hold the same dims)
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
        for (int j = 0; j < PMAX; ++j) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m[j], off);
            const float l2 = __shfl_xor_sync(0xffffffffu, l[j], off);
            const float mn = fmaxf(m[j], m2);
            const float c1 = m[j] == -INFINITY ? 0.f : exp2f(m[j] - mn);
            const float c2 = m2 == -INFINITY ? 0.f : exp2f(m2 - mn);
            l[j] = l[j] * c1 + l2 * c2;
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
                const float o2 = __shfl_xor_sync(0xffffffffu, o[j][e], off);
                o[j][e] = o[j][e] * c1 + o2 * c2;
            }
            m[j] = mn;
        }
    }
    // merge the 4 warps through shared memory: [warp][j] (m, l) and [warp][j][d] o
    __shared__ float sm_ml[4][PMAX][2];
    __shared__ float sm_o[4][PMAX][d];
    if (grp == 0) {
#pragma unroll
        for (int j = 0; j < PMAX; ++j) {
            if (gl == 0) {
                sm_ml[warp][j][0] = m[j];
                sm_ml[warp][j][1] = l[j];
            }
#pragma unroll
            for (int e = 0; e < DPL; ++e) sm_o[warp][j][gl * DPL + e] = o[j][e];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < P * d; i += blockDim.x) {
        const int j = i / d, c = i % d;
        float mn = -INFINITY;
        for (int w = 0; w < 4; ++w) mn = fmaxf(mn, sm_ml[w][j][0]);
        float lt = 0.f, ot = 0.f;
        for (int w = 0; w < 4; ++w) {
            const float mw = sm_ml[w][j][0];
            const float cw = mw == -INFINITY ? 0.f : exp2f(mw - mn);
            lt += sm_ml[w][j][1] * cw;
            ot += sm_o[w][j][c] * cw;
        }
        const size_t pidx = ((size_t)bh * nch + chunk) * P + j;
        part_o[pidx * d + c] = ot;
        if (c == 0) {
            part_ml[pidx * 2] = mn;
            part_ml[pidx * 2 + 1] = lt;
        }
    }
}

// ---------------------------------------------------------------------------------------
// 4. merge the chunks, normalise, R contraction; one CTA per b
// ---------------------------------------------------------------------------------------
__global__ void decode_combine(const float *__restrict__ part_ml, const float *__restrict__ part_o,
                               const float *__restrict__ R, int H, int d, int P, int nch, __nv_bfloat16 *__restrict__ out) {
    extern __shared__ float pb[];   // Pbar[b] as [H*P][d], fp32
    const int b = blockIdx.x, HP = H * P;
    for (int i = threadIdx.x; i < HP * d; i += blockDim.x) {
        const int k = i / d, c = i % d;             // k = h'*P + j
        const size_t base = ((size_t)b * H + k / P) * nch;
        const int j = k % P;
        float mn = -INFINITY;
        for (int ch = 0; ch < nch; ++ch) mn = fmaxf(mn, part_ml[((base + ch) * P + j) * 2]);
        float lt = 0.f, ot = 0.f;
        for (int ch = 0; ch < nch; ++ch) {
            const size_t pidx = (base + ch) * P + j;
            const float mc = part_ml[pidx * 2];
            const float cw = mc == -INFINITY ? 0.f : exp2f(mc - mn);
            lt += part_ml[pidx * 2 + 1] * cw;
            ot += part_o[pidx * d + c] * cw;
        }
        pb[i] = lt > 0.f ? ot / lt : 0.f;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < H * d; i += blockDim.x) {
        const int h = i / d, c = i % d;
        float v = 0.f;
        for (int k = 0; k < HP; ++k) v = fmaf(R[(size_t)h * HP + k], pb[k * d + c], v);
        out[(size_t)b * H * d + i] = __float2bfloat16_rn(v);
    }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
bool decode_supported(int H, int d, int P) {
    return (d == 64 && P <= 8) || (d == 128 && P <= 4);
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
                          cudaStream_t st) {
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
    const size_t smem1 = (size_t)DC_BMAX * krows * 4 + (size_t)8 * DC_BMAX * 256 * 4;
    cudaError_t e = cudaFuncSetAttribute(decode_proj, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    if (e != cudaSuccess) return e;
    decode_proj<<<dim3(3 * ((D + 255) / 256), DC_KS), 256, smem1, st>>>(
        (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)WQ, (const __nv_bfloat16 *)WK, (const __nv_bfloat16 *)WV, B,
        D, Yp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 2. mixing + append
    decode_mix<<<dim3(B, 3, H), d, 0, st>>>(Yp, aQ, aK, aV, B, H, d, P, t, cache_rows, qt, (__nv_bfloat16 *)Kc,
                                            (__half *)Vc);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 3. attention over the readable cached rows [lo, hi]
    const long long hi = (t + 1) * P - 1;
    long long lo = 0;
    if (mask_mode == 2) lo = (t - window + 1) * P > 0 ? (t - window + 1) * P : 0;
    const long long rows = hi - lo + 1;
    long long nch = (3LL * device_sm_count() + (long long)B * H - 1) / ((long long)B * H);
    if (nch > (rows + 63) / 64) nch = (rows + 63) / 64;
    if (nch > DC_NCH_MAX) nch = DC_NCH_MAX;
    if (nch < 1) nch = 1;
    const int rpc = (int)((rows + nch - 1) / nch);
    nch = (rows + rpc - 1) / rpc;
    const float sl2 = 1.4426950408889634f / sqrtf((float)d);
    const dim3 g3((unsigned)nch, H, B);
    if (d == 128)
        decode_attn<16, 4><<<g3, DC_ATT_THREADS, 0, st>>>(qt, (const __nv_bfloat16 *)Kc, (const __half *)Vc, H, P,
                                                          cache_rows, lo, hi, rpc, sl2, part_ml, part_o);
    else
        decode_attn<8, 8><<<g3, DC_ATT_THREADS, 0, st>>>(qt, (const __nv_bfloat16 *)Kc, (const __half *)Vc, H, P,
                                                         cache_rows, lo, hi, rpc, sl2, part_ml, part_o);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 4. combine + contraction
    const size_t smem4 = (size_t)H * P * d * 4;
    e = cudaFuncSetAttribute(decode_combine, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem4);
    if (e != cudaSuccess) return e;
    decode_combine<<<B, 256, smem4, st>>>(part_ml, part_o, R, H, d, P, (int)nch, (__nv_bfloat16 *)out);
    return cudaGetLastError();
}

}  // namespace iha
