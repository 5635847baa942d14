// k_rowmix.cu -- a per-token "row mixing" kernel, out[t][r][:] = sum_k coef[k][r] in[t][k][:],
// used for the unstack + contraction step of Algorithm 1 ("Interleaved Head Attention"
// section 4, "反堆疊與收縮"): in = Pbar[t][h'*P + j][:] (k = h'P + j, H*P rows),
// coef[k][h] = R[h][k], out = O[t][h][:] (heads concatenated).  (The kernel also supports a
// mixing mode that writes the stacked pseudo-head layout.)
//
// An HBM-bound stream with little arithmetic per byte.  Design: persistent CTAs
// (two per SM); a tile is a few whole tokens whose input rows (contiguous d-element rows)
// arrive by cp.async.bulk into a 3-stage shared-memory ring, so the next tiles' bytes are
// in flight while the current one is computed.  A thread computes a register tile of R
// output rows x 4 consecutive columns: per input row one 8-byte shared load of 4 bf16 and
// broadcast float4 loads of the coefficients feed 2R packed f32x2 FMAs.  The 32 threads of
// a warp cover 128 consecutive columns of one output row, so stores are coalesced.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "iha_internal.h"
#include "ptx.cuh"

namespace iha {

constexpr int RM_THREADS = 256, RM_STAGES = 3, RM_C = 4, RM_STAGE_TARGET = 32768;

struct RowMixParams {
    const __nv_bfloat16 *in;
    __nv_bfloat16 *out;
    long long ntok;           // B*N
    int N_tok, H, P, d;
    int K, NR, NRr;           // input rows, output rows (padded to R) per token
    int tok;                  // tokens per tile
    long long in_tok_stride;  // elements between consecutive tokens' input blocks
    long long s_stride;       // mixing: elements of one of Qbar/Kbar/Vbar
    int nsets;                // mixing: 3 coefficient sets (Q, K, V); contraction: 1
    long long num_tiles;
    int *status;
};

__device__ __forceinline__ void bf16x4_to_f32(uint2 u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xffff0000u);
}

template <bool MIX, int R>
__global__ void __launch_bounds__(RM_THREADS)
rowmix_kernel(const float *__restrict__ c0, const float *__restrict__ c1, const float *__restrict__ c2,
              const RowMixParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int K = p.K, NRr = p.NRr, d = p.d;
    float *coef = reinterpret_cast<float *>(smem);                              // [nsets][K][NRr]
    const size_t coef_bytes = ((size_t)p.nsets * K * NRr * 4 + 127) & ~size_t(127);
    const size_t tok_bytes = (size_t)K * d * 2, stage_bytes = (size_t)p.tok * tok_bytes;
    uint8_t *stages = smem + coef_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(stages + RM_STAGES * stage_bytes);
    __shared__ int abort_flag;

    // coefficients: mixing -> alpha_s[m][h*P + j] as stored; contraction -> coef[k][h] = R[h][k]
    for (int set = 0; set < p.nsets; ++set) {
        const float *src = set == 0 ? c0 : (set == 1 ? c1 : c2);
        for (int idx = threadIdx.x; idx < K * NRr; idx += blockDim.x) {
            const int k = idx / NRr, r = idx % NRr;
            float v = 0.f;
            if (r < p.NR) v = MIX ? src[(size_t)k * p.NR + r] : src[(size_t)r * K + k];
            coef[((size_t)set * K + k) * NRr + r] = v;
        }
    }
    if (threadIdx.x == 0) {
        for (int st = 0; st < RM_STAGES; ++st) mbar_init(&full[st], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const long long ntb = (p.ntok + p.tok - 1) / p.tok;   // token blocks
    auto issue = [&](long long tile, int st) {
        const long long tb = MIX ? tile / 3 : tile;
        const int s = MIX ? (int)(tile % 3) : 0;
        const long long t0 = tb * p.tok;
        const int nt = (int)min((long long)p.tok, p.ntok - t0);
        mbar_arrive_expect_tx(&full[st], (uint32_t)(nt * tok_bytes));
        uint8_t *dst = stages + st * stage_bytes;
        if (MIX) {   // Y rows of consecutive tokens are 3*H*d apart: one copy per token
            for (int i = 0; i < nt; ++i)
                bulk_load(dst + i * tok_bytes, p.in + (t0 + i) * p.in_tok_stride + (long long)s * K * d,
                          (uint32_t)tok_bytes, &full[st]);
        } else {     // Pbar blocks of consecutive tokens are contiguous: one copy
            bulk_load(dst, p.in + t0 * p.in_tok_stride, (uint32_t)(nt * tok_bytes), &full[st]);
        }
    };
    (void)ntb;
    if (threadIdx.x == 0)
        for (int i = 0; i < RM_STAGES; ++i) {
            const long long tile = blockIdx.x + (long long)i * gridDim.x;
            if (tile < p.num_tiles) issue(tile, i);
        }

    const int cgs = d / RM_C, rbs = NRr / R;
    const int units = p.tok * rbs * cgs;
    const long long Pd = (long long)p.P * d;
    int it = 0;
    for (long long tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
        const int st = it % RM_STAGES;
        if (!mbar_wait(&full[st], (it / RM_STAGES) & 1, p.status, kSiteRowMix, &abort_flag)) break;
        const long long tb = MIX ? tile / 3 : tile;
        const int s = MIX ? (int)(tile % 3) : 0;
        const long long t0 = tb * p.tok;
        const int nt = (int)min((long long)p.tok, p.ntok - t0);
        const __nv_bfloat16 *in_s = reinterpret_cast<const __nv_bfloat16 *>(stages + st * stage_bytes);
        const float *cs = coef + (size_t)s * K * NRr;
        for (int u = threadIdx.x; u < units; u += blockDim.x) {
            const int cg = u % cgs, rest = u / cgs, rb = rest % rbs, ti = rest / rbs;
            if (ti >= nt) continue;
            uint64_t acc2[R / 2][RM_C];
#pragma unroll
            for (int rp = 0; rp < R / 2; ++rp)
#pragma unroll
                for (int c = 0; c < RM_C; ++c) acc2[rp][c] = 0ull;
            const __nv_bfloat16 *yrow = in_s + (size_t)ti * K * d + cg * RM_C;
            const float *crow = cs + rb * R;
#pragma unroll 4
            for (int k = 0; k < K; ++k) {
                float y[4];
                bf16x4_to_f32(*reinterpret_cast<const uint2 *>(yrow + (size_t)k * d), y);
                uint64_t ap[R / 2];
#pragma unroll
                for (int q = 0; q < R / 4; ++q) {
                    const ulonglong2 a = *reinterpret_cast<const ulonglong2 *>(crow + (size_t)k * NRr + 4 * q);
                    ap[2 * q] = a.x;
                    ap[2 * q + 1] = a.y;
                }
#pragma unroll
                for (int c = 0; c < RM_C; ++c) {
                    uint64_t yy;
                    asm("mov.b64 %0, {%1, %1};" : "=l"(yy) : "f"(y[c]));
#pragma unroll
                    for (int rp = 0; rp < R / 2; ++rp)
                        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[rp][c]) : "l"(ap[rp]), "l"(yy));
                }
            }
            const long long t = t0 + ti;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int row = rb * R + r;
                if (row >= p.NR) break;
                float v4[4];
#pragma unroll
                for (int c = 0; c < RM_C; ++c) {
                    float lo, hi;
                    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc2[r / 2][c]));
                    v4[c] = (r & 1) ? hi : lo;
                }
                uint2 v;
                __nv_bfloat16 *dst;
                if (MIX) {
                    const int h = row / p.P, j = row % p.P;
                    const long long b = t / p.N_tok, tt = t % p.N_tok;
                    // stacked row tt*P + j of head h: ((b*H + h)*N + tt)*P*d + j*d
                    dst = p.out + (long long)s * p.s_stride + ((b * p.H + h) * p.N_tok + tt) * Pd + (long long)j * d +
                          cg * RM_C;
                } else {
                    dst = p.out + (t * p.NR + row) * (long long)d + cg * RM_C;
                }
                if (MIX && s == 2) {   // Vbar in f16
                    __half2 h0 = __floats2half2_rn(v4[0], v4[1]), h1 = __floats2half2_rn(v4[2], v4[3]);
                    v.x = *reinterpret_cast<uint32_t *>(&h0);
                    v.y = *reinterpret_cast<uint32_t *>(&h1);
                } else {
                    __nv_bfloat162 b0 = __floats2bfloat162_rn(v4[0], v4[1]), b1 = __floats2bfloat162_rn(v4[2], v4[3]);
                    v.x = *reinterpret_cast<uint32_t *>(&b0);
                    v.y = *reinterpret_cast<uint32_t *>(&b1);
                }
                *reinterpret_cast<uint2 *>(dst) = v;
            }
        }
        __syncthreads();   // every thread is done with stage st
        if (threadIdx.x == 0) {
            const long long next = tile + (long long)RM_STAGES * gridDim.x;
            if (next < p.num_tiles) {
                fence_proxy_async_smem();
                issue(next, st);
            }
        }
    }
}

// Shared memory the row-mixing kernel needs for K input rows of d columns (0 if it fits in
// no CTA).
static size_t rowmix_smem(int K, int NR, int d, int nsets, int R) {
    const int NRr = (NR + R - 1) / R * R;
    const size_t tok_bytes = (size_t)K * d * 2;
    size_t tok = RM_STAGE_TARGET / tok_bytes;
    if (tok < 1) tok = 1;
    const size_t coef_bytes = ((size_t)nsets * K * NRr * 4 + 127) & ~size_t(127);
    const size_t smem = 128 + coef_bytes + RM_STAGES * tok * tok_bytes + RM_STAGES * 8;
    return smem <= 227 * 1024 ? smem : 0;
}

bool contract_rowmix_fits(const Shape &sh) { return rowmix_smem(sh.H * sh.P, sh.H, sh.d, 1, 4) != 0; }

template <bool MIX, int R>
static cudaError_t launch_rowmix(const float *c0, const float *c1, const float *c2, RowMixParams p, cudaStream_t st) {
    p.NRr = (p.NR + R - 1) / R * R;
    const size_t tok_bytes = (size_t)p.K * p.d * 2;
    p.tok = (int)(RM_STAGE_TARGET / tok_bytes);
    if (p.tok < 1) p.tok = 1;
    const long long ntb = (p.ntok + p.tok - 1) / p.tok;
    p.num_tiles = MIX ? ntb * 3 : ntb;
    const size_t smem = rowmix_smem(p.K, p.NR, p.d, p.nsets, R);
    if (smem == 0) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(rowmix_kernel<MIX, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long maxgrid = 2LL * device_sm_count();
    const unsigned grid = (unsigned)(p.num_tiles < maxgrid ? p.num_tiles : maxgrid);
    rowmix_kernel<MIX, R><<<grid, RM_THREADS, smem, st>>>(c0, c1, c2, p);
    return cudaGetLastError();
}

cudaError_t launch_contract_rowmix(const void *Pbar, const float *R, const Shape &sh, void *out, cudaStream_t st,
                                   int *status) {
    if (sh.d % 8 != 0) return cudaErrorInvalidValue;
    RowMixParams p{};
    p.in = (const __nv_bfloat16 *)Pbar;
    p.out = (__nv_bfloat16 *)out;
    p.ntok = (long long)sh.B * sh.N;
    p.N_tok = sh.N;
    p.H = sh.H;
    p.P = sh.P;
    p.d = sh.d;
    p.K = sh.H * sh.P;
    p.NR = sh.H;
    p.in_tok_stride = (long long)sh.H * sh.P * sh.d;
    p.nsets = 1;
    p.status = status;
    return launch_rowmix<false, 4>(R, R, R, p, st);
}

}  // namespace iha
