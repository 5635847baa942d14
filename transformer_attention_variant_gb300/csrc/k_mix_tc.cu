// k_mix_tc.cu -- pseudo-head mixing ("Interleaved Head Attention" section 4, Algorithm 1,
// step "偽頭混合") on the unfolded route, as the small dense contraction it is:
//
//     S~_s[t][(h,j)][c] = sum_m alpha_s[m][h][j] * Y_s[t][m][c],   s in {Q, K, V},
//
// i.e. for each projection s and token t the product alpha_s^T (H*P x H) * Y_s[t] (H x d).
// The result is written straight into the stacked layout QKV[s][b][h][t*P + j][c] (Qbar,
// Kbar bf16; Vbar f16).
//
// Design (sm_103a): persistent CTAs, one per SM.  H*P is often far below the 128 rows of a
// tcgen05 accumulator, so G = min(4, 128 / (H*P)) token groups are stacked along M with a
// block-diagonal A:  rows g*H*P + rho (rho = j*H + h) hold group g's pseudo-heads, and
// k-step g (16 columns, heads m < H) carries alpha_s^T only in group g's rows.  One tile is
// (s, G groups of 128/d tokens): the warp-0 producer TMA-loads each group's Y rows as
// [16 m][64 c] boxes (128B swizzle, an MN-major B operand; m >= H reads as zero) into a
// 4-stage ring; warp 1 issues G tcgen05.mma (M=128, N=128, K=16), one per group, into one
// of four TMEM accumulators; eight epilogue warps drain it (two per lane quarter, 64
// columns each).  The epilogue writes the converted tile into a ring of 2-4 shared staging
// buffers laid out as the output ([h][token][j][c], one 16-byte pad per head: lanes hold
// consecutive h, so their stores hit different banks), then one lane per head sends the
// head's contiguous run to global memory with a bulk copy.  Direct scattered 16-byte
// stores from registers (one line per lane) ran at a quarter of the copy rate, and with
// one group per tile most accumulator lanes were idle.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "iha_internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace iha {

constexpr int MX_M = 128, MX_N = 128, MX_K = 16, MX_GMAX = 4, MX_STAGES = 4, MX_NACC = 4;
constexpr int MX_EPI_WARPS = 8, MX_THREADS = 64 + 32 * MX_EPI_WARPS;   // producer, MMA, 8 epilogue warps
constexpr int MX_A_BYTES = MX_M * 128;             // one SW128 K-major tile, K = 16 per group
constexpr int MX_GROUP_BYTES = MX_N * MX_K * 2;    // one group's B: [16 m][128 n], 64-column chunks
constexpr int MX_B_BYTES = MX_GMAX * MX_GROUP_BYTES;
constexpr int MX_EPI_BAR = 1;                      // named barrier of the epilogue warps

__host__ __device__ constexpr int mix_groups(int HP) { return MX_M / HP < MX_GMAX ? MX_M / HP : MX_GMAX; }
// Staging bytes of one head for one tile: G*128/d tokens x P rows x d values, plus the
// 16-byte bank pad.
__host__ __device__ constexpr int mix_head_stride(int G, int P) { return G * MX_N * P * 2 + 16; }
constexpr int MX_SMEM_FIXED = 3 * MX_A_BYTES + MX_STAGES * MX_B_BYTES + 256 + 1024;
constexpr int MX_SMEM_MAX = 232448;                 // the opt-in maximum per block
// As many staging buffers (2..4) as fit: more of them keep more bulk copies in flight.
inline int mix_staging_buffers(int stg_bytes) {
    int n = (MX_SMEM_MAX - MX_SMEM_FIXED) / stg_bytes;
    return n > 4 ? 4 : n;
}

struct MixParams {
    __nv_bfloat16 *qkv;
    long long s_stride;   // elements of one of Qbar/Kbar/Vbar
    long long ntok;       // B*N
    int N_tok, H, P, d;
    int G;                // token groups per tile
    int tpg;              // tokens per group (MX_N / d)
    int tpt;              // tokens per tile (G * tpg)
    int stg_bytes;        // one staging buffer: H * mix_head_stride(G, P)
    int nstg;             // staging buffers (2..4)
    int nsets;            // mixed projections: 3 (Q, K, V) or 1
    int f16_set;          // the set written as f16 (-1: none)
    long long num_tiles;  // nsets * ceil(ntok / tpt)
    int *status;
};

__global__ void __launch_bounds__(MX_THREADS, 1)
mix_tc(const __grid_constant__ CUtensorMap tmY, const float *__restrict__ aQ, const float *__restrict__ aK,
       const float *__restrict__ aV, const MixParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;                          // [3][MX_A_BYTES]
    uint8_t *sB = smem + 3 * MX_A_BYTES;         // [MX_STAGES][MX_B_BYTES]
    uint8_t *sStg = sB + MX_STAGES * MX_B_BYTES;  // [nstg][H][mix_head_stride(G, P)]
    uint64_t *full = reinterpret_cast<uint64_t *>(sStg + p.nstg * p.stg_bytes);
    uint64_t *empty = full + MX_STAGES;
    uint64_t *tfull = empty + MX_STAGES;
    uint64_t *tempty = tfull + MX_NACC;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + MX_NACC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = warp_id(), lane = lane_id();
    const int H = p.H, HP = p.H * p.P, G = p.G;

    // alpha_Q, alpha_K, alpha_V (3 x H x H*P floats, at most 24 KB) into shared memory,
    // parked in the B ring before the producer starts: all of a thread's loads in flight
    // at once.
    float *sAl = reinterpret_cast<float *>(sB);
    {
        constexpr int kPer = (3 * MX_K * MX_M + MX_THREADS - 1) / MX_THREADS;
        const int n1 = H * HP, n = 3 * n1;
        float v[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int idx = threadIdx.x + k * MX_THREADS;
            v[k] = 0.f;
            if (idx < n) v[k] = idx < n1 ? aQ[idx] : (idx < 2 * n1 ? aK[idx - n1] : aV[idx - 2 * n1]);
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int idx = threadIdx.x + k * MX_THREADS;
            if (idx < n) sAl[idx] = v[k];
        }
    }
    __syncthreads();
    // A_s: a 128-row, 128-byte-row K-major tile with the 128B swizzle: 16-byte chunk cp of
    // row r holds columns k = 8*((cp ^ r) % 8) + e.  Row r = g*H*P + j*H + h, column
    // k = g'*16 + m holds alpha_s[m][h][j] when g' == g and m < H, else zero.
    for (int idx = threadIdx.x; idx < 3 * MX_M * 8; idx += blockDim.x) {
        const int s = idx / (MX_M * 8), r = (idx / 8) % MX_M, cp = idx % 8;
        const int kc = cp ^ (r % 8), gk = kc / 2, m0 = (kc % 2) * 8;
        const int g = r / HP, rho = r % HP, jj = rho / H, hh = rho % H;
        const float *al = sAl + s * H * HP;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const int m = m0 + e;
            const bool on = g < G && gk == g;
            const float x0 = on && m < H ? al[m * HP + hh * p.P + jj] : 0.f;   // alpha_s[m][h][j]
            const float x1 = on && m + 1 < H ? al[(m + 1) * HP + hh * p.P + jj] : 0.f;
            w[e / 2] = pack_bf16x2(x0, x1);
        }
        *reinterpret_cast<uint4 *>(sA + s * MX_A_BYTES + (r / 8) * 1024 + (r % 8) * 128 + cp * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();   // the B ring is the TMA's from here on
    fence_proxy_async_smem();   // generic-proxy writes of A before the tensor core reads them
    if (threadIdx.x == 0) {
        for (int i = 0; i < MX_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int a = 0; a < MX_NACC; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 32 * MX_EPI_WARPS);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&tmY);
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int halves = p.d / 64;   // 64-column boxes per token

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (long long tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
                const long long tb = tile / p.nsets;
                const int s = (int)(tile % p.nsets);
                if (!mbar_wait_lazy(&empty[stage], phase ^ 1, p.status, kSiteMixProducer, abort_flag)) break;
                mbar_arrive_expect_tx(&full[stage], G * MX_GROUP_BYTES);
                // group g, token i, c half hf -> 64-column chunk i*halves + hf of group g's B
                // (tokens past the end read as zero)
                for (int g = 0; g < G; ++g)
                    for (int i = 0; i < p.tpg; ++i)
                        for (int hf = 0; hf < halves; ++hf)
                            tma_load_3d(&tmY, &full[stage],
                                        sB + stage * MX_B_BYTES + g * MX_GROUP_BYTES + (i * halves + hf) * (16 * 128),
                                        hf * 64, 0, (int)((tb * p.tpt + g * p.tpg + i) * p.nsets + s));
                if (++stage == MX_STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(MX_M, MX_N, 0, 1);   // A K-major, B MN-major
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            for (long long tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
                const int s = (int)(tile % p.nsets);
                const int acc = it % MX_NACC;
                if (!mbar_wait(&tempty[acc], ((it / MX_NACC) & 1) ^ 1, p.status, kSiteMixMma, abort_flag)) break;
                if (!mbar_wait(&full[stage], phase, p.status, kSiteMixMma, abort_flag)) break;
                tc_fence_after();
                // k-step g: A columns 16g.. (32 bytes into the swizzled rows), group g's B
                // (64-column chunks 2 KB apart as the leading byte offset, 8 k-rows 1 KB apart)
                for (int g = 0; g < G; ++g)
                    mma_ss(tmem + acc * MX_N, sdesc_sw128(smem_u32(sA + s * MX_A_BYTES) + g * 32, 16, 1024),
                           sdesc_sw128(smem_u32(sB + stage * MX_B_BYTES + g * MX_GROUP_BYTES), 16 * 128, 1024),
                           idesc, g > 0 ? 1u : 0u);
                mma_commit(&empty[stage]);
                mma_commit(&tfull[acc]);
                if (++stage == MX_STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else {
        // epilogue: warps 2..9; lane quarter q = warp % 4, column half colh = (warp - 2) / 4
        const int q = warp & 3, colh = (warp - 2) / 4;
        const int r = q * 32 + lane;                 // the accumulator row this thread drains
        const int g = r / HP, rho = r % HP, j = rho / H, h = rho % H;
        const bool row_ok = g < G;
        const int hstride = mix_head_stride(G, p.P);
        const long long Pd = (long long)p.P * p.d;
        const bool issuer = warp == 2 && lane < H;   // sends head `lane`'s run of each tile
        int it = 0, sb = 0;
        for (long long tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
            const long long tb = tile / p.nsets;
            const int s = (int)(tile % p.nsets);
            const int acc = it % MX_NACC;
            uint8_t *stg = sStg + sb * p.stg_bytes;
            if (++sb == p.nstg) sb = 0;
            const bool ok = mbar_wait(&tfull[acc], (it / MX_NACC) & 1, p.status, kSiteMixEpilogue, abort_flag);
            if (ok) {
                tc_fence_after();
                uint32_t u[2][32];
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    tmem_ld32(tmem + acc * MX_N + colh * 64 + c * 32 + (uint32_t(q * 32) << 16), u[c]);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(&tempty[acc]);   // the accumulator is in registers: the MMA may reuse it
                // The bulk copies that last read this buffer (tile it-nstg) were waited for
                // before the barrier of tile it-1.
                if (row_ok) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int col = colh * 64 + c * 32;
                        const int ti = g * p.tpg + col / p.d, cc = col % p.d;   // token within the tile
                        uint4 v[4];
                        uint32_t *vw = reinterpret_cast<uint32_t *>(v);
                        if (s == p.f16_set) {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                vw[i] = pack_f16x2(__uint_as_float(u[c][2 * i]), __uint_as_float(u[c][2 * i + 1]));
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                vw[i] = pack_bf16x2(__uint_as_float(u[c][2 * i]), __uint_as_float(u[c][2 * i + 1]));
                        }
                        uint4 *d4 = reinterpret_cast<uint4 *>(stg + h * hstride + ((ti * p.P + j) * p.d + cc) * 2);
#pragma unroll
                        for (int i = 0; i < 4; ++i) d4[i] = v[i];
                    }
                }
                fence_proxy_async_smem();   // staging writes -> the bulk copy's reads
            }
            // Before the barrier the issuers make sure the buffer of the next tile is free
            // again (its copies, tile it+1-nstg, are all but the newest nstg-2 groups), so
            // that after it every thread may fill it.
            if (issuer) bulk_wait_read(p.nstg - 2);
            if (named_bar_or(MX_EPI_BAR, 32 * MX_EPI_WARPS, !ok)) break;   // a uniform decision
            if (issuer) {
                const long long t0 = tb * p.tpt;
                int ti = 0;
                while (ti < p.tpt && t0 + ti < p.ntok) {
                    const long long t = t0 + ti, b = t / p.N_tok, tt = t - b * p.N_tok;
                    // tokens of the same batch entry are contiguous in the stacked layout
                    long long n = p.tpt - ti;
                    if (n > p.N_tok - tt) n = p.N_tok - tt;
                    if (n > p.ntok - t) n = p.ntok - t;
                    // stacked row tt*P of head `lane`: ((b*H + h)*N + tt)*P*d
                    bulk_store(p.qkv + s * p.s_stride + ((b * H + lane) * p.N_tok + tt) * Pd,
                               stg + lane * hstride + (long long)ti * Pd * 2, (uint32_t)(n * Pd * 2));
                    ti += (int)n;
                }
                bulk_commit();
            }
        }
        if (issuer) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

cudaError_t launch_mix_sets(const void *Y, const float *aQ, const float *aK, const float *aV, const Shape &sh,
                            int nsets, void *QKV, cudaStream_t st, int *status, int y_sets, int f16_set) {
    if (y_sets < 0) y_sets = nsets;
    if (nsets != y_sets && nsets != 1) return cudaErrorInvalidValue;
    if ((sh.d != 64 && sh.d != 128) || sh.H > MX_K || sh.H * sh.P > MX_M) return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(QKV) & 15) != 0) return cudaErrorInvalidValue;   // bulk-copy alignment
    const long long ntok = (long long)sh.B * sh.N;
    CUtensorMap tmY;
    {
        // Y [t][s][m][c] viewed as (c, m, t*nsets + s); boxes of [16 m][64 c].  One set out
        // of y_sets: the row stride skips the other sets.
        const uint64_t dims[3] = {(uint64_t)sh.d, (uint64_t)sh.H, (uint64_t)(ntok * nsets)};
        const uint64_t strides[2] = {(uint64_t)sh.d * 2, (uint64_t)(nsets == y_sets ? 1 : y_sets) * sh.H * sh.d * 2};
        const uint32_t box[3] = {64, (uint32_t)MX_K, 1};
        if (!make_tmap_bf16(&tmY, Y, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    MixParams p{};
    p.qkv = (__nv_bfloat16 *)QKV;
    p.s_stride = sh.qkv_elems();
    p.ntok = ntok;
    p.N_tok = sh.N;
    p.H = sh.H;
    p.P = sh.P;
    p.d = sh.d;
    p.G = mix_groups(sh.H * sh.P);
    p.tpg = MX_N / sh.d;
    p.tpt = p.G * p.tpg;
    p.stg_bytes = sh.H * mix_head_stride(p.G, sh.P);
    p.nstg = mix_staging_buffers(p.stg_bytes);
    if (p.nstg < 2) return cudaErrorInvalidValue;
    p.nsets = nsets;
    p.f16_set = f16_set;
    p.num_tiles = nsets * ((ntok + p.tpt - 1) / p.tpt);
    p.status = status;
    const int smem = MX_SMEM_FIXED + p.nstg * p.stg_bytes;
    cudaError_t e = cudaFuncSetAttribute(mix_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long grid = p.num_tiles < device_sm_count() ? p.num_tiles : device_sm_count();
    mix_tc<<<(unsigned)grid, MX_THREADS, smem, st>>>(tmY, aQ, aK, aV, p);
    return cudaGetLastError();
}

}  // namespace iha

namespace iha {
cudaError_t launch_mix(const void *Y, const float *aQ, const float *aK, const float *aV, const Shape &sh, void *QKV,
                       cudaStream_t st, int *status) {
    return launch_mix_sets(Y, aQ, aK, aV, sh, 3, QKV, st, status);
}
}  // namespace iha
