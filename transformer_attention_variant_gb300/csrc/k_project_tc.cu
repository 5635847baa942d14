// k_project_tc.cu -- projection + pseudo-head mixing + stacking as one tcgen05 GEMM.
//
// "Interleaved Head Attention" section 4, Algorithm 1, steps "偽頭混合" and "偽主堆疊":
// with the mixing folded into the weights (Wt = transposed sum_m alpha[m,h,j] W^(m)), every
// pseudo-query/key/value of every head is one column block of  C = X Wt^T  (M = B*N rows,
// K = D, N = 3*H*P*d columns).  The epilogue writes each column block straight into the
// stacked layout QKV[s][b][h][t*P + j][c], so no separate stacking pass exists.
//
// A second mode (PLAIN) is the same GEMM without the fold: Y = X [W_Q | W_K | W_V], the
// per-head projections X W_s^(m) of all heads, with the weights read as they are stored
// ([D][H*d], N contiguous: an MN-major B operand) and Y written row-major [B*N][3*H*d]; the
// pseudo-head mixing then runs as a separate pass (mix_kernel).  For P >= 2 this does 1/P of
// the folded GEMM's tensor work.
//
// Design (sm_103a): persistent CTAs, one per SM; warp 0 = TMA producer (128B-swizzled
// A and B tiles, 4-stage ring), warp 1 = MMA issuer (tcgen05.mma kind::f16, M=128 N=256
// K=16, fp32 accumulators in TMEM, double-buffered so the epilogue of one tile overlaps
// the main loop of the next), warps 2-5 = epilogue (tcgen05.ld -> bf16 -> global; the
// Vbar third is written as f16, the type the attention kernel's P V product uses; in the
// PLAIN mode each 64-column chunk is staged 128B-swizzled in shared memory and sent with one
// TMA tensor store -- stores straight from registers, one row per lane, cost 13-15% of the
// GEMM's time).
#include <cuda_bf16.h>

#include "iha_internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace iha {

constexpr int PG_M = 128, PG_N = 256, PG_K = 64, PG_STAGES = 4;
constexpr int PG_A_BYTES = PG_M * PG_K * 2;   // 16 KB
constexpr int PG_B_BYTES = PG_N * PG_K * 2;   // 32 KB
constexpr int PG_THREADS = 192;
constexpr int PG_SMEM = PG_STAGES * (PG_A_BYTES + PG_B_BYTES) + 256 + 1024;
constexpr int PG_STG_BYTES = PG_M * 128;   // one staged 64-column chunk of the plain epilogue
constexpr int PG_SMEM_PLAIN = PG_SMEM + 2 * PG_STG_BYTES;
static_assert(PG_SMEM_PLAIN <= 232448, "shared memory");

struct ProjParams {
    __nv_bfloat16 *qkv;   // folded mode: stacked output
    __nv_bfloat16 *y;     // plain mode: [M][3 * hd] output
    int hd;               // plain mode: H*d columns per projection
    int ntps;             // plain mode: N tiles per projection
    long long s_stride;   // elements of one of Qbar/Kbar/Vbar
    int M, Ncols, K;
    int N_tok, H, P, d;
    int num_m_tiles, num_tiles;
    int *status;
};

template <bool PLAIN>
__global__ void __launch_bounds__(PG_THREADS, 1)
proj_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
             const __grid_constant__ CUtensorMap tmY, const ProjParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + PG_STAGES * PG_A_BYTES;
    uint8_t *sStg = sB + PG_STAGES * PG_B_BYTES;   // plain epilogue: 2 staged chunks
    uint64_t *full = reinterpret_cast<uint64_t *>(sStg + (PLAIN ? 2 * PG_STG_BYTES : 0));
    uint64_t *empty = full + PG_STAGES;
    uint64_t *tfull = empty + PG_STAGES;
    uint64_t *tempty = tfull + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = warp_id(), lane = lane_id();
    if (threadIdx.x == 0) {
        for (int s = 0; s < PG_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (PLAIN) {
            tma_prefetch_desc(&tmB1);
            tma_prefetch_desc(&tmB2);
            tma_prefetch_desc(&tmY);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int nk = (p.K + PG_K - 1) / PG_K;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
                const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, p.status, kSiteProjProducer, abort_flag)) goto producer_done;
                    mbar_arrive_expect_tx(&full[stage], PG_A_BYTES + PG_B_BYTES);
                    tma_load_2d(&tmA, &full[stage], sA + stage * PG_A_BYTES, kb * PG_K, mt * PG_M);
                    if (PLAIN) {
                        // B tile = 4 chunks of [64 k][64 n] of W_s (n contiguous, MN-major), one
                        // rank-3 copy (four rank-2 copies per stage ran 8-12% slower)
                        const int s = nt / p.ntps, n0 = (nt % p.ntps) * PG_N;
                        const CUtensorMap *mb = s == 0 ? &tmB : (s == 1 ? &tmB1 : &tmB2);
                        tma_load_3d(mb, &full[stage], sB + stage * PG_B_BYTES, 0, kb * PG_K, n0 / 64);
                    } else {
                        tma_load_2d(&tmB, &full[stage], sB + stage * PG_B_BYTES, kb * PG_K, nt * PG_N);
                    }
                    if (++stage == PG_STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        producer_done:;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(PG_M, PG_N, 0, PLAIN ? 1 : 0);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1, p.status, kSiteProjMmaAcc, abort_flag)) break;
                tc_fence_after();
                const uint32_t dt = tmem_base + acc * PG_N;
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&full[stage], phase, p.status, kSiteProjMma, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * PG_A_BYTES);
                    const uint32_t b0 = smem_u32(sB + stage * PG_B_BYTES);
#pragma unroll
                    for (int k = 0; k < PG_K / 16; ++k) {
                        // K-major B: the next 16 k are 32 bytes along the row; MN-major B: 16 rows of
                        // 128 bytes further, 64-column chunks 8 KB apart (leading byte offset)
                        const uint64_t bdesc = PLAIN ? sdesc_sw128(b0 + k * 2048, 64 * PG_K * 2, 1024)
                                                     : sdesc_sw128(b0 + k * 32, 16, 1024);
                        mma_ss(dt, sdesc_sw128(a0 + k * 32, 16, 1024), bdesc, idesc, (kb | k) != 0);
                    }
                    mma_commit(&empty[stage]);
                    if (++stage == PG_STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
            }
        }
    } else {
        // epilogue: warps 2..5 -> TMEM lane quarters 2, 3, 0, 1
        const int q = warp & 3;
        const int row_in_tile = q * 32 + lane;
        const long long HPd = (long long)p.H * p.P * p.d, Pd = (long long)p.P * p.d;
        const bool issuer = warp == 2 && lane == 0;   // sends the staged chunks (plain mode)
        int staged = 0;                               // chunks staged so far (plain mode)
        int it = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            if (!mbar_wait(&tfull[acc], acc_phase, p.status, kSiteProjEpilogue, abort_flag)) break;
            tc_fence_after();
            const int mt = tile % p.num_m_tiles, nt = tile / p.num_m_tiles;
            if (PLAIN) {
                // Y tile -> bf16 -> a 128B-swizzled chunk of 64 columns in shared memory (each
                // thread writes its row) -> one TMA store per chunk (rows past M are clipped);
                // two chunk buffers, so a chunk is converted while the previous one is sent
                const int s = nt / p.ntps;
                const int ncol0 = (nt % p.ntps) * PG_N;
#pragma unroll 1
                for (int cc = 0; cc < PG_N / 64 && ncol0 + cc * 64 < p.hd; ++cc, ++staged) {
                    uint8_t *stg = sStg + (staged & 1) * PG_STG_BYTES;
                    if (issuer) bulk_wait_read(1);   // the store that last read this buffer is done
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    uint32_t r[2][32];
                    tmem_ld32(tmem_base + acc * PG_N + cc * 64 + (uint32_t(q * 32) << 16), r[0]);
                    tmem_ld32(tmem_base + acc * PG_N + cc * 64 + 32 + (uint32_t(q * 32) << 16), r[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 8; ++u) {   // 16-byte unit u of the row: columns 8u .. 8u+7
                        const uint32_t *rr = r[u / 4] + (u % 4) * 8;
                        *reinterpret_cast<uint4 *>(stg + row_in_tile * 128 + ((u ^ (row_in_tile & 7)) << 4)) =
                            make_uint4(pack_bf16x2(__uint_as_float(rr[0]), __uint_as_float(rr[1])),
                                       pack_bf16x2(__uint_as_float(rr[2]), __uint_as_float(rr[3])),
                                       pack_bf16x2(__uint_as_float(rr[4]), __uint_as_float(rr[5])),
                                       pack_bf16x2(__uint_as_float(rr[6]), __uint_as_float(rr[7])));
                    }
                    fence_proxy_async_smem();   // the staging writes before the TMA store reads them
                    asm volatile("bar.sync 1, 128;" ::: "memory");
                    if (issuer) {
                        tma_store_2d(&tmY, stg, s * p.hd + ncol0 + cc * 64, mt * PG_M);
                        bulk_commit();
                    }
                }
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
                continue;
            }
            const long long m = (long long)mt * PG_M + row_in_tile;
            const bool row_ok = m < p.M;
            const long long b = m / p.N_tok, t = m % p.N_tok;
#pragma unroll 1
            for (int c0 = 0; c0 < PG_N; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem_base + acc * PG_N + c0 + (uint32_t(q * 32) << 16), r);
                tmem_ld_wait();
                const long long n = (long long)nt * PG_N + c0;
                if (row_ok && n < p.Ncols) {
                    // columns n..n+31 lie in one (s, h) block because P*d is a multiple of 32
                    const long long s = n / HPd, rem = n % HPd, h = rem / Pd, jc = rem % Pd;
                    __nv_bfloat16 *dst = p.qkv + s * p.s_stride + ((b * p.H + h) * p.N_tok + t) * Pd + jc;
                    uint4 v[4];
                    uint32_t *vw = reinterpret_cast<uint32_t *>(v);
                    if (s == 2) {   // Vbar is stored as f16 (the P V product runs in f16)
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            vw[i] = pack_f16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            vw[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                    }
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                    for (int i = 0; i < 4; ++i) d4[i] = v[i];
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
        if (PLAIN && issuer) bulk_wait_all();   // the staged chunks are read and written before exit
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

cudaError_t launch_project_f32(const void *X, const void *Wt, const Shape &sh, void *QKV, cudaStream_t st);

cudaError_t launch_project(const void *X, const void *Wt, const Shape &sh, int dtype, void *QKV,
                           cudaStream_t st, int *status) {
    if (dtype == 0) return launch_project_f32(X, Wt, sh, QKV, st);
    const long long M = (long long)sh.B * sh.N, Ncols = sh.wt_rows(), K = sh.D();
    CUtensorMap tmA, tmB;
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)K * 2};
        const uint32_t box[2] = {PG_K, PG_M};
        if (!make_tmap_bf16(&tmA, X, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)Ncols};
        const uint64_t strides[1] = {(uint64_t)K * 2};
        const uint32_t box[2] = {PG_K, PG_N};
        if (!make_tmap_bf16(&tmB, Wt, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    ProjParams p{};
    p.qkv = (__nv_bfloat16 *)QKV;
    p.s_stride = sh.qkv_elems();
    p.M = (int)M;
    p.Ncols = (int)Ncols;
    p.K = (int)K;
    p.N_tok = sh.N;
    p.H = sh.H;
    p.P = sh.P;
    p.d = sh.d;
    p.num_m_tiles = (int)((M + PG_M - 1) / PG_M);
    const int num_n_tiles = (int)((Ncols + PG_N - 1) / PG_N);
    p.num_tiles = p.num_m_tiles * num_n_tiles;
    p.status = status;
    cudaError_t e = cudaFuncSetAttribute(proj_gemm_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, PG_SMEM);
    if (e != cudaSuccess) return e;
    const int grid = p.num_tiles < device_sm_count() ? p.num_tiles : device_sm_count();
    proj_gemm_tc<false><<<grid, PG_THREADS, PG_SMEM, st>>>(tmA, tmB, tmB, tmB, tmA, p);
    return cudaGetLastError();
}

cudaError_t launch_project_heads(const void *X, const void *WQ, const void *WK, const void *WV, const Shape &sh,
                                 void *Y, cudaStream_t st, int *status) {
    const long long M = (long long)sh.B * sh.N, K = sh.D(), hd = (long long)sh.H * sh.d;
    if (hd % 64 != 0) return cudaErrorInvalidValue;
    CUtensorMap tmA, tmW[3];
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)K * 2};
        const uint32_t box[2] = {PG_K, PG_M};
        if (!make_tmap_bf16(&tmA, X, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    const void *W[3] = {WQ, WK, WV};
    for (int s = 0; s < 3; ++s) {
        // (n % 64, k, n / 64): one box = 4 chunks of [64 k][64 n]
        const uint64_t dims[3] = {64, (uint64_t)K, (uint64_t)(hd / 64)};
        const uint64_t strides[2] = {(uint64_t)hd * 2, 128};
        const uint32_t box[3] = {64, PG_K, PG_N / 64};
        if (!make_tmap_bf16(&tmW[s], W[s], 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    CUtensorMap tmY;   // Y [M][3*hd] in 64-column x 128-row boxes (the epilogue's stores)
    {
        const uint64_t dims[2] = {(uint64_t)(3 * hd), (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)(3 * hd) * 2};
        const uint32_t box[2] = {64, PG_M};
        if (!make_tmap_bf16(&tmY, Y, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    ProjParams p{};
    p.y = (__nv_bfloat16 *)Y;
    p.hd = (int)hd;
    p.ntps = (int)((hd + PG_N - 1) / PG_N);
    p.M = (int)M;
    p.K = (int)K;
    p.N_tok = sh.N;
    p.H = sh.H;
    p.P = sh.P;
    p.d = sh.d;
    p.num_m_tiles = (int)((M + PG_M - 1) / PG_M);
    p.num_tiles = p.num_m_tiles * 3 * p.ntps;
    p.status = status;
    cudaError_t e =
        cudaFuncSetAttribute(proj_gemm_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, PG_SMEM_PLAIN);
    if (e != cudaSuccess) return e;
    const int grid = p.num_tiles < device_sm_count() ? p.num_tiles : device_sm_count();
    proj_gemm_tc<true><<<grid, PG_THREADS, PG_SMEM_PLAIN, st>>>(tmA, tmW[0], tmW[1], tmW[2], tmY, p);
    return cudaGetLastError();
}

}  // namespace iha
