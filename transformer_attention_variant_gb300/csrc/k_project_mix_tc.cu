// k_project_mix_tc.cu -- steps 1 and 2 of "Interleaved Head Attention" (section 4,
// Algorithm 1, "偽頭混合") in one kernel: the head projections X W_s^(m) on the tcgen05 tensor
// cores, and the pseudo-head mixing  S~_{h,j} = sum_m alpha_s[m,h,j] X W_s^(m)  in the GEMM
// epilogue, written straight into the stacked layout QKV[s][b][h][t*P + j][c] (step
// "偽主堆疊").  The head projections never reach global memory (unless asked for).
//
// The mixing of output column c of one token reads column c of every head m, so a GEMM tile
// holds ALL H heads for one slice of CW columns: N = H*CW columns ordered (m, c), with CW the
// widest of 64, 32, 16 for which H*CW <= 256 (CW = 16 at H = 16).  A small first kernel
// (slice_weights) writes each W_s slice-major, Wp_s[k][slice][m][c] = W_s[k][m*d + slice*CW + c]
// (each slice padded to a multiple of 64 columns), so that a B tile is a plain [64 k][N]
// block loaded exactly like an ordinary GEMM's MN-major operand (128-byte rows, 128B swizzle).
// Loading the slices straight from W needs boxes with 32-byte rows, which TMA pads to the
// swizzle span (a 128B-swizzled 32-byte-row box takes 4x its size in shared memory), and
// a 32-byte-swizzled operand made the main loop about 60% slower.
//
// Design (sm_103a): persistent CTAs, one per SM.  Warp 0: TMA producer (A = 128 tokens x 64 k
// of X, B = 64 k x N of Wp_s, both 128B swizzle; 4-stage ring).  Warp 1: MMA issuer (M=128, N=H*CW, K=16,
// fp32 accumulators in TMEM, two buffers of 256 columns, so one tile's epilogue overlaps the
// next tile's main loop); warps 2-3 idle.  Warps 4-11: epilogue, one token row per thread;
// the two warps of a TMEM lane quarter take alternate 8-column groups.  A group's
// projections of all H heads are loaded from TMEM once, mixed into every pseudo-head with
// alpha_s (fp32, staged in shared memory) by packed fp32x2 FMAs, rounded (bf16; f16 for
// Vbar, the type the attention kernel's P V product reads) and stored 16 bytes at a time.
// Tiles are ordered column-slice fastest, so the CTAs working at one time write every
// slice of the same token rows and each stacked row's pieces meet in L2 (ordered the other
// way, the 32-byte pieces of a row were written waves apart and DRAM saw partial lines).
// The mixing costs H*P*H*CW FMAs per token and tile, on the CUDA cores while the tensor
// cores run the next tile.
// Register split (setmaxnreg): launched at PM_LAUNCH_REGS per thread (the build checks the
// count); the control warpgroup drops to PM_REGS_CONTROL, the epilogue warpgroups rise to
// PM_REGS_EPILOGUE.
#include <cuda_bf16.h>

#include "iha_internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace iha {

constexpr int PM_M = 128, PM_K = 64, PM_MAX_STAGES = 4;
constexpr int PM_A_BYTES = PM_M * PM_K * 2;      // 16 KB
constexpr int PM_B_BYTES_MAX = 256 * PM_K * 2;   // 32 KB (N = H*CW <= 256)
constexpr int PM_THREADS = 384;                  // producer, MMA, 2 idle, 8 epilogue warps
constexpr int PM_EPI_THREADS = 256;
constexpr int PM_LAUNCH_REGS = 168, PM_REGS_CONTROL = 56, PM_REGS_EPILOGUE = 224;
static_assert(128 * PM_REGS_CONTROL + 256 * PM_REGS_EPILOGUE <= PM_THREADS * PM_LAUNCH_REGS, "register split");
constexpr int PM_MAXH = 16, PM_MAXHP = 128;
constexpr int PM_STAGE_BYTES = PM_A_BYTES + PM_B_BYTES_MAX;
// Output staging of the TMA-store epilogue: per TMEM lane quarter, PM_OUT_BUFS buffers of
// [4 pseudo-heads][32 tokens][16 columns] bf16.
constexpr int PM_OUT_BUF_BYTES = 4 * 32 * 16 * 2, PM_OUT_BUFS = 3;
constexpr int PM_OUT_BYTES = 4 * PM_OUT_BUFS * PM_OUT_BUF_BYTES;   // 48 KB
// alpha_s[m][hj], fp32: 3*H*HPp*4 bytes.
// Direct-store epilogue: a 4-stage ring when alpha takes at most 24 KB (H*P <= 64), else 3;
// TMA-store epilogue: 3 stages and the staging buffers.
static int pm_alpha_bytes(int H, int HPp) { return 3 * H * HPp * 4; }
static int pm_stages(int H, int HPp, bool tma_out) {
    return tma_out ? 3 : (pm_alpha_bytes(H, HPp) <= 24576 ? 4 : 3);
}
static int pm_smem(int H, int HPp, bool tma_out) {
    return pm_stages(H, HPp, tma_out) * PM_STAGE_BYTES + pm_alpha_bytes(H, HPp) + (tma_out ? PM_OUT_BYTES : 0) + 512 +
           1024;
}
static_assert(4 * PM_STAGE_BYTES + 24576 + 1536 <= 232448 && 3 * PM_STAGE_BYTES + 49152 + 1536 <= 232448 &&
                  3 * PM_STAGE_BYTES + 24576 + PM_OUT_BYTES + 1536 <= 232448,
              "shared memory");

struct PMParams {
    __nv_bfloat16 *qkv;       // stacked output [3][B][H][N*P][d] (Vbar as f16)
    __nv_bfloat16 *y;         // optional: the head projections Y [B*N][3][H*d] (bf16), or NULL
    long long s_stride;       // elements of one of Qbar/Kbar/Vbar
    const float *alpha[3];    // alpha_Q, alpha_K, alpha_V: [H(m)][H(h)][P(j)]
    int M;                    // token rows of this launch
    long long tok0;           // flat token index (b*N + t) of row 0
    int K;                    // D
    int N_tok, H, P, d;
    int HPp;                  // H*P rounded up to a multiple of 4 (alpha row stride in shared memory)
    int stages;               // TMA ring depth (3 or 4)
    int nslices;              // column slices per projection (d / CW)
    int slice_cols;           // columns of one slice in Wp (H*CW rounded up to 64)
    int num_m_tiles, num_n_tiles, num_tiles;
    int *status;
};

// HT: the head count at compile time (0: taken from p.H at run time, up to PM_MAXH).
// TMA_OUT: results leave through shared-memory staging and TMA tensor stores (tmO0..2, rank 5
// over [B][H][P][N][d] of each set: a box is 16 columns x 32 tokens x 4 pseudo-heads); else
// by 16-byte stores from registers.
template <int CW, int HT, bool TMA_OUT>
__global__ void __launch_bounds__(PM_THREADS, 1)
proj_mix_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
            const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
            const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1,
            const __grid_constant__ CUtensorMap tmO2, const PMParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int NH = HT > 0 ? HT : PM_MAXH;
    const int H = HT > 0 ? HT : p.H;
    const int NS = p.stages;
    uint8_t *sA = smem;
    uint8_t *sB = sA + NS * PM_A_BYTES;
    uint8_t *sOut = sB + NS * PM_B_BYTES_MAX;                             // TMA_OUT staging (1 KB aligned)
    float *sAl = reinterpret_cast<float *>(sOut + (TMA_OUT ? PM_OUT_BYTES : 0));   // [s][m][HPp]
    uint64_t *full = reinterpret_cast<uint64_t *>(sAl + 3 * H * p.HPp);
    uint64_t *empty = full + PM_MAX_STAGES;
    uint64_t *tfull = empty + PM_MAX_STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *blk_full = tempty + 2;                       // [4 quarters][PM_OUT_BUFS] (TMA_OUT)
    uint64_t *blk_free = blk_full + 4 * PM_OUT_BUFS;       // [4 quarters][PM_OUT_BUFS]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(blk_free + 4 * PM_OUT_BUFS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = warp_id(), lane = lane_id();
    const int HP = H * p.P;
    const int b_bytes = p.slice_cols * PM_K * 2;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], PM_EPI_THREADS);
        }
        for (int i = 0; i < 4 * PM_OUT_BUFS; ++i) {
            mbar_init(&blk_full[i], 64);   // every thread of the quarter's two epilogue warps
            mbar_init(&blk_free[i], 1);    // the thread that sent the buffer's store
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB0);
        tma_prefetch_desc(&tmB1);
        tma_prefetch_desc(&tmB2);
        if (TMA_OUT) {
            tma_prefetch_desc(&tmO0);
            tma_prefetch_desc(&tmO1);
            tma_prefetch_desc(&tmO2);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    // alpha of the three projections, zero-padded to HPp pseudo-heads per row
    for (int i = threadIdx.x; i < 3 * H * p.HPp; i += PM_THREADS) {
        const int s = i / (H * p.HPp), r = i % (H * p.HPp), m = r / p.HPp, hj = r % p.HPp;
        const float *al = s == 0 ? p.alpha[0] : (s == 1 ? p.alpha[1] : p.alpha[2]);
        const float a = hj < HP ? al[m * HP + hj] : 0.f;
        sAl[(s * H + m) * p.HPp + hj] = a;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int nk = (p.K + PM_K - 1) / PM_K;

    if (warp < 4) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PM_REGS_CONTROL));
      if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
                const int nt = tile % p.num_n_tiles, mt = tile / p.num_n_tiles;
                const int s = nt / p.nslices;
                const CUtensorMap *mb = s == 0 ? &tmB0 : (s == 1 ? &tmB1 : &tmB2);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, p.status, kSiteProjProducer, abort_flag)) goto producer_done;
                    mbar_arrive_expect_tx(&full[stage], PM_A_BYTES + b_bytes);
                    tma_load_2d(&tmA, &full[stage], sA + stage * PM_A_BYTES, kb * PM_K, mt * PM_M);
                    // [slice_cols/64 chunks][64 k][64 n] of Wp_s, one rank-3 copy
                    tma_load_3d(mb, &full[stage], sB + stage * PM_B_BYTES_MAX, 0, kb * PM_K,
                                (nt % p.nslices) * (p.slice_cols / 64));
                    if (++stage == NS) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        producer_done:;
        }
      } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(PM_M, p.H * CW, 0, 1);   // B MN-major
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1, p.status, kSiteProjMmaAcc, abort_flag)) break;
                tc_fence_after();
                const uint32_t dt = tmem_base + acc * 256;
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&full[stage], phase, p.status, kSiteProjMma, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * PM_A_BYTES);
                    const uint32_t b0 = smem_u32(sB + stage * PM_B_BYTES_MAX);
#pragma unroll
                    for (int k = 0; k < PM_K / 16; ++k) {
                        // MN-major B: the next 16 k are 16 rows of 128 bytes further, 64-column
                        // chunks 8 KB apart (leading byte offset)
                        const uint64_t bdesc = sdesc_sw128(b0 + k * 2048, 64 * PM_K * 2, 1024);
                        mma_ss(dt, sdesc_sw128(a0 + k * 32, 16, 1024), bdesc, idesc, (kb | k) != 0);
                    }
                    mma_commit(&empty[stage]);
                    if (++stage == NS) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
            }
        }
      } else if (TMA_OUT && lane == 0) {
        // ------------------------- TMA stores of the staged output -------------------------
        // Warp 2 serves lane quarters 0 and 1, warp 3 quarters 2 and 3, taking their blocks
        // in the order the epilogue fills them: for each block, wait until the quarter's two
        // warps have filled the staging buffer, send it, and free the buffer of the store
        // sent before once that store has read it (so two stores are in flight).
        const int jb = p.P < 4 ? p.P : 4;
        (void)jb;
        int n = 0;               // blocks taken so far (per quarter: n / 2)
        int prev = -1;           // barrier index of the previous store still being read
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
            const int nt = tile % p.num_n_tiles, mt = tile / p.num_n_tiles;
            const int s = nt / p.nslices, c0 = (nt % p.nslices) * CW;
            const CUtensorMap *mo = s == 0 ? &tmO0 : (s == 1 ? &tmO1 : &tmO2);
            for (int k = 0; ok && k < CW / 16; ++k) {
                for (int hb = 0; ok && hb < p.HPp; hb += 4) {
                    for (int qq = 0; qq < 2; ++qq, ++n) {
                        const int q = 2 * (warp - 2) + qq;
                        const int blk = n / 2;                         // the quarter's block number
                        const int bi = q * PM_OUT_BUFS + blk % PM_OUT_BUFS;
                        if (!mbar_wait(&blk_full[bi], (blk / PM_OUT_BUFS) & 1, p.status, kSiteProjStore, abort_flag)) {
                            ok = false;
                            break;
                        }
                        const int g0 = mt * PM_M + q * 32;
                        if (g0 < p.M && hb < HP) {
                            const long long gq = p.tok0 + g0;
                            const uint8_t *stg = sOut + bi * PM_OUT_BUF_BYTES;
                            tma_store_5d(mo, stg, c0 + 16 * k, (int)(gq % p.N_tok), hb % p.P, hb / p.P,
                                         (int)(gq / p.N_tok));
                        }
                        bulk_commit();                                 // an empty group keeps the count
                        bulk_wait_read(1);                             // the previous store has read its buffer
                        if (prev >= 0) mbar_arrive(&blk_free[prev]);
                        prev = bi;
                    }
                }
            }
        }
        bulk_wait_all();
        if (prev >= 0) mbar_arrive(&blk_free[prev]);
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(PM_REGS_EPILOGUE));
        // ------------------------------- epilogue ---------------------------------
        const int q = warp & 3;              // TMEM lane quarter this warp may read
        const int half = (warp - 4) >> 2;    // pseudo-head blocks 4*half, 4*half + 8, ...
        const int row = q * 32 + lane;
        const uint32_t lane_addr = uint32_t(q * 32) << 16;
        const long long Pd = (long long)p.P * p.d;
        int out_blk = 0;   // staging blocks this quarter has filled (TMA_OUT)
        int it = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            // the two warps of a quarter leave together (TMA_OUT: they share a barrier)
            const bool got = mbar_wait(&tfull[acc], acc_phase, p.status, kSiteProjEpilogue, abort_flag);
            if (TMA_OUT ? named_bar_or(1 + q, 64, !got) : !got) break;
            tc_fence_after();
            const int nt = tile % p.num_n_tiles, mt = tile / p.num_n_tiles;
            const int s = nt / p.nslices, c0 = (nt % p.nslices) * CW;
            const bool f16 = s == 2;
            const int mrow = mt * PM_M + row;
            const bool valid = mrow < p.M;
            const long long g = p.tok0 + mrow, b = g / p.N_tok, t = g % p.N_tok;
            // row (b, h, t*P + j) of set s starts at base + (b*H + h)*N*P*d + t*P*d + j*d
            __nv_bfloat16 *base = p.qkv + s * p.s_stride + (b * p.H * p.N_tok + t) * Pd + c0;
            const long long h_stride = (long long)p.N_tok * Pd;
            const float *al_s = sAl + s * H * p.HPp;
            const uint32_t tacc = tmem_base + lane_addr + acc * 256;
            if (p.y && half == 0) {   // the head projections themselves, when asked for
                const long long D = (long long)H * p.d;
#pragma unroll 1
                for (int cc = 0; cc < CW; cc += 16) {
#pragma unroll 1
                    for (int m = 0; m < H; ++m) {
                        uint32_t r[16];
                        tmem_ld16(tacc + m * CW + cc, r);
                        tmem_ld_wait();
                        reg_fence16(r);
                        if (valid) {
                            uint4 *yr = reinterpret_cast<uint4 *>(p.y + g * 3 * D + s * D + (long long)m * p.d + c0 + cc);
                            yr[0] = make_uint4(pack_bf16x2(__uint_as_float(r[0]), __uint_as_float(r[1])),
                                               pack_bf16x2(__uint_as_float(r[2]), __uint_as_float(r[3])),
                                               pack_bf16x2(__uint_as_float(r[4]), __uint_as_float(r[5])),
                                               pack_bf16x2(__uint_as_float(r[6]), __uint_as_float(r[7])));
                            yr[1] = make_uint4(pack_bf16x2(__uint_as_float(r[8]), __uint_as_float(r[9])),
                                               pack_bf16x2(__uint_as_float(r[10]), __uint_as_float(r[11])),
                                               pack_bf16x2(__uint_as_float(r[12]), __uint_as_float(r[13])),
                                               pack_bf16x2(__uint_as_float(r[14]), __uint_as_float(r[15])));
                        }
                    }
                }
            }
            if (TMA_OUT) {
                // The two warps of the quarter take the two 8-column halves of each 16-column
                // chunk; per block of 4 pseudo-heads they fill one staging buffer
                // [4][32 tokens][16 columns] and arrive on its barrier; a thread of warp 2 or 3
                // sends it with a TMA store (its 32-byte rows are whole sectors of stacked rows)
                // and frees it once the store has read it.
#pragma unroll 1
                for (int k = 0; k < CW / 16; ++k) {
                    const int grp = 2 * k + half;
                    float2 y[NH][4];   // [head][column pair]
#pragma unroll
                    for (int m = 0; m < NH; ++m) {
                        if (HT > 0 || m < H)
                            tmem_ld8(tacc + m * CW + grp * 8, *reinterpret_cast<uint32_t (*)[8]>(y[m]));
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int m = 0; m < NH; m += 2) reg_fence16(*reinterpret_cast<uint32_t (*)[16]>(y[m]));
#pragma unroll 1
                    for (int hb = 0; hb < p.HPp; hb += 4, ++out_blk) {
                        float2 o[4][4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int e = 0; e < 4; ++e) o[i][e] = make_float2(0.f, 0.f);
                        // alpha of the block, four heads ahead of its use (the shared-memory load
                        // latency stays off the FMA chain)
                        const float *al_b = al_s + hb;
                        float4 qr[4];
#pragma unroll
                        for (int m = 0; m < 4; ++m)
                            if (HT > 0 || m < H) qr[m] = *reinterpret_cast<const float4 *>(al_b + m * p.HPp);
#pragma unroll
                        for (int m = 0; m < NH; ++m) {
                            if (HT > 0 || m < H) {
                                const float4 q4 = qr[m & 3];
                                if (m + 4 < NH && (HT > 0 || m + 4 < H))
                                    qr[m & 3] = *reinterpret_cast<const float4 *>(al_b + (m + 4) * p.HPp);
                                const float2 a[4] = {make_float2(q4.x, q4.x), make_float2(q4.y, q4.y),
                                                     make_float2(q4.z, q4.z), make_float2(q4.w, q4.w)};
#pragma unroll
                                for (int i = 0; i < 4; ++i)
#pragma unroll
                                    for (int e = 0; e < 4; ++e) o[i][e] = __ffma2_rn(a[i], y[m][e], o[i][e]);
                            }
                        }
                        const int bi = q * PM_OUT_BUFS + out_blk % PM_OUT_BUFS;
                        uint8_t *stg = sOut + bi * PM_OUT_BUF_BYTES;
                        // the store that last read this buffer is done (its first use needs no wait)
                        if (out_blk >= PM_OUT_BUFS &&
                            !mbar_wait(&blk_free[bi], ((out_blk / PM_OUT_BUFS) - 1) & 1, p.status, kSiteProjEpilogue,
                                       abort_flag))
                            break;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                w[e] = f16 ? pack_f16x2(o[i][e].x, o[i][e].y) : pack_bf16x2(o[i][e].x, o[i][e].y);
                            // 32-byte rows, 16-byte halves swapped on every other group of four rows
                            // (the tensor map's 32-byte swizzle): the warp's 32 stores hit 8
                            // different bank groups
                            const int row = i * 32 + lane;
                            *reinterpret_cast<uint4 *>(stg + row * 32 + ((half ^ ((row >> 2) & 1)) << 4)) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                        fence_proxy_async_smem();   // the staging writes before the TMA store reads them
                        mbar_arrive(&blk_full[bi]);
                    }
                }
            } else {
            // Each thread takes the 8-column groups half, half + 2, ... of the slice: the group's
                // projections of all H heads are loaded from TMEM once and every pseudo-head is mixed
                // from them (blocks of 4 pseudo-heads), each leaving as one 16-byte store.
#pragma unroll 1
                for (int grp = half; grp < CW / 8; grp += 2) {
                    float2 y[NH][4];   // [head][column pair]
#pragma unroll
                    for (int m = 0; m < NH; ++m) {
                        if (HT > 0 || m < H) tmem_ld8(tacc + m * CW + grp * 8, *reinterpret_cast<uint32_t (*)[8]>(y[m]));
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int m = 0; m < NH; m += 2) reg_fence16(*reinterpret_cast<uint32_t (*)[16]>(y[m]));
#pragma unroll 1
                    for (int hb = 0; hb < p.HPp; hb += 4) {
                        float2 o[4][4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int e = 0; e < 4; ++e) o[i][e] = make_float2(0.f, 0.f);
#pragma unroll
                        for (int m = 0; m < NH; ++m) {
                            if (HT > 0 || m < H) {
                                const float4 q4 = *reinterpret_cast<const float4 *>(al_s + m * p.HPp + hb);
                                const float2 a[4] = {make_float2(q4.x, q4.x), make_float2(q4.y, q4.y),
                                                     make_float2(q4.z, q4.z), make_float2(q4.w, q4.w)};
#pragma unroll
                                for (int i = 0; i < 4; ++i)
#pragma unroll
                                    for (int e = 0; e < 4; ++e) o[i][e] = __ffma2_rn(a[i], y[m][e], o[i][e]);
                            }
                        }
                        if (valid) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int hj = hb + i;
                                if (hj < HP) {
                                    uint32_t w[4];
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        w[e] = f16 ? pack_f16x2(o[i][e].x, o[i][e].y) : pack_bf16x2(o[i][e].x, o[i][e].y);
                                    const int h = hj / p.P, j = hj % p.P;
                                    *reinterpret_cast<uint4 *>(base + h * h_stride + (long long)j * p.d + grp * 8) =
                                        make_uint4(w[0], w[1], w[2], w[3]);
                                }
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// The column-slice width for H heads: the widest of 64, 32, 16 that keeps N = H*CW <= 256 and
// CW <= d.
static int pm_slice_width(int H, int d) {
    for (int cw = 64; cw >= 16; cw /= 2)
        if (H * cw <= 256 && cw <= d) return cw;
    return 0;
}

bool project_mix_supported(const Shape &sh) {
    return sh.H >= 1 && sh.H <= PM_MAXH && sh.H * sh.P <= PM_MAXHP && (sh.d == 64 || sh.d == 128) &&
           pm_slice_width(sh.H, sh.d) > 0;
}

// Columns of one slice in the slice-major weights: H*CW rounded up to whole 64-column chunks.
static int pm_slice_cols(int H, int cw) { return (H * cw + 63) / 64 * 64; }

size_t sliced_weights_bytes(const Shape &sh) {
    const int cw = pm_slice_width(sh.H, sh.d);
    if (cw == 0) return 0;
    return 3 * (size_t)sh.D() * (size_t)(sh.d / cw) * pm_slice_cols(sh.H, cw) * 2;
}

// Wp_s[k][sl*SC + m*CW + c] = W_s[k][m*d + sl*CW + c] (zero in a slice's padding columns),
// SC = slice columns.  A block moves SW_ROWS whole rows (row = (s, k)); each thread takes
// the same 16-byte unit of every one of them, so their loads are in flight together, and
// consecutive threads write consecutive units.  A warp's loads are whole 32-byte sectors
// (the two 16-byte units of a head's slice).  Indices fit 32 bits: 3*D rows of at most
// d/16 * 256 / 8 units.
constexpr int SW_ROWS = 4;
__global__ void __launch_bounds__(256)
slice_weights_kernel(const uint4 *__restrict__ W0, const uint4 *__restrict__ W1, const uint4 *__restrict__ W2,
                     uint4 *__restrict__ Wp, int D, int H, int d, int cw, int sc, int nslices) {
    const int units_per_slice = sc / 8, row_out = nslices * units_per_slice, row_in = H * d / 8;
    for (int row0 = blockIdx.x * SW_ROWS; row0 < 3 * D; row0 += gridDim.x * SW_ROWS) {
        for (int un = threadIdx.x; un < row_out; un += blockDim.x) {
            const int sl = un / units_per_slice, n = (un % units_per_slice) * 8;   // column within the slice
            const bool live = n < H * cw;
            const int src = live ? ((n / cw) * d + sl * cw + n % cw) / 8 : 0;
            uint4 v[SW_ROWS];
#pragma unroll
            for (int u = 0; u < SW_ROWS; ++u) {
                const int row = row0 + u, s = row / D, k = row - s * D;
                const uint4 *W = s == 0 ? W0 : (s == 1 ? W1 : W2);
                v[u] = (live && row < 3 * D) ? W[(long long)k * row_in + src] : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < SW_ROWS; ++u)
                if (row0 + u < 3 * D) Wp[(long long)(row0 + u) * row_out + un] = v[u];
        }
    }
}

cudaError_t launch_slice_weights(const void *WQ, const void *WK, const void *WV, const Shape &sh, void *Wp,
                                 cudaStream_t st) {
    if (!project_mix_supported(sh)) return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(WQ) | reinterpret_cast<uintptr_t>(WK) | reinterpret_cast<uintptr_t>(WV) |
         reinterpret_cast<uintptr_t>(Wp)) & 15)
        return cudaErrorInvalidValue;
    const int cw = pm_slice_width(sh.H, sh.d), sc = pm_slice_cols(sh.H, cw);
    const long long rows = 3LL * sh.D();
    long long blocks = (rows + SW_ROWS - 1) / SW_ROWS;
    const long long cap = 16LL * device_sm_count();
    if (blocks > cap) blocks = cap;
    slice_weights_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint4 *>(WQ), static_cast<const uint4 *>(WK),
                                                           static_cast<const uint4 *>(WV), static_cast<uint4 *>(Wp),
                                                           (int)sh.D(), sh.H, sh.d, cw, sc, sh.d / cw);
    return cudaGetLastError();
}

template <int CW, int HT, bool TMA_OUT>
static cudaError_t launch_pm(const CUtensorMap &tmA, const void *Wp, const PMParams &p0, const Shape &sh,
                             cudaStream_t st) {
    PMParams p = p0;
    p.stages = pm_stages(sh.H, p.HPp, TMA_OUT);
    const int smem = pm_smem(sh.H, p.HPp, TMA_OUT);
    p.nslices = sh.d / CW;
    p.slice_cols = pm_slice_cols(sh.H, CW);
    p.num_n_tiles = 3 * p.nslices;
    p.num_tiles = p.num_m_tiles * p.num_n_tiles;
    const long long row = (long long)p.nslices * p.slice_cols;   // columns of a Wp_s row
    CUtensorMap tmB[3], tmO[3];
    for (int s = 0; s < 3; ++s) {
        // Wp_s [D][row] as (n % 64, k, n / 64): one box = slice_cols/64 chunks of [64 k][64 n]
        const uint64_t dims[3] = {64, (uint64_t)sh.D(), (uint64_t)(row / 64)};
        const uint64_t strides[2] = {(uint64_t)row * 2, 128};
        const uint32_t box[3] = {64, (uint32_t)PM_K, (uint32_t)(p.slice_cols / 64)};
        if (!make_tmap_bf16(&tmB[s], static_cast<const __nv_bfloat16 *>(Wp) + s * sh.D() * row, 3, dims, strides,
                            box))
            return cudaErrorInvalidValue;
        if (TMA_OUT) {
            // set s of QKV [B][H][N*P][d] as (c, t, j, h, b); a box = 16 columns x 32 tokens x 4
            // pseudo-heads (min(P,4) values of j times 4/min(P,4) heads), 32-byte swizzle
            const int jb = sh.P < 4 ? sh.P : 4;
            const uint64_t dims5[5] = {(uint64_t)sh.d, (uint64_t)sh.N, (uint64_t)sh.P, (uint64_t)sh.H, (uint64_t)sh.B};
            const uint64_t str5[4] = {(uint64_t)sh.P * sh.d * 2, (uint64_t)sh.d * 2,
                                      (uint64_t)sh.N * sh.P * sh.d * 2, (uint64_t)sh.H * sh.N * sh.P * sh.d * 2};
            const uint32_t box5[5] = {16, 32, (uint32_t)jb, (uint32_t)(4 / jb), 1};
            if (!make_tmap_bf16(&tmO[s], p.qkv + s * p.s_stride, 5, dims5, str5, box5, false, 32))
                return cudaErrorInvalidValue;
        } else {
            tmO[s] = tmB[s];   // unused
        }
    }
    auto kern = proj_mix_tc<CW, HT, TMA_OUT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = check_register_contract(kern, PM_LAUNCH_REGS);
    if (e != cudaSuccess) return e;
    const int grid = p.num_tiles < device_sm_count() ? p.num_tiles : device_sm_count();
    kern<<<grid, PM_THREADS, smem, st>>>(tmA, tmB[0], tmB[1], tmB[2], tmO[0], tmO[1], tmO[2], p);
    return cudaGetLastError();
}

// Token rows [tok0, tok0 + ntok) of X [B*N][D] (flat b*N + t) -> their rows of the stacked
// QKV [3][B][H][N*P][d] (Qbar, Kbar bf16; Vbar f16), and, when Y is not NULL, of the head
// projections Y [B*N][3][H*d] (bf16).  Wp: the slice-major weights of launch_slice_weights.
// QKV 32-byte aligned, Y 16-byte aligned.
cudaError_t launch_project_mix(const void *X, const void *Wp, const float *aQ, const float *aK, const float *aV,
                               const Shape &sh, long long tok0, long long ntok, void *QKV, void *Y, cudaStream_t st,
                               int *status) {
    if (!project_mix_supported(sh)) return cudaErrorInvalidValue;
    if (ntok <= 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(QKV) & 31) || (reinterpret_cast<uintptr_t>(Y) & 15)) return cudaErrorInvalidValue;
    const long long K = sh.D();
    CUtensorMap tmA;
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)ntok};
        const uint64_t strides[1] = {(uint64_t)K * 2};
        const uint32_t box[2] = {PM_K, PM_M};
        if (!make_tmap_bf16(&tmA, static_cast<const __nv_bfloat16 *>(X) + tok0 * K, 2, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    PMParams p{};
    p.qkv = (__nv_bfloat16 *)QKV;
    p.y = (__nv_bfloat16 *)Y;
    p.s_stride = sh.qkv_elems();
    p.alpha[0] = aQ;
    p.alpha[1] = aK;
    p.alpha[2] = aV;
    p.M = (int)ntok;
    p.tok0 = tok0;
    p.K = (int)K;
    p.N_tok = sh.N;
    p.H = sh.H;
    p.P = sh.P;
    p.d = sh.d;
    p.HPp = (sh.H * sh.P + 3) / 4 * 4;
    p.num_m_tiles = (int)((ntok + PM_M - 1) / PM_M);
    p.status = status;
    // TMA-store epilogue: whole 32-token groups of one batch element, blocks of 4 pseudo-heads
    // that a box can hold, and alpha within 24 KB; otherwise direct stores
    const bool tma_out = sh.N % 32 == 0 && tok0 % 32 == 0 && ntok % 32 == 0 &&
                         (sh.P == 1 || sh.P == 2 || sh.P == 4 || sh.P == 8) && (sh.H * sh.P) % 4 == 0 &&
                         pm_alpha_bytes(sh.H, p.HPp) <= 24576;
    switch (pm_slice_width(sh.H, sh.d)) {
        case 64: return tma_out ? launch_pm<64, 0, true>(tmA, Wp, p, sh, st) : launch_pm<64, 0, false>(tmA, Wp, p, sh, st);
        case 32: return tma_out ? launch_pm<32, 0, true>(tmA, Wp, p, sh, st) : launch_pm<32, 0, false>(tmA, Wp, p, sh, st);
        case 16:
            if (sh.H == 16)
                return tma_out ? launch_pm<16, 16, true>(tmA, Wp, p, sh, st) : launch_pm<16, 16, false>(tmA, Wp, p, sh, st);
            return tma_out ? launch_pm<16, 0, true>(tmA, Wp, p, sh, st) : launch_pm<16, 0, false>(tmA, Wp, p, sh, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace iha
