// k_backward_tc.cu -- the dense contractions of the IHA backward pass on the tcgen05
// tensor cores: the attention gradients and the weight/input GEMMs.
//
// Attention gradients ("Interleaved Head Attention" section 4, Algorithm 1, the attention
// step differentiated; the softmax part follows "注意力机制" eqs. (5.24)-(5.31)).  Per head,
// over the stacked rows (r = t*P + j) with the forward's per-row log2 normaliser lse
// (p = 2^(s*log2(e)/sqrt(d) - lse)) and D_r = dPbar_r . Pbar_r:
//
//     s_rc = q_r . k_c,   p_rc = 2^(s_rc log2(e)/sqrt(d) - lse_r),   dp_rc = dPbar_r . v_c
//     ds_rc = p_rc (dp_rc - D_r)
//     dv_c = sum_r p_rc dPbar_r,   dk_c = sum_r ds_rc q_r / sqrt(d),   dq_r = sum_c ds_rc k_c / sqrt(d)
//
// over the readable pairs only (c's original position t' <= t, and t - t' < window).  Two
// launches of one kernel, which differ in which side stays resident:
//   - KV: a CTA owns 128 key rows (K, V resident) and streams the query rows that can read
//     them in blocks of 64 (Q, dPbar, lse, D): S^T = K Q^T and dP^T = V dPbar^T (SS MMAs,
//     M=128 N=64), then dV += P^T dPbar and dK += dS^T Q (TS MMAs with P^T / dS^T read
//     from TMEM, M=128 N=d);
//   - Q: a CTA owns 128 query rows (Q, dPbar resident, lse and D per thread) and streams the
//     readable key rows in blocks of 64: S = Q K^T, dP = dPbar V^T, dQ += dS K.
// The scores S and dP are computed in both launches (7 products instead of 5): no atomics,
// and every gradient is written once, in a fixed order.
//
// Roles (384 threads): warps 0-3 and 4-7 are two softmax warpgroups, one thread per
// resident row, taking alternate blocks (TMEM buffers 0 / 1) so that one group's
// exponentials overlap the other's MMAs; warp 8 = TMA producer (128B-swizzled tiles, a
// 4-stage ring of moving blocks; in the KV launch each slot also receives the block's lse
// and D by bulk copy, on the same barrier); warp 9 = MMA issuer.  The MMA order S(i),
// dP(i), [wait P(i-1)] acc(i-1), S(i+1), ... keeps the tensor pipe busy while a block's
// exponentials run.
// Each CTA loads every streamed block for itself; CTAs of neighbouring tiles read the same
// blocks, which L2 serves (the score products, not L2 streaming, bound these kernels).
// TMEM: buffer b: S at 128b, dP at 128b+64 (P^T / dS overwrite their first 32 columns as
// bf16 pairs); accumulators at 256 (dK or dQ) and 256+d (dV).  512 columns.
//
// Weight and input GEMMs (the projection step differentiated):
//     dX = sum_s dY_s W_s^T     (A = dY_s K-major, B = W_s K-major, 3 segments of K)
//     dW_s = X^T dY_s           (A = X^T MN-major, B = dY_s MN-major, 3 problems)
// as one persistent tcgen05 GEMM (M=128 N=256 K=64 tiles, 4-stage TMA ring, two TMEM
// accumulators so that a tile's epilogue overlaps the next tile's main loop), bf16 out
// through shared-memory staging and TMA tensor stores.
#include <cuda_bf16.h>

#include "iha_internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace iha {

// =========================================================================================
// attention gradients
// =========================================================================================
constexpr int BA_ROWS = 128;       // resident rows per CTA
constexpr int BA_BLK = 64;         // streamed rows per block
constexpr int BA_STAGES = 4;       // moving-block ring
constexpr int BA_THREADS = 384;
constexpr int BA_LAUNCH_REGS = 168, BA_REGS_SOFTMAX = 216, BA_REGS_CONTROL = 72;
static_assert(128 * BA_REGS_CONTROL + 256 * BA_REGS_SOFTMAX <= BA_THREADS * BA_LAUNCH_REGS, "register split");

template <int DH>
struct BwdAttnCfg {
    static constexpr int CHUNKS = DH / 64;
    static constexpr int STAT_BYTES = BA_ROWS * DH * 2;   // one resident tile
    static constexpr int MOV_BYTES = BA_BLK * DH * 2;     // one streamed block
    static constexpr int NBARS = 1 + 2 * BA_STAGES + 2 + 2 + 2 + 1 + 1;
    static constexpr int LD_BYTES = BA_STAGES * 2 * BA_BLK * 4;   // lse and D of each ring slot
    static constexpr int CTRL_BYTES = 256;
    static constexpr int SMEM = 2 * STAT_BYTES + BA_STAGES * 2 * MOV_BYTES + LD_BYTES + CTRL_BYTES + 1024;
    static_assert(NBARS * 8 + 8 <= CTRL_BYTES, "control area");
    static_assert(SMEM <= 232448, "shared memory");
    static constexpr uint32_t G_COL = 256, V_COL = 256 + DH;
};

struct BwdAttnParams {
    const float *lse;        // [B*H][ld]
    const float *Dv;         // [B*H][ld]
    __nv_bfloat16 *out0;     // KV: dV, Q: dQ   (token-major [B*N][H*P][d])
    __nv_bfloat16 *out1;     // KV: dK
    int N, H, P, L;
    int mask_mode, window;
    int ntiles;              // resident tiles per head
    int ld;                  // row stride of lse and D: L rounded up to BA_BLK (zero padding)
    float sl2;               // log2(e)/sqrt(d)
    float scale;             // 1/sqrt(d)
    int *status;
};

// readable key rows of query row r: [lo, hi]
__device__ __forceinline__ void ba_key_interval(const BwdAttnParams &p, int r, int &lo, int &hi) {
    const int t = r / p.P;
    lo = 0;
    hi = p.L - 1;
    if (p.mask_mode >= 1) hi = min(hi, (t + 1) * p.P - 1);
    if (p.mask_mode == 2) lo = max(lo, (t - p.window + 1) * p.P);
}
// query rows that read key row c: [lo, hi]
__device__ __forceinline__ void ba_query_interval(const BwdAttnParams &p, int c, int &lo, int &hi) {
    const int t = c / p.P;
    lo = 0;
    hi = p.L - 1;
    if (p.mask_mode >= 1) lo = t * p.P;
    if (p.mask_mode == 2) hi = min(hi, (t + p.window) * p.P - 1);
}

// The resident tile of this CTA and the blocks it streams: [mb0, mb0 + nmov).  Both
// interval ends are nondecreasing in the row, so the union of the tile's rows' ranges runs
// from the first row's lower end to the last row's upper end.
template <bool KV>
__device__ __forceinline__ void ba_range(const BwdAttnParams &p, int &tile, int &mb0, int &nmov) {
    // KV: early key tiles are read by the most queries (causal), Q: late query tiles read
    // the most keys -- heaviest tiles first
    tile = KV ? (int)blockIdx.x : (int)gridDim.x - 1 - (int)blockIdx.x;
    const int r0 = tile * BA_ROWS, r1 = min((tile + 1) * BA_ROWS - 1, p.L - 1);
    int lo0, hi0, lo1, hi1;
    if (KV) {
        ba_query_interval(p, r0, lo0, hi0);
        ba_query_interval(p, r1, lo1, hi1);
    } else {
        ba_key_interval(p, r0, lo0, hi0);
        ba_key_interval(p, r1, lo1, hi1);
    }
    mb0 = lo0 / BA_BLK;
    nmov = lo0 <= hi1 ? hi1 / BA_BLK - mb0 + 1 : 0;
}

__device__ __forceinline__ float ba_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// tmS1/tmS2: resident operands of the score and dP products (KV: K, V; Q: Q, dPbar), box
// 128 rows; tmM1/tmM2: streamed (KV: Q, dPbar; Q: K, V), box 64 rows.  All [B*H][L][d] bf16.
template <int DH, bool KV>
__global__ void __launch_bounds__(BA_THREADS, 1)
bwd_attn_tc(const __grid_constant__ CUtensorMap tmS1, const __grid_constant__ CUtensorMap tmS2,
            const __grid_constant__ CUtensorMap tmM1, const __grid_constant__ CUtensorMap tmM2,
            const BwdAttnParams p) {
    using C = BwdAttnCfg<DH>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sS = smem;                                  // 2 resident tiles (S1, S2)
    uint8_t *sM = sS + 2 * C::STAT_BYTES;                // [stage][M1, M2] blocks
    float *sLD = reinterpret_cast<float *>(sM + BA_STAGES * 2 * C::MOV_BYTES);   // [stage][lse 64 | D 64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(sLD) + C::LD_BYTES);
    uint64_t *stat_full = bars;                    // [1]
    uint64_t *mov_full = stat_full + 1;            // [BA_STAGES]
    uint64_t *mov_empty = mov_full + BA_STAGES;    // [BA_STAGES]
    uint64_t *s_full = mov_empty + BA_STAGES;      // [2]
    uint64_t *dp_full = s_full + 2;                // [2]
    uint64_t *p_full = dp_full + 2;                // [2]
    uint64_t *acc_full = p_full + 2;               // [1]
    uint64_t *drain = acc_full + 1;                // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = warp_id(), lane = lane_id();
    const int bh = blockIdx.y;
    int tile, mb0, nmov;
    ba_range<KV>(p, tile, mb0, nmov);
    const int row0 = tile * BA_ROWS;

    if (threadIdx.x == 0) {
        mbar_init(stat_full, 1);
        for (int s = 0; s < BA_STAGES; ++s) {
            mbar_init(&mov_full[s], 1);
            mbar_init(&mov_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&dp_full[b], 1);
            mbar_init(&p_full[b], 4);   // lane 0 of each warp of the group
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tmS1);
        tma_prefetch_desc(&tmS2);
        tma_prefetch_desc(&tmM1);
        tma_prefetch_desc(&tmM2);
    }
    if (warp == 9) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BA_REGS_CONTROL));
        const bool leader = elect_one();
        if (warp == 8 && nmov > 0) {
            // ----------------------------- TMA producer -----------------------------
            auto wait = [&](uint64_t *bar, uint32_t par) -> bool {
                return __all_sync(0xffffffffu, mbar_wait_lazy(bar, par, p.status, kSiteBwdProducer, abort_flag));
            };
            if (leader) {
                mbar_arrive_expect_tx(stat_full, 2 * C::STAT_BYTES);
                for (int c = 0; c < C::CHUNKS; ++c) {
                    tma_load_3d(&tmS1, stat_full, sS + c * (BA_ROWS * 128), c * 64, row0, bh);
                    tma_load_3d(&tmS2, stat_full, sS + C::STAT_BYTES + c * (BA_ROWS * 128), c * 64, row0, bh);
                }
            }
            int issued = 0;
            for (int i = 0; i < nmov; ++i) {
                const int st = i % BA_STAGES;
                if (!wait(&mov_empty[st], ((i / BA_STAGES) & 1) ^ 1)) break;
                const int rb = (mb0 + i) * BA_BLK;
                if (leader) {
                    mbar_arrive_expect_tx(&mov_full[st], 2 * C::MOV_BYTES + (KV ? 2 * BA_BLK * 4 : 0));
                    if (KV) {
                        // lse and D of the block's 64 query rows (this CTA's own copy; rows past
                        // the end are zero padding, and every pair with them is masked)
                        float *ld = sLD + st * 2 * BA_BLK;
                        bulk_load(ld, p.lse + (size_t)bh * p.ld + rb, BA_BLK * 4, &mov_full[st]);
                        bulk_load(ld + BA_BLK, p.Dv + (size_t)bh * p.ld + rb, BA_BLK * 4, &mov_full[st]);
                    }
                    uint8_t *dst = sM + st * 2 * C::MOV_BYTES;
                    for (int c = 0; c < C::CHUNKS; ++c) {
                        tma_load_3d(&tmM1, &mov_full[st], dst + c * (BA_BLK * 128), c * 64, rb, bh);
                        tma_load_3d(&tmM2, &mov_full[st], dst + C::MOV_BYTES + c * (BA_BLK * 128), c * 64, rb, bh);
                    }
                }
                ++issued;
            }
            // every copy into this CTA has landed before the CTA may exit (the normal path has
            // consumed them all already)
            for (int k = issued - BA_STAGES > 0 ? issued - BA_STAGES : 0; k < issued; ++k)
                mbar_wait(&mov_full[k % BA_STAGES], (k / BA_STAGES) & 1, p.status, kSiteBwdProducer, nullptr,
                          kWaitLimitNs);
            mbar_wait(stat_full, 0, p.status, kSiteBwdProducer, nullptr, kWaitLimitNs);
        } else if (warp == 9 && nmov > 0) {
            // ------------------------------- MMA issuer -------------------------------
            auto wait = [&](uint64_t *bar, uint32_t par) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(bar, par, p.status, kSiteBwdMma, abort_flag));
            };
            constexpr uint32_t idesc_s = idesc_bf16_f32(BA_ROWS, BA_BLK, 0, 0);   // both K-major
            constexpr uint32_t idesc_a = idesc_bf16_f32(BA_ROWS, DH, 0, 1);       // B MN-major
            const uint32_t hi = sdesc_sw128_hi(1024);
            const uint32_t s1_lo = sdesc_sw128_lo(smem_u32(sS), 16);
            const uint32_t s2_lo = sdesc_sw128_lo(smem_u32(sS + C::STAT_BYTES), 16);
            const uint32_t mk_lo = sdesc_sw128_lo(smem_u32(sM), 16);               // K-major view
            const uint32_t mn_lo = sdesc_sw128_lo(smem_u32(sM), BA_BLK * 128);     // MN-major view
            // S(i) then dP(i) into buffer i&1, each committed on its own barrier so that the
            // exponentials of S start while dP is still being computed
            auto issue_scores = [&](int i) {
                const int st = i % BA_STAGES, b = i & 1;
                const uint32_t m1 = (st * 2 * C::MOV_BYTES) >> 4, m2 = (st * 2 * C::MOV_BYTES + C::MOV_BYTES) >> 4;
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk) {
                    const uint32_t oa = ((kk / 4) * (BA_ROWS * 128) + (kk % 4) * 32) >> 4;
                    const uint32_t ob = ((kk / 4) * (BA_BLK * 128) + (kk % 4) * 32) >> 4;
                    mma_ss_w(tmem + b * 128, s1_lo + oa, mk_lo + m1 + ob, hi, idesc_s, kk > 0);
                }
                mma_commit(&s_full[b]);
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk) {
                    const uint32_t oa = ((kk / 4) * (BA_ROWS * 128) + (kk % 4) * 32) >> 4;
                    const uint32_t ob = ((kk / 4) * (BA_BLK * 128) + (kk % 4) * 32) >> 4;
                    mma_ss_w(tmem + b * 128 + 64, s2_lo + oa, mk_lo + m2 + ob, hi, idesc_s, kk > 0);
                }
                mma_commit(&dp_full[b]);
            };
            auto issue_acc = [&](int i) {
                const int st = i % BA_STAGES, b = i & 1;
                const uint32_t m1 = (st * 2 * C::MOV_BYTES) >> 4, m2 = (st * 2 * C::MOV_BYTES + C::MOV_BYTES) >> 4;
#pragma unroll
                for (int kk = 0; kk < BA_BLK / 16; ++kk) {
                    // A = dS (bf16 pairs over the dP columns); B = 16 streamed rows x d
                    const uint32_t ob = (kk * 16 * 128) >> 4;
                    mma_ts_w(tmem + C::G_COL, tmem + b * 128 + 64 + kk * 8, mn_lo + m1 + ob, hi, idesc_a,
                             (i > 0 || kk > 0) ? 1u : 0u);
                    if (KV)   // A = P^T over the S columns, B = dPbar rows
                        mma_ts_w(tmem + C::V_COL, tmem + b * 128 + kk * 8, mn_lo + m2 + ob, hi, idesc_a,
                                 (i > 0 || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = wait(stat_full, 0);
            for (int i = 0; ok && i <= nmov; ++i) {
                if (i < nmov) {
                    const int st = i % BA_STAGES;
                    ok = wait(&mov_full[st], (i / BA_STAGES) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    if (leader) issue_scores(i);
                }
                if (i >= 1) {
                    const int j = i - 1;
                    ok = wait(&p_full[j & 1], (j >> 1) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    if (leader) {
                        issue_acc(j);
                        mma_commit(&mov_empty[j % BA_STAGES]);
                        if (j == nmov - 1) mma_commit(acc_full);
                    }
                }
            }
            // the tensor core is idle before TMEM can be released
            if (leader) mma_commit(drain);
            __syncwarp();
            mbar_wait(drain, 0, p.status, kSiteBwdMma, nullptr, kWaitLimitNs);
        }
    } else {
        // ------------------------------ softmax warps ------------------------------
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(BA_REGS_SOFTMAX));
        const int grp = warp >> 2, q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_addr = uint32_t(q * 32) << 16;
        const int R = row0 + row;   // this thread's resident stacked row
        const bool valid = R < p.L;
        int lo = 1, hi = 0;         // readable streamed rows (empty for padding rows)
        if (valid) {
            if (KV) ba_query_interval(p, R, lo, hi);
            else ba_key_interval(p, R, lo, hi);
        }
        float lse_r = 0.f, D_r = 0.f;
        if (!KV && valid) {
            lse_r = p.lse[(size_t)bh * p.ld + R];
            D_r = p.Dv[(size_t)bh * p.ld + R];
        }
        const float sl2 = p.sl2;
        bool ok = true;
        for (int jj = 0;; ++jj) {
            const int i = grp + 2 * jj;
            if (i >= nmov) break;
            const int st = i % BA_STAGES;
            ok = mbar_wait(&s_full[grp], jj & 1, p.status, kSiteBwdSoftmax, abort_flag);
            if (ok && KV) ok = mbar_wait(&mov_full[st], (i / BA_STAGES) & 1, p.status, kSiteBwdSoftmax, abort_flag);
            if (!ok) break;
            tc_fence_after();
            const uint32_t sc = tmem + lane_addr + grp * 128;
            float pv[BA_BLK];   // the scores, then the probabilities
            {
                uint32_t (&u)[BA_BLK] = *reinterpret_cast<uint32_t (*)[BA_BLK]>(pv);
                tmem_ld32(sc, *reinterpret_cast<uint32_t (*)[32]>(u));
                tmem_ld32(sc + 32, *reinterpret_cast<uint32_t (*)[32]>(u + 32));
                tmem_ld_wait();
            }
            {
                const int rb = (mb0 + i) * BA_BLK;
                const int a = lo - rb, b = hi - rb;
                if (__any_sync(0xffffffffu, a > 0 || b < BA_BLK - 1)) {
#pragma unroll
                    for (int c = 0; c < BA_BLK; ++c)
                        if (c < a || c > b) pv[c] = -INFINITY;
                }
            }
            const float4 *l4 = reinterpret_cast<const float4 *>(sLD + st * 2 * BA_BLK);
            const float4 *d4 = l4 + BA_BLK / 4;
            if (KV) {
                uint32_t pw[BA_BLK / 2];
#pragma unroll
                for (int c4 = 0; c4 < BA_BLK / 4; ++c4) {
                    const float4 l = l4[c4];
                    float x0, x1, x2, x3;   // exponents by packed fp32x2 FMAs
                    ffma2(x0, x1, pv[4 * c4 + 0], pv[4 * c4 + 1], sl2, sl2, -l.x, -l.y);
                    ffma2(x2, x3, pv[4 * c4 + 2], pv[4 * c4 + 3], sl2, sl2, -l.z, -l.w);
                    pv[4 * c4 + 0] = ba_exp2(x0);
                    pv[4 * c4 + 1] = ba_exp2(x1);
                    pv[4 * c4 + 2] = ba_exp2(x2);
                    pv[4 * c4 + 3] = ba_exp2(x3);
                    pw[2 * c4] = pack_bf16x2(pv[4 * c4], pv[4 * c4 + 1]);
                    pw[2 * c4 + 1] = pack_bf16x2(pv[4 * c4 + 2], pv[4 * c4 + 3]);
                }
                tmem_st32(sc, pw);   // P^T over the S columns (dP is in other columns)
            } else {
#pragma unroll
                for (int c = 0; c < BA_BLK; c += 2) {
                    float x0, x1;
                    ffma2(x0, x1, pv[c], pv[c + 1], sl2, sl2, -lse_r, -lse_r);
                    pv[c] = ba_exp2(x0);
                    pv[c + 1] = ba_exp2(x1);
                }
            }
            if (!mbar_wait(&dp_full[grp], jj & 1, p.status, kSiteBwdSoftmax, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t dw[BA_BLK / 2];
            {
                float dp[BA_BLK];
                uint32_t (&u)[BA_BLK] = *reinterpret_cast<uint32_t (*)[BA_BLK]>(dp);
                tmem_ld32(sc + 64, *reinterpret_cast<uint32_t (*)[32]>(u));
                tmem_ld32(sc + 96, *reinterpret_cast<uint32_t (*)[32]>(u + 32));
                tmem_ld_wait();
                if (KV) {
#pragma unroll
                    for (int c4 = 0; c4 < BA_BLK / 4; ++c4) {
                        const float4 dd = d4[c4];
                        float t0, t1, t2, t3;   // dp - D, then p (dp - D), by packed fp32x2 operations
                        fadd2(t0, t1, dp[4 * c4], dp[4 * c4 + 1], -dd.x, -dd.y);
                        fadd2(t2, t3, dp[4 * c4 + 2], dp[4 * c4 + 3], -dd.z, -dd.w);
                        ffma2(t0, t1, pv[4 * c4], pv[4 * c4 + 1], t0, t1, 0.f, 0.f);
                        ffma2(t2, t3, pv[4 * c4 + 2], pv[4 * c4 + 3], t2, t3, 0.f, 0.f);
                        dw[2 * c4] = pack_bf16x2(t0, t1);
                        dw[2 * c4 + 1] = pack_bf16x2(t2, t3);
                    }
                } else {
#pragma unroll
                    for (int c2 = 0; c2 < BA_BLK / 2; ++c2) {
                        float t0, t1;
                        fadd2(t0, t1, dp[2 * c2], dp[2 * c2 + 1], -D_r, -D_r);
                        ffma2(t0, t1, pv[2 * c2], pv[2 * c2 + 1], t0, t1, 0.f, 0.f);
                        dw[c2] = pack_bf16x2(t0, t1);
                    }
                }
            }
            tmem_st32(sc + 64, dw);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[grp]);
        }
        // --------------------------------- epilogue ---------------------------------
        // KV: group 0 writes dV, group 1 dK; Q: each group writes half of dQ's columns.
        const bool have = nmov > 0 && ok && mbar_wait(acc_full, 0, p.status, kSiteBwdEpilogue, abort_flag);
        if (have) tc_fence_after();
        const int ncol = KV ? DH : DH / 2;
        const int col0 = KV ? 0 : grp * (DH / 2);
        const uint32_t acc = tmem + lane_addr + (KV ? (grp == 0 ? C::V_COL : C::G_COL) : C::G_COL) + col0;
        const float sc_out = (KV && grp == 0) ? 1.f : p.scale;
        __nv_bfloat16 *out = (KV && grp == 1) ? p.out1 : p.out0;
        const int b = bh / p.H, h = bh % p.H;
        const long long t = R / p.P, j = R % p.P;
        uint4 *dst = reinterpret_cast<uint4 *>(out + ((((long long)b * p.N + t) * p.H + h) * p.P + j) * DH + col0);
        if (nmov == 0 || have) {
#pragma unroll 1
            for (int c = 0; c < ncol; c += 32) {
                uint32_t u[32];
                if (have) {
                    tmem_ld32(acc + c, u);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) u[e] = 0u;
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(u[2 * e]) * sc_out, __uint_as_float(u[2 * e + 1]) * sc_out);
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        dst[c / 8 + e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int DH, bool KV>
static cudaError_t launch_bwd_attn_kernel(const CUtensorMap (&tm)[4], const BwdAttnParams &p, int BH,
                                          cudaStream_t st) {
    using C = BwdAttnCfg<DH>;
    auto kern = bwd_attn_tc<DH, KV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess) e = check_register_contract(kern, BA_LAUNCH_REGS);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.ntiles, (unsigned)BH);
    cfg.blockDim = dim3(BA_THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    if (KV) e = cudaLaunchKernelEx(&cfg, kern, tm[1], tm[2], tm[0], tm[3], p);
    else e = cudaLaunchKernelEx(&cfg, kern, tm[0], tm[3], tm[1], tm[2], p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Row stride of the lse and D arrays the attention-gradient kernels read: whole 64-row
// blocks, so that each block is one 256-byte bulk copy.
int bwd_ld_stride(long long L) { return (int)((L + BA_BLK - 1) / BA_BLK * BA_BLK); }

// Q, K, Vb (bf16 copy of Vbar), dPst: stacked [B*H][L][d] bf16; lse, Dv [B*H][ld] (ld =
// bwd_ld_stride(L), 256-byte aligned, padding zero);
// dQ, dK, dV token-major [B*N][H*P][d] bf16.
cudaError_t launch_bwd_attention_tc(const void *Q, const void *K, const void *Vb, const void *dPst, const float *lse,
                                    const float *Dv, const Shape &sh, int mask_mode, int window, void *dQ, void *dK,
                                    void *dV, cudaStream_t st, int *status) {
    if (sh.d != 64 && sh.d != 128) return cudaErrorInvalidValue;
    const long long L = sh.L(), BH = (long long)sh.B * sh.H;
    if (BH > 65535) return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(lse) & 15) || (reinterpret_cast<uintptr_t>(Dv) & 15)) return cudaErrorInvalidValue;
    // maps [0] Q, [1] K, [2] Vb, [3] dPst with 128-row boxes (resident) and 64-row boxes
    // (a streamed block)
    const void *src[4] = {Q, K, Vb, dPst};
    CUtensorMap big[4], small[4];
    for (int s = 0; s < 4; ++s) {
        const uint64_t dims[3] = {(uint64_t)sh.d, (uint64_t)L, (uint64_t)BH};
        const uint64_t strides[2] = {(uint64_t)sh.d * 2, (uint64_t)L * sh.d * 2};
        const uint32_t box_b[3] = {64, BA_ROWS, 1}, box_s[3] = {64, BA_BLK, 1};
        if (!make_tmap_bf16(&big[s], src[s], 3, dims, strides, box_b)) return cudaErrorInvalidValue;
        if (!make_tmap_bf16(&small[s], src[s], 3, dims, strides, box_s)) return cudaErrorInvalidValue;
    }
    BwdAttnParams p{};
    p.lse = lse;
    p.Dv = Dv;
    p.N = sh.N;
    p.H = sh.H;
    p.P = sh.P;
    p.L = (int)L;
    p.mask_mode = mask_mode;
    p.window = window;
    p.ntiles = (int)((L + BA_ROWS - 1) / BA_ROWS);
    p.ld = bwd_ld_stride(L);
    p.scale = 1.f / sqrtf((float)sh.d);
    p.sl2 = 1.4426950408889634f * p.scale;
    p.status = status;
    // KV launch: resident K (S1), Vb (S2); streamed Q (M1), dPst (M2)
    const CUtensorMap kv[4] = {small[0], big[1], big[2], small[3]};
    // Q launch: resident Q (S1), dPst (S2); streamed K (M1), Vb (M2)
    const CUtensorMap qm[4] = {big[0], small[1], small[2], big[3]};
    p.out0 = (__nv_bfloat16 *)dV;
    p.out1 = (__nv_bfloat16 *)dK;
    cudaError_t e = sh.d == 128 ? launch_bwd_attn_kernel<128, true>(kv, p, (int)BH, st)
                                : launch_bwd_attn_kernel<64, true>(kv, p, (int)BH, st);
    if (e != cudaSuccess) return e;
    p.out0 = (__nv_bfloat16 *)dQ;
    p.out1 = nullptr;
    return sh.d == 128 ? launch_bwd_attn_kernel<128, false>(qm, p, (int)BH, st)
                       : launch_bwd_attn_kernel<64, false>(qm, p, (int)BH, st);
}

// =========================================================================================
// weight and input GEMMs
// =========================================================================================
constexpr int BG_M = 128, BG_N = 256, BG_K = 64, BG_STAGES = 4;
constexpr int BG_A_BYTES = BG_M * BG_K * 2;   // 16 KB
constexpr int BG_B_BYTES = BG_N * BG_K * 2;   // 32 KB
constexpr int BG_THREADS = 192;
constexpr int BG_STG_BYTES = BG_M * 128;   // one staged 64-column chunk of the epilogue
constexpr int BG_SMEM = BG_STAGES * (BG_A_BYTES + BG_B_BYTES) + 2 * BG_STG_BYTES + 256 + 1024;
static_assert(BG_SMEM <= 232448, "shared memory");

struct BwdGemmParams {
    __nv_bfloat16 *c[3];   // outputs [M][N] row-major, one per problem
    int M, N, K;           // per problem; K per segment
    int nseg;              // K segments summed into one output (operand maps by segment)
    int nprob;             // independent problems (operand maps by problem)
    int num_m_tiles, num_n_tiles, num_tiles;
    int *status;
};

// A_MN: A is stored K-rows x M-contiguous (read through a (m%64, k, m/64) view);
// B_MN: B is stored K-rows x N-contiguous (a (n%64, k, n/64) view).  Otherwise both are
// row-major with K contiguous.
template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(BG_THREADS, 1)
bwd_gemm_tc(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
            const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB0,
            const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
            const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
            const __grid_constant__ CUtensorMap tmC2, const BwdGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + BG_STAGES * BG_A_BYTES;
    uint8_t *sStg = sB + BG_STAGES * BG_B_BYTES;   // 2 staged output chunks
    uint64_t *full = reinterpret_cast<uint64_t *>(sStg + 2 * BG_STG_BYTES);
    uint64_t *empty = full + BG_STAGES;
    uint64_t *tfull = empty + BG_STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = warp_id(), lane = lane_id();
    if (threadIdx.x == 0) {
        for (int s = 0; s < BG_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int nkb = (p.K + BG_K - 1) / BG_K;   // k blocks per segment
    const int nk = nkb * p.nseg;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
                const int prob = tile / (p.num_m_tiles * p.num_n_tiles);
                const int rem = tile % (p.num_m_tiles * p.num_n_tiles);
                const int mt = rem % p.num_m_tiles, nt = rem / p.num_m_tiles;
                for (int kb = 0; kb < nk; ++kb) {
                    const int seg = kb / nkb, k0 = (kb % nkb) * BG_K;
                    const int oi = prob + seg;   // one of the two is always 0
                    const CUtensorMap *ma = oi == 0 ? &tmA0 : (oi == 1 ? &tmA1 : &tmA2);
                    const CUtensorMap *mb = oi == 0 ? &tmB0 : (oi == 1 ? &tmB1 : &tmB2);
                    if (!mbar_wait(&empty[stage], phase ^ 1, p.status, kSiteBwdGemmProducer, abort_flag))
                        goto producer_done;
                    mbar_arrive_expect_tx(&full[stage], BG_A_BYTES + BG_B_BYTES);
                    if (A_MN) tma_load_3d(ma, &full[stage], sA + stage * BG_A_BYTES, 0, k0, mt * (BG_M / 64));
                    else tma_load_2d(ma, &full[stage], sA + stage * BG_A_BYTES, k0, mt * BG_M);
                    if (B_MN) tma_load_3d(mb, &full[stage], sB + stage * BG_B_BYTES, 0, k0, nt * (BG_N / 64));
                    else tma_load_2d(mb, &full[stage], sB + stage * BG_B_BYTES, k0, nt * BG_N);
                    ++issued;
                    if (++stage == BG_STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        producer_done:
            // the copies in flight land before the CTA may exit
            for (int k = issued - BG_STAGES > 0 ? issued - BG_STAGES : 0; k < issued; ++k)
                mbar_wait(&full[k % BG_STAGES], (k / BG_STAGES) & 1, p.status, kSiteBwdGemmProducer, nullptr,
                          kWaitLimitNs);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BG_M, BG_N, A_MN ? 1 : 0, B_MN ? 1 : 0);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                if (!mbar_wait(&tempty[acc], ((it >> 1) & 1) ^ 1, p.status, kSiteBwdGemmMma, abort_flag)) break;
                tc_fence_after();
                const uint32_t dt = tmem_base + acc * BG_N;
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&full[stage], phase, p.status, kSiteBwdGemmMma, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * BG_A_BYTES);
                    const uint32_t b0 = smem_u32(sB + stage * BG_B_BYTES);
#pragma unroll
                    for (int k = 0; k < BG_K / 16; ++k) {
                        // K-major: the next 16 k are 32 bytes along the row; MN-major: 16 rows of
                        // 128 bytes further, 64-wide chunks 8 KB apart (leading byte offset)
                        const uint64_t ad = A_MN ? sdesc_sw128(a0 + k * 2048, 64 * BG_K * 2, 1024)
                                                 : sdesc_sw128(a0 + k * 32, 16, 1024);
                        const uint64_t bd = B_MN ? sdesc_sw128(b0 + k * 2048, 64 * BG_K * 2, 1024)
                                                 : sdesc_sw128(b0 + k * 32, 16, 1024);
                        mma_ss(dt, ad, bd, idesc, (kb | k) != 0);
                    }
                    mma_commit(&empty[stage]);
                    if (++stage == BG_STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
            }
            mma_commit(drain);
            mbar_wait(drain, 0, p.status, kSiteBwdGemmMma, nullptr, kWaitLimitNs);
        }
    } else {
        // epilogue: warps 2..5 -> TMEM lane quarters 2, 3, 0, 1.  Each 64-column chunk of a tile
        // is converted to bf16, staged 128B-swizzled in shared memory (each thread writes its
        // row) and sent with one TMA tensor store (rows past M are clipped); two chunk buffers.
        const int q = warp & 3;
        const int row_in_tile = q * 32 + lane;
        const bool issuer = warp == 2 && lane == 0;
        int staged = 0;
        int it = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
            const int acc = it & 1;
            if (!mbar_wait(&tfull[acc], (it >> 1) & 1, p.status, kSiteBwdGemmEpilogue, abort_flag)) break;
            tc_fence_after();
            const int prob = tile / (p.num_m_tiles * p.num_n_tiles);
            const int rem = tile % (p.num_m_tiles * p.num_n_tiles);
            const int mt = rem % p.num_m_tiles, nt = rem / p.num_m_tiles;
            const CUtensorMap *mc = prob == 0 ? &tmC0 : (prob == 1 ? &tmC1 : &tmC2);
#pragma unroll 1
            for (int cc = 0; cc < BG_N / 64 && nt * BG_N + cc * 64 < p.N; ++cc, ++staged) {
                uint8_t *stg = sStg + (staged & 1) * BG_STG_BYTES;
                if (issuer) bulk_wait_read(1);   // the store that last read this buffer is done
                asm volatile("bar.sync 1, 128;" ::: "memory");
                uint32_t r[2][32];
                tmem_ld32(tmem_base + acc * BG_N + cc * 64 + (uint32_t(q * 32) << 16), r[0]);
                tmem_ld32(tmem_base + acc * BG_N + cc * 64 + 32 + (uint32_t(q * 32) << 16), r[1]);
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
                    tma_store_2d(mc, stg, nt * BG_N + cc * 64, mt * BG_M);
                    bulk_commit();
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
        if (issuer) bulk_wait_all();   // the staged chunks are read and written before exit
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// A row-major [rows][cols] bf16 output map, box [64 cols][BG_M rows] (the epilogue's stores)
static bool out_map(CUtensorMap *m, const void *base, long long rows, long long cols) {
    const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)cols * 2};
    const uint32_t box[2] = {64, BG_M};
    return make_tmap_bf16(m, base, 2, dims, strides, box);
}

template <bool A_MN, bool B_MN>
static cudaError_t launch_bwd_gemm_kernel(const CUtensorMap (&ta)[3], const CUtensorMap (&tb)[3], BwdGemmParams &p,
                                          cudaStream_t st) {
    CUtensorMap tc[3];
    for (int k = 0; k < 3; ++k)
        if (!out_map(&tc[k], p.c[k], p.M, p.N)) return cudaErrorInvalidValue;
    p.num_m_tiles = (p.M + BG_M - 1) / BG_M;
    p.num_n_tiles = (p.N + BG_N - 1) / BG_N;
    p.num_tiles = p.nprob * p.num_m_tiles * p.num_n_tiles;
    cudaError_t e = cudaFuncSetAttribute(bwd_gemm_tc<A_MN, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize, BG_SMEM);
    if (e != cudaSuccess) return e;
    const int grid = p.num_tiles < device_sm_count() ? p.num_tiles : device_sm_count();
    bwd_gemm_tc<A_MN, B_MN><<<grid, BG_THREADS, BG_SMEM, st>>>(ta[0], ta[1], ta[2], tb[0], tb[1], tb[2], tc[0], tc[1],
                                                               tc[2], p);
    return cudaGetLastError();
}

// A row-major [rows][K] bf16 tile map (K contiguous), box [64 k][box_rows]
static bool kmajor_map(CUtensorMap *m, const void *base, long long rows, long long K, uint32_t box_rows) {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {BG_K, box_rows};
    return make_tmap_bf16(m, base, 2, dims, strides, box);
}
// A [K][cols] bf16 tensor (cols contiguous, a multiple of 64) viewed as (c%64, k, c/64),
// box [64 c][64 k][box_cols/64]
static bool mnmajor_map(CUtensorMap *m, const void *base, long long K, long long cols, uint32_t box_cols) {
    const uint64_t dims[3] = {64, (uint64_t)K, (uint64_t)(cols / 64)};
    const uint64_t strides[2] = {(uint64_t)cols * 2, 128};
    const uint32_t box[3] = {64, BG_K, box_cols / 64};
    return make_tmap_bf16(m, base, 3, dims, strides, box);
}

// dX [T][D] = sum_s dY_s [T][D] W_s^T (W_s [D][D], row-major: row = input feature)
cudaError_t launch_bwd_dx_tc(const void *const dY[3], const void *const W[3], long long T, int D, void *dX,
                             cudaStream_t st, int *status) {
    if (D % 64 != 0) return cudaErrorInvalidValue;
    CUtensorMap ta[3], tb[3];
    for (int s = 0; s < 3; ++s) {
        if (!kmajor_map(&ta[s], dY[s], T, D, BG_M)) return cudaErrorInvalidValue;
        if (!kmajor_map(&tb[s], W[s], D, D, BG_N)) return cudaErrorInvalidValue;
    }
    BwdGemmParams p{};
    p.c[0] = p.c[1] = p.c[2] = (__nv_bfloat16 *)dX;
    p.M = (int)T;
    p.N = D;
    p.K = D;
    p.nseg = 3;
    p.nprob = 1;
    p.status = status;
    return launch_bwd_gemm_kernel<false, false>(ta, tb, p, st);
}

// dW_s [D][D] = X^T dY_s  (X [T][D], dY_s [T][D]), s = 0, 1, 2
cudaError_t launch_bwd_dw_tc(const void *X, const void *const dY[3], long long T, int D, void *const dW[3],
                             cudaStream_t st, int *status) {
    if (D % 64 != 0) return cudaErrorInvalidValue;
    CUtensorMap ta[3], tb[3];
    if (!mnmajor_map(&ta[0], X, T, D, BG_M)) return cudaErrorInvalidValue;
    ta[1] = ta[2] = ta[0];
    for (int s = 0; s < 3; ++s)
        if (!mnmajor_map(&tb[s], dY[s], T, D, BG_N)) return cudaErrorInvalidValue;
    BwdGemmParams p{};
    for (int s = 0; s < 3; ++s) p.c[s] = (__nv_bfloat16 *)dW[s];
    p.M = D;
    p.N = D;
    p.K = (int)T;
    p.nseg = 1;
    p.nprob = 3;
    p.status = status;
    return launch_bwd_gemm_kernel<true, true>(ta, tb, p, st);
}

}  // namespace iha

namespace iha {

// =========================================================================================
// token gram: out[a][b] = sum over tokens t and c < d of U(t, a, c) V(t, b, c)
// =========================================================================================
// The gradients of the mixing matrices (alpha_s from Y_s and dS_s, R from dO and Pbar) are
// sums over every token of a small product of two head blocks.  As one contraction over
// K = (token, c) it is a GEMM with M = NB <= 128 rows (V, H*P head rows per token), N = NA
// <= 16 (U, H head rows per token, padded to 16) and a very long K: the tensor cores do it
// in a few cycles per token, so the kernel is a stream of both operands from HBM.  Each CTA
// owns a contiguous token range, accumulates in TMEM and writes its partial [NA][NB]; a
// second pass sums the partials in a fixed order.  Rows past NB / NA in a tile (the next
// token's rows, or zero fill) only produce accumulator rows / columns that are ignored.
constexpr int TG_M = 128, TG_N = 16, TG_STAGES = 8;
constexpr int TG_A_BYTES = TG_M * 128, TG_B_BYTES = TG_N * 128;   // one 64-column chunk each
constexpr int TG_THREADS = 192;
constexpr int TG_SMEM = TG_STAGES * (TG_A_BYTES + TG_B_BYTES) + 256 + 1024;

struct GramParams {
    float *part;        // [gridDim.x][NA][NB]
    int NA, NB, chunks; // chunks = d / 64
    long long ntok;
    int u_rows, v_rows; // rows of U / V per token in the tensor maps' row views
    int *status;
};

__global__ void __launch_bounds__(TG_THREADS, 1)
gram_tc(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmV, const GramParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + TG_STAGES * TG_A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + TG_STAGES * TG_B_BYTES);
    uint64_t *empty = full + TG_STAGES;
    uint64_t *done = empty + TG_STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = warp_id(), lane = lane_id();
    if (threadIdx.x == 0) {
        for (int s = 0; s < TG_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // this CTA's tokens
    const long long per = (p.ntok + gridDim.x - 1) / gridDim.x;
    const long long t0 = (long long)blockIdx.x * per, t1 = min(p.ntok, t0 + per);
    const int nk = t1 > t0 ? (int)(t1 - t0) * p.chunks : 0;
    const uint32_t bytes = (uint32_t)(p.NB + TG_N) * 128;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int k = 0; k < nk; ++k) {
                const int st = k % TG_STAGES;
                if (!mbar_wait_lazy(&empty[st], ((k / TG_STAGES) & 1) ^ 1, p.status, kSiteGramProducer, abort_flag))
                    break;
                const long long t = t0 + k / p.chunks;
                const int c = (k % p.chunks) * 64;
                mbar_arrive_expect_tx(&full[st], bytes);
                tma_load_2d(&tmV, &full[st], sA + st * TG_A_BYTES, c, (int)(t * p.v_rows));
                tma_load_2d(&tmU, &full[st], sB + st * TG_B_BYTES, c, (int)(t * p.u_rows));
                ++issued;
            }
            for (int k = issued - TG_STAGES > 0 ? issued - TG_STAGES : 0; k < issued; ++k)
                mbar_wait(&full[k % TG_STAGES], (k / TG_STAGES) & 1, p.status, kSiteGramProducer, nullptr, kWaitLimitNs);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(TG_M, TG_N, 0, 0);
            bool ok = true;
            for (int k = 0; k < nk; ++k) {
                const int st = k % TG_STAGES;
                if (!mbar_wait(&full[st], (k / TG_STAGES) & 1, p.status, kSiteGramMma, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(sA + st * TG_A_BYTES), b0 = smem_u32(sB + st * TG_B_BYTES);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem, sdesc_sw128(a0 + kk * 32, 16, 1024), sdesc_sw128(b0 + kk * 32, 16, 1024), idesc,
                           (k | kk) != 0);
                mma_commit(&empty[st]);
            }
            // arrives once every MMA issued above is done: the accumulator is final (and, if a
            // wait gave up, no MMA is still writing TMEM when it is released)
            mma_commit(done);
            (void)ok;
            mbar_wait(done, 0, p.status, kSiteGramMma, nullptr, kWaitLimitNs);
        }
    } else {
        // epilogue: warps 2..5 -> TMEM lane quarters 2, 3, 0, 1; row m = b (V row), column n = a
        const int q = warp & 3;
        const int m = q * 32 + lane;
        const bool have = nk > 0 && mbar_wait(done, 0, p.status, kSiteGramEpilogue, abort_flag);
        uint32_t r[16];
        if (have) {
            tc_fence_after();
            tmem_ld16(tmem + (uint32_t(q * 32) << 16), r);
            tmem_ld_wait();
        } else {
#pragma unroll
            for (int n = 0; n < 16; ++n) r[n] = 0u;   // no tokens: a zero partial
        }
        if (m < p.NB) {
            float *dst = p.part + (size_t)blockIdx.x * p.NA * p.NB;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                if (n < p.NA) dst[n * p.NB + m] = __uint_as_float(r[n]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 32);
    }
}

__global__ void gram_sum(const float *__restrict__ part, int nparts, int n, float *__restrict__ out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float v = 0.f;
    for (int k = 0; k < nparts; ++k) v += part[(size_t)k * n + i];
    out[i] = v;
}

static int gram_ctas(long long ntok) {
    const long long g = device_sm_count();
    return (int)(ntok < g ? (ntok > 0 ? ntok : 1) : g);
}

size_t bwd_gram_part_floats(long long ntok, int NA, int NB) { return (size_t)gram_ctas(ntok) * NA * NB; }

// out[a][b] = sum_t sum_c U[t*us + a*d + c] V[t*vs + b*d + c]  (bf16 U, V; us, vs multiples
// of d; NA <= 16, NB <= 128, d in {64, 128}); part holds bwd_gram_part_floats floats.
cudaError_t launch_bwd_gram(const void *U, long long us, int NA, const void *V, long long vs, int NB, int d,
                            long long ntok, float *part, float *out, cudaStream_t st, int *status) {
    if (NA < 1 || NA > TG_N || NB < 1 || NB > TG_M || (d != 64 && d != 128) || us % d || vs % d || ntok < 1)
        return cudaErrorInvalidValue;
    GramParams p{};
    p.part = part;
    p.NA = NA;
    p.NB = NB;
    p.chunks = d / 64;
    p.ntok = ntok;
    p.u_rows = (int)(us / d);
    p.v_rows = (int)(vs / d);
    p.status = status;
    if ((long long)ntok * p.u_rows >= (1LL << 31) || (long long)ntok * p.v_rows >= (1LL << 31))
        return cudaErrorInvalidValue;
    CUtensorMap tmU, tmV;
    {
        // U as rows of d: row t*u_rows + a; only the rows up to the last token's are mapped
        const uint64_t dims[2] = {(uint64_t)d, (uint64_t)((ntok - 1) * p.u_rows + NA)};
        const uint64_t strides[1] = {(uint64_t)d * 2};
        const uint32_t box[2] = {64, TG_N};
        if (!make_tmap_bf16(&tmU, U, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[2] = {(uint64_t)d, (uint64_t)((ntok - 1) * p.v_rows + NB)};
        const uint64_t strides[1] = {(uint64_t)d * 2};
        const uint32_t box[2] = {64, (uint32_t)NB};
        if (!make_tmap_bf16(&tmV, V, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(gram_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, TG_SMEM);
    if (e != cudaSuccess) return e;
    const int g = gram_ctas(ntok);
    gram_tc<<<g, TG_THREADS, TG_SMEM, st>>>(tmU, tmV, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int n = NA * NB;
    gram_sum<<<(n + 255) / 256, 256, 0, st>>>(part, g, n, out);
    return cudaGetLastError();
}

}  // namespace iha
