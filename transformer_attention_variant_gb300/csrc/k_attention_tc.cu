// k_attention_tc.cu -- masked softmax attention over each head's stacked pseudo-token
// sequence ("Interleaved Head Attention" section 4, Algorithm 1, step "注意力計算":
// S_h = Qbar_h Kbar_h^T / sqrt(d), Pbar_h = softmax(S_h) Vbar_h), computed without ever
// materialising S (online softmax: "注意力机制" eq. (5.11) evaluated tile by tile with a
// running maximum and sum).
//
// Stacked rows are t-major (row t*P + j).  The mask reads the original position t only
// (t' <= t, and t - t' < window), so for query row r the readable key rows form ONE
// contiguous interval  [lo(r), hi(r)] = [max(0,(t-w+1)P), min(L-1,(t+1)P-1)];  KV tiles
// outside the union of intervals of a CTA's rows are skipped and tiles inside every row's
// interval run without any mask arithmetic.
//
// Design (sm_103a, one CTA per SM):
//   - a CTA owns 256 query rows of one (b, h): two 128-row tiles Q0, Q1 that ping-pong so
//     the tensor cores work on one tile while the softmax warps work on the other;
//   - warp 8: TMA producer (Q once; K and V tiles through a 2-stage ring, 128B swizzle);
//   - warp 9: MMA issuer: S_i = Q_i K^T (SS, M=128 N=128) into TMEM, then O_i += P_i V
//     with P_i read from TMEM (TS form, M=128 N=d, f16 P and f16 V) -- P never touches
//     shared memory;
//   - warps 0-3 / 4-7: softmax of Q0 / Q1, one thread per row (32x32b TMEM loads): row
//     max, exp2 (two per MUFU op in f16x2), row sum, f16 P written back over its S columns.  The running max is only
//     raised when a tile's max exceeds it by more than 8 (log2 units), so O (in TMEM) is
//     rarely rescaled; values stay <= 2^8 before normalisation;
//   - epilogue: O / l -> bf16 -> Pbar[b][t][h][j][:].
// TMEM: S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [256+d,256+2d)  (512 columns allocated).
#include <cuda_bf16.h>

#include "iha_internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace iha {

constexpr int AT_BM = 128;         // query rows per tile
constexpr int AT_BN = 128;         // key rows per tile
constexpr int AT_THREADS = 384;    // 2 softmax warpgroups + 1 warpgroup (producer, MMA, 2 idle)
// Register split (setmaxnreg): the kernel is compiled to exactly AT_LAUNCH_REGS per thread
// (384 x 168 = 64512 registers allocated at launch); the producer/MMA warpgroup gives
// registers back, the softmax warpgroups take them: 128 x 56 + 256 x 224 = 64512.
constexpr int AT_LAUNCH_REGS = 168, AT_REGS_SOFTMAX = 224, AT_REGS_CONTROL = 56;
static_assert(128 * AT_REGS_CONTROL + 256 * AT_REGS_SOFTMAX <= AT_THREADS * AT_LAUNCH_REGS, "register split");
constexpr float AT_RESCALE_THRESHOLD = 8.0f;

template <int DH>
struct AttnCfg {
    static constexpr int CHUNKS = DH / 64;               // 64-column (128-byte) swizzle chunks
    static constexpr int Q_BYTES = AT_BM * DH * 2;
    static constexpr int KV_BYTES = AT_BN * DH * 2;
    // K tiles are freed as soon as the second S-MMA has read them, V tiles only after the
    // second PV-MMA: K gets the deeper ring so the next K is resident before it is needed.
    static constexpr int KSTAGES = DH == 128 ? 3 : 4;
    static constexpr int VSTAGES = DH == 128 ? 2 : 4;
    static constexpr int SMEM = 2 * Q_BYTES + (KSTAGES + VSTAGES) * KV_BYTES + 256 + 1024;
    __device__ static constexpr uint32_t s_col(int i) { return uint32_t(i) * 128u; }
    __device__ static constexpr uint32_t o_col(int i) { return 256u + uint32_t(i) * DH; }
};

struct AttnParams {
    __nv_bfloat16 *pbar;   // [B][N][H][P][d]
    int N, H, P, L;        // L = N*P
    int mask_mode, window;
    float scale_log2;      // log2(e) / sqrt(d)
    int num_qblocks;
    int num_heads;         // B * H
    int head_group;        // heads per scheduling group
    int *status;
};

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// readable stacked key rows of query row r: [lo, hi]
__device__ __forceinline__ void key_interval(const AttnParams &p, long long r, long long &lo, long long &hi) {
    const long long t = r / p.P;
    lo = 0;
    hi = p.L - 1;
    if (p.mask_mode >= 1) {
        const long long h2 = (t + 1) * p.P - 1;
        if (h2 < hi) hi = h2;
    }
    if (p.mask_mode == 2) {
        const long long l2 = (t - p.window + 1) * p.P;
        if (l2 > lo) lo = l2;
    }
}

template <int DH>
__global__ void __launch_bounds__(AT_THREADS, 1)
attn_fwd_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
            const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using C = AttnCfg<DH>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem;                                  // 2 tiles
    uint8_t *sK = sQ + 2 * C::Q_BYTES;                   // KSTAGES tiles
    uint8_t *sV = sK + C::KSTAGES * C::KV_BYTES;         // VSTAGES tiles
    uint64_t *bars = reinterpret_cast<uint64_t *>(sV + C::VSTAGES * C::KV_BYTES);
    uint64_t *q_full = bars;
    uint64_t *k_full = bars + 1;               // [KSTAGES]
    uint64_t *k_empty = k_full + C::KSTAGES;   // [KSTAGES]
    uint64_t *v_full = k_empty + C::KSTAGES;   // [VSTAGES]
    uint64_t *v_empty = v_full + C::VSTAGES;   // [VSTAGES]
    uint64_t *s_full = v_empty + C::VSTAGES;   // [2]
    uint64_t *p_full = s_full + 2;            // [2]
    uint64_t *o_full = p_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(o_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = warp_id(), lane = lane_id();
    // Work order: heads in groups of p.head_group (chosen so a group's K and V fit in L2);
    // within a group, query blocks heaviest (latest) first across the group's heads.  The
    // CTAs resident at one time then share one group's K/V in L2, and the light blocks of
    // each group fill the tail of its wave.
    int bh, qb;
    {
        const long long i = blockIdx.x;
        const long long per_group = (long long)p.head_group * p.num_qblocks;
        const int g = (int)(i / per_group);
        const int j = (int)(i % per_group);
        const int g_heads = min(p.head_group, p.num_heads - g * p.head_group);
        bh = g * p.head_group + j % g_heads;
        qb = p.num_qblocks - 1 - j / g_heads;
    }
    const long long r0 = (long long)qb * 2 * AT_BM;

    // KV tiles this CTA needs: union of the readable intervals of its rows
    long long lo_first, hi_first, lo_last, hi_last;
    const long long r_last = (r0 + 2 * AT_BM - 1 < p.L - 1) ? r0 + 2 * AT_BM - 1 : p.L - 1;
    key_interval(p, r0, lo_first, hi_first);
    key_interval(p, r_last, lo_last, hi_last);
    const int kv_begin = (int)(lo_first / AT_BN);
    const int kv_end = (int)(hi_last / AT_BN);
    const int nkv = kv_end - kv_begin + 1;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < C::KSTAGES; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < C::VSTAGES; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);   // one arrive per softmax warp
        }
        mbar_init(o_full, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
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
      // control warpgroup: gives registers back, then warp 8 = TMA, warp 9 = MMA
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(AT_REGS_CONTROL));
      if (warp == 8) {
        // ------------------------------- TMA producer -------------------------------
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, 2 * C::Q_BYTES);
            for (int i = 0; i < 2; ++i)
                for (int c = 0; c < C::CHUNKS; ++c)
                    tma_load_3d(&tmQ, q_full, sQ + i * C::Q_BYTES + c * (AT_BM * 128), c * 64,
                                (int)(r0 + i * AT_BM), bh);
            // K runs one tile ahead of V: K(k) is issued before V(k-1)
            for (int k = 0; k <= nkv; ++k) {
                if (k < nkv) {
                    const int st = k % C::KSTAGES;
                    if (!mbar_wait_lazy(&k_empty[st], ((k / C::KSTAGES) & 1) ^ 1, p.status, kSiteAttnProducer, abort_flag))
                        break;
                    mbar_arrive_expect_tx(&k_full[st], C::KV_BYTES);
                    for (int c = 0; c < C::CHUNKS; ++c)
                        tma_load_3d(&tmK, &k_full[st], sK + st * C::KV_BYTES + c * (AT_BN * 128), c * 64,
                                    (kv_begin + k) * AT_BN, bh);
                }
                if (k >= 1) {
                    const int kv = k - 1, st = kv % C::VSTAGES;
                    if (!mbar_wait_lazy(&v_empty[st], ((kv / C::VSTAGES) & 1) ^ 1, p.status, kSiteAttnProducer, abort_flag))
                        break;
                    mbar_arrive_expect_tx(&v_full[st], C::KV_BYTES);
                    for (int c = 0; c < C::CHUNKS; ++c)
                        tma_load_3d(&tmV, &v_full[st], sV + st * C::KV_BYTES + c * (AT_BN * 128), c * 64,
                                    (kv_begin + kv) * AT_BN, bh);
                }
            }
        }
      } else if (warp == 9) {
        // ------------------------------- MMA issuer ---------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(AT_BM, AT_BN, 0, 0);   // Q K^T: both K-major
            constexpr uint32_t idesc_o = idesc_f16_f32(AT_BM, DH, 0, 1);       // P V (f16): V is MN-major
            const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
            auto issue_s = [&](int i, int st) {
                const uint32_t d = tmem + C::s_col(i);
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk) {
                    const uint32_t off = (kk / 4) * (AT_BM * 128) + (kk % 4) * 32;
                    mma_ss(d, sdesc_sw128(q_addr + i * C::Q_BYTES + off, 16, 1024),
                           sdesc_sw128(k_addr + st * C::KV_BYTES + off, 16, 1024), idesc_s, kk > 0);
                }
            };
            auto issue_pv = [&](int i, int st, bool acc) {
                const uint32_t d = tmem + C::o_col(i);
#pragma unroll
                for (int kk = 0; kk < AT_BN / 16; ++kk) {
                    // A = P (bf16 pairs in TMEM, 8 columns per 16 keys); B = 16 keys x d of V:
                    // leading (MN) byte offset = one 64-column chunk, stride = 8 keys.
                    mma_ts(d, tmem + C::s_col(i) + kk * 8,
                           sdesc_sw128(v_addr + st * C::KV_BYTES + kk * 16 * 128, AT_BN * 128, 1024), idesc_o,
                           (acc || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = mbar_wait(q_full, 0, p.status, kSiteAttnMmaQ, abort_flag) &&
                      mbar_wait(&k_full[0], 0, p.status, kSiteAttnMmaK, abort_flag);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                mma_commit(&s_full[0]);
                issue_s(1, 0);
                mma_commit(&s_full[1]);
                mma_commit(&k_empty[0]);
            }
            for (int k = 0; ok && k < nkv; ++k) {
                const int vst = k % C::VSTAGES;
                const int kst2 = (k + 1) % C::KSTAGES;
                const bool more = k + 1 < nkv;
                // tile 0: O0 += P0 V(k), then S0(k+1)
                ok = mbar_wait(&p_full[0], k & 1, p.status, kSiteAttnMmaP, abort_flag) &&
                     mbar_wait(&v_full[vst], (k / C::VSTAGES) & 1, p.status, kSiteAttnMmaV, abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_pv(0, vst, k > 0);
                if (more) {
                    ok = mbar_wait(&k_full[kst2], ((k + 1) / C::KSTAGES) & 1, p.status, kSiteAttnMmaK, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(0, kst2);
                    mma_commit(&s_full[0]);
                }
                // tile 1: O1 += P1 V(k) (then V(k) is free), S1(k+1) (then K(k+1) is free)
                ok = mbar_wait(&p_full[1], k & 1, p.status, kSiteAttnMmaP, abort_flag);
                if (!ok) break;
                tc_fence_after();
                issue_pv(1, vst, k > 0);
                mma_commit(&v_empty[vst]);
                if (more) {
                    issue_s(1, kst2);
                    mma_commit(&s_full[1]);
                    mma_commit(&k_empty[kst2]);
                }
            }
            mma_commit(o_full);
        }
      }
    } else {
        // ------------------------------- softmax warps ------------------------------
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(AT_REGS_SOFTMAX));
        const int tile = warp >> 2;           // 0: rows [r0, r0+128), 1: [r0+128, r0+256)
        const int q = warp & 3;               // TMEM lane quarter
        const int row = q * 32 + lane;
        const long long r = r0 + tile * AT_BM + row;
        const uint32_t lane_addr = uint32_t(q * 32) << 16;
        const uint32_t s_col = tmem + lane_addr + C::s_col(tile);
        const uint32_t o_col = tmem + lane_addr + C::o_col(tile);
        long long lo, hi;
        key_interval(p, r, lo, hi);
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int k = 0; k < nkv; ++k) {
            if (!mbar_wait(&s_full[tile], k & 1, p.status, kSiteAttnSoftmax, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[AT_BN];
#pragma unroll
            for (int c = 0; c < AT_BN / 32; ++c) {
                uint32_t u[32];
                tmem_ld32(s_col + c * 32, u);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(u[i]);
            }
            tmem_ld_wait();
            // mask columns outside [lo, hi] (only when some row of the warp needs it)
            {
                const long long kr0 = (long long)(kv_begin + k) * AT_BN;
                const bool need_mask = (kr0 < lo) || (kr0 + AT_BN - 1 > hi);
                if (__any_sync(0xffffffffu, need_mask)) {
                    const long long a = lo - kr0, b = hi - kr0;
#pragma unroll
                    for (int c = 0; c < AT_BN; ++c)
                        if (c < a || c > b) s[c] = -INFINITY;
                }
            }
            // row max: 8 independent chains of 3-input max, then a tree (max is exact)
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
            for (int c = 8; c < AT_BN; c += 16)
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = fmax3(mx[i], s[c + i], s[c + 8 + i]);
            const float mt = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7]));
            const float m_cand = mt * sl2;
            const bool raise = m_cand > m_run + AT_RESCALE_THRESHOLD;
            float factor = 1.f;
            if (raise) {
                factor = fast_exp2(m_run - m_cand);   // m_run = -inf -> 0
                l_run *= factor;
                m_run = m_cand;
            }
            if (k > 0 && __any_sync(0xffffffffu, raise)) {
                // O (previous tiles) is complete: S(k) was issued after PV(k-1)
#pragma unroll 1
                for (int c = 0; c < DH / 32; ++c) {
                    uint32_t u[32];
                    tmem_ld32(o_col + c * 32, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * factor);
                    tmem_st32(o_col + c * 32, u);
                }
            }
            const float mu = (m_run == -INFINITY) ? 0.f : m_run;
            // p = 2^(s * log2(e)/sqrt(d) - m): the exponent by a packed fp32x2 FMA, rounded to
            // f16x2, then one ex2.f16x2 per pair.  P goes to TMEM as f16 (the PV product is f16).
            uint32_t pk[AT_BN / 64][32];
#pragma unroll
            for (int c = 0; c < AT_BN / 64; ++c) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x0, x1;
                    ffma2(x0, x1, s[c * 64 + 2 * i], s[c * 64 + 2 * i + 1], sl2, sl2, -mu, -mu);
                    pk[c][i] = ex2_f16x2(pack_f16x2(x0, x1));
                }
                tmem_st32(s_col + c * 32, pk[c]);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[tile]);
            // row sum off the critical path (the MMA warp already has P).  Each p <= 2^8
            // (threshold rule), so an f16 partial over 16 values stays below 2^12.
            uint32_t hs[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) hs[i] = hadd2_f16(pk[0][i], pk[0][i + 8]);
#pragma unroll
            for (int i = 0; i < 8; ++i) hs[i] = hadd2_f16(hs[i], hadd2_f16(pk[0][i + 16], pk[0][i + 24]));
            float lsum = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) lsum += f16x2_sum_to_f32(hs[i]);
#pragma unroll
            for (int c = 1; c < AT_BN / 64; ++c) {
#pragma unroll
                for (int i = 0; i < 8; ++i) hs[i] = hadd2_f16(pk[c][i], pk[c][i + 8]);
#pragma unroll
                for (int i = 0; i < 8; ++i) hs[i] = hadd2_f16(hs[i], hadd2_f16(pk[c][i + 16], pk[c][i + 24]));
#pragma unroll
                for (int i = 0; i < 8; ++i) lsum += f16x2_sum_to_f32(hs[i]);
            }
            l_run += lsum;
        }
        // ------------------------------- epilogue -----------------------------------
        if (ok && mbar_wait(o_full, 0, p.status, kSiteAttnEpilogue, abort_flag)) {
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            const bool row_ok = r < p.L;
            const long long t = r / p.P, j = r % p.P;
            const long long b = bh / p.H, h = bh % p.H;
            __nv_bfloat16 *dst = p.pbar + (((b * p.N + t) * p.H + h) * p.P + j) * DH;
#pragma unroll 1
            for (int c = 0; c < DH / 32; ++c) {
                uint32_t u[32];
                tmem_ld32(o_col + c * 32, u);
                tmem_ld_wait();
                if (row_ok) {
                    uint4 v[4];
                    uint32_t *vw = reinterpret_cast<uint32_t *>(v);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        vw[i] = pack_bf16x2(__uint_as_float(u[2 * i]) * inv, __uint_as_float(u[2 * i + 1]) * inv);
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) d4[i] = v[i];
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

cudaError_t launch_attention_f32(const void *QKV, const Shape &sh, int mask_mode, int window, void *Pbar,
                                 cudaStream_t st);

template <int DH>
static cudaError_t launch_attn_tc(const void *QKV, const Shape &sh, int mask_mode, int window, void *Pbar,
                                  cudaStream_t st, int *status) {
    using C = AttnCfg<DH>;
    const long long L = sh.L(), BH = (long long)sh.B * sh.H;
    const __nv_bfloat16 *base = (const __nv_bfloat16 *)QKV;
    const long long sstride = sh.qkv_elems();
    CUtensorMap tm[3];
    for (int s = 0; s < 3; ++s) {
        const uint64_t dims[3] = {(uint64_t)DH, (uint64_t)L, (uint64_t)BH};
        const uint64_t strides[2] = {(uint64_t)DH * 2, (uint64_t)L * DH * 2};
        const uint32_t box[3] = {64, AT_BM, 1};
        if (!make_tmap_bf16(&tm[s], base + s * sstride, 3, dims, strides, box, /*f16=*/s == 2))
            return cudaErrorInvalidValue;
    }
    AttnParams p;
    p.pbar = (__nv_bfloat16 *)Pbar;
    p.N = sh.N;
    p.H = sh.H;
    p.P = sh.P;
    p.L = (int)L;
    p.mask_mode = mask_mode;
    p.window = window;
    p.scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
    p.num_qblocks = (int)((L + 2 * AT_BM - 1) / (2 * AT_BM));
    p.status = status;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    // the register split above is only valid for exactly AT_LAUNCH_REGS registers per thread
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attn_fwd_tc<DH>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != AT_LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    p.num_heads = (int)BH;
    {
        const long long kv_bytes_per_head = 2LL * L * DH * 2;   // K and V of one (b, h)
        long long g = (48LL << 20) / (kv_bytes_per_head > 0 ? kv_bytes_per_head : 1);
        p.head_group = (int)(g < 1 ? 1 : (g > BH ? BH : g));
    }
    const unsigned grid = (unsigned)(BH * p.num_qblocks);
    attn_fwd_tc<DH><<<grid, AT_THREADS, C::SMEM, st>>>(tm[0], tm[1], tm[2], p);
    return cudaGetLastError();
}

cudaError_t launch_attention(const void *QKV, const Shape &sh, int mask_mode, int window, int dtype, void *Pbar,
                             cudaStream_t st, int *status) {
    if (dtype == 0) return launch_attention_f32(QKV, sh, mask_mode, window, Pbar, st);
    if (sh.d == 128) return launch_attn_tc<128>(QKV, sh, mask_mode, window, Pbar, st, status);
    if (sh.d == 64) return launch_attn_tc<64>(QKV, sh, mask_mode, window, Pbar, st, status);
    return cudaErrorInvalidValue;
}

}  // namespace iha
