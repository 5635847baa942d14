// k_decode_tc.cu -- the attention of one decoding step on the tcgen05 tensor cores (d = 128
// with P <= 4, d = 64 with P <= 8): the P pseudo-queries of the new token t against the cached pseudo-keys and
// pseudo-values it may read ("Interleaved Head Attention" section 4, Algorithm 1, the
// attention step for the rows of token t; the mask is by original position, so every
// pseudo-query of t reads the same cached rows [lo, hi]).
//
// A CTA takes a chunk of the readable rows of one (b, h) and walks it in tiles of 128 rows:
//   S^T  = K_tile Q^T     (M = 128 cached rows, N = 16 -- the P queries padded with zero
//                          rows, K = d; bf16, fp32 in TMEM)
//   O^T_tile = V_tile^T P^T (M = 128 >= d, N = 16, K = 128 rows; f16 V and P)
// so every cached row costs the tensor cores a few cycles and the softmax warps a handful
// of instructions per tile: the kernel streams K and V at HBM speed instead of spending
// ~65 SIMT instructions per row on dot products and lane reductions.
//
// Roles (192 threads): warps 0-3 = softmax, thread i <-> TMEM lane i (cached row i of a tile
// for S, output column i for O); warp 4 = TMA producer (K and V tiles, 128B-swizzled, a
// 3-stage ring of 64 KB); warp 5 = MMA issuer.  Per tile the softmax warps take the tile's
// per-query maximum across the 128 rows (warp shuffles + one named barrier), update the
// running maximum m_q and each thread's share of the normaliser, and write P^T (f16) into a
// double-buffered shared-memory B operand.  Each tile's O^T goes to its own TMEM columns
// (two buffers), and thread i folds it into its register copy of output column i,
// o_q = o_q * 2^(m_q(prev) - m_q) + O^T_tile[i][q], one tile behind the MMA -- no rescaling
// of TMEM.  The chunk's (m, l, o) go to the workspace, and decode_combine (k_decode.cu)
// merges the chunks.
//
// Rows of a tile past the chunk's end are masked out of the softmax (p = 0), and their V rows
// in shared memory are cleared before the output product: a cache row that has not been
// written yet may hold any bits, and 0 * NaN would reach the output.  Everything up to the
// first K/V loads runs before the wait for the mixing kernel (dependent launch); a tile is
// loaded before that wait only if every row the chunk reads from it predates token t, since
// the mixing kernel writes token t's rows while this kernel may already be running.
// TMEM: S buffers at columns 0 and 16, O^T buffers at 32 and 48 (64 columns).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "iha_internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace iha {

constexpr int DT_ROWS = 128;    // cached rows per tile
constexpr int DT_N = 16;        // queries per MMA (P <= 8, zero-padded)
constexpr int DT_STAGES = 3;
constexpr int DT_THREADS = 192;
constexpr int DT_PT_BYTES = DT_N * DT_ROWS * 2;          // one P^T buffer: 4 KB
constexpr int DT_CHUNK = DT_ROWS * 128;                  // one 64-column chunk of a tile: 16 KB

// d = 128 (P <= 4) or d = 64 (P <= 8).  The output product always has M = 128 rows, two
// 64-row d-chunks DT_CHUNK apart in shared memory: for d = 64 a stage is K, V and a block of
// zeros after V, so that the second chunk reads zeros and the rows past d of O^T are 0.
template <int DH>
struct DtCfg {
    static constexpr int PMAX = DH == 128 ? 4 : 8;
    static constexpr int KV_BYTES = DT_ROWS * DH * 2;                           // 32 KB or 16 KB
    static constexpr int STAGE_BYTES = DH == 128 ? 2 * KV_BYTES : 3 * KV_BYTES;   // K, V (, zeros)
    static constexpr int Q_BYTES = DT_N * DH * 2;
    static constexpr int SMEM = DT_STAGES * STAGE_BYTES + Q_BYTES + 2 * DT_PT_BYTES + 512 + 1024;
    static_assert(SMEM <= 232448, "shared memory");
};

struct DecodeTcParams {
    const __nv_bfloat16 *qt;   // [B][H][P][d]
    int H, P;
    long long lo, hi;          // readable stacked rows
    int rows_per_chunk;        // a multiple of DT_ROWS
    float scale_log2;
    float *part_ml, *part_o;
    int *status;
};

__device__ __forceinline__ float dt_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The first N columns (N = 4 or 8: the queries a kernel instance serves) of this warp's lane
// quarter.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
    static_assert(N == 4 || N == 8, "4 or 8 columns");
    if constexpr (N == 4) tmem_ld4(taddr, r);
    else tmem_ld8(taddr, r);
}

// Byte offset of element (row r, column k) in a K-major SW128 tile of 16-bit values whose
// rows hold 64 elements per 128-byte chunk and whose chunks are `chunk_bytes` apart.
__device__ __forceinline__ uint32_t sw128_off(int r, int k, int chunk_bytes) {
    const int c = k >> 6, kc = k & 63;
    return c * chunk_bytes + (r >> 3) * 1024 + (r & 7) * 128 + ((((kc >> 3) ^ (r & 7))) << 4) + (kc & 7) * 2;
}

template <int DH>
__global__ void __launch_bounds__(DT_THREADS, 1)
decode_attn_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const DecodeTcParams p) {
    using C = DtCfg<DH>;
    constexpr int DT_PMAX = C::PMAX;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sKV = smem;                                       // [stage][K tile | V tile]
    uint8_t *sQ = sKV + DT_STAGES * C::STAGE_BYTES;            // B operand of S: [16 q][d]
    uint8_t *sPT = sQ + C::Q_BYTES;                            // 2 x B operand of O: [16 q][128 rows]
    float *red = reinterpret_cast<float *>(sPT + 2 * DT_PT_BYTES);   // [2][4 warps][DT_PMAX]
    uint64_t *bars = reinterpret_cast<uint64_t *>(red + 2 * 4 * DT_PMAX);
    uint64_t *kv_full = bars;                  // [DT_STAGES]
    uint64_t *kv_empty = kv_full + DT_STAGES;  // [DT_STAGES]
    uint64_t *s_full = kv_empty + DT_STAGES;   // [2]
    uint64_t *p_full = s_full + 2;             // [2]
    uint64_t *o_full = p_full + 2;             // [2]
    uint64_t *drain = o_full + 2;              // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = warp_id(), lane = lane_id();
    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z, nch = gridDim.x;
    const long long bh = (long long)b * p.H + h;
    const long long r_begin = p.lo + (long long)chunk * p.rows_per_chunk;
    const long long r_end = min(p.hi + 1, r_begin + p.rows_per_chunk);
    const int ntiles = (int)((r_end - r_begin + DT_ROWS - 1) / DT_ROWS);
    const int P = p.P;

    pdl_trigger();
    // Q (bf16) and zeroed P^T buffers: the rows past P stay zero; for d = 64 the zero block of
    // every stage (never written by TMA)
    for (int i = threadIdx.x; i < (C::Q_BYTES + 2 * DT_PT_BYTES) / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(sQ)[i] = make_uint4(0, 0, 0, 0);
    if (DH == 64)
        for (int i = threadIdx.x; i < DT_STAGES * (DT_CHUNK / 16); i += blockDim.x)
            reinterpret_cast<uint4 *>(sKV + (i / (DT_CHUNK / 16)) * C::STAGE_BYTES + 2 * C::KV_BYTES)[i % (DT_CHUNK / 16)] =
                make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < DT_STAGES; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);   // lane 0 of each softmax warp
            mbar_init(&o_full[i], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, 64);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // one stage of the K/V ring: tile i of the chunk (a fresh stage needs no empty wait)
    auto load_tile = [&](int i) {
        const int st = i % DT_STAGES;
        const int row0 = (int)(r_begin + (long long)i * DT_ROWS);
        uint8_t *dst = sKV + st * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&kv_full[st], 2 * C::KV_BYTES);
        for (int c = 0; c < DH / 64; ++c) {
            tma_load_3d(&tmK, &kv_full[st], dst + c * DT_CHUNK, c * 64, row0, (int)bh);
            tma_load_3d(&tmV, &kv_full[st], dst + C::KV_BYTES + c * DT_CHUNK, c * 64, row0, (int)bh);
        }
    };
    // tiles whose readable rows all predate token t (rows hi-P+1 .. hi are token t's) go out
    // before the wait for the mixing kernel
    int early = 0;
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        const long long first_new = p.hi - P + 1;
        while (early < DT_STAGES && early < ntiles &&
               min(r_begin + (long long)(early + 1) * DT_ROWS, r_end) <= first_new)
            load_tile(early++);
    }
    pdl_wait();   // the mixing kernel's q~ and appended cache rows
    for (int i = threadIdx.x; i < P * DH; i += blockDim.x) {
        const int q = i / DH, c = i % DH;
        *reinterpret_cast<__nv_bfloat16 *>(sQ + sw128_off(q, c, DT_N * 128)) = p.qt[(bh * P + q) * DH + c];
    }
    fence_proxy_async_smem();   // generic writes of Q, P^T and the zero blocks before the tensor core reads them
    __syncthreads();

    if (warp == 4) {
        // ------------------------------- TMA producer -------------------------------
        if (lane == 0) {
            int issued = early;
            for (int i = early; i < ntiles; ++i) {
                const int st = i % DT_STAGES;
                if (!mbar_wait_lazy(&kv_empty[st], ((i / DT_STAGES) & 1) ^ 1, p.status, kSiteDecodeTcProducer,
                                    abort_flag))
                    break;
                load_tile(i);
                ++issued;
            }
            for (int k = issued - DT_STAGES > 0 ? issued - DT_STAGES : 0; k < issued; ++k)
                mbar_wait(&kv_full[k % DT_STAGES], (k / DT_STAGES) & 1, p.status, kSiteDecodeTcProducer, nullptr,
                          kWaitLimitNs);
        }
    } else if (warp == 5) {
        // ------------------------------- MMA issuer ---------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(DT_ROWS, DT_N, 0, 0);   // K rows x Q: both K-major
            constexpr uint32_t idesc_o = idesc_f16_f32(128, DT_N, 1, 0);        // V^T (MN-major) x P^T
            const uint32_t q0 = smem_u32(sQ), pt0 = smem_u32(sPT), kv0 = smem_u32(sKV);
            bool ok = true;
            auto issue_pv = [&](int j) -> bool {
                const int bj = j & 1, st = j % DT_STAGES;
                if (!mbar_wait(&p_full[bj], (j >> 1) & 1, p.status, kSiteDecodeTcMma, abort_flag)) return false;
                tc_fence_after();
                const uint32_t v0 = kv0 + st * C::STAGE_BYTES + C::KV_BYTES;
#pragma unroll
                for (int kk = 0; kk < DT_ROWS / 16; ++kk) {
                    // A = V^T: 16 cached rows of 128-byte d-chunks 16 KB apart (leading offset;
                    // for d = 64 the second chunk is the zero block)
                    const uint64_t a = sdesc_sw128(v0 + kk * 2048, DT_CHUNK, 1024);
                    const uint64_t bd = sdesc_sw128(pt0 + bj * DT_PT_BYTES + (kk / 4) * (DT_N * 128) + (kk % 4) * 32, 16,
                                                    1024);
                    mma_ss(tmem + 32 + bj * 16, a, bd, idesc_o, kk > 0 ? 1u : 0u);
                }
                mma_commit(&o_full[bj]);
                mma_commit(&kv_empty[st]);
                return true;
            };
            for (int i = 0; ok && i < ntiles; ++i) {
                const int st = i % DT_STAGES, bi = i & 1;
                if (!mbar_wait(&kv_full[st], (i / DT_STAGES) & 1, p.status, kSiteDecodeTcMma, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t k0 = kv0 + st * C::STAGE_BYTES;
#pragma unroll
                for (int kk = 0; kk < DH / 16; ++kk) {
                    const uint64_t a = sdesc_sw128(k0 + (kk / 4) * DT_CHUNK + (kk % 4) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(q0 + (kk / 4) * (DT_N * 128) + (kk % 4) * 32, 16, 1024);
                    mma_ss(tmem + bi * 16, a, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[bi]);
                if (i >= 1) ok = issue_pv(i - 1);
            }
            if (ok && ntiles > 0) issue_pv(ntiles - 1);
            mma_commit(drain);
            mbar_wait(drain, 0, p.status, kSiteDecodeTcMma, nullptr, kWaitLimitNs);
        }
    } else {
        // ------------------------------ softmax warps ------------------------------
        const int i_row = warp * 32 + lane;   // TMEM lane: cached row of a tile, output column c
        const uint32_t lane_addr = uint32_t(warp * 32) << 16;
        const float sl2 = p.scale_log2;
        float m[DT_PMAX], l[DT_PMAX], o[DT_PMAX], fprev[DT_PMAX];
#pragma unroll
        for (int q = 0; q < DT_PMAX; ++q) {
            m[q] = -INFINITY;
            l[q] = 0.f;
            o[q] = 0.f;
            fprev[q] = 1.f;
        }
        bool ok = true;
        // fold tile j's O^T into o (its factor: from the running max before tile j to after it)
        auto fold = [&](int j, const float (&f)[DT_PMAX]) -> bool {
            if (!mbar_wait(&o_full[j & 1], (j >> 1) & 1, p.status, kSiteDecodeTc, abort_flag)) return false;
            tc_fence_after();
            uint32_t u[DT_PMAX];
            tmem_ld_cols<DT_PMAX>(tmem + lane_addr + 32 + (j & 1) * 16, u);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < DT_PMAX; ++q) o[q] = fmaf(o[q], f[q], __uint_as_float(u[q]));
            return true;
        };
        for (int i = 0; i < ntiles; ++i) {
            const int bi = i & 1;
            ok = ok && mbar_wait(&s_full[bi], (i >> 1) & 1, p.status, kSiteDecodeTc, abort_flag);
            uint32_t u[DT_PMAX] = {};
            if (ok) {
                tc_fence_after();
                tmem_ld_cols<DT_PMAX>(tmem + lane_addr + bi * 16, u);
                tmem_ld_wait();
            }
            const long long row = r_begin + (long long)i * DT_ROWS + i_row;
            const bool valid = row < r_end;
            float x[DT_PMAX], tm[DT_PMAX];
#pragma unroll
            for (int q = 0; q < DT_PMAX; ++q) {
                x[q] = valid ? __uint_as_float(u[q]) * sl2 : -INFINITY;
                float v = x[q];
#pragma unroll
                for (int o2 = 16; o2 >= 1; o2 >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o2));
                tm[q] = v;
            }
            float *rb = red + bi * 4 * DT_PMAX;
            if (lane == 0) {
#pragma unroll
                for (int q = 0; q < DT_PMAX; ++q) rb[warp * DT_PMAX + q] = tm[q];
            }
            // the tile maxima are shared, and the four warps leave together if a wait gave up
            if (named_bar_or(1, 128, !ok)) {
                ok = false;
                break;
            }
            float f[DT_PMAX];
#pragma unroll
            for (int q = 0; q < DT_PMAX; ++q) {
                const float t4 = fmaxf(fmaxf(rb[q], rb[DT_PMAX + q]), fmaxf(rb[2 * DT_PMAX + q], rb[3 * DT_PMAX + q]));
                const float mn = fmaxf(m[q], t4);
                // nothing readable so far: keep the (zero) sums as they are
                f[q] = mn == -INFINITY ? 1.f : dt_ex2(m[q] - mn);
                const float pq = mn == -INFINITY ? 0.f : dt_ex2(x[q] - mn);
                l[q] = fmaf(l[q], f[q], pq);
                m[q] = mn;
                if (q < P)
                    *reinterpret_cast<__half *>(sPT + bi * DT_PT_BYTES + sw128_off(q, i_row, DT_N * 128)) =
                        __float2half_rn(pq);
            }
            if (!valid) {   // this row's V: cleared, so that p = 0 meets zeros, whatever the cache held
                uint4 *vrow = reinterpret_cast<uint4 *>(sKV + (i % DT_STAGES) * C::STAGE_BYTES + C::KV_BYTES + i_row * 128);
#pragma unroll
                for (int c = 0; c < DH / 64; ++c)
#pragma unroll
                    for (int e = 0; e < 8; ++e) vrow[c * (DT_CHUNK / 16) + e] = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();   // P^T and cleared V rows before the tensor core reads them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[bi]);
            // the previous tile's O^T, one tile behind the MMA (a failed wait is acted on at
            // the next tile's barrier)
            if (i >= 1) ok = fold(i - 1, fprev);
#pragma unroll
            for (int q = 0; q < DT_PMAX; ++q) fprev[q] = f[q];
        }
        if (ok && ntiles > 0) ok = fold(ntiles - 1, fprev);
        // the chunk's normalisers: sum l over the 128 rows
        float lt[DT_PMAX];
#pragma unroll
        for (int q = 0; q < DT_PMAX; ++q) {
            float v = l[q];
#pragma unroll
            for (int o2 = 16; o2 >= 1; o2 >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o2);
            lt[q] = v;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");   // the last tile's maxima are read
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < DT_PMAX; ++q) red[warp * DT_PMAX + q] = lt[q];
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        for (int q = 0; q < P; ++q) {
            const size_t pidx = ((size_t)bh * nch + chunk) * P + q;
            if (i_row < DH) p.part_o[pidx * DH + i_row] = ok ? o[q] : 0.f;
            if (i_row == 0) {
                p.part_ml[pidx * 2] = ok ? m[q] : -INFINITY;
                p.part_ml[pidx * 2 + 1] =
                    ok ? red[q] + red[DT_PMAX + q] + red[2 * DT_PMAX + q] + red[3 * DT_PMAX + q] : 0.f;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

bool decode_tc_supported(int d, int P, const void *Kc, const void *Vc) {
    return ((d == 128 && P <= DtCfg<128>::PMAX) || (d == 64 && P <= DtCfg<64>::PMAX)) &&
           (reinterpret_cast<uintptr_t>(Kc) & 15) == 0 && (reinterpret_cast<uintptr_t>(Vc) & 15) == 0;
}

// Chunks per (b, h): one wave of CTAs (one per SM), whole tiles per chunk.
int decode_tc_chunks(int B, int H, long long rows, int max_chunks, int &rows_per_chunk) {
    long long nch = (long long)device_sm_count() / ((long long)B * H);
    const long long tiles = (rows + DT_ROWS - 1) / DT_ROWS;
    if (nch > tiles) nch = tiles;
    if (nch > max_chunks) nch = max_chunks;
    if (nch < 1) nch = 1;
    const long long tpc = (tiles + nch - 1) / nch;
    rows_per_chunk = (int)(tpc * DT_ROWS);
    return (int)((rows + rows_per_chunk - 1) / rows_per_chunk);
}

template <int DH>
static cudaError_t launch_decode_attn_tc_d(const void *qt, const void *Kc, const void *Vc, int B, int H, int P,
                                          long long cache_rows, long long lo, long long hi, int nch,
                                          int rows_per_chunk, float *part_ml, float *part_o, cudaStream_t st,
                                          int *status) {
    using C = DtCfg<DH>;
    const long long BH = (long long)B * H;
    if (cache_rows >= (1LL << 31) || BH >= (1LL << 31)) return cudaErrorInvalidValue;
    CUtensorMap tmK, tmV;
    const uint64_t dims[3] = {(uint64_t)DH, (uint64_t)cache_rows, (uint64_t)BH};
    const uint64_t strides[2] = {(uint64_t)DH * 2, (uint64_t)cache_rows * DH * 2};
    const uint32_t box[3] = {64, DT_ROWS, 1};
    if (!make_tmap_bf16(&tmK, Kc, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tmV, Vc, 3, dims, strides, box, /*f16=*/true)) return cudaErrorInvalidValue;
    DecodeTcParams p{};
    p.qt = (const __nv_bfloat16 *)qt;
    p.H = H;
    p.P = P;
    p.lo = lo;
    p.hi = hi;
    p.rows_per_chunk = rows_per_chunk;
    p.scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
    p.part_ml = part_ml;
    p.part_o = part_o;
    p.status = status;
    cudaError_t e = cudaFuncSetAttribute(decode_attn_tc<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    // programmatic stream serialization: the launch and prologue overlap the mixing kernel
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nch, H, B);
    cfg.blockDim = dim3(DT_THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_attn_tc<DH>, tmK, tmV, p);
}

cudaError_t launch_decode_attn_tc(const void *qt, const void *Kc, const void *Vc, int B, int H, int d, int P,
                                  long long cache_rows, long long lo, long long hi, int nch, int rows_per_chunk,
                                  float *part_ml, float *part_o, cudaStream_t st, int *status) {
    if (d == 128)
        return launch_decode_attn_tc_d<128>(qt, Kc, Vc, B, H, P, cache_rows, lo, hi, nch, rows_per_chunk, part_ml,
                                            part_o, st, status);
    if (d == 64)
        return launch_decode_attn_tc_d<64>(qt, Kc, Vc, B, H, P, cache_rows, lo, hi, nch, rows_per_chunk, part_ml,
                                           part_o, st, status);
    return cudaErrorInvalidValue;
}

}  // namespace iha
