// k_contract_tc.cu -- unstack + R contraction ("Interleaved Head Attention" section 4,
// Algorithm 1, step "反堆疊與收縮") on tensor cores:
//
//     out[t][h][c] = sum_k R[h][k] * Pbar[t][k][c],   k = h'*P + j  (K = H*P terms),
//
// i.e. per token out_t^T (d x H) = Pbar_t^T (d x H*P) * R^T (H*P x H).  As a tcgen05 MMA the
// accumulator rows are the output columns c (M = 128 rows = 128/d tokens x d), the N = 16
// accumulator columns are the output heads (H <= 16, rows h >= H of R^T are zero) and the
// reduction runs over the K = H*P pseudo-heads, padded to KP (a multiple of 16) by the
// tensor map's zero fill.
//
// Design (sm_103a): persistent CTAs, one per SM.  A tile is G = 128/KP token groups; the
// warp-0 producer TMA-loads each group's Pbar rows as two [KP k][64 c] boxes (128B swizzle,
// an MN-major A operand) into a 4-stage ring; warp 1 issues KP/16 MMAs (M=128, N=16, K=16)
// per group into one of four TMEM accumulators (G x 16 columns each); eight epilogue warps
// (two per lane quarter, half of the groups each) convert the accumulator to bf16 into a
// shared staging buffer laid out as the output and one thread sends the tile -- consecutive
// tokens, contiguous in out -- with one bulk copy.  R^T (bf16, K-major, 128B swizzle) stays
// in shared memory.  HBM-bound: the bytes are Pbar once and out once.
#include <cuda_bf16.h>

#include "iha_internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace iha {

constexpr int CT_M = 128, CT_N = 16, CT_STAGES = 4, CT_NACC = 4;
constexpr int CT_EPI_WARPS = 8, CT_THREADS = 64 + 32 * CT_EPI_WARPS;
constexpr int CT_STAGE_BYTES = 2 * CT_M * 128;      // G groups x 2 boxes x KP rows x 128 B, G*KP = 128
constexpr int CT_R_BYTES = 2 * CT_N * 128;          // R^T: up to 2 K-atoms of [16 rows][64 k]
constexpr int CT_EPI_BAR = 1;

struct ContractParams {
    __nv_bfloat16 *out;
    long long ntok;       // B*N
    int H, HP, d;
    int KP;               // H*P rounded up to 16
    int G;                // token groups per tile (128 / KP)
    int tpg;              // tokens per group (128 / d)
    int tpt;              // tokens per tile (G * tpg)
    int stg_bytes;        // one output staging buffer: tpt * H * d * 2
    int nstg;             // staging buffers (2..4)
    long long num_tiles;
    int *status;
};

inline int contract_smem_fixed() { return CT_R_BYTES + CT_STAGES * CT_STAGE_BYTES + 256 + 1024; }

bool contract_tc_fits(const Shape &sh) {
    return (sh.d == 64 || sh.d == 128) && sh.H <= CT_N && sh.H * sh.P <= CT_M;
}

__global__ void __launch_bounds__(CT_THREADS, 1)
contract_tc(const __grid_constant__ CUtensorMap tmP, const float *__restrict__ R, const ContractParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;                                   // [CT_STAGES][CT_STAGE_BYTES]
    uint8_t *sR = sA + CT_STAGES * CT_STAGE_BYTES;        // R^T, 1024-aligned
    uint8_t *sStg = sR + CT_R_BYTES;                      // [nstg][stg_bytes]
    uint64_t *full = reinterpret_cast<uint64_t *>(sStg + p.nstg * p.stg_bytes);
    uint64_t *empty = full + CT_STAGES;
    uint64_t *tfull = empty + CT_STAGES;
    uint64_t *tempty = tfull + CT_NACC;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + CT_NACC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = warp_id(), lane = lane_id();
    const int H = p.H, HP = p.HP, d = p.d, G = p.G;

    // R^T as the K-major B operand: row n = output head h, column k = pseudo-head h'*P + j;
    // K-atom a = k / 64 is a [16 rows][128 B] block at a*2 KB; in a row, 16-byte chunk
    // (k%64)/8 sits at position ((k%64)/8) ^ (n%8).  Zero outside h < H, k < H*P.
    for (int idx = threadIdx.x; idx < 2 * CT_N * 8; idx += blockDim.x) {
        const int a = idx / (CT_N * 8), n = (idx / 8) % CT_N, cp = idx % 8;
        const int kc = cp ^ (n % 8);            // logical 16-byte chunk held at position cp
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const int k = a * 64 + kc * 8 + e;
            const float x0 = (n < H && k < HP) ? R[(size_t)n * HP + k] : 0.f;
            const float x1 = (n < H && k + 1 < HP) ? R[(size_t)n * HP + k + 1] : 0.f;
            w[e / 2] = pack_bf16x2(x0, x1);
        }
        *reinterpret_cast<uint4 *>(sR + a * (CT_N * 128) + (n / 8) * 1024 + (n % 8) * 128 + cp * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();   // generic-proxy writes of R^T before the tensor core reads them
    if (threadIdx.x == 0) {
        for (int i = 0; i < CT_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int a = 0; a < CT_NACC; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 32 * CT_EPI_WARPS);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&tmP);
    if (warp == 1) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int box_bytes = p.KP * 128;   // one [KP k][64 c] box

    if (warp == 0) {
        // ------------------------------- TMA producer -------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (long long tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
                if (!mbar_wait_lazy(&empty[stage], phase ^ 1, p.status, kSiteContractProducer, abort_flag)) break;
                mbar_arrive_expect_tx(&full[stage], G * 2 * box_bytes);
                // group g, box i: d=128 -> token tile*tpt + g, columns i*64..; d=64 -> token
                // tile*tpt + 2g + i, columns 0..63 (tokens past the end read as zero)
                for (int g = 0; g < G; ++g)
                    for (int i = 0; i < 2; ++i) {
                        const long long t = tile * p.tpt + (long long)g * p.tpg + (d == 64 ? i : 0);
                        tma_load_3d(&tmP, &full[stage], sA + stage * CT_STAGE_BYTES + (g * 2 + i) * box_bytes,
                                    d == 128 ? i * 64 : 0, 0, (int)t);
                    }
                if (++stage == CT_STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------- MMA issuer ---------------------------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(CT_M, CT_N, 1, 0);   // A MN-major, B K-major
            const uint32_t hi = sdesc_sw128_hi(1024);                       // 8 k-rows 1 KB apart
            const uint32_t r_lo = sdesc_sw128_lo(smem_u32(sR), 16);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            for (long long tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
                const int acc = it % CT_NACC;
                if (!mbar_wait(&tempty[acc], ((it / CT_NACC) & 1) ^ 1, p.status, kSiteContractMma, abort_flag)) break;
                if (!mbar_wait(&full[stage], phase, p.status, kSiteContractMma, abort_flag)) break;
                tc_fence_after();
                for (int g = 0; g < G; ++g) {
                    // A: the group's two boxes are the two 64-row chunks of M (leading byte
                    // offset = one box); k-step s starts 16 rows (2 KB) further
                    const uint32_t a_lo =
                        sdesc_sw128_lo(smem_u32(sA + stage * CT_STAGE_BYTES + g * 2 * box_bytes), box_bytes);
                    for (int s = 0; s < p.KP / 16; ++s) {
                        // B: K-atom s/4, 32 bytes per k-step inside it
                        const uint32_t b_lo = r_lo + (((s / 4) * (CT_N * 128) + (s % 4) * 32) >> 4);
                        mma_ss_w(tmem + acc * (G * CT_N) + g * CT_N, a_lo + ((s * 16 * 128) >> 4), b_lo, hi, idesc,
                                 s > 0 ? 1u : 0u);
                    }
                }
                mma_commit(&empty[stage]);
                mma_commit(&tfull[acc]);
                if (++stage == CT_STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else {
        // ------------------------------- epilogue -----------------------------------
        // warps 2..9: lane quarter q = warp % 4 (accumulator rows 32q..32q+31), half hf of
        // the groups.  Row r: d=128 -> column c = r of the group's token; d=64 -> token
        // 2g + r/64, column r%64.
        const int q = warp & 3, hf = (warp - 2) / 4;
        const int r = q * 32 + lane;
        const int tsub = d == 64 ? r / 64 : 0, c = r % d;
        const int gpe = (G + 1) / 2;                     // groups per epilogue half
        const bool issuer = warp == 2 && lane == 0;
        int it = 0, sb = 0;
        for (long long tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
            const int acc = it % CT_NACC;
            uint8_t *stg = sStg + sb * p.stg_bytes;
            if (++sb == p.nstg) sb = 0;
            const bool ok = mbar_wait(&tfull[acc], (it / CT_NACC) & 1, p.status, kSiteContractEpilogue, abort_flag);
            if (ok) {
                tc_fence_after();
                for (int g = hf * gpe; g < G && g < (hf + 1) * gpe; ++g) {
                    uint32_t u[16];
                    tmem_ld16(tmem + acc * (G * CT_N) + g * CT_N + (uint32_t(q * 32) << 16), u);
                    tmem_ld_wait();
                    // token g*tpg + tsub of the tile, heads 0..H-1 at column c
                    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(stg) +
                                       ((size_t)(g * p.tpg + tsub) * H) * d + c;
#pragma unroll
                    for (int h = 0; h < CT_N; ++h)
                        if (h < H) o[(size_t)h * d] = __float2bfloat16_rn(__uint_as_float(u[h]));
                }
                tc_fence_before();
                mbar_arrive(&tempty[acc]);   // the accumulator has been read
                fence_proxy_async_smem();    // staging writes before the bulk copy reads them
            }
            // Before the barrier the issuer makes sure the buffer of the next tile is free
            // again (its copy, tile it+1-nstg, is among all but the newest nstg-2 groups),
            // so that after it every thread may fill it.
            if (issuer) bulk_wait_read(p.nstg - 2);
            if (named_bar_or(CT_EPI_BAR, 32 * CT_EPI_WARPS, !ok)) break;   // a uniform decision
            if (issuer) {
                const long long t0 = tile * p.tpt;
                long long n = p.ntok - t0;
                if (n > p.tpt) n = p.tpt;
                bulk_store(p.out + t0 * H * d, stg, (uint32_t)(n * H * d * 2));
                bulk_commit();
            }
        }
        if (issuer) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

cudaError_t launch_contract_tc(const void *Pbar, const float *R, const Shape &sh, void *out, cudaStream_t st,
                               int *status) {
    if (!contract_tc_fits(sh)) return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(out) & 15) != 0) return cudaErrorInvalidValue;   // bulk-copy alignment
    const long long ntok = (long long)sh.B * sh.N;
    ContractParams p{};
    p.out = (__nv_bfloat16 *)out;
    p.ntok = ntok;
    p.H = sh.H;
    p.HP = sh.H * sh.P;
    p.d = sh.d;
    p.KP = (p.HP + 15) / 16 * 16;
    p.G = CT_M / p.KP;                       // KP <= 128
    if (p.G > 4) p.G = 4;                    // 4 groups x 16 columns per accumulator
    p.tpg = CT_M / sh.d;
    p.tpt = p.G * p.tpg;
    p.stg_bytes = p.tpt * sh.H * sh.d * 2;
    p.nstg = 3;
    p.num_tiles = (ntok + p.tpt - 1) / p.tpt;
    p.status = status;
    CUtensorMap tmP;
    {
        // Pbar [t][k][c] as (c, k, t); boxes of [KP k][64 c], k >= H*P read as zero
        const uint64_t dims[3] = {(uint64_t)sh.d, (uint64_t)p.HP, (uint64_t)ntok};
        const uint64_t strides[2] = {(uint64_t)sh.d * 2, (uint64_t)p.HP * sh.d * 2};
        const uint32_t box[3] = {64, (uint32_t)p.KP, 1};
        if (!make_tmap_bf16(&tmP, Pbar, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    const int smem = contract_smem_fixed() + p.nstg * p.stg_bytes;
    cudaError_t e = cudaFuncSetAttribute(contract_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const long long grid = p.num_tiles < device_sm_count() ? p.num_tiles : device_sm_count();
    if (grid == 0) return cudaSuccess;
    contract_tc<<<(unsigned)grid, CT_THREADS, smem, st>>>(tmP, R, p);
    return cudaGetLastError();
}

}  // namespace iha
