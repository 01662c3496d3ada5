// Grouped MXFP4 expert GEMM on the 5th-generation tensor cores (tcgen05 + TMA).
//
// D[m, n] = sum_k W[m, k] B[n, k] for one expert's weight rows m (M tile of
// 128) and its token rows n (N tile <= BN), where W is stored MXFP4 (two E2M1
// codes per byte, low nibble first, one E8M0 exponent per 32 values: "Kimi K3,
// as released", Gate 3 section) and B holds f16 activation rows.
//
// Exact decoding into f16: each row m is scaled by 2^(emax_m - 127), emax_m =
// the row's largest exponent byte, so a block with exponent e becomes
// E2M1 x 2^(e - emax_m) in f16 -- exact for e >= emax_m - 23 -- and the factor
// 2^(emax_m - 127) is applied to the fp32 accumulator in the epilogue.
//
// A packed stage feeds four 64-K MMA sub-steps; activation tiles have their
// own ring so packed prefetch never waits on them.
//
// Roles (one CTA per SM, persistent over the tile list):
//   warp 0            TMA producer of the packed FP4 tiles: 128 rows x 128 bytes
//                     (256 K values) per stage, per-expert tensor maps, 128-byte swizzle
//   warp 2            TMA producer of the f16 activation sub-tiles (64 K x N rows)
//   warp 1            TMEM allocator and the single MMA-issuing thread
//   warps 4..4+4*NMAT dequant: one thread per weight row, FP4 -> f16 into the
//                     128-byte-swizzled K-major layout the MMA reads, or into TMEM
//   last 8 or 12      epilogue: TMEM -> registers -> scaled outputs, two or three
//   warps             warps per TMEM lane quarter taking 16-token chunks in turn
// Every wait is bounded; on expiry the CTA records K3MOE_ERR_TIMEOUT, drains
// its copies and MMAs, frees TMEM and returns.
#pragma once
#include <cudaTypedefs.h>

#include "k3moe_internal.h"
#include "ptx.cuh"
#include "wait.cuh"

namespace k3 {

enum ExpertOut { OUT_GLU_F16 = 0, OUT_BF16 = 1, OUT_BF16_ADD = 2 };

struct ExpertGemmArgs {
    const CUtensorMap *amaps;        // global: maps of group g, matrix m at amaps[g * amap_stride + amap_off[m]]
    int amap_stride;
    int amap_off[2];
    const uint8_t *const *scales[2]; // device tables [groups] of scale arrays [rows, K/32]
    const uint8_t *rowmax[2];        // [groups * rows] per-row max exponent byte
    int rows;                        // weight rows per group (multiple of 128)
    int K;                           // reduction length (multiple of 512)
    const int4 *tiles;               // (group, row0, nrows, -) per token tile
    const int *n_tiles;              // device count of tiles
    const float *rscale;             // per B-row factor: GLU, of the inputs (h scaling); other modes, of the outputs; or nullptr
    const float *ascale;             // GLU: per B-row power of two 2^k the f16 output is divided by, or nullptr
    void *out;                       // GLU: f16 [R, rows]; BF16 and BF16_ADD: BF16 [R, rows]
    const float *addend;             // BF16_ADD: fp32 [R, rows] added before the rounding to BF16
    int *status;
    uint32_t spin_limit;
    K3Act act;                       // GLU activation
    int a8;                          // GLU: 1 rounds the output to MXFP8 (blocks of 32 rows per token)
};

// Epilogue variants of the GLU mode (a template argument of the kernel).
enum { EPI_SILU = 0, EPI_SITU = 1, EPI_A8 = 2 };

constexpr int EX_BM = 128;           // weight rows per tile (MMA M)
constexpr int EX_KP = 256;           // K per packed stage (128-byte FP4 rows)
constexpr int EX_KS = 64;            // K per MMA sub-step (one 128-byte f16 row)
constexpr int EX_NSUB = EX_KP / EX_KS;
constexpr int EX_BBOX = 16;          // activation rows per small TMA box: a tile loads only the rows it needs,
constexpr int EX_BBIG = 64;          // as 64-row boxes plus at most three 16-row boxes
constexpr int EX_BBOX_BYTES = EX_BBOX * EX_KS * 2;

// Tensor maps of one f16 activation matrix [rows, K] with 64- and 16-row boxes.
struct ActMaps {
    CUtensorMap big, small;
};

template <int NMAT, int BN, int NS, int NB, int NA, bool ATMEM = false>
struct ExpertSmem {
    static constexpr int PK_BYTES = EX_BM * EX_KP / 2;      // 16384 packed bytes per matrix
    static constexpr int B_BYTES = BN * EX_KS * 2;          // activation sub-tile
    static constexpr int A_BYTES = EX_BM * EX_KS * 2;       // 16384 f16 tile
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + (ATMEM ? 0 : NA * NMAT * A_BYTES);   // ATMEM: A lives in TMEM
    static constexpr int OFF_PK = OFF_B + NB * B_BYTES;
    static constexpr int OFF_BAR = OFF_PK + NS * NMAT * PK_BYTES;
    static constexpr int N_BAR = 2 * NS + 2 * NB + 2 * NA + 4 + 1 + 2;
    static constexpr int OFF_RS = (OFF_BAR + N_BAR * 8 + 16 + 15) & ~15;   // after the tmem holder and abort flag; 16-byte reads
    // per-token factors (fp32), then the GLU output divisors' exponents: as fp32 factors
    // already multiplied into the input factor (RSA) where shared memory allows, else as bytes
    static constexpr bool RSA = OFF_RS + BN * 8 + 1024 <= 227 * 1024;
    static constexpr int BYTES = OFF_RS + BN * 4 + (RSA ? BN * 4 : BN) + 1024;   // + align slack
};

__device__ __forceinline__ uint32_t f16_pow2_bits(int d)
{
    // 2^d as f16 bits for d <= 0 (subnormals for d < -14, zero below -24)
    if (d >= -14) return (uint32_t)(d + 15) << 10;
    if (d >= -24) return 1u << (d + 24);
    return 0u;
}

// Threads per CTA: 4 control warps, 4 dequant warps per weight matrix (one thread
// per weight row) and the epilogue warps, ex_nepi of them (two or three per TMEM lane
// quarter, taking 16-token chunks in turn).  The kernels with one accumulator set, whose
// drain holds back the next job's MMAs, take three per quarter where their registers
// fit the 80 a thread gets at 768 threads: the 192-token kernels (with their dequant
// warps reading each sub-step's bytes when needed) and the SiLU GLU kernel of 256-token
// tiles.  The others keep two.
__host__ __device__ constexpr int ex_nepi(int bn, int mode, int epi)
{
    return bn == 192 || (bn == 256 && mode == 0 && epi == 0) ? 12 : 8;
}
__host__ __device__ constexpr int ex_threads(int nmat, int nepi) { return (4 + 4 * nmat + nepi) * 32; }

template <int NMAT, int BN, int NS, int NB, int NA, int NACC, int MODE, bool ATMEM = false, int EPI = 0>
__global__ void __launch_bounds__(ex_threads(NMAT, ex_nepi(BN, MODE, EPI)), 1)
expert_gemm_kernel(const __grid_constant__ ActMaps bmaps, const ExpertGemmArgs args)
{
    griddep_enter();
    using SM = ExpertSmem<NMAT, BN, NS, NB, NA, ATMEM>;
    constexpr int DQW = 4, NEPI = ex_nepi(BN, MODE, EPI);
    constexpr int EPI_WARP0 = 4 + DQW * NMAT;
    // TMEM columns: NACC accumulator sets (2: the epilogue overlaps the next tile),
    // then with ATMEM the NA x NMAT decoded A sub-tiles (128 lanes x 32 columns each)
    constexpr int ACOL0 = NACC * NMAT * BN;
    constexpr int COLS = ACOL0 + (ATMEM ? NA * NMAT * EX_KS / 2 : 0);
    constexpr uint32_t TMEM_COLS = (COLS <= 32) ? 32 : (COLS <= 64) ? 64 : (COLS <= 128) ? 128
                                 : (COLS <= 256) ? 256 : 512;
    static_assert(COLS <= 512 && (NACC == 1 || NACC == 2), "TMEM columns");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(smem + SM::OFF_BAR);
    uint64_t *pfull = bars, *pempty = pfull + NS;
    uint64_t *bfull = pempty + NS, *bempty = bfull + NB;
    uint64_t *afull = bempty + NB, *aempty = afull + NA;
    uint64_t *tfull = aempty + NA, *tempty = tfull + 2, *drain = tempty + 2;
    uint64_t *rsfull = drain + 1, *rsempty = drain + 2;      // per-token factor staging (epilogue only)
    uint32_t *tmem_holder = (uint32_t *)(drain + 3);
    volatile int *abort_flag = (volatile int *)(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = args.K, nkp = K / EX_KP;
    // SiLU: the GLU output divisor 2^-k is staged multiplied into the up branch's input factor
    // (SiTU soft-limits the up branch, so its factor stays apart)
    constexpr bool RSA = SM::RSA && MODE == OUT_GLU_F16 && EPI == EPI_SILU;
    // GLU: the two matrices share the job's 128 rows.  Otherwise NMAT = 2 takes two
    // 128-row blocks of the same matrix, so each activation tile feeds 256 rows.
    constexpr bool ROWPAIR = MODE != OUT_GLU_F16 && NMAT == 2;
    constexpr int JOB_ROWS = ROWPAIR ? 2 * EX_BM : EX_BM;
    const int m_tiles = args.rows / JOB_ROWS;
    const int total = __ldg(args.n_tiles) * m_tiles;
    const uint32_t lim = args.spin_limit;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(pfull + i), 1);
            mbar_init(smem_u32(pempty + i), DQW * NMAT);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(smem_u32(bfull + i), 1);
            mbar_init(smem_u32(bempty + i), 1);
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(smem_u32(afull + i), 4 * NMAT);
            mbar_init(smem_u32(aempty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(tfull + i), 1);
            mbar_init(smem_u32(tempty + i), NEPI);
        }
        mbar_init(smem_u32(drain), 1);
        mbar_init(smem_u32(rsfull), NEPI * 32);
        mbar_init(smem_u32(rsempty), NEPI);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA: packed FP4 tiles
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            uint32_t pit = 0;
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
                const int4 tile = __ldg(args.tiles + t / m_tiles);
                const int g = tile.x, m0 = (t % m_tiles) * JOB_ROWS;
                const CUtensorMap *am0 = args.amaps + (size_t)g * args.amap_stride + args.amap_off[0];
                const CUtensorMap *am1 = args.amaps + (size_t)g * args.amap_stride + args.amap_off[NMAT - 1];
                bool ok = true;
                for (int s = 0; s < nkp; ++s, ++pit) {
                    const int slot = pit % NS;
                    if (!role_wait(smem_u32(pempty + slot), ((pit / NS) & 1) ^ 1, abort_flag, lim,
                                   args.status, 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(pfull + slot);
                    mbar_expect_tx(fb, NMAT * SM::PK_BYTES);
                    uint8_t *pk = smem + SM::OFF_PK + slot * NMAT * SM::PK_BYTES;
                    tma_load_2d_hint(smem_u32(pk), am0, fb, s * (EX_KP / 2), m0, pol_w);
                    if (NMAT == 2)
                        tma_load_2d_hint(smem_u32(pk + SM::PK_BYTES), am1, fb, s * (EX_KP / 2),
                                         m0 + (ROWPAIR ? EX_BM : 0), pol_w);
                }
                if (!ok) break;
            }
            drain_ring(pfull, pit, NS);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ TMA: activation sub-tiles
        if (lane == 0) {
            prefetch_tmap(&bmaps.big);
            prefetch_tmap(&bmaps.small);
            const uint64_t pol_b = policy_evict_last();
            uint32_t bit = 0;
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
                const int4 tile = __ldg(args.tiles + t / m_tiles);
                const int row0 = tile.y;
                const int n16 = min(BN, max(16, (tile.z + 15) & ~15)) / EX_BBOX;    // = MMA N / 16
                const int nbig = n16 / (EX_BBIG / EX_BBOX), nsmall = n16 % (EX_BBIG / EX_BBOX);
                bool ok = true;
                for (int ks = 0; ks < K / EX_KS; ++ks, ++bit) {
                    const int slot = bit % NB;
                    if (!role_wait(smem_u32(bempty + slot), ((bit / NB) & 1) ^ 1, abort_flag, lim,
                                   args.status, 8)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(bfull + slot);
                    mbar_expect_tx(fb, n16 * EX_BBOX_BYTES);
                    const uint32_t dst = smem_u32(smem + SM::OFF_B + slot * SM::B_BYTES);
                    for (int b = 0; b < nbig; ++b)
                        tma_load_2d_hint(dst + b * (EX_BBIG * EX_KS * 2), &bmaps.big, fb, ks * EX_KS,
                                         row0 + b * EX_BBIG, pol_b);
                    for (int b = 0; b < nsmall; ++b)
                        tma_load_2d_hint(dst + nbig * (EX_BBIG * EX_KS * 2) + b * EX_BBOX_BYTES, &bmaps.small, fb,
                                         ks * EX_KS, row0 + nbig * EX_BBIG + b * EX_BBOX, pol_b);
                }
                if (!ok) break;
            }
            drain_ring(bfull, bit, NB);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t bit = 0, ait = 0, tc = 0;
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++tc) {
                const int4 tile = __ldg(args.tiles + t / m_tiles);
                const int nrows = tile.z;
                const int nmma = min(BN, max(16, (nrows + 15) & ~15));
                const uint32_t idesc = idesc_f16(EX_BM, nmma, 0);
                const int acc = (int)(tc % NACC);
                if (!role_wait(smem_u32(tempty + acc), ((tc / NACC) & 1) ^ 1, abort_flag, lim, args.status, 2))
                    break;
                tc_fence_after();
                const uint32_t dcol = tmem + acc * NMAT * BN;
                bool ok = true;
                for (int ks = 0; ks < K / EX_KS; ++ks, ++bit, ++ait) {
                    const int bslot = bit % NB, aslot = ait % NA;
                    if (!role_wait(smem_u32(bfull + bslot), (bit / NB) & 1, abort_flag, lim, args.status, 3) ||
                        !role_wait(smem_u32(afull + aslot), (ait / NA) & 1, abort_flag, lim, args.status, 4)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(smem + SM::OFF_B + bslot * SM::B_BYTES));
#pragma unroll
                    for (int mt = 0; mt < NMAT; ++mt) {
                        if (ATMEM) {
                            const uint32_t acol = tmem + ACOL0 + (aslot * NMAT + mt) * (EX_KS / 2);
#pragma unroll
                            for (int kk = 0; kk < EX_KS / 16; ++kk)   // 16 K = 8 columns
                                tc_mma_f16_ts(dcol + mt * BN, acol + 8 * kk, bdesc + 2 * kk, idesc,
                                              (ks > 0 || kk > 0) ? 1u : 0u);
                        } else {
                            const uint64_t adesc =
                                smem_desc_sw128(smem_u32(smem + SM::OFF_A + (aslot * NMAT + mt) * SM::A_BYTES));
#pragma unroll
                            for (int kk = 0; kk < EX_KS / 16; ++kk)
                                tc_mma_f16(dcol + mt * BN, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                                           (ks > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    tc_commit(smem_u32(bempty + bslot));
                    tc_commit(smem_u32(aempty + aslot));
                }
                if (!ok) break;
                tc_commit(smem_u32(tfull + acc));
            }
            // all issued MMAs complete before TMEM is released
            tc_commit(smem_u32(drain));
            mbar_wait(smem_u32(drain), 0, 0xFFFFFFFFu);
        }
    } else if (warp >= 4 && warp < EPI_WARP0) {
        // ------------------------------------------------------------ dequant FP4 -> f16
        const int d = warp - 4;
        const int mat = d / DQW;
        const int r = (d % DQW) * 32 + lane;               // weight row within the tile
        const int kblk = K / 32;
        uint32_t pit = 0, ait = 0;
        // 16 scale bytes cover two packed stages; the next group is read one
        // group ahead, and the next tile's first group during the current
        // tile's last group
        int t = blockIdx.x;
        const uint8_t *srow = nullptr;
        int emax = 0, emax_next = 0;
        uint4 sc_cur = make_uint4(0, 0, 0, 0), sc_next = sc_cur;
        if (t < total) {
            const int4 tile = __ldg(args.tiles + t / m_tiles);
            const int row = (t % m_tiles) * JOB_ROWS + (ROWPAIR ? mat * EX_BM : 0) + r;
            emax = __ldg(args.rowmax[mat] + (size_t)tile.x * args.rows + row);
            srow = args.scales[mat][tile.x] + (size_t)row * kblk;
            sc_cur = __ldg(reinterpret_cast<const uint4 *>(srow));
        }
        for (; t < total && !*abort_flag; t += gridDim.x) {
            const int tn = t + gridDim.x;
            const uint8_t *srow_next = nullptr;
            if (tn < total) {
                const int4 tile = __ldg(args.tiles + tn / m_tiles);
                const int row = (tn % m_tiles) * JOB_ROWS + (ROWPAIR ? mat * EX_BM : 0) + r;
                srow_next = args.scales[mat][tile.x] + (size_t)row * kblk;
                emax_next = __ldg(args.rowmax[mat] + (size_t)tile.x * args.rows + row);
            }
            bool ok = true;
            for (int s = 0; s < nkp; ++s, ++pit) {
                if ((s & 1) == 0) {
                    if (s > 0) sc_cur = sc_next;
                    if (s + 2 < nkp) sc_next = __ldg(reinterpret_cast<const uint4 *>(srow) + (s >> 1) + 1);
                    else if (srow_next) sc_next = __ldg(reinterpret_cast<const uint4 *>(srow_next));
                }
                const int slot = pit % NS;
                if (!role_wait(smem_u32(pfull + slot), (pit / NS) & 1, abort_flag, lim, args.status, 5)) {
                    ok = false;
                    break;
                }
                // the row's 128 packed bytes (128-byte swizzle of the TMA box)
                const uint8_t *pk = smem + SM::OFF_PK + (slot * NMAT + mat) * SM::PK_BYTES + r * 128;
                // A in shared memory: the row's 128 bytes are read at once and the stage is
                // released; ATMEM: each sub-step reads its own 32 bytes (fewer live registers,
                // which leaves room for more epilogue warps) and the last one releases it
                uint4 c[ATMEM ? 1 : 8];
                if constexpr (!ATMEM) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) c[j] = *reinterpret_cast<const uint4 *>(pk + 16 * (j ^ (r & 7)));
                    // the stage is refilled by TMA (async proxy): order these generic reads before it
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(pempty + slot));
                }
                const uint32_t sw_lo = (s & 1) ? sc_cur.z : sc_cur.x;
                const uint32_t sw_hi = (s & 1) ? sc_cur.w : sc_cur.y;
#pragma unroll
                for (int q = 0; q < EX_NSUB; ++q, ++ait) {
                    const uint32_t sw32 = q < 2 ? sw_lo : sw_hi;
                    const int e0 = (sw32 >> (16 * (q & 1))) & 0xFF, e1 = (sw32 >> (16 * (q & 1) + 8)) & 0xFF;
                    const uint32_t f0 = f16_pow2_bits(e0 - emax), f1 = f16_pow2_bits(e1 - emax);
                    const __half2 s0 = __halves2half2(__ushort_as_half((unsigned short)f0),
                                                      __ushort_as_half((unsigned short)f0));
                    const __half2 s1 = __halves2half2(__ushort_as_half((unsigned short)f1),
                                                      __ushort_as_half((unsigned short)f1));
                    const int aslot = ait % NA;
                    if (!role_wait(smem_u32(aempty + aslot), ((ait / NA) & 1) ^ 1, abort_flag, lim,
                                   args.status, 6)) {
                        ok = false;
                        break;
                    }
                    uint8_t *arow = smem + SM::OFF_A + (aslot * NMAT + mat) * SM::A_BYTES + r * 128;
                    uint4 lo, hi;
                    if constexpr (ATMEM) {
                        lo = *reinterpret_cast<const uint4 *>(pk + 16 * ((2 * q) ^ (r & 7)));
                        hi = *reinterpret_cast<const uint4 *>(pk + 16 * ((2 * q + 1) ^ (r & 7)));
                        if (q == EX_NSUB - 1) {
                            fence_proxy_async_smem();       // before the stage's refill by TMA
                            __syncwarp();
                            if (lane == 0) mbar_arrive(smem_u32(pempty + slot));
                        }
                    } else {
                        lo = c[2 * q];
                        hi = c[2 * q + 1];
                    }
                    const uint32_t words[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                    uint32_t tv[ATMEM ? 32 : 1];                 // ATMEM: the row's 64 values in K order
                    if (ATMEM) tc_fence_after();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t h0, h1, h2, h3;
                        asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
                            "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
                            "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
                            : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
                            : "r"(words[j]));
                        const __half2 sc = j < 4 ? s0 : s1;
                        __half2 q0 = __hmul2(*reinterpret_cast<__half2 *>(&h0), sc);
                        __half2 q1 = __hmul2(*reinterpret_cast<__half2 *>(&h1), sc);
                        __half2 q2 = __hmul2(*reinterpret_cast<__half2 *>(&h2), sc);
                        __half2 q3 = __hmul2(*reinterpret_cast<__half2 *>(&h3), sc);
                        uint4 v;
                        v.x = *reinterpret_cast<uint32_t *>(&q0);
                        v.y = *reinterpret_cast<uint32_t *>(&q1);
                        v.z = *reinterpret_cast<uint32_t *>(&q2);
                        v.w = *reinterpret_cast<uint32_t *>(&q3);
                        if (ATMEM) {
                            tv[(4 * j + 0) % (ATMEM ? 32 : 1)] = v.x;
                            tv[(4 * j + 1) % (ATMEM ? 32 : 1)] = v.y;
                            tv[(4 * j + 2) % (ATMEM ? 32 : 1)] = v.z;
                            tv[(4 * j + 3) % (ATMEM ? 32 : 1)] = v.w;
                        } else {
                            *reinterpret_cast<uint4 *>(arow + 16 * (j ^ (r & 7))) = v;
                        }
                    }
                    if (ATMEM) {
                        // lanes 32 (warp % 4) .. +31 = rows r of this warp; columns of A slot (aslot, mat)
                        const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + ACOL0 +
                                            (aslot * NMAT + mat) * (EX_KS / 2);
                        tmem_st16(ta, tv);
                        tmem_st16(ta + 16, tv + (ATMEM ? 16 : 0));
                        tc_wait_st();
                        tc_fence_before();
                    } else {
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(afull + aslot));
                }
                if (!ok) break;
            }
            if (!ok) break;
            srow = srow_next;
            emax = emax_next;
            sc_cur = sc_next;
        }
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                            // TMEM lanes 32q .. 32q+31
        const int half = (warp - EPI_WARP0) >> 2;          // chunks c with c % (NEPI / 4) == half
        const int eth = (warp - EPI_WARP0) * 32 + lane;
        const int r = q * 32 + lane;
        float *srs = reinterpret_cast<float *>(smem + SM::OFF_RS);
        uint32_t tc = 0;
        bool bad = false;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++tc) {
            const int4 tile = __ldg(args.tiles + t / m_tiles);
            const int g = tile.x, row0 = tile.y, nrows = tile.z;
            const int m0 = (t % m_tiles) * JOB_ROWS, row = m0 + r;
            const int row1 = row + (ROWPAIR ? EX_BM : 0);          // output row of matrix slot 1
            const int acc = (int)(tc % NACC);
            const float fw0 = e8m0_to_f32(__ldg(args.rowmax[0] + (size_t)g * args.rows + row));
            const float fw1 = NMAT == 2 ? e8m0_to_f32(__ldg(args.rowmax[NMAT - 1] + (size_t)g * args.rows + row1)) : 0.f;
            {
                // the tile's per-token factors, staged while its MMAs run, once the
                // epilogue warps have finished with the previous tile's: the input
                // factor (GLU) or output factor (other modes), and for the GLU the
                // inverse 2^-k of the power of two its f16 outputs are divided by
                if (tc > 0 && !role_wait(smem_u32(rsempty), (tc - 1) & 1, abort_flag, lim, args.status, 9)) break;
                uint8_t *sas = reinterpret_cast<uint8_t *>(srs + BN);
                for (int i = eth; i < nrows; i += NEPI * 32) {
                    srs[i] = args.rscale ? __ldg(args.rscale + row0 + i) : 1.f;
                    if (MODE == OUT_GLU_F16) {   // k of the output's divisor 2^k
                        const uint32_t k = args.ascale ? (__float_as_uint(__ldg(args.ascale + row0 + i)) >> 23) - 127 : 0;
                        if constexpr (RSA)
                            reinterpret_cast<float *>(sas)[i] = srs[i] * __uint_as_float((127u - k) << 23);
                        else
                            sas[i] = (uint8_t)k;
                    }
                }
                mbar_arrive(smem_u32(rsfull));
                if (!role_wait(smem_u32(rsfull), tc & 1, abort_flag, lim, args.status, 9)) break;
            }
            if (!role_wait(smem_u32(tfull + acc), (tc / NACC) & 1, abort_flag, lim, args.status, 7)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + acc * NMAT * BN;
            const int nchunks = (nrows + 15) >> 4;
            // the GLU variant (SiLU, SiTU, A8) is a template argument: each kernel carries one
            constexpr int KIND = MODE == OUT_GLU_F16 ? EPI : EPI_SILU;
            for (int c = half; c < nchunks; c += NEPI / 4) {
                // BF16_ADD: the chunk's addends are read before the TMEM loads, so
                // their latency overlaps them
                float ad0[16], ad1[16];
                if (MODE == OUT_BF16_ADD) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = c * 16 + j;
                        const float *ar = args.addend + (size_t)(row0 + (n < nrows ? n : 0)) * args.rows;
                        ad0[j] = ar[row];
                        ad1[j] = ROWPAIR ? ar[row1] : 0.f;
                    }
                }
                // SiLU and SiTU: the chunk's 16 per-token factors, read from shared memory
                // before any of the chunk's global stores (through generic pointers the
                // compiler cannot order a shared read above an earlier store); A8 reads them
                // in its first pass, which stores nothing
                float rsv[16], asv[16];
                if constexpr (MODE != OUT_GLU_F16 || KIND != EPI_A8) {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float4 f = reinterpret_cast<const float4 *>(srs + c * 16)[w];
                        rsv[4 * w] = f.x;
                        rsv[4 * w + 1] = f.y;
                        rsv[4 * w + 2] = f.z;
                        rsv[4 * w + 3] = f.w;
                    }
                }
                if constexpr (MODE == OUT_GLU_F16 && RSA) {
                    // the input factor times 2^-k, for the up branch
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float4 f = reinterpret_cast<const float4 *>(srs + BN + c * 16)[w];
                        asv[4 * w] = f.x;
                        asv[4 * w + 1] = f.y;
                        asv[4 * w + 2] = f.z;
                        asv[4 * w + 3] = f.w;
                    }
                } else if constexpr (MODE == OUT_GLU_F16 && KIND != EPI_A8) {
                    const uint4 e = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(srs + BN) + c * 16);
                    const uint32_t ew[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
                    for (int j = 0; j < 16; ++j)     // 2^-k
                        asv[j] = __uint_as_float((127u - ((ew[j >> 2] >> (8 * (j & 3))) & 0xFFu)) << 23);
                }
                uint32_t v0[16], v1[16];
                tmem_ld16(tbase + c * 16, v0);
                if (NMAT == 2) tmem_ld16(tbase + BN + c * 16, v1);
                tc_wait_ld();
                if constexpr (MODE == OUT_GLU_F16 && KIND == EPI_A8) {
                    // A8: the accurate activation, rounded to MXFP8 over the 32 consecutive
                    // weight rows this warp's lanes hold (one block of the down projection's K
                    // for each token): the 16 tokens' largest exponent fields, packed four to a
                    // word, are reduced over the lanes with byte-wise maxima
                    float av[16];
                    uint32_t pk[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = c * 16 + j;
                        float a = 0.f;
                        if (n < nrows) {
                            const float rs = srs[n];
                            const float gv = __uint_as_float(v0[j]) * (fw0 * rs);
                            const float uv = __uint_as_float(v1[j]) * (fw1 * rs);
                            a = args.act.kind == K3MOE_ACT_SITU ? k3_glu(gv, uv, args.act)
                                                                : __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                        }
                        av[j] = a;
                        pk[j >> 2] |= ((__float_as_uint(a) >> 23) & 0xFFu) << (8 * (j & 3));
                    }
#pragma unroll
                    for (int o = 16; o; o >>= 1)
#pragma unroll
                        for (int w = 0; w < 4; ++w) pk[w] = __vmaxu4(pk[w], __shfl_xor_sync(0xffffffffu, pk[w], o));
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = c * 16 + j;
                        if (n < nrows) {
                            const float a = mx8_round_x(av[j], mx8_scale_exp((pk[j >> 2] >> (8 * (j & 3))) & 0xFFu));
                            bad |= !(fabsf(a) <= 65504.f);
                            reinterpret_cast<__half *>(args.out)[(size_t)(row0 + n) * args.rows + row] =
                                __float2half_rn(a);
                        }
                    }
                } else {
                    // the chunk's 16 results first, without branches, so that their dependency
                    // chains interleave (columns past the tile's rows give values that are never
                    // stored), then the stores of the columns the tile holds
                    uint32_t o0[16], o1[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (MODE == OUT_GLU_F16) {
                            // sigmoid(gv) = (1 + tanh(hv)) / 2 with hv = gv / 2, so
                            // SiLU(gv) = hv + hv tanh(hv); SiTU multiplies the sigmoid by
                            // beta tanh(gv / beta) and soft-limits the up branch the same way
                            const float rs = rsv[j];
                            const float hv = __uint_as_float(v0[j]) * (0.5f * fw0 * rs);
                            // RSA (SiLU): 2^-k is already in the up factor (an exact power of two)
                            const float uv = __uint_as_float(v1[j]) * (fw1 * (RSA ? asv[j] : rs));
                            float a;
                            if constexpr (KIND == EPI_SITU)
                                a = fmaf(0.5f, tanh_approx(hv), 0.5f) * args.act.beta *
                                    tanh_approx(hv * (2.0f * args.act.inv_beta)) *
                                    (args.act.linear_beta * tanh_approx(uv * args.act.inv_linear_beta));
                            else
                                a = fmaf(hv, tanh_approx(hv), hv) * uv;
                            if (!RSA) a *= asv[j];      // exact power of two keeping |a| inside f16
                            bad |= (c * 16 + j < nrows) && !(fabsf(a) <= 65504.f);
                            o0[j] = __half_as_ushort(__float2half_rn(a));
                        } else if (MODE == OUT_BF16) {
                            o0[j] = f32_to_bf16(__uint_as_float(v0[j]) * (fw0 * rsv[j]));
                            if (ROWPAIR) o1[j] = f32_to_bf16(__uint_as_float(v1[j]) * (fw1 * rsv[j]));
                        } else {
                            o0[j] = f32_to_bf16(ad0[j] + __uint_as_float(v0[j]) * (fw0 * rsv[j]));
                            if (ROWPAIR) o1[j] = f32_to_bf16(ad1[j] + __uint_as_float(v1[j]) * (fw1 * rsv[j]));
                        }
                    }
                    uint16_t *o = reinterpret_cast<uint16_t *>(args.out) + (size_t)(row0 + c * 16) * args.rows;
                    const int nv = nrows - c * 16;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (j < nv) {
                            o[(size_t)j * args.rows + row] = (uint16_t)o0[j];
                            if (MODE != OUT_GLU_F16 && ROWPAIR) o[(size_t)j * args.rows + row1] = (uint16_t)o1[j];
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(tempty + acc));
                mbar_arrive(smem_u32(rsempty));
            }
        }
        if (bad) set_status(args.status, K3MOE_ERR_RANGE, 2);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace k3
