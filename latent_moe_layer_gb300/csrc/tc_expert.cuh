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
// Roles (one CTA per SM, persistent over the tile list):
//   warp 0            TMA producer: packed FP4 tiles (per-expert tensor maps,
//                     32-byte swizzle) and activation rows (128-byte swizzle)
//   warp 1            TMEM allocator and the single MMA-issuing thread
//   warps 4..4+4*NMAT dequant: one thread per weight row, FP4 -> f16 into the
//                     128-byte-swizzled K-major layout the MMA reads
//   last 4 warps      epilogue: TMEM -> registers -> scaled outputs
// Every wait is bounded; on expiry the CTA records K3MOE_ERR_TIMEOUT, drains
// its copies and MMAs, frees TMEM and returns.
#pragma once
#include <cudaTypedefs.h>

#include "k3moe_internal.h"
#include "ptx.cuh"

namespace k3 {

enum ExpertOut { OUT_GLU_F16 = 0, OUT_BF16 = 1, OUT_F32_ADD = 2 };

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
    const float *rscale;             // per B-row factor (GLU input scaling) or nullptr
    void *out;                       // GLU: f16 [R, rows]; BF16: [R, rows]; F32_ADD: fp32 [R, rows]
    int *status;
    uint32_t spin_limit;
};

constexpr int EX_BM = 128;           // weight rows per tile (MMA M)
constexpr int EX_BK = 64;            // K per stage (one 128-byte f16 row)

template <int NMAT, int BN, int NS>
struct ExpertSmem {
    static constexpr int NA = 4 / NMAT;                     // f16 A slots (each NMAT tiles)
    static constexpr int PK_BYTES = EX_BM * EX_BK / 2;      // 4096 packed bytes per matrix
    static constexpr int B_BYTES = BN * EX_BK * 2;          // activation tile
    static constexpr int A_BYTES = EX_BM * EX_BK * 2;       // 16384 f16 tile
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + NA * NMAT * A_BYTES;
    static constexpr int OFF_PK = OFF_B + NS * B_BYTES;
    static constexpr int OFF_BAR = OFF_PK + NS * NMAT * PK_BYTES;
    static constexpr int N_BAR = 2 * NS + 2 * NA + 4 + 1;
    static constexpr int BYTES = OFF_BAR + N_BAR * 8 + 16 + 1024;   // + tmem holder/flag + align slack
};

__device__ __forceinline__ uint32_t f16_pow2_bits(int d)
{
    // 2^d as f16 bits for d <= 0 (subnormals for d < -14, zero below -24)
    if (d >= -14) return (uint32_t)(d + 15) << 10;
    if (d >= -24) return 1u << (d + 24);
    return 0u;
}

// Wait with the CTA abort flag: returns false on timeout or abort.
__device__ __forceinline__ bool role_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          uint32_t limit, int *status, int where)
{
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer();
    for (uint32_t i = 1; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((i & 255u) == 0 && globaltimer() - t0 > kWaitCapNs) break;
    }
    set_status(status, K3MOE_ERR_TIMEOUT, where);
    *abort_flag = 1;
    return false;
}

template <int NMAT, int BN, int NS, int MODE>
__global__ void __launch_bounds__((8 + 4 * NMAT) * 32, 1)
expert_gemm_kernel(const __grid_constant__ CUtensorMap bmap, const ExpertGemmArgs args)
{
    using SM = ExpertSmem<NMAT, BN, NS>;
    constexpr int NA = SM::NA;
    constexpr int EPI_WARP0 = 4 + 4 * NMAT;
    constexpr uint32_t TMEM_COLS = (2 * NMAT * BN <= 32) ? 32 : (2 * NMAT * BN <= 64) ? 64
                                 : (2 * NMAT * BN <= 128) ? 128 : (2 * NMAT * BN <= 256) ? 256 : 512;
    static_assert(2 * NMAT * BN <= 512, "TMEM columns");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(smem + SM::OFF_BAR);
    uint64_t *full = bars, *empty = bars + NS, *afull = bars + 2 * NS, *aempty = bars + 2 * NS + NA;
    uint64_t *tfull = bars + 2 * NS + 2 * NA, *tempty = tfull + 2, *drain = tempty + 2;
    uint32_t *tmem_holder = (uint32_t *)(drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = args.K, nk = K / EX_BK;
    const int m_tiles = args.rows / EX_BM;
    const int total = __ldg(args.n_tiles) * m_tiles;
    const uint32_t lim = args.spin_limit;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), 4 * NMAT + 1);
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(smem_u32(afull + i), 4 * NMAT);
            mbar_init(smem_u32(aempty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(tfull + i), 1);
            mbar_init(smem_u32(tempty + i), 4);
        }
        mbar_init(smem_u32(drain), 1);
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
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&bmap);
            const uint64_t pol_w = policy_evict_first(), pol_b = policy_evict_last();
            uint32_t it = 0;
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
                const int4 tile = __ldg(args.tiles + t / m_tiles);
                const int g = tile.x, row0 = tile.y, m0 = (t % m_tiles) * EX_BM;
                const CUtensorMap *am0 = args.amaps + (size_t)g * args.amap_stride + args.amap_off[0];
                const CUtensorMap *am1 = args.amaps + (size_t)g * args.amap_stride + args.amap_off[NMAT - 1];
                for (int s = 0; s < nk; ++s, ++it) {
                    const int slot = it % NS;
                    if (!role_wait(smem_u32(empty + slot), ((it / NS) & 1) ^ 1, abort_flag, lim,
                                   args.status, 1))
                        break;
                    const uint32_t fb = smem_u32(full + slot);
                    mbar_expect_tx(fb, NMAT * SM::PK_BYTES + SM::B_BYTES);
                    uint8_t *pk = smem + SM::OFF_PK + slot * NMAT * SM::PK_BYTES;
                    tma_load_2d_hint(smem_u32(pk), am0, fb, s * (EX_BK / 2), m0, pol_w);
                    if (NMAT == 2)
                        tma_load_2d_hint(smem_u32(pk + SM::PK_BYTES), am1, fb, s * (EX_BK / 2), m0, pol_w);
                    tma_load_2d_hint(smem_u32(smem + SM::OFF_B + slot * SM::B_BYTES), &bmap, fb,
                                     s * EX_BK, row0, pol_b);
                }
            }
            // drain: every issued stage must have landed before the CTA exits
            const uint32_t n = it < (uint32_t)NS ? it : (uint32_t)NS;
            for (uint32_t q = 0; q < n; ++q) {
                const uint32_t i2 = it - 1 - q;
                mbar_wait(smem_u32(full + i2 % NS), (i2 / NS) & 1, 0xFFFFFFFFu);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, ait = 0, tc = 0;
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++tc) {
                const int4 tile = __ldg(args.tiles + t / m_tiles);
                const int nrows = tile.z;
                const int nmma = min(BN, max(16, (nrows + 15) & ~15));
                const uint32_t idesc = idesc_f16(EX_BM, nmma, 0);
                const int acc = tc & 1;
                if (!role_wait(smem_u32(tempty + acc), ((tc >> 1) & 1) ^ 1, abort_flag, lim, args.status, 2))
                    break;
                tc_fence_after();
                const uint32_t dcol = tmem + acc * NMAT * BN;
                bool ok = true;
                for (int s = 0; s < nk; ++s, ++it, ++ait) {
                    const int slot = it % NS, aslot = ait % NA;
                    if (!role_wait(smem_u32(full + slot), (it / NS) & 1, abort_flag, lim, args.status, 3) ||
                        !role_wait(smem_u32(afull + aslot), (ait / NA) & 1, abort_flag, lim, args.status, 4)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b_addr = smem_u32(smem + SM::OFF_B + slot * SM::B_BYTES);
                    const uint64_t bdesc = smem_desc_sw128(b_addr);
#pragma unroll
                    for (int mt = 0; mt < NMAT; ++mt) {
                        const uint32_t a_addr =
                            smem_u32(smem + SM::OFF_A + (aslot * NMAT + mt) * SM::A_BYTES);
                        const uint64_t adesc = smem_desc_sw128(a_addr);
#pragma unroll
                        for (int kk = 0; kk < EX_BK / 16; ++kk)
                            tc_mma_f16(dcol + mt * BN, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                                       (s > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(smem_u32(empty + slot));
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
        const int mat = d / 4;
        const int r = (d % 4) * 32 + lane;                 // weight row within the tile
        const int kblk = K / 32;
        uint32_t it = 0, ait = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
            const int4 tile = __ldg(args.tiles + t / m_tiles);
            const int g = tile.x, m0 = (t % m_tiles) * EX_BM;
            const int row = m0 + r;
            const int emax = __ldg(args.rowmax[mat] + (size_t)g * args.rows + row);
            const uint8_t *srow = args.scales[mat][g] + (size_t)row * kblk;
            uint4 sc_cur = __ldg(reinterpret_cast<const uint4 *>(srow));
            uint4 sc_next = make_uint4(0, 0, 0, 0);
            bool ok = true;
            for (int s = 0; s < nk; ++s, ++it, ++ait) {
                if ((s & 7) == 0) {
                    if (s > 0) sc_cur = sc_next;
                    if (s + 8 < nk) sc_next = __ldg(reinterpret_cast<const uint4 *>(srow) + (s >> 3) + 1);
                }
                const int slot = it % NS, aslot = ait % NA;
                if (!role_wait(smem_u32(full + slot), (it / NS) & 1, abort_flag, lim, args.status, 5)) {
                    ok = false;
                    break;
                }
                const uint8_t *pk = smem + SM::OFF_PK + (slot * NMAT + mat) * SM::PK_BYTES + r * 32;
                const int sw = (r >> 2) & 1;                   // 32-byte swizzle of the TMA box
                const uint4 lo = *reinterpret_cast<const uint4 *>(pk + 16 * (0 ^ sw));
                const uint4 hi = *reinterpret_cast<const uint4 *>(pk + 16 * (1 ^ sw));
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(empty + slot));
                // the two E8M0 bytes of this stage
                const uint32_t sw32 = (&sc_cur.x)[(s & 7) >> 1];
                const int e0 = (sw32 >> (16 * (s & 1))) & 0xFF, e1 = (sw32 >> (16 * (s & 1) + 8)) & 0xFF;
                const uint32_t f0 = f16_pow2_bits(e0 - emax), f1 = f16_pow2_bits(e1 - emax);
                const __half2 s0 = __halves2half2(__ushort_as_half((unsigned short)f0), __ushort_as_half((unsigned short)f0));
                const __half2 s1 = __halves2half2(__ushort_as_half((unsigned short)f1), __ushort_as_half((unsigned short)f1));
                if (!role_wait(smem_u32(aempty + aslot), ((ait / NA) & 1) ^ 1, abort_flag, lim, args.status, 6)) {
                    ok = false;
                    break;
                }
                uint8_t *arow = smem + SM::OFF_A + (aslot * NMAT + mat) * SM::A_BYTES + r * 128;
                const uint32_t words[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
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
                    *reinterpret_cast<uint4 *>(arow + 16 * (j ^ (r & 7))) = v;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(afull + aslot));
            }
            if (!ok) break;
        }
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------------------ epilogue
        const int q = warp - EPI_WARP0;                    // TMEM lanes 32q .. 32q+31
        const int r = q * 32 + lane;
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++tc) {
            const int4 tile = __ldg(args.tiles + t / m_tiles);
            const int g = tile.x, row0 = tile.y, nrows = tile.z;
            const int m0 = (t % m_tiles) * EX_BM, row = m0 + r;
            const int acc = tc & 1;
            const float fw0 = e8m0_to_f32(__ldg(args.rowmax[0] + (size_t)g * args.rows + row));
            const float fw1 = NMAT == 2 ? e8m0_to_f32(__ldg(args.rowmax[NMAT - 1] + (size_t)g * args.rows + row)) : 0.f;
            if (!role_wait(smem_u32(tfull + acc), (tc >> 1) & 1, abort_flag, lim, args.status, 7)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + acc * NMAT * BN;
            const int nchunks = (nrows + 15) >> 4;
            for (int c = 0; c < nchunks; ++c) {
                uint32_t v0[16], v1[16];
                tmem_ld16(tbase + c * 16, v0);
                if (NMAT == 2) tmem_ld16(tbase + BN + c * 16, v1);
                tc_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = c * 16 + j;
                    if (n < nrows) {
                        const size_t orow = (size_t)(row0 + n);
                        if (MODE == OUT_GLU_F16) {
                            const float rs = args.rscale ? __ldg(args.rscale + row0 + n) : 1.f;
                            const float gv = __uint_as_float(v0[j]) * fw0 * rs;
                            const float uv = __uint_as_float(v1[j]) * fw1 * rs;
                            const float a = gv / (1.0f + expf(-gv)) * uv;
                            if (!(fabsf(a) <= 65504.f)) set_status(args.status, K3MOE_ERR_RANGE, 2);
                            reinterpret_cast<__half *>(args.out)[orow * args.rows + row] = __float2half_rn(a);
                        } else if (MODE == OUT_BF16) {
                            const float y = __uint_as_float(v0[j]) * fw0;
                            reinterpret_cast<uint16_t *>(args.out)[orow * args.rows + row] = f32_to_bf16(y);
                        } else {
                            const float y = __uint_as_float(v0[j]) * fw0;
                            float *o = reinterpret_cast<float *>(args.out) + orow * args.rows + row;
                            *o += y;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(tempty + acc));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace k3
