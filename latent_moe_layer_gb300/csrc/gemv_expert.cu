// Decode-batch expert kernels: streaming MXFP4 GEMV for experts with few tokens.
//
// When each touched expert sees only a handful of tokens the layer is bound by
// reading the touched experts' packed bytes once from HBM.  These kernels
// decode FP4 in registers straight from 64-bit coalesced global loads -- the
// packed bytes never go through shared memory, and nothing is expanded there
// -- and feed the warp-level tensor-core MMA (m16n8k16, f16 inputs, fp32
// accumulate) with the decoded weights as the A fragment and up to 16 token
// rows as B.
//
// Exactness: as in the tcgen05 path, row m's weights are decoded as
// E2M1 x 2^(e - emax_m) in f16 (exact for e >= emax_m - 23) and 2^(emax_m - 127)
// is applied to the fp32 result; activation rows are the per-token
// power-of-two scaled f16 copies prepared for the tensor path.
//
// K order: for each 64-wide K step, thread (g = lane/4, c = lane%4) loads bytes
// [8c, 8c+8) of rows g and g+8, i.e. 16 consecutive codes of one MX block, and
// uses its pairs 2s and 2s+1 as MMA k-step s's pair slots c and c+4.  The B
// fragment reads the matching activation elements (K = 16c + 4s .. +3), so the
// contraction covers every K exactly once in a permuted order.
#include "gemv_expert.h"
#include "tc_expert.cuh"

namespace k3 {

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint2 ldg_stream(const uint8_t *p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// 8 codes (one 32-bit word, low nibble first) -> 4 f16x2 of E2M1 values times `sc`.
__device__ __forceinline__ void decode8(uint32_t w, __half2 sc, uint32_t (&o)[4])
{
    uint32_t h0, h1, h2, h3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
    __half2 q0 = __hmul2(*reinterpret_cast<__half2 *>(&h0), sc);
    __half2 q1 = __hmul2(*reinterpret_cast<__half2 *>(&h1), sc);
    __half2 q2 = __hmul2(*reinterpret_cast<__half2 *>(&h2), sc);
    __half2 q3 = __hmul2(*reinterpret_cast<__half2 *>(&h3), sc);
    o[0] = *reinterpret_cast<uint32_t *>(&q0);
    o[1] = *reinterpret_cast<uint32_t *>(&q1);
    o[2] = *reinterpret_cast<uint32_t *>(&q2);
    o[3] = *reinterpret_cast<uint32_t *>(&q3);
}

__device__ __forceinline__ __half2 pow2_h2(int d)
{
    // 2^d (d <= 0) as f16x2: built exactly in fp32 (d clamped at -126, far below
    // f16's range) and rounded once to f16 -- subnormals below 2^-14, zero below 2^-24
    const float f = __int_as_float((max(d, -126) + 127) << 23);
    return __float2half2_rn(f);
}

// Packed FP4 rows arrive by TMA (per-expert tensor maps: 128 rows x 128 bytes
// = 256 K values per stage, 128-byte swizzle) into a ring of NS stages; eight
// consumer warps, 16 weight rows each, read their bytes out of shared memory,
// decode them in registers and run the MMAs.  Work items are (token tile of the
// permutation, 128-row block); activation fragments come from global memory
// (the few token rows of a tile stay in L1/L2).
constexpr int GV_STAGE_BYTES = 128 * 128;    // one matrix, one stage
constexpr int GV_B_BYTES = 4 * 16 * 128;     // 16 activation rows x 256 K (four 64-K boxes)

template <int NMAT, int NS>
struct GvSmem {
    static constexpr int STAGE = NMAT * GV_STAGE_BYTES + GV_B_BYTES;
    static constexpr int OFF_BAR = NS * STAGE;
    static constexpr int BYTES = OFF_BAR + 2 * NS * 8 + 16 + 1024;
};

template <int NMAT, int NS, int MODE>
__global__ void __launch_bounds__(288, 2) gemv_expert_kernel(const __grid_constant__ CUtensorMap bmap,
                                                             const GemvArgs a)
{
    griddep_enter();
    using SM = GvSmem<NMAT, NS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + SM::OFF_BAR), *empty = full + NS;
    volatile int *abort_flag = (volatile int *)(empty + NS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = a.rows / 128;
    const int total = __ldg(a.n_tiles) * m_tiles;
    const int nkp = a.K / 256;                // packed stages per tile
    const int kb = a.K / 32;                  // scale bytes per row
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), 8);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&bmap);
            const uint64_t pol = policy_evict_first(), polb = policy_evict_last();
            uint32_t it = 0;
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
                const int4 tile = __ldg(a.tiles + t / m_tiles);
                const int m0 = (t % m_tiles) * 128;
                const CUtensorMap *am0 = a.amaps + (size_t)tile.x * a.amap_stride + a.amap_off[0];
                const CUtensorMap *am1 = a.amaps + (size_t)tile.x * a.amap_stride + a.amap_off[NMAT - 1];
                bool ok = true;
                for (int s = 0; s < nkp; ++s, ++it) {
                    const int slot = it % NS;
                    if (!role_wait(smem_u32(empty + slot), ((it / NS) & 1) ^ 1, abort_flag, 0xFFFFFFFFu,
                                   a.status, 11)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(full + slot);
                    mbar_expect_tx(fb, SM::STAGE);
                    uint8_t *dst = smem + slot * SM::STAGE;
                    tma_load_2d_hint(smem_u32(dst), am0, fb, s * 128, m0, pol);
                    if (NMAT == 2)
                        tma_load_2d_hint(smem_u32(dst + GV_STAGE_BYTES), am1, fb, s * 128, m0, pol);
                    uint8_t *bdst = dst + NMAT * GV_STAGE_BYTES;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tma_load_2d_hint(smem_u32(bdst + q * 16 * 128), &bmap, fb, s * 256 + q * 64, tile.y, polb);
                }
                if (!ok) break;
            }
            drain_ring(full, it, NS);
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int cw = warp - 1;                 // 0..7: rows 16 cw .. 16 cw + 15 of the 128-row block
        const int g8 = lane >> 2, c = lane & 3;
        const int ra_l = 16 * cw + g8, rb_l = ra_l + 8;       // local rows (ra_l & 7 == g8)
        uint32_t it = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
            const int4 tile = __ldg(a.tiles + t / m_tiles);
            const int grp = tile.x, b_first = tile.y, nt = tile.z;
            const int m0 = (t % m_tiles) * 128;
            const int ra = m0 + ra_l, rb = m0 + rb_l;
            const uint8_t *sa[NMAT], *sb[NMAT];
            int ea[NMAT], eb[NMAT];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                const uint8_t *S = a.scales[m][grp];
                sa[m] = S + (size_t)ra * kb;
                sb[m] = S + (size_t)rb * kb;
                ea[m] = __ldg(a.rowmax[m] + (size_t)grp * a.rows + ra);
                eb[m] = __ldg(a.rowmax[m] + (size_t)grp * a.rows + rb);
            }
            const int nnb = (nt + 7) >> 3;           // n-blocks of 8 tokens (<= 2)
            float acc[NMAT][2][4];
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[m][h][q] = 0.f;
            // scale bytes: 8 per row and stage (blocks 8s .. 8s+7), read one stage ahead
            uint2 sca[NMAT], scb[NMAT], nsa[NMAT], nsb[NMAT];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                nsa[m] = __ldg(reinterpret_cast<const uint2 *>(sa[m]));
                nsb[m] = __ldg(reinterpret_cast<const uint2 *>(sb[m]));
            }
            bool ok = true;
            for (int s = 0; s < nkp; ++s, ++it) {
#pragma unroll
                for (int m = 0; m < NMAT; ++m) {
                    sca[m] = nsa[m];
                    scb[m] = nsb[m];
                    if (s + 1 < nkp) {
                        nsa[m] = __ldg(reinterpret_cast<const uint2 *>(sa[m]) + s + 1);
                        nsb[m] = __ldg(reinterpret_cast<const uint2 *>(sb[m]) + s + 1);
                    }
                }
                const int slot = it % NS;
                if (!role_wait(smem_u32(full + slot), (it / NS) & 1, abort_flag, 0xFFFFFFFFu, a.status, 12)) {
                    ok = false;
                    break;
                }
                const uint8_t *sbase = smem + slot * SM::STAGE;
                const uint8_t *bbase = sbase + NMAT * GV_STAGE_BYTES;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    // this thread's bytes: rows ra/rb, bytes [32 ks + 8 c, +8) of the 128-byte row
                    uint2 pa[NMAT], pb[NMAT];
                    const int chunk = 2 * ks + (c >> 1);
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) {
                        const uint8_t *base = sbase + m * GV_STAGE_BYTES;
                        pa[m] = *reinterpret_cast<const uint2 *>(base + ra_l * 128 + 16 * (chunk ^ (ra_l & 7)) + 8 * (c & 1));
                        pb[m] = *reinterpret_cast<const uint2 *>(base + rb_l * 128 + 16 * (chunk ^ (rb_l & 7)) + 8 * (c & 1));
                    }
                    // activation fragments of tokens 8 nb + g8: K = 64 ks + 16 c .. + 15 of this
                    // stage = 16-byte chunks 2c, 2c+1 of row (8 nb + g8) in box ks (128-byte swizzle)
                    uint4 hb[2][2];
#pragma unroll
                    for (int nb = 0; nb < 2; ++nb) {
                        if (nb < nnb) {                  // tokens 8..15 only when the tile has them
                            const int br = 8 * nb + g8;
                            const uint8_t *bx = bbase + ks * 16 * 128 + br * 128;
                            hb[nb][0] = *reinterpret_cast<const uint4 *>(bx + 16 * ((2 * c) ^ (br & 7)));
                            hb[nb][1] = *reinterpret_cast<const uint4 *>(bx + 16 * ((2 * c + 1) ^ (br & 7)));
                        }
                    }
                    if (ks == 3) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(empty + slot));
                    }
                    // block of this thread's codes in this stage: 2 ks + c / 2 (byte of the 8)
                    const int bsh = 8 * (2 * (ks & 1) + (c >> 1));
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) {
                        const uint32_t wsa = (ks >> 1) ? sca[m].y : sca[m].x;
                        const uint32_t wsb = (ks >> 1) ? scb[m].y : scb[m].x;
                        const __half2 fa = pow2_h2((int)((wsa >> bsh) & 0xFF) - ea[m]);
                        const __half2 fb = pow2_h2((int)((wsb >> bsh) & 0xFF) - eb[m]);
                        uint32_t qa[8], qb[8];
                        decode8(pa[m].x, fa, *reinterpret_cast<uint32_t(*)[4]>(&qa[0]));
                        decode8(pa[m].y, fa, *reinterpret_cast<uint32_t(*)[4]>(&qa[4]));
                        decode8(pb[m].x, fb, *reinterpret_cast<uint32_t(*)[4]>(&qb[0]));
                        decode8(pb[m].y, fb, *reinterpret_cast<uint32_t(*)[4]>(&qb[4]));
#pragma unroll
                        for (int st = 0; st < 4; ++st) {
                            const uint32_t af[4] = {qa[2 * st], qb[2 * st], qa[2 * st + 1], qb[2 * st + 1]};
#pragma unroll
                            for (int nb = 0; nb < 2; ++nb) {
                                if (nb < nnb) {
                                    const uint4 &h0 = hb[nb][st >> 1];
                                    const uint32_t b0 = (st & 1) ? h0.z : h0.x, b1 = (st & 1) ? h0.w : h0.y;
                                    mma16816(acc[m][nb], af, b0, b1);
                                }
                            }
                        }
                    }
                }
            }
            if (!ok) break;
            // epilogue: acc[m][nb][0..1] = (row ra, tokens 8 nb + 2c, +1); [2..3] = (row rb, same tokens)
#pragma unroll
            for (int nb = 0; nb < 2; ++nb)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int tok = 8 * nb + 2 * c + (q & 1);
                    const int row = (q < 2) ? ra : rb;
                    if (tok < nt) {
                        const size_t orow = (size_t)(b_first + tok);
                        const float f0 = e8m0_to_f32((uint32_t)((q < 2) ? ea[0] : eb[0]));
                        if (MODE == GV_GLU_F16) {
                            const float f1 = e8m0_to_f32((uint32_t)((q < 2) ? ea[NMAT - 1] : eb[NMAT - 1]));
                            const float rs = a.rscale ? __ldg(a.rscale + orow) : 1.f;
                            const float gv = acc[0][nb][q] * f0 * rs;
                            const float uv = acc[NMAT - 1][nb][q] * f1 * rs;
                            const float av = gv / (1.0f + expf(-gv)) * uv;
                            if (!(fabsf(av) <= 65504.f)) set_status(a.status, K3MOE_ERR_RANGE, 3);
                            reinterpret_cast<__half *>(a.out)[orow * a.rows + row] = __float2half_rn(av);
                        } else {
                            reinterpret_cast<uint16_t *>(a.out)[orow * a.rows + row] =
                                f32_to_bf16(acc[0][nb][q] * f0);
                        }
                    }
                }
        }
    }
}

}  // namespace k3

using namespace k3;

template <int NMAT, int NS, int MODE>
static int launch_gemv(const CUtensorMap &bmap, const GemvArgs &args, int max_items, int num_sms, cudaStream_t st)
{
    using SM = GvSmem<NMAT, NS>;
    static_assert(2 * SM::BYTES <= 228 * 1024, "two CTAs per SM");
    auto kern = gemv_expert_kernel<NMAT, NS, MODE>;
    static unsigned long long attr_set = 0;
    if (!k3_smem_attr(kern, SM::BYTES, attr_set)) return K3MOE_ERR_CUDA;
    const int grid = max(1, min(max_items, 2 * num_sms));
    k3_launch(kern, grid, 288, SM::BYTES, st, bmap, args);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

int k3_launch_gemv_expert(int glu, int mode, const CUtensorMap &bmap, const GemvArgs &args, int max_items,
                          int num_sms, cudaStream_t st)
{
    if (glu) return launch_gemv<2, 2, GV_GLU_F16>(bmap, args, max_items, num_sms, st);
    if (mode == GV_BF16) return launch_gemv<1, 4, GV_BF16>(bmap, args, max_items, num_sms, st);
    return K3MOE_ERR_UNSUPPORTED;
}
