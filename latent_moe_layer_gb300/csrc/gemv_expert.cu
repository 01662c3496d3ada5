// Decode-batch expert kernels: streaming MXFP4 GEMV for experts with few tokens.
//
// When each touched expert sees only a handful of tokens the layer is bound by
// reading the touched experts' packed bytes once from HBM.  A TMA warp streams
// the packed rows (and the tile's few activation rows) into a shared-memory
// ring; consumer warps decode FP4 in registers (nothing is expanded in shared
// memory) and feed the warp-level tensor-core MMA (m16n8k16, f16 inputs, fp32
// accumulate) with the decoded weights as the A fragment and up to 16 token
// rows as B.  Activation rows are the per-token power-of-two scaled f16 copies
// prepared for the tensor path.
//
// Block scales (OCP MX v1.0: value = E2M1 x 2^(e - 127), e the block's E8M0
// byte): each MMA covers one MX block only.  Thread (g = lane/4, c = lane%4)
// holds bytes [4c, 4c+4) of the block for weight rows g and g+8, i.e.
// block-local K = 8c .. 8c+7, used as the k-steps {8c, 8c+1 | 8c+2, 8c+3} and
// {8c+4, 8c+5 | 8c+6, 8c+7}; the B fragments read the activations at the same
// K.  The MMAs run on the plain E2M1 values (exact in f16) and the block's fp32
// partial sum is multiplied by 2^(e - 127) (exact in fp32; code 0 is taken as 0)
// and added to the row's accumulator (packed fp32x2 FMAs: the two token columns a
// thread holds for one row share the row's scale).
#include "gemv_expert.h"
#include "wait.cuh"

namespace k3 {

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 8 codes (one 32-bit word, low nibble first) -> 4 f16x2 of the plain E2M1 values.
__device__ __forceinline__ void decode8(uint32_t w, uint32_t (&o)[4])
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}

// ldmatrix of 8x8 b16 tiles: lane t receives bytes [4 (t % 4), +4) of row t / 4 of
// each tile; lanes 8i .. 8i + 7 give the row addresses of tile i.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// {d0, d1} += {a0, a1} * s: two fp32 FMAs, each rounded once (as fmaf), in one packed instruction.
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float s)
{
    asm("{\n\t.reg .b64 d, a, s;\n\tmov.b64 d, {%0, %1};\n\tmov.b64 a, {%2, %3};\n\tmov.b64 s, {%4, %4};\n\t"
        "fma.rn.f32x2 d, a, s, d;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1), "f"(s));
}

// Token row of B (within an 8-token block) that MMA column n reads: 0, 4, 1, 5, 2, 6, 3, 7.
__device__ __forceinline__ int tok_perm(int n) { return (n >> 1) | ((n & 1) << 2); }

// 2^(e - 127) for the E8M0 byte `e`, exact in fp32 (e = 0 is taken as 0).
__device__ __forceinline__ float e8m0_f32_noden(uint32_t e) { return __uint_as_float(e << 23); }

// Packed FP4 rows arrive by TMA (per-expert tensor maps: boxes of 128 rows x 128
// bytes = 256 K values per stage, 128-byte swizzle) into a ring of NS stages; WPC
// consumer warps, 16 weight rows each, read their bytes out of shared memory,
// decode them in registers and run the MMAs.  Work items are (token tile of the
// permutation, 16 WPC-row block); each stage also carries the tile's activation
// rows (16 rows x 256 K, four 64-K boxes), which stay L2-resident across the
// row blocks of an expert.
constexpr int GV_B_BYTES = 4 * 16 * 128;     // 16 activation rows x 256 K (four 64-K boxes)

// WPC consumer warps per CTA: 16 WPC weight rows per work item and stage.
template <int NMAT, int NS, int WPC>
struct GvSmem {
    static constexpr int ROWS = 16 * WPC;
    static constexpr int MAT_BYTES = ROWS * 128;          // one matrix, one stage
    static constexpr int STAGE = NMAT * MAT_BYTES + GV_B_BYTES;
    static constexpr int OFF_BAR = NS * STAGE;
    static constexpr int BYTES = OFF_BAR + 2 * NS * 8 + 16 + 1024;
};

// One work item's K loop for a tile of NNB x 8 token rows (the token count is a
// template argument so that the unrolled loop carries no branches).  The stages have
// the layout of LM >= NMAT matrices (the activation rows after them).  PRE: the next
// work item's first-stage scale bytes (rows at sa_next, nullptr if none) are read
// during the last stage and handed over in `carry`; with carry_in this item's come
// from there.
template <int NMAT, int LM, int NS, int WPC, int NNB, bool PRE>
__device__ __forceinline__ bool gemv_k_loop(const uint8_t *smem, const uint64_t *full, uint64_t *empty,
                                            volatile int *abort_flag, const GemvArgs &a, int nkp, int ra_l,
                                            int g8, int c, int lane, const uint2 *const (&sa)[NMAT],
                                            const uint2 *const (&sa_next)[NMAT], bool carry_in,
                                            uint2 (&carry)[2][NMAT], int rbo, uint32_t &it,
                                            float (&acc)[NMAT][2][4])
{
    const int tr = tok_perm(g8);
    using SM = GvSmem<LM, NS, WPC>;
    // scale bytes: 8 per row and stage (blocks 8s .. 8s+7), read one stage ahead
    uint2 sca[NMAT], scb[NMAT], nsa[NMAT], nsb[NMAT];
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
        if (PRE && carry_in) {
            nsa[m] = carry[0][m];
            nsb[m] = carry[1][m];
        } else {
            nsa[m] = __ldg(sa[m]);
            nsb[m] = __ldg(sa[m] + rbo);
        }
    }
    for (int s = 0; s < nkp; ++s, ++it) {
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            sca[m] = nsa[m];
            scb[m] = nsb[m];
            if (s + 1 < nkp) {
                nsa[m] = __ldg(sa[m] + s + 1);
                nsb[m] = __ldg(sa[m] + rbo + s + 1);
            } else if (PRE && sa_next[0]) {
                nsa[m] = __ldg(sa_next[m]);
                nsb[m] = __ldg(sa_next[m] + rbo);
            }
        }
        const int slot = it % NS;
        if (!role_wait(smem_u32(full + slot), (it / NS) & 1, abort_flag, 0xFFFFFFFFu, a.status, 12)) return false;
        const uint8_t *sbase = smem + slot * SM::STAGE;
        const uint8_t *bbase = sbase + LM * SM::MAT_BYTES;
        // ldmatrix row base of this lane: tile (lane >> 3) = (matrix, rows ra or rb)
        const int cw_rows = ra_l >> 4;                   // this warp's 16-row group
        const uint32_t sld = smem_u32(sbase) + ((lane >> 4) & (NMAT - 1)) * SM::MAT_BYTES +
                             (16 * cw_rows + 8 * ((lane >> 3) & 1) + (lane & 7)) * 128;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int bl = 0; bl < 2; ++bl) {
                // MX block j = 2 ks + bl of the stage = 16-byte chunk j of each 128-byte row;
                // this thread takes bytes [4c, 4c + 4) of it
                const int j = 2 * ks + bl;
                // gate/up: one ldmatrix for tiles (rows ra, matrix 0), (rows rb, 0), (ra, 1),
                // (rb, 1), this lane's row address being row (lane & 7) of its tile, chunk j
                // (128-byte swizzle); down: two plain loads (measured faster than ldmatrix.x2)
                uint32_t pa[NMAT], pb[NMAT];
                if (NMAT == 2) {
                    ldsm_x4(sld + 16 * (j ^ (lane & 7)), pa[0], pb[0], pa[NMAT - 1], pb[NMAT - 1]);
                } else {
                    const uint8_t *base = sbase + 16 * cw_rows * 128 + 16 * (j ^ g8) + 4 * c;
                    pa[0] = *reinterpret_cast<const uint32_t *>(base + g8 * 128);
                    pb[0] = *reinterpret_cast<const uint32_t *>(base + (g8 + 8) * 128);
                }
                // MMA column g8 takes token row 8 nb + tr (tr = tok_perm(g8)) at block-local
                // K = 8c .. 8c + 7: 16-byte chunk 4 bl + c of that row in box ks (128-byte
                // swizzle).  The two rows a quarter-warp reads differ by 4, so their chunks
                // fall in disjoint bank groups
                uint4 hb[NNB];
#pragma unroll
                for (int nb = 0; nb < NNB; ++nb)
                    hb[nb] = *reinterpret_cast<const uint4 *>(bbase + ks * 16 * 128 + (8 * nb + tr) * 128 +
                                                              16 * ((4 * bl + c) ^ tr));
                if (ks == 3 && bl == 1) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(empty + slot));
                }
#pragma unroll
                for (int m = 0; m < NMAT; ++m) {
                    const uint32_t wsa = (j >> 2) ? sca[m].y : sca[m].x;
                    const uint32_t wsb = (j >> 2) ? scb[m].y : scb[m].x;
                    const float fa = e8m0_f32_noden((wsa >> (8 * (j & 3))) & 0xFFu);
                    const float fb = e8m0_f32_noden((wsb >> (8 * (j & 3))) & 0xFFu);
                    uint32_t qa[4], qb[4];
                    decode8(pa[m], qa);
                    decode8(pb[m], qb);
                    const uint32_t a0[4] = {qa[0], qb[0], qa[1], qb[1]};
                    const uint32_t a1[4] = {qa[2], qb[2], qa[3], qb[3]};
#pragma unroll
                    for (int nb = 0; nb < NNB; ++nb) {
                        float p[4] = {0.f, 0.f, 0.f, 0.f};
                        mma16816(p, a0, hb[nb].x, hb[nb].y);
                        mma16816(p, a1, hb[nb].z, hb[nb].w);
                        ffma2(acc[m][nb][0], acc[m][nb][1], p[0], p[1], fa);
                        ffma2(acc[m][nb][2], acc[m][nb][3], p[2], p[3], fb);
                    }
                }
            }
        }
    }
    if (PRE) {
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            carry[0][m] = nsa[m];
            carry[1][m] = nsb[m];
        }
    }
    return true;
}

// Output of one work item: acc[m][nb][0..1] = (row ra, tokens 8 nb + 2c, +1),
// [2..3] = (row rb, same tokens).  PRE: pf holds each of the thread's two token
// columns' input and output factors, read ahead.
template <int NMAT, int MODE, int MAXNB, bool PRE>
__device__ __forceinline__ void gemv_epilogue(const GemvArgs &a, const float (&acc)[NMAT][2][4],
                                              const float (&pf)[2][2], int c, int ra, int rb, int b_first, int nt)
{
#pragma unroll
    for (int nb = 0; nb < MAXNB; ++nb)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int tok = 8 * nb + tok_perm(2 * c + (q & 1));
            const int row = (q < 2) ? ra : rb;
            if (tok < nt) {
                const size_t orow = (size_t)(b_first + tok);
                if (MODE == GV_GLU_F16) {
                    const float rs = PRE ? pf[q & 1][0] : (a.rscale ? __ldg(a.rscale + orow) : 1.f);
                    const float gv = acc[0][nb][q] * rs;
                    const float uv = acc[NMAT - 1][nb][q] * rs;
                    const float av = k3_glu(gv, uv, a.act);
                    if (a.out_f32) {
                        reinterpret_cast<float *>(a.out)[orow * a.rows + row] = av;
                    } else {
                        // an exact power of two keeps |a| inside the f16 range
                        const float asv = PRE ? pf[q & 1][1] : (a.ascale ? __ldg(a.ascale + orow) : 1.f);
                        const float as = av * pow2_inverse(asv);
                        if (!(fabsf(as) <= 65504.f)) set_status(a.status, K3MOE_ERR_RANGE, 3);
                        reinterpret_cast<__half *>(a.out)[orow * a.rows + row] = __float2half_rn(as);
                    }
                } else {
                    const float asv = PRE ? pf[q & 1][1] : (a.ascale ? __ldg(a.ascale + orow) : 1.f);
                    const float y = acc[0][nb][q] * asv;
                    reinterpret_cast<uint16_t *>(a.out)[orow * a.rows + row] = f32_to_bf16(y);
                }
            }
        }
}

// MAXNB = 2: the K loop exists for 8- and 16-token tiles.  MAXNB = 1: for 8 only (tiles of
// at most 8 tokens), which leaves the compiler more registers for the one loop.
// WPC = 8: 128-row work items, two CTAs per SM; WPC = 16: 256-row items, one CTA per SM
// (the ring shared by twice the warps, with deeper stages in flight).
template <int NMAT, int NS, int MODE, int MAXNB, int WPC>
__global__ void __launch_bounds__((WPC + 1) * 32, 16 / WPC) gemv_expert_kernel(const __grid_constant__ CUtensorMap bmap,
                                                                                const GemvArgs a)
{
    griddep_enter();
    using SM = GvSmem<NMAT, NS, WPC>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + SM::OFF_BAR), *empty = full + NS;
    volatile int *abort_flag = (volatile int *)(empty + NS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = a.rows / SM::ROWS;
    const int total = __ldg(a.n_tiles) * m_tiles;
    const int nkp = a.K / 256;                // packed stages per tile
    const int kb = a.K / 32;                  // scale bytes per row
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), WPC);
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
                const int m0 = (t % m_tiles) * SM::ROWS;
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
#pragma unroll
                    for (int h = 0; h < SM::ROWS / 128; ++h) {          // 128-row boxes
                        tma_load_2d_hint(smem_u32(dst + h * 16384), am0, fb, s * 128, m0 + 128 * h, pol);
                        if (NMAT == 2)
                            tma_load_2d_hint(smem_u32(dst + SM::MAT_BYTES + h * 16384), am1, fb, s * 128,
                                             m0 + 128 * h, pol);
                    }
                    uint8_t *bdst = dst + NMAT * SM::MAT_BYTES;
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
        const int ra_l = 16 * cw + g8;           // local rows ra_l and ra_l + 8 (both = g8 mod 8)
        // The 8-token down kernel reads ahead: the next work item's first-stage scale bytes
        // during this one's last stage, and this item's per-token epilogue factors at its start
        // (a thread's two token columns).  Measured at T=16: down 0.2238 -> 0.2221 ms; the
        // gate/up kernel, with twice the scale registers, went from 0.435 to 0.440 ms with it.
        constexpr bool PRE = MAXNB == 1 && NMAT == 1;
        uint2 carry[2][NMAT];
        bool have_carry = false;
        uint32_t it = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
            const int4 tile = __ldg(a.tiles + t / m_tiles);
            const int grp = tile.x, b_first = tile.y, nt = tile.z;
            const int m0 = (t % m_tiles) * SM::ROWS;
            const int ra = m0 + ra_l, rb = ra + 8;
            const uint2 *sa[NMAT];               // row ra's scale bytes; row rb's follow 8 rows later
            const uint2 *sa_next[NMAT];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                sa[m] = reinterpret_cast<const uint2 *>(a.scales[m][grp] + (size_t)ra * kb);
                sa_next[m] = nullptr;
            }
            float pf[2][2] = {{1.f, 1.f}, {1.f, 1.f}};   // per token column: input factor, output factor
            if (PRE) {
                const int tn = t + gridDim.x;
                if (tn < total) {
                    const int gn = __ldg(a.tiles + tn / m_tiles).x;
                    const size_t rn = (size_t)((tn % m_tiles) * SM::ROWS + ra_l);
#pragma unroll
                    for (int m = 0; m < NMAT; ++m)
                        sa_next[m] = reinterpret_cast<const uint2 *>(a.scales[m][gn] + rn * kb);
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int tok = tok_perm(2 * c + j);
                    if (tok < nt) {
                        const size_t orow = (size_t)(b_first + tok);
                        if (MODE == GV_GLU_F16 && a.rscale) pf[j][0] = __ldg(a.rscale + orow);
                        if (a.ascale) pf[j][1] = __ldg(a.ascale + orow);
                    }
                }
            }
            float acc[NMAT][2][4];
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[m][h][q] = 0.f;
            const bool ok = (MAXNB == 2 && nt > 8)
                                ? gemv_k_loop<NMAT, NMAT, NS, WPC, 2, PRE>(smem, full, empty, abort_flag, a, nkp, ra_l, g8, c, lane,
                                                                sa, sa_next, have_carry, carry, kb, it, acc)
                                : gemv_k_loop<NMAT, NMAT, NS, WPC, 1, PRE>(smem, full, empty, abort_flag, a, nkp, ra_l, g8, c, lane,
                                                                sa, sa_next, have_carry, carry, kb, it, acc);
            if (!ok) break;
            have_carry = PRE && sa_next[0] != nullptr;
            gemv_epilogue<NMAT, MODE, MAXNB, PRE>(a, acc, pf, c, ra, rb, b_first, nt);
        }
    }
}

// ---- The decode gate/up and down GEMVs of one routing as one persistent launch
// (8-token tiles, two CTAs of 8 consumer warps per SM).  Separate launches each end in
// a partly idle round (the work items rarely divide evenly over the CTAs) and the down
// launch starts only when the last gate/up CTA has finished.  Here each CTA's producer
// takes work items in ticket order from a counter: first every (tile, 128-row block)
// of gate/up, then every (tile, 256-row block) of down (two 128-row blocks of w2 in the
// stage's two matrix slots, against the same activation rows, so that every stage has
// the gate/up shape), and hands each to its consumer warps through a small ring in
// shared memory.  A down item reads its tile's GLU output, so its producer first waits
// until all gate/up items of that tile are stored: each consumer warp counts each
// gate/up item it finished in the tile's counter, after a fence that it issues just
// before its next item's epilogue (by then the stores are long done and the fence is
// cheap), or at once when its next item is a down item or the end.  Tickets are taken
// in order by running CTAs and a producer publishes an item before it waits on it, so
// the gate/up items a down item waits for are held by running CTAs whose warps finish
// and count them without waiting on anything.
constexpr int GF_NI = 4;    // item ring slots

template <int NS>
struct GfSmem {
    using SM = GvSmem<2, NS, 8>;
    // the stage ring of the gate/up layout (down items use its first matrix slot), then
    // full[NS], empty[NS], ifull[GF_NI], iempty[GF_NI], the abort flag and the item slots
    static constexpr int OFF_BAR = SM::OFF_BAR;
    static constexpr int OFF_FLAG = OFF_BAR + (2 * NS + 2 * GF_NI) * 8;
    static constexpr int OFF_ITEMS = OFF_FLAG + 16;
    static constexpr int BYTES = OFF_ITEMS + GF_NI * 4 + 1024;
};

// Waits (bounded) until the counter at p reaches target.
__device__ __forceinline__ bool gf_wait_count(const int *p, int target, volatile int *abort_flag, int *status)
{
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v >= target) return true;
        if (*abort_flag) return false;
        if (i == 0) {
            t0 = globaltimer();
        } else if ((i & 255u) == 0 && globaltimer() - t0 > kWaitCapNs) {
            set_status(status, K3MOE_ERR_TIMEOUT, 15);
            *abort_flag = 1;
            return false;
        }
        __nanosleep(64);
    }
}

// a1: gate/up (GLU, f16 output, no read-ahead factors), a2: down (BF16 output); the same
// tile list.  sync[0]: ticket counter; sync[1 + t]: finished gate/up item-warps of tile
// t; both zero before the launch.
template <int NS>
__global__ void __launch_bounds__(288, 2) gemv_fused_kernel(const __grid_constant__ CUtensorMap bmap1,
                                                            const __grid_constant__ CUtensorMap bmap2,
                                                            const GemvArgs a1, const GemvArgs a2, int *sync)
{
    griddep_enter();
    using SM = GvSmem<2, NS, 8>;
    using GF = GfSmem<NS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + GF::OFF_BAR), *empty = full + NS;
    uint64_t *ifull = empty + NS, *iempty = ifull + GF_NI;
    volatile int *abort_flag = (volatile int *)(smem + GF::OFF_FLAG);
    volatile int *items = (volatile int *)(smem + GF::OFF_ITEMS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = __ldg(a1.n_tiles);
    const int mt1 = a1.rows / 128, mt2 = a2.rows / 256;
    const int total1 = n_tiles * mt1, total = total1 + n_tiles * mt2;
    const int nkp1 = a1.K / 256, nkp2 = a2.K / 256;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), 8);
        }
        for (int i = 0; i < GF_NI; ++i) {
            mbar_init(smem_u32(ifull + i), 1);
            mbar_init(smem_u32(iempty + i), 8);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ tickets and TMA
        if (lane == 0) {
            prefetch_tmap(&bmap1);
            prefetch_tmap(&bmap2);
            const uint64_t pol = policy_evict_first(), polb = policy_evict_last();
            uint32_t it = 0, ii = 0;
            // one ticket at a time: taking the next one an item ahead measured slower (0.7033 vs
            // 0.6995 ms per T=16 step): a ticket held ahead cannot go to a CTA that is idle
            while (!*abort_flag) {
                const int islot = ii % GF_NI;
                if (!role_wait(smem_u32(iempty + islot), ((ii / GF_NI) & 1) ^ 1, abort_flag, 0xFFFFFFFFu,
                               a1.status, 13))
                    break;
                const int item = atomicAdd(sync, 1);
                items[islot] = item < total ? item : -1;
                mbar_arrive(smem_u32(ifull + islot));
                ++ii;
                if (item >= total) break;
                const bool up = item < total1;
                const int d = up ? item : item - total1, mt = up ? mt1 : mt2;
                const int ti = d / mt, m0 = (d % mt) * (up ? 128 : 256);
                const int4 tile = __ldg((up ? a1.tiles : a2.tiles) + ti);
                const CUtensorMap *am = up ? a1.amaps + (size_t)tile.x * a1.amap_stride
                                           : a2.amaps + (size_t)tile.x * a2.amap_stride;
                const CUtensorMap *am0 = am + (up ? a1.amap_off[0] : a2.amap_off[0]);
                const CUtensorMap *am1 = am + (up ? a1.amap_off[1] : a2.amap_off[0]);
                const int m1 = up ? m0 : m0 + 128;                  // matrix slot 1: w3, or w2's next block
                if (!up) {
                    // the tile's GLU output, written by the gate/up items through the generic
                    // proxy, is read here by TMA
                    if (!gf_wait_count(sync + 1 + ti, 8 * mt1, abort_flag, a2.status)) break;
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                const CUtensorMap *bm = up ? &bmap1 : &bmap2;
                const int nkp = up ? nkp1 : nkp2;
                bool ok = true;
                for (int s = 0; s < nkp; ++s, ++it) {
                    const int slot = it % NS;
                    if (!role_wait(smem_u32(empty + slot), ((it / NS) & 1) ^ 1, abort_flag, 0xFFFFFFFFu,
                                   a1.status, 11)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(full + slot);
                    mbar_expect_tx(fb, SM::STAGE);
                    uint8_t *dst = smem + slot * SM::STAGE;
                    tma_load_2d_hint(smem_u32(dst), am0, fb, s * 128, m0, pol);
                    tma_load_2d_hint(smem_u32(dst + SM::MAT_BYTES), am1, fb, s * 128, m1, pol);
                    uint8_t *bdst = dst + 2 * SM::MAT_BYTES;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tma_load_2d_hint(smem_u32(bdst + q * 16 * 128), bm, fb, s * 256 + q * 64, tile.y, polb);
                }
                if (!ok) break;
            }
            drain_ring(full, it, NS);
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int cw = warp - 1;
        const int g8 = lane >> 2, c = lane & 3;
        const int ra_l = 16 * cw + g8;
        const float pf[2][2] = {{1.f, 1.f}, {1.f, 1.f}};
        int owed = -1;                          // tile whose counter this warp owes its last gate/up item
        auto pay = [&]() {
            if (owed >= 0) {
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(sync + 1 + owed, 1);
                owed = -1;
            }
        };
        uint32_t it = 0, ii = 0;
        for (;;) {
            const int islot = ii % GF_NI;
            if (!role_wait(smem_u32(ifull + islot), (ii / GF_NI) & 1, abort_flag, 0xFFFFFFFFu, a1.status, 14))
                break;
            const int item = items[islot];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(iempty + islot));
            ++ii;
            if (item < total1) {
                if (item < 0) break;
                const int ti = item / mt1, m0 = (item % mt1) * 128;
                const int4 tile = __ldg(a1.tiles + ti);
                const int ra = m0 + ra_l, rb = ra + 8;
                const int kb = a1.K / 32;
                const uint2 *sa[2], *sn[2] = {nullptr, nullptr};
                uint2 carry[2][2];
#pragma unroll
                for (int m = 0; m < 2; ++m)
                    sa[m] = reinterpret_cast<const uint2 *>(a1.scales[m][tile.x] + (size_t)ra * kb);
                float acc[2][2][4];
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[m][h][q] = 0.f;
                if (!gemv_k_loop<2, 2, NS, 8, 1, false>(smem, full, empty, abort_flag, a1, nkp1, ra_l, g8, c, lane,
                                                        sa, sn, false, carry, kb, it, acc))
                    break;
                pay();
                gemv_epilogue<2, GV_GLU_F16, 1, false>(a1, acc, pf, c, ra, rb, tile.y, tile.z);
                owed = ti;
            } else {
                pay();
                const int d = item - total1;
                const int ti = d / mt2, m0 = (d % mt2) * 256;
                const int4 tile = __ldg(a2.tiles + ti);
                const int ra = m0 + ra_l, rb = ra + 8;
                const int kb = a2.K / 32;
                // matrix slot m: w2 rows m0 + 128 m ..
                const uint2 *sa[2] = {reinterpret_cast<const uint2 *>(a2.scales[0][tile.x] + (size_t)ra * kb),
                                      reinterpret_cast<const uint2 *>(a2.scales[0][tile.x] + (size_t)(ra + 128) * kb)};
                const uint2 *sn[2] = {nullptr, nullptr};
                uint2 carry[2][2];
                float acc[2][2][4];
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[m][h][q] = 0.f;
                if (!gemv_k_loop<2, 2, NS, 8, 1, false>(smem, full, empty, abort_flag, a2, nkp2, ra_l, g8, c, lane,
                                                        sa, sn, false, carry, kb, it, acc))
                    break;
                gemv_epilogue<1, GV_BF16, 1, false>(a2, reinterpret_cast<const float(&)[1][2][4]>(acc[0]), pf, c,
                                                    ra, rb, tile.y, tile.z);
                gemv_epilogue<1, GV_BF16, 1, false>(a2, reinterpret_cast<const float(&)[1][2][4]>(acc[1]), pf, c,
                                                    ra + 128, rb + 128, tile.y, tile.z);
            }
        }
        pay();
    }
}

}  // namespace k3

using namespace k3;

// max_items counts 128-row work items
template <int NMAT, int NS, int MODE, int MAXNB, int WPC>
static int launch_gemv(const CUtensorMap &bmap, const GemvArgs &args, int max_items, int num_sms, cudaStream_t st)
{
    using SM = GvSmem<NMAT, NS, WPC>;
    static_assert((16 / WPC) * SM::BYTES <= 228 * 1024, "CTAs per SM");
    if (args.rows % SM::ROWS) return K3MOE_ERR_SHAPE;
    auto kern = gemv_expert_kernel<NMAT, NS, MODE, MAXNB, WPC>;
    static unsigned long long attr_set = 0;
    if (!k3_smem_attr(kern, SM::BYTES, attr_set)) return K3MOE_ERR_CUDA;
    const int items = (int)(((long long)max_items * 128 + SM::ROWS - 1) / SM::ROWS);
    const int grid = max(1, min(items, (16 / WPC) * num_sms));
    k3_launch(kern, grid, (WPC + 1) * 32, SM::BYTES, st, bmap, args);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

int k3_launch_gemv_expert(int glu, int mode, int max_nb, const CUtensorMap &bmap, const GemvArgs &args,
                          int max_items, int num_sms, cudaStream_t st)
{
    if (max_nb == 1) {
        if (glu) return launch_gemv<2, 2, GV_GLU_F16, 1, 8>(bmap, args, max_items, num_sms, st);
        // down: one CTA of 16 consumer warps per SM (measured at T=16: 0.218 vs 0.2225 ms; the
        // gate/up kernel in that form took 0.456 vs 0.433 ms)
        if (mode == GV_BF16 && args.rows % 256 == 0)
            return launch_gemv<1, 4, GV_BF16, 1, 16>(bmap, args, max_items, num_sms, st);
        if (mode == GV_BF16) return launch_gemv<1, 4, GV_BF16, 1, 8>(bmap, args, max_items, num_sms, st);
    } else {
        if (glu) return launch_gemv<2, 2, GV_GLU_F16, 2, 8>(bmap, args, max_items, num_sms, st);
        if (mode == GV_BF16) return launch_gemv<1, 4, GV_BF16, 2, 8>(bmap, args, max_items, num_sms, st);
    }
    return K3MOE_ERR_UNSUPPORTED;
}

int k3_launch_gemv_fused(const CUtensorMap &bmap1, const CUtensorMap &bmap2, const GemvArgs &a1, const GemvArgs &a2,
                         int32_t *sync, int max_items, int num_sms, cudaStream_t st)
{
    using GF = GfSmem<2>;
    static_assert(2 * GF::BYTES <= 228 * 1024, "two CTAs per SM");
    if (a1.rows % 128 || a2.rows % 256 || a1.amap_off[0] == a1.amap_off[1]) return K3MOE_ERR_SHAPE;
    auto kern = gemv_fused_kernel<2>;
    static unsigned long long attr_set = 0;
    if (!k3_smem_attr(kern, GF::BYTES, attr_set)) return K3MOE_ERR_CUDA;
    const int grid = max(1, min(max_items, 2 * num_sms));
    k3_launch(kern, grid, 288, GF::BYTES, st, bmap1, bmap2, a1, a2, sync);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}
