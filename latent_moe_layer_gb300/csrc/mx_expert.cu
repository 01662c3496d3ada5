// Block-scaled grouped expert GEMMs of the A8 option on the 5th-generation
// tensor cores: D = W B^T with W the expert's MXFP4 weights (E2M1 codes, one
// E8M0 scale per 32 values, the checkpoint's shard layout: "Kimi K3, as
// released", Gate 3 section) and B MXFP8 activations (E4M3, one E8M0 scale per
// 32 values: the K3 report review's post-training section, routed experts
// served with MXFP4 weights and MXFP8 input activations).
//
// tcgen05.mma kind::mxf8f6f4 multiplies E2M1 x E4M3 exactly and applies both
// operands' block scales itself, so nothing is dequantised: TMA unpacks the FP4
// weight rows into 16-byte groups (16U4_ALIGN16B) in the 128-byte-swizzled
// K-major layout the MMA reads, and the scale bytes move into tensor memory.
//
// One CTA per SM, persistent over jobs = (token tile, weight-row block):
//   warp 0       TMA: per 128-K stage the weight tile (two 64-row boxes) and the
//                activation rows of the tile; per 512-K group the raw scale bytes
//                (16 per row) of both operands
//   warp 1       TMEM allocation and the single MMA-issuing thread
//   warps 4..7   scale movers, one per TMEM lane quarter: per stage the stage's
//                4 scale bytes of each weight row and each token into a TMEM slot
//   warps 8..15  epilogue, two per lane quarter on alternate 16-token chunks
// Gate/up (MX_GLU): the 128-row weight tile holds 64 rows of w1 (lanes 0..63) over
// the same 64 rows of w3 (lanes 64..127), so one M = 128 MMA feeds both halves of
// the GLU and two accumulator sets of N <= 224 fit in tensor memory: the epilogue
// of one job overlaps the MMAs of the next.  The gate and up warps of a lane pair
// swap half a chunk each through shared memory, each computes the GLU output of 8
// tokens for its 32 rows, rounds it to MXFP8 over those 32 rows (one block of the
// down projection's K) and writes E4M3 bytes and the block's E8M0 scale.
// Down (MX_DOWN): 128 rows of w2 per job, BF16 outputs.
// Every wait is bounded; on expiry the CTA records K3MOE_ERR_TIMEOUT, drains its
// copies and MMAs, frees tensor memory and returns.
#include <cuda_fp8.h>

#include "mx_expert.h"
#include "ptx.cuh"

namespace k3 {

namespace {

constexpr int NS = 4;               // pipeline stages (weight tile + activation rows)
constexpr int NG = 2;               // raw scale groups in shared memory
constexpr int NSS = 5;              // scale slots in tensor memory
constexpr int SLOT_COLS = 12;       // per slot: 4 columns of weight scales (lane quarter q uses column q), 8 of token scales
constexpr int ACC_COLS = MX_BN;     // per accumulator set
constexpr int SCOL0 = 2 * ACC_COLS; // first scale slot column
static_assert(SCOL0 + NSS * SLOT_COLS <= 512, "tensor memory columns");
constexpr int NEPI = 8;
constexpr int THREADS = (8 + NEPI) * 32;

constexpr int A_BYTES = 128 * MX_KS;            // 16 KB: 128 weight rows x 128 unpacked bytes
constexpr int B_BYTES = MX_BN * MX_KS;          // 28 KB: token rows x 128 bytes
constexpr int SA_BYTES = 128 * 16;              // raw weight scales of one group
constexpr int SB_BYTES = MX_BN * 16;            // raw token scales of one group
constexpr int X_FLOATS = 4 * 2 * 2 * 32 * 8;    // GLU exchange: pairs x parity x direction x lanes x 8

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + NS * A_BYTES;
constexpr int OFF_SA = OFF_B + NS * B_BYTES;
constexpr int OFF_SB = OFF_SA + NG * SA_BYTES;
constexpr int OFF_X = OFF_SB + NG * SB_BYTES;
constexpr int OFF_BAR = OFF_X + X_FLOATS * 4;
constexpr int N_BAR = 2 * NS + 2 * NG + 2 * NSS + 4 + 8 + 1;
constexpr int SMEM_BYTES = OFF_BAR + N_BAR * 8 + 16 + 1024;
static_assert(SMEM_BYTES <= kMaxSmem, "shared memory");
static_assert(OFF_B % 1024 == 0 && B_BYTES % 1024 == 0 && OFF_SA % 1024 == 0, "swizzle atoms");

__device__ __forceinline__ bool mx_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, uint32_t limit,
                                        int *status, int where)
{
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer();
    for (uint32_t i = 1; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((i & 255u) == 0 && globaltimer() - t0 > kWaitCapNs) break;
    }
    set_status(status, K3MOE_ERR_TIMEOUT, 40 + where);
    *abort_flag = 1;
    return false;
}

__device__ __forceinline__ void mx_drain(uint64_t *full, uint32_t issued, int ring)
{
    const uint32_t n = issued < (uint32_t)ring ? issued : (uint32_t)ring;
    for (uint32_t q = 0; q < n; ++q) {
        const uint32_t i2 = issued - 1 - q;
        mbar_wait(smem_u32(full + i2 % ring), (i2 / ring) & 1, 0xFFFFFFFFu);
    }
}

// E4M3 byte of v (nearest even, saturating at +-448).
__device__ __forceinline__ uint32_t e4m3_byte(float v)
{
    return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// 2^-X as fp32 for a block scale exponent -127 <= X <= 127.
__device__ __forceinline__ float pow2_neg(int X) { return __uint_as_float((uint32_t)(127 - X) << 23); }

// CL CTAs of a cluster take the same token tile and CL consecutive weight-row
// blocks; each loads 1 / CL of the tile's activation boxes and multicasts them to
// all CL, so the activation rows cross from L2 once per cluster, not once per CTA.
template <int MODE, int CL>
__global__ void __launch_bounds__(THREADS, 1)
mx_expert_kernel(const __grid_constant__ MxActMaps bmaps, const MxGemmArgs args)
{
    griddep_enter();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(smem + OFF_BAR);
    uint64_t *full = bars, *empty = full + NS;
    uint64_t *gfull = empty + NS, *gempty = gfull + NG;
    uint64_t *sfull = gempty + NG, *sempty = sfull + NSS;
    uint64_t *tfull = sempty + NSS, *tempty = tfull + 2;
    uint64_t *xbar = tempty + 2;                                   // [4 pairs][2 parities]
    uint64_t *drain = xbar + 8;
    uint32_t *tmem_holder = (uint32_t *)(drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = args.K, nst = K / MX_KS;
    constexpr int JOB_ROWS = MODE == MX_GLU ? 64 : 128;
    const int m_tiles = args.rows / JOB_ROWS;
    const uint32_t lim = args.spin_limit;
    // job order: group jg = (tile, CL row blocks), cluster c takes groups c, c + nclusters, ...;
    // rank r of the cluster takes row block (jg % groups per tile) CL + r of the group's tile
    const int crank = CL > 1 ? (int)cluster_ctarank() : 0;
    const int cid = CL > 1 ? (int)cluster_id_x() : (int)blockIdx.x;
    const int ncl = CL > 1 ? (int)ncluster_x() : (int)gridDim.x;
    const int mg = m_tiles / CL;
    const int groups = __ldg(args.n_tiles) * mg;
    auto job_of = [&](int jg) { return (jg / mg) * m_tiles + (jg % mg) * CL + crank; };
    constexpr uint16_t CL_MASK = (uint16_t)((1u << CL) - 1u);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), CL);        // every CTA of the cluster read the slot's activations
        }
        for (int i = 0; i < NG; ++i) {
            mbar_init(smem_u32(gfull + i), 1);
            mbar_init(smem_u32(gempty + i), 4);
        }
        for (int i = 0; i < NSS; ++i) {
            mbar_init(smem_u32(sfull + i), 4);
            mbar_init(smem_u32(sempty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(tfull + i), 1);
            mbar_init(smem_u32(tempty + i), NEPI);
        }
        for (int i = 0; i < 8; ++i) mbar_init(smem_u32(xbar + i), 64);
        mbar_init(smem_u32(drain), 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    if (CL > 1) cluster_sync();          // the cluster's barriers exist before any multicast reaches them
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&bmaps.big);
            prefetch_tmap(&bmaps.small);
            prefetch_tmap(&bmaps.sbig);
            prefetch_tmap(&bmaps.ssmall);
            const uint64_t pol_w = policy_evict_first(), pol_b = policy_evict_last();
            uint32_t it = 0, git = 0;
            bool ok = true;
            // weight maps and rows of job t (the second 64-row box: up rows, or w2's next 64)
            auto job_w = [&](int t, const CUtensorMap *&w0, const CUtensorMap *&w1, int &m0, int &m1) {
                const int g = __ldg(args.tiles + t / m_tiles).x;
                w0 = args.wmaps + (size_t)g * args.map_stride + args.map_off[0];
                w1 = args.wmaps + (size_t)g * args.map_stride + args.map_off[1];
                m0 = (t % m_tiles) * JOB_ROWS;
                m1 = MODE == MX_GLU ? m0 : m0 + MX_WBOX;
            };
            for (int jg = cid; jg < groups && ok && !*abort_flag; jg += ncl) {
                const int t = job_of(jg);
                const int4 tile = __ldg(args.tiles + t / m_tiles);
                const int g = tile.x, row0 = tile.y;
                const CUtensorMap *w0, *w1;
                int m0, m1;
                job_w(t, w0, w1, m0, m1);
                const int n16 = min(MX_BN, max(16, (tile.z + 15) & ~15)) / 16;
                const int nbig = n16 / 4, nsmall = n16 % 4;
                const CUtensorMap *s0 = args.smaps + (size_t)g * args.map_stride + args.map_off[0];
                const CUtensorMap *s1 = args.smaps + (size_t)g * args.map_stride + args.map_off[1];
                for (int s = 0; s < nst; ++s, ++it) {
                    if ((s & 3) == 0) {
                        const int gs = git % NG;
                        if (!mx_wait(smem_u32(gempty + gs), ((git / NG) & 1) ^ 1, abort_flag, lim, args.status, 0)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = smem_u32(gfull + gs);
                        mbar_expect_tx(fb, SA_BYTES + n16 * 16 * 16);
                        const int x = 16 * (s >> 2);
                        const uint32_t sa = smem_u32(smem + OFF_SA + gs * SA_BYTES);
                        const uint32_t sb = smem_u32(smem + OFF_SB + gs * SB_BYTES);
                        tma_load_2d(sa, s0, fb, x, m0);
                        tma_load_2d(sa + MX_WBOX * 16, s1, fb, x, m1);
                        for (int b = 0; b < nbig; ++b) tma_load_2d(sb + b * 64 * 16, &bmaps.sbig, fb, x, row0 + 64 * b);
                        for (int b = 0; b < nsmall; ++b)
                            tma_load_2d(sb + nbig * 64 * 16 + b * 16 * 16, &bmaps.ssmall, fb, x,
                                        row0 + 64 * nbig + 16 * b);
                        ++git;
                    }
                    const int slot = it % NS;
                    if (!mx_wait(smem_u32(empty + slot), ((it / NS) & 1) ^ 1, abort_flag, lim, args.status, 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(full + slot);
                    // FP4 boxes count their packed global bytes (64 rows x 64 bytes each)
                    mbar_expect_tx(fb, 2 * MX_WBOX * (MX_KS / 2) + n16 * 16 * MX_KS);
                    const uint32_t a = smem_u32(smem + OFF_A + slot * A_BYTES);
                    const uint32_t bb = smem_u32(smem + OFF_B + slot * B_BYTES);
                    tma_load_2d_hint(a, w0, fb, MX_KS * s, m0, pol_w);
                    tma_load_2d_hint(a + MX_WBOX * MX_KS, w1, fb, MX_KS * s, m1, pol_w);
                    // activation boxes: box i from rank i % CL, multicast to the whole cluster
                    for (int i = crank; i < nbig + nsmall; i += CL) {
                        const bool big = i < nbig;
                        const uint32_t dst = bb + (big ? i * 64 * MX_KS : nbig * 64 * MX_KS + (i - nbig) * 16 * MX_KS);
                        const CUtensorMap *bm = big ? &bmaps.big : &bmaps.small;
                        const int r = big ? row0 + 64 * i : row0 + 64 * nbig + 16 * (i - nbig);
                        if (CL > 1)
                            tma_load_2d_mc(dst, bm, fb, MX_KS * s, r, CL_MASK, pol_b);
                        else
                            tma_load_2d_hint(dst, bm, fb, MX_KS * s, r, pol_b);
                    }
                }
            }
            mx_drain(full, it, NS);
            mx_drain(gfull, git, NG);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, sit = 0, tc = 0;
            bool ok = true;
            for (int jg = cid; jg < groups && ok && !*abort_flag; jg += ncl, ++tc) {
                const int t = job_of(jg);
                const int4 tile = __ldg(args.tiles + t / m_tiles);
                const int nmma = min(MX_BN, max(16, (tile.z + 15) & ~15));
                uint32_t idesc[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) idesc[kk] = idesc_mx(128, nmma, MX_E2M1, MX_E4M3, kk, kk);
                const int acc = (int)(tc & 1);
                if (!mx_wait(smem_u32(tempty + acc), ((tc >> 1) & 1) ^ 1, abort_flag, lim, args.status, 2)) break;
                tc_fence_after();
                const uint32_t dcol = tmem + acc * ACC_COLS;
                for (int s = 0; s < nst; ++s, ++it, ++sit) {
                    const int slot = it % NS, ss = sit % NSS;
                    if (!mx_wait(smem_u32(full + slot), (it / NS) & 1, abort_flag, lim, args.status, 3) ||
                        !mx_wait(smem_u32(sfull + ss), (sit / NSS) & 1, abort_flag, lim, args.status, 4)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = smem_desc_sw128(smem_u32(smem + OFF_A + slot * A_BYTES));
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(smem + OFF_B + slot * B_BYTES));
                    const uint32_t sfa = tmem + SCOL0 + ss * SLOT_COLS;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)        // 32 K (32 bytes of both operands) per MMA
                        tc_mma_mx(dcol, adesc + 2 * kk, bdesc + 2 * kk, idesc[kk], sfa, sfa + 4,
                                  (s > 0 || kk > 0) ? 1u : 0u);
                    if (CL > 1)
                        tc_commit_mc(smem_u32(empty + slot), CL_MASK);   // the slot's activations came from every rank
                    else
                        tc_commit(smem_u32(empty + slot));
                    tc_commit(smem_u32(sempty + ss));
                }
                if (!ok) break;
                tc_commit(smem_u32(tfull + acc));
            }
            tc_commit(smem_u32(drain));
            mbar_wait(smem_u32(drain), 0, 0xFFFFFFFFu);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ scale movers
        const int q = warp & 3;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        uint32_t sit = 0, git = 0;
        bool ok = true;
        for (int jg = cid; jg < groups && ok && !*abort_flag; jg += ncl) {
            const int t = job_of(jg);
            const int4 tile = __ldg(args.tiles + t / m_tiles);
            const int nmma = min(MX_BN, max(16, (tile.z + 15) & ~15));
            const int nsfb = (nmma + 31) >> 5;
            for (int s = 0; s < nst; ++s, ++sit) {
                const int gs = git % NG;
                if ((s & 3) == 0 &&
                    !mx_wait(smem_u32(gfull + gs), (git / NG) & 1, abort_flag, lim, args.status, 5)) {
                    ok = false;
                    break;
                }
                const int ss = sit % NSS;
                if (!mx_wait(smem_u32(sempty + ss), ((sit / NSS) & 1) ^ 1, abort_flag, lim, args.status, 6)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t *sa = smem + OFF_SA + gs * SA_BYTES;
                const uint8_t *sb = smem + OFF_SB + gs * SB_BYTES;
                const int sub = 4 * (s & 3);
                // weight row 32 q + lane -> lane 32 q + lane, column q of the slot
                const uint32_t wa = *reinterpret_cast<const uint32_t *>(sa + (32 * q + lane) * 16 + sub);
                uint32_t wb[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)                 // token 32 j + lane -> column 4 + j of this quarter
                    wb[j] = j < nsfb ? *reinterpret_cast<const uint32_t *>(sb + (32 * j + lane) * 16 + sub) : 0u;
                const uint32_t col = SCOL0 + ss * SLOT_COLS;
                tmem_st1(lane_base + col + q, wa);
                tmem_st8(lane_base + col + 4, wb);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(sfull + ss));
                if ((s & 3) == 3 || s == nst - 1) {
                    // the raw bytes were read with generic loads; TMA refills the group next
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(gempty + gs));
                    ++git;
                }
            }
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                            // TMEM lanes 32 q .. 32 q + 31
        const int half = (warp - 8) >> 2;                  // chunks c with c % 2 == half
        const int p = q & 1;                               // GLU: lane pair (gate quarter p, up quarter p + 2)
        const bool gate = q < 2;
        const int pair = p + 2 * half;
        float *xbuf = reinterpret_cast<float *>(smem + OFF_X);
        uint32_t tc = 0, xit = 0;
        bool bad = false, ok = true;
        for (int jg = cid; jg < groups && ok && !*abort_flag; jg += ncl, ++tc) {
            const int t = job_of(jg);
            const int4 tile = __ldg(args.tiles + t / m_tiles);
            const int row0 = tile.y, nrows = tile.z;
            const int m0 = (t % m_tiles) * JOB_ROWS;
            const int acc = (int)(tc & 1);
            if (!mx_wait(smem_u32(tfull + acc), (tc >> 1) & 1, abort_flag, lim, args.status, 7)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + acc * ACC_COLS;
            const int nchunks = (nrows + 15) >> 4;
            for (int c = half; c < nchunks; c += 2) {
                uint32_t v[16];
                tmem_ld16(tbase + c * 16, v);
                tc_wait_ld();
                if constexpr (MODE == MX_DOWN) {
                    const int orow = m0 + 32 * q + lane;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = c * 16 + j;
                        if (n < nrows)
                            args.out_bf16[(size_t)(row0 + n) * args.rows + orow] = f32_to_bf16(__uint_as_float(v[j]));
                    }
                } else {
                    // gate lanes keep tokens 0..7 of the chunk and send 8..15; up lanes the reverse
                    const int par = xit & 1;
                    float *mine = xbuf + (((pair * 2 + par) * 2 + (gate ? 0 : 1)) * 32 + lane) * 8;
                    const float *theirs = xbuf + (((pair * 2 + par) * 2 + (gate ? 1 : 0)) * 32 + lane) * 8;
                    const int so = gate ? 8 : 0, ko = gate ? 0 : 8;
                    reinterpret_cast<float4 *>(mine)[0] = make_float4(__uint_as_float(v[so]), __uint_as_float(v[so + 1]),
                                                                      __uint_as_float(v[so + 2]), __uint_as_float(v[so + 3]));
                    reinterpret_cast<float4 *>(mine)[1] = make_float4(__uint_as_float(v[so + 4]), __uint_as_float(v[so + 5]),
                                                                      __uint_as_float(v[so + 6]), __uint_as_float(v[so + 7]));
                    const uint32_t xb = smem_u32(xbar + pair * 2 + par);
                    mbar_arrive(xb);
                    if (!mx_wait(xb, (xit >> 1) & 1, abort_flag, lim, args.status, 8)) {
                        ok = false;
                        break;
                    }
                    const float4 o0 = reinterpret_cast<const float4 *>(theirs)[0];
                    const float4 o1 = reinterpret_cast<const float4 *>(theirs)[1];
                    const float other[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
                    ++xit;
                    const int nb = c * 16 + ko;                  // first token of this warp's 8
                    float a[8];
                    uint32_t pk[2] = {0u, 0u};
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float g = gate ? __uint_as_float(v[j]) : other[j];
                        const float u = gate ? other[j] : __uint_as_float(v[8 + j]);
                        float av = args.act.kind == K3MOE_ACT_SITU ? k3_glu(g, u, args.act)
                                                                    : __fdividef(g, 1.0f + __expf(-g)) * u;
                        if (nb + j >= nrows) av = 0.f;
                        bad |= !(fabsf(av) <= 3.0e38f);
                        a[j] = av;
                        pk[j >> 2] |= ((__float_as_uint(av) >> 23) & 0xFFu) << (8 * (j & 3));
                    }
                    // the block's largest exponent field per token: byte-wise maxima over the 32 rows
#pragma unroll
                    for (int o = 16; o; o >>= 1) {
                        pk[0] = __vmaxu4(pk[0], __shfl_xor_sync(0xffffffffu, pk[0], o));
                        pk[1] = __vmaxu4(pk[1], __shfl_xor_sync(0xffffffffu, pk[1], o));
                    }
                    const int orow = m0 + 32 * p + lane;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int n = nb + j;
                        if (n < nrows) {
                            const int X = mx8_scale_exp((pk[j >> 2] >> (8 * (j & 3))) & 0xFFu);
                            args.out_q[(size_t)(row0 + n) * args.rows + orow] = (uint8_t)e4m3_byte(a[j] * pow2_neg(X));
                            if (lane == 0)
                                args.out_s[(size_t)(row0 + n) * (args.rows / 32) + orow / 32] = (uint8_t)(X + 127);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(tempty + acc));
        }
        if (bad) set_status(args.status, K3MOE_ERR_RANGE, 3);
    }

    tc_fence_before();
    __syncthreads();
    // no CTA leaves while another rank may still multicast into its shared memory
    if (CL > 1) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// One CTA (128 threads) per token and copy group: thread b takes MX block b of
// the row (32 BF16 values), gives it the OCP MX scale 2^X, X = floor(log2 amax) - 8,
// and writes the E4M3 bytes and the scale byte to every expert-ordered copy of
// the token this CTA serves.
__global__ void __launch_bounds__(128) prep_mx8_kernel(const uint16_t *__restrict__ h, int L,
                                                       const int32_t *__restrict__ row_of, int K,
                                                       uint8_t *__restrict__ q, uint8_t *__restrict__ s)
{
    griddep_enter();
    const int t = blockIdx.x, nblk = L / 32;
    for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(h + (size_t)t * L + 32 * b);
        float v[32];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 w = src[i];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * i + 2 * j] = __uint_as_float(ww[j] << 16);
                v[8 * i + 2 * j + 1] = __uint_as_float(ww[j] & 0xffff0000u);
                amax = fmaxf(amax, fmaxf(fabsf(v[8 * i + 2 * j]), fabsf(v[8 * i + 2 * j + 1])));
            }
        }
        const int X = mx8_scale_exp((__float_as_uint(amax) >> 23) & 0xFFu);
        const float down = pow2_neg(X);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            o[i] = e4m3_byte(v[4 * i] * down) | e4m3_byte(v[4 * i + 1] * down) << 8 |
                   e4m3_byte(v[4 * i + 2] * down) << 16 | e4m3_byte(v[4 * i + 3] * down) << 24;
        for (int kk = blockIdx.y; kk < K; kk += gridDim.y) {
            const size_t row = (size_t)row_of[(size_t)t * K + kk];
            uint4 *dst = reinterpret_cast<uint4 *>(q + row * L + 32 * b);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            s[row * nblk + b] = (uint8_t)(X + 127);
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 mx_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &r) ==
                cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

bool encode_bytes(CUtensorMap *m, const void *base, int rows, int width, int box_w, int box_rows, bool swizzle)
{
    auto fn = mx_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)width};
    cuuint32_t box[2] = {(cuuint32_t)box_w, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// FP4 weights [rows, cols] (packed bytes [rows, cols / 2], base 32-byte aligned, cols / 2 a
// multiple of 32): boxes of 128 values x 64 rows, unpacked by TMA into 16-byte groups.
bool k3_encode_mx_weight(CUtensorMap *m, const void *packed, int rows, int cols)
{
    auto fn = mx_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols / 2)};
    cuuint32_t box[2] = {MX_KS, MX_WBOX};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void *>(packed), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E8M0 weight scales [rows, cols / 32]: boxes of 16 bytes x 64 rows.
bool k3_encode_mx_scale(CUtensorMap *m, const void *scale, int rows, int cols)
{
    return encode_bytes(m, scale, rows, cols / 32, 16, MX_WBOX, false);
}

bool k3_encode_mx_act(MxActMaps *m, const uint8_t *q, const uint8_t *s, int rows, int K)
{
    return encode_bytes(&m->big, q, rows, K, MX_KS, 64, true) && encode_bytes(&m->small, q, rows, K, MX_KS, 16, true) &&
           encode_bytes(&m->sbig, s, rows, K / 32, 16, 64, false) &&
           encode_bytes(&m->ssmall, s, rows, K / 32, 16, 16, false);
}

template <int MODE, int CL>
static int launch_mx(const MxActMaps &b, const MxGemmArgs &a, int max_jobs, cudaStream_t st)
{
    auto kern = mx_expert_kernel<MODE, CL>;
    static unsigned long long attr_set = 0;
    static int max_clusters[64] = {};
    if (!k3_smem_attr(kern, SMEM_BYTES, attr_set)) return K3MOE_ERR_CUDA;
    int dev = 0;
    K3_CUDA_TRY(cudaGetDevice(&dev));
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = THREADS;
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cfg.attrs = attr;
    if (dev >= 64) return K3MOE_ERR_UNSUPPORTED;
    if (!max_clusters[dev]) {
        // how many clusters of CL one-CTA-per-SM blocks the GPU holds at once
        int sms = 0;
        K3_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        cfg.gridDim = dim3(CL * (sms / CL), 1, 1);
        cfg.numAttrs = 1;
        int n = 0;
        K3_CUDA_TRY(cudaOccupancyMaxActiveClusters(&n, kern, &cfg));
        if (n < 1) return K3MOE_ERR_CUDA;
        max_clusters[dev] = n;
    }
    const int groups = max(1, (max_jobs + CL - 1) / CL);
    cfg.gridDim = dim3(CL * min(max_clusters[dev], groups), 1, 1);
    cfg.numAttrs = 2;
    K3_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, b, a));
    k3_note_launch();
    return K3MOE_OK;
}

int k3_launch_mx_expert(int mode, const MxActMaps &b, const MxGemmArgs &a, int max_jobs, int num_sms,
                        cudaStream_t st)
{
    (void)num_sms;
    // clusters of 4 where the weight-row blocks split evenly (the K3 shapes: 48 and 28 blocks)
    const int blocks = a.rows / (mode == MX_GLU ? 64 : 128);
    if (blocks % 4 == 0)
        return mode == MX_GLU ? launch_mx<MX_GLU, 4>(b, a, max_jobs, st) : launch_mx<MX_DOWN, 4>(b, a, max_jobs, st);
    if (blocks % 2 == 0)
        return mode == MX_GLU ? launch_mx<MX_GLU, 2>(b, a, max_jobs, st) : launch_mx<MX_DOWN, 2>(b, a, max_jobs, st);
    return mode == MX_GLU ? launch_mx<MX_GLU, 1>(b, a, max_jobs, st) : launch_mx<MX_DOWN, 1>(b, a, max_jobs, st);
}

int k3_launch_prep_mx8(const uint16_t *h, int T, int L, const int32_t *row_of, int K, uint8_t *q, uint8_t *s,
                       int num_sms, cudaStream_t st)
{
    if (T <= 0) return K3MOE_OK;
    // the K copies of a row spread over up to K CTAs while the grid is below 4 CTAs per SM
    int split = 1;
    while (split < K && (long)T * split * 2 <= 4L * num_sms) split *= 2;
    k3_launch(prep_mx8_kernel, dim3(T, min(split, K)), 128, 0, st, h, L, row_of, K, q, s);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

}  // namespace k3
