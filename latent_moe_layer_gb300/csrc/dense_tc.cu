// Dense BF16 GEMMs of the layer on tcgen05: router logits, routed_expert_down_proj
// and routed_expert_up_proj ("Kimi K3, as released": the latent MoE's two dense
// projections around the expert block; the router reads the same x).
//
// out[t, n] = sum_k X[t, k] W[n, k]: MMA M = 128 token rows (TMA; rows beyond T
// are zero-filled by the copy engine), N = BN weight rows (TMA), K in 64-wide
// steps, fp32 accumulators in TMEM.  Up to two segments of N share a launch,
// each with its own weight tensor map, K and output: the router (fp32 weights
// held as BF16 hi + lo, contracted over K' = 2H against x read twice, which
// keeps the logits fp32-accurate) and the down projection run together.
// Split-K writes fp32 partials that k3_launch_dense_reduce sums in a fixed order, or
// (weight-stationary kernel) the last split of each tile to finish sums them.
#include <cudaTypedefs.h>

#include "dense_tc.h"
#include "ptx.cuh"

namespace k3 {

constexpr int DN_BM = 128;
constexpr int DN_BK = 64;

template <int BN, int NS>
struct DenseSmem {
    static constexpr int A_BYTES = DN_BM * DN_BK * 2;   // 16 KB
    static constexpr int B_BYTES = BN * DN_BK * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int OFF_BAR = NS * STAGE;
    static constexpr int N_BAR = 2 * NS + 4 + 1;          // full/empty per stage, tfull/tempty x 2, drain
    static constexpr int BYTES = OFF_BAR + N_BAR * 8 + 16 + 1024;
};

constexpr int DN_THREADS = 320;    // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue (two per TMEM lane quarter)

__device__ __forceinline__ bool dn_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *status,
                                        int where)
{
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((i & 255u) == 0 && globaltimer() - t0 > kWaitCapNs) break;
    }
    set_status(status, K3MOE_ERR_TIMEOUT, where);
    *abort_flag = 1;
    return false;
}

struct DnTile {
    int seg, split, n0, m0, k0, ks;
};

// segment by value (a select between the two parameter copies, no indexed access)
__device__ __forceinline__ DenseSeg dn_seg(const DenseArgs &args, int seg) { return seg ? args.seg[1] : args.seg[0]; }

// tile index -> (segment, split, n tile, m tile); segment 0's tiles come first
__device__ __forceinline__ DnTile dn_tile(const DenseArgs &args, int t, int mt_n, int BN)
{
    DnTile r;
    const int per0 = args.seg[0].n_tiles * mt_n * args.seg[0].splits;
    r.seg = 0;
    if (t >= per0) {
        r.seg = 1;
        t -= per0;
    }
    const DenseSeg S = dn_seg(args, r.seg);
    r.split = t % S.splits;
    t /= S.splits;
    // groups of G token tiles, token tile fastest within a group
    const int G = S.m_group > 0 && S.m_group < mt_n ? S.m_group : mt_n;
    const int per = G * S.n_tiles, g = t / per, w = t % per;
    const int gs = min(G, mt_n - g * G);
    r.m0 = (g * G + w % gs) * DN_BM;
    r.n0 = (w / gs) * BN;
    // split s of KS K steps covers [s KS / splits, (s + 1) KS / splits): sizes differ by at most one
    const int KS = S.K / DN_BK;
    r.k0 = r.split * KS / S.splits;
    r.ks = (r.split + 1) * KS / S.splits - r.k0;
    return r;
}

// Persistent over the output tiles: the TMA ring runs across tile boundaries,
// and two TMEM accumulator sets let the epilogue of one tile overlap the
// MMAs of the next.
template <int BN, int NS>
__global__ void __launch_bounds__(DN_THREADS, 2) dense_gemm_kernel(const __grid_constant__ CUtensorMap amap,
                                                                 const __grid_constant__ CUtensorMap bmap0,
                                                                 const __grid_constant__ CUtensorMap bmap1,
                                                                 const DenseArgs args)
{
    griddep_enter();
    using SM = DenseSmem<BN, NS>;
    constexpr uint32_t TMEM_COLS = 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128 : 2 * BN <= 256 ? 256 : 512;
    static_assert(2 * BN <= 512, "two accumulator sets");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + SM::OFF_BAR), *empty = full + NS;
    uint64_t *tfull = empty + NS, *tempty = tfull + 2, *drain = tempty + 2;
    uint32_t *tmem_holder = (uint32_t *)(drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_holder + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt_n = (args.M + DN_BM - 1) / DN_BM;
    const int total = args.seg[0].n_tiles * mt_n * args.seg[0].splits +
                      (args.nseg > 1 ? args.seg[1].n_tiles * mt_n * args.seg[1].splits : 0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(tfull + i), 1);
            mbar_init(smem_u32(tempty + i), 8);
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

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        prefetch_tmap(&amap);
        prefetch_tmap(&bmap0);
        if (args.nseg > 1) prefetch_tmap(&bmap1);
        const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
        uint32_t it = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
            const DnTile d = dn_tile(args, t, mt_n, BN);
            const DenseSeg S = dn_seg(args, d.seg);
            const CUtensorMap *bm = d.seg == 0 ? &bmap0 : &bmap1;
            bool ok = true;
            for (int s = 0; s < d.ks; ++s, ++it) {
                const int slot = it % NS;
                if (!dn_wait(smem_u32(empty + slot), ((it / NS) & 1) ^ 1, abort_flag, args.status, 21)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(full + slot);
                mbar_expect_tx(fb, SM::STAGE);
                uint8_t *st = smem + slot * SM::STAGE;
                const int k = (d.k0 + s) * DN_BK;
                tma_load_2d_hint(smem_u32(st), &amap, fb, k % S.a_kmod, d.m0, pol_a);
                tma_load_2d_hint(smem_u32(st + SM::A_BYTES), bm, fb, k, d.n0, pol_w);
            }
            if (!ok) break;
        }
        const uint32_t n = it < (uint32_t)NS ? it : (uint32_t)NS;
        for (uint32_t q = 0; q < n; ++q) {
            const uint32_t i2 = it - 1 - q;
            mbar_wait(smem_u32(full + i2 % NS), (i2 / NS) & 1, 0xFFFFFFFFu);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc = idesc_f16(DN_BM, BN, 1);
        uint32_t it = 0, tc = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++tc) {
            const DnTile d = dn_tile(args, t, mt_n, BN);
            const int acc = (int)(tc & 1);
            if (!dn_wait(smem_u32(tempty + acc), ((tc >> 1) & 1) ^ 1, abort_flag, args.status, 24)) break;
            tc_fence_after();
            const uint32_t dcol = tmem + acc * BN;
            bool ok = true;
            for (int s = 0; s < d.ks; ++s, ++it) {
                const int slot = it % NS;
                if (!dn_wait(smem_u32(full + slot), (it / NS) & 1, abort_flag, args.status, 22)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + slot * SM::STAGE);
                const uint64_t adesc = smem_desc_sw128(a_addr), bdesc = smem_desc_sw128(a_addr + SM::A_BYTES);
#pragma unroll
                for (int kk = 0; kk < DN_BK / 16; ++kk)
                    tc_mma_f16(dcol, adesc + 2 * kk, bdesc + 2 * kk, idesc, (s > 0 || kk > 0) ? 1u : 0u);
                tc_commit(smem_u32(empty + slot));
            }
            if (!ok) break;
            tc_commit(smem_u32(tfull + acc));
        }
        // every issued MMA completes before TMEM is released
        tc_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, 0xFFFFFFFFu);
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue (warps 2..9)
        const int q = warp & 3;                       // TMEM lanes 32q .. 32q + 31
        const int half = (warp - 2) >> 2;             // chunks c with c % 2 == half
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++tc) {
            const DnTile d = dn_tile(args, t, mt_n, BN);
            const DenseSeg S = dn_seg(args, d.seg);
            const int acc = (int)(tc & 1);
            const int m = d.m0 + 32 * q + lane;
            if (!dn_wait(smem_u32(tfull + acc), (tc >> 1) & 1, abort_flag, args.status, 23)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + acc * BN;
            for (int c = half; c < BN / 16; c += 2) {
                uint32_t v[16];
                tmem_ld16(tbase + c * 16, v);
                tc_wait_ld();
                const int n = d.n0 + 16 * c;
                const int nv = S.n_out - n;                 // valid columns in this chunk
                if (m < args.M && nv > 0) {
                    if (S.mode == DN_OUT_F32) {
                        float *o = reinterpret_cast<float *>(S.out) + ((size_t)d.split * args.M + m) * S.ldo +
                                   S.col0 + n;
                        if (nv >= 16 && ((uintptr_t)o & 15) == 0) {
#pragma unroll
                            for (int j = 0; j < 16; j += 4)
                                *reinterpret_cast<float4 *>(o + j) = make_float4(
                                    __uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                    __uint_as_float(v[j + 3]));
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (j < nv) o[j] = __uint_as_float(v[j]);
                        }
                    } else {
                        uint16_t *o = reinterpret_cast<uint16_t *>(S.out) + (size_t)m * S.ldo + S.col0 + n;
                        if (nv >= 16 && ((uintptr_t)o & 15) == 0) {
                            uint32_t pk[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                pk[j] = (uint32_t)f32_to_bf16(__uint_as_float(v[2 * j])) |
                                        ((uint32_t)f32_to_bf16(__uint_as_float(v[2 * j + 1])) << 16);
                            *reinterpret_cast<uint4 *>(o) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            *reinterpret_cast<uint4 *>(o + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (j < nv) o[j] = f32_to_bf16(__uint_as_float(v[j]));
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

// Decode sizes (T <= TNS tokens): weight-stationary form of the same product.
// The MMA's M is 128 weight rows and its N the token count rounded to 16, so a
// stage holds a 16 KB weight tile plus only TNS activation rows, and the ring
// can be NS deep.  TMEM lanes are weight rows and columns tokens; the epilogue
// writes fp32 partials [split][token][col0 + n] (split-K mode only).
template <int TNS, int NS>
struct DenseWsSmem {
    static constexpr int A_BYTES = DN_BM * DN_BK * 2;   // 16 KB of weights
    static constexpr int B_BYTES = TNS * DN_BK * 2;     // activation rows
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int OFF_BAR = NS * STAGE;
    static constexpr int N_BAR = 2 * NS + 4 + 1;
    static constexpr int BYTES = OFF_BAR + N_BAR * 8 + 16 + 1024;
};

// Named barrier 1 over the 8 epilogue warps (256 threads); the _and form returns
// whether every thread passed a true predicate.
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool epi_bar_and(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred p, 1, 256, q;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v)
                 : "memory");
    return r != 0;
}

template <int TNS, int NS>
__global__ void __launch_bounds__(DN_THREADS, 2) dense_ws_kernel(const __grid_constant__ CUtensorMap amap,
                                                               const __grid_constant__ CUtensorMap bmap0,
                                                               const __grid_constant__ CUtensorMap bmap1,
                                                               const DenseArgs args)
{
    griddep_enter();
    using SM = DenseWsSmem<TNS, NS>;
    constexpr uint32_t TMEM_COLS = 2 * TNS <= 32 ? 32 : 2 * TNS <= 64 ? 64 : 2 * TNS <= 128 ? 128 : 2 * TNS <= 256 ? 256 : 512;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + SM::OFF_BAR), *empty = full + NS;
    uint64_t *tfull = empty + NS, *tempty = tfull + 2, *drain = tempty + 2;
    uint32_t *tmem_holder = (uint32_t *)(drain + 1);
    volatile int *abort_flag = (volatile int *)(tmem_holder + 1);
    volatile int *last_flag = (volatile int *)(tmem_holder + 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tn = min(TNS, max(16, (args.M + 15) & ~15));      // MMA N
    const int total = args.seg[0].n_tiles * args.seg[0].splits +
                      (args.nseg > 1 ? args.seg[1].n_tiles * args.seg[1].splits : 0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(tfull + i), 1);
            mbar_init(smem_u32(tempty + i), 8);
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

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------ TMA producer
        prefetch_tmap(&amap);
        prefetch_tmap(&bmap0);
        if (args.nseg > 1) prefetch_tmap(&bmap1);
        const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
        uint32_t it = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
            const DnTile d = dn_tile(args, t, 1, DN_BM);
            const DenseSeg S = dn_seg(args, d.seg);
            const CUtensorMap *bm = d.seg == 0 ? &bmap0 : &bmap1;
            bool ok = true;
            for (int s = 0; s < d.ks; ++s, ++it) {
                const int slot = it % NS;
                if (!dn_wait(smem_u32(empty + slot), ((it / NS) & 1) ^ 1, abort_flag, args.status, 25)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = smem_u32(full + slot);
                mbar_expect_tx(fb, SM::STAGE);
                uint8_t *st = smem + slot * SM::STAGE;
                const int k = (d.k0 + s) * DN_BK;
                tma_load_2d_hint(smem_u32(st), bm, fb, k, d.n0, pol_w);
                tma_load_2d_hint(smem_u32(st + SM::A_BYTES), &amap, fb, k % S.a_kmod, 0, pol_a);
            }
            if (!ok) break;
        }
        const uint32_t n = it < (uint32_t)NS ? it : (uint32_t)NS;
        for (uint32_t q = 0; q < n; ++q) {
            const uint32_t i2 = it - 1 - q;
            mbar_wait(smem_u32(full + i2 % NS), (i2 / NS) & 1, 0xFFFFFFFFu);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc = idesc_f16(DN_BM, tn, 1);
        uint32_t it = 0, tc = 0;
        for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++tc) {
            const DnTile d = dn_tile(args, t, 1, DN_BM);
            const int acc = (int)(tc & 1);
            if (!dn_wait(smem_u32(tempty + acc), ((tc >> 1) & 1) ^ 1, abort_flag, args.status, 26)) break;
            tc_fence_after();
            const uint32_t dcol = tmem + acc * TNS;
            bool ok = true;
            for (int s = 0; s < d.ks; ++s, ++it) {
                const int slot = it % NS;
                if (!dn_wait(smem_u32(full + slot), (it / NS) & 1, abort_flag, args.status, 27)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t w_addr = smem_u32(smem + slot * SM::STAGE);
                const uint64_t adesc = smem_desc_sw128(w_addr), bdesc = smem_desc_sw128(w_addr + SM::A_BYTES);
#pragma unroll
                for (int kk = 0; kk < DN_BK / 16; ++kk)
                    tc_mma_f16(dcol, adesc + 2 * kk, bdesc + 2 * kk, idesc, (s > 0 || kk > 0) ? 1u : 0u);
                tc_commit(smem_u32(empty + slot));
            }
            if (!ok) break;
            tc_commit(smem_u32(tfull + acc));
        }
        tc_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, 0xFFFFFFFFu);
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue (warps 2..9)
        const int q = warp & 3;                       // TMEM lanes 32q .. 32q + 31 = weight rows
        const int half = (warp - 2) >> 2;             // token chunks c with c % 2 == half
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const DnTile d = dn_tile(args, t, 1, DN_BM);
            const DenseSeg S = dn_seg(args, d.seg);
            const int acc = (int)(tc & 1);
            const int n = d.n0 + 32 * q + lane;          // output column (weight row)
            const bool ok = !*abort_flag && dn_wait(smem_u32(tfull + acc), (tc >> 1) & 1, abort_flag, args.status, 28);
            if (ok) {
                tc_fence_after();
                const uint32_t tbase = tmem + ((uint32_t)(32 * q) << 16) + acc * TNS;
                for (int c = half; c < tn / 16; c += 2) {
                    uint32_t v[16];
                    tmem_ld16(tbase + c * 16, v);
                    tc_wait_ld();
                    if (n < S.n_out) {
                        float *o = reinterpret_cast<float *>(S.out) + ((size_t)d.split * args.M) * S.ldo + S.col0 + n;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int m = 16 * c + j;               // token
                            if (m < args.M) o[(size_t)m * S.ldo] = __uint_as_float(v[j]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(tempty + acc));
            }
            if (!args.tile_cnt) {
                if (!ok) break;
                continue;
            }
            // The tile's last split to arrive sums the partials of all splits in split order
            // (the fixed order of the separate reduction).  The 256 epilogue threads agree on
            // continuing before any of them waits at the named barrier again.
            __threadfence();
            if (!epi_bar_and(ok)) break;
            const int id = (d.seg ? args.seg[0].n_tiles : 0) + d.n0 / DN_BM;
            if (warp == 2 && lane == 0) *last_flag = atomicAdd(args.tile_cnt + id, 1) == S.splits - 1;
            epi_bar();
            if (*last_flag) {
                // thread i: columns d.n0 + 4 (i % 32) .. +3 of token rows i / 32 + 8 j; every
                // split's 16-byte partial is loaded before the sum in split order
                __threadfence();
                const int i = threadIdx.x - 64;              // 0 .. 255
                const int col = d.n0 + 4 * (i & 31);
                if (col < S.n_out) {
                    const float *p = reinterpret_cast<const float *>(S.out) + S.col0 + col;
                    for (int m = i >> 5; m < args.M; m += 8) {
                        float r[4] = {0.f, 0.f, 0.f, 0.f};
                        for (int s0 = 0; s0 < S.splits; s0 += 8) {     // 8 splits' loads in flight
                            float4 v[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (s0 + j < S.splits)
                                    v[j] = __ldcg(reinterpret_cast<const float4 *>(
                                        p + ((size_t)(s0 + j) * args.M + m) * S.ldo));
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (s0 + j < S.splits) {
                                    r[0] += v[j].x;
                                    r[1] += v[j].y;
                                    r[2] += v[j].z;
                                    r[3] += v[j].w;
                                }
                        }
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2) {
                            if (col + q2 >= S.n_out) break;
                            const size_t o = (size_t)m * S.red_ldo + col + q2;
                            if (S.red_mode == DN_OUT_BF16)
                                reinterpret_cast<uint16_t *>(S.red_out)[o] = f32_to_bf16(r[q2]);
                            else
                                reinterpret_cast<float *>(S.red_out)[o] = r[q2];
                        }
                    }
                }
                if (i == 0) args.tile_cnt[id] = 0;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Sum split-K partials [splits][M][ldp] (columns [c0, c0 + n)) in split order.
__global__ void dense_reduce_kernel(const float *__restrict__ part, int splits, int M, int ldp, int c0, int n,
                                   float *__restrict__ out32, uint16_t *__restrict__ out16, int ldo)
{
    griddep_enter();
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)M * n) return;
    const int m = (int)(i / n), j = (int)(i % n);
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) acc += part[((size_t)s * M + m) * ldp + c0 + j];
    if (out32) out32[(size_t)m * ldo + j] = acc;
    if (out16) out16[(size_t)m * ldo + j] = f32_to_bf16(acc);
}

// Router weights fp32 [E, H] -> [E, 2H] BF16: hi = bf16(w) in columns [0, H), lo = bf16(w - hi) in [H, 2H).
__global__ void split_hilo_kernel(const float *__restrict__ w, int E, int H, uint16_t *__restrict__ out)
{
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)E * H) return;
    const size_t e = i / H, k = i % H;
    const float v = w[i];
    const uint16_t hi = f32_to_bf16(v);
    const uint16_t lo = f32_to_bf16(v - bf16_to_f32(hi));
    out[e * 2 * H + k] = hi;
    out[e * 2 * H + H + k] = lo;
}

}  // namespace k3

using namespace k3;

bool k3_encode_bf16_rows(CUtensorMap *m, const void *base, int rows, int cols, int box_rows)
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
        fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int NS>
static int launch_dense(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1, const DenseArgs &args,
                        int num_sms, cudaStream_t st)
{
    using SM = DenseSmem<BN, NS>;
    static_assert(SM::BYTES <= 227 * 1024, "shared memory");
    auto kern = dense_gemm_kernel<BN, NS>;
    static unsigned long long attr_set = 0;
    if (!k3_smem_attr(kern, SM::BYTES, attr_set)) return K3MOE_ERR_CUDA;
    const int mt = (args.M + DN_BM - 1) / DN_BM;
    int tiles = 0;
    for (int s = 0; s < args.nseg; ++s) tiles += args.seg[s].n_tiles * mt * args.seg[s].splits;
    if (tiles == 0) return K3MOE_OK;
    // persistent: as many CTAs as fit on the GPU at once (shared memory bound)
    const int per_sm = (228 * 1024) / (SM::BYTES + 1024) > 1 ? 2 : 1;
    const int grid = std::min(tiles, per_sm * num_sms);
    k3_launch(kern, grid, DN_THREADS, SM::BYTES, st, a, b0, b1, args);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

template <int TNS, int NS>
static int launch_dense_ws(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                           const DenseArgs &args, int num_sms, cudaStream_t st)
{
    using SM = DenseWsSmem<TNS, NS>;
    static_assert(2 * (SM::BYTES + 1024) <= 228 * 1024, "two CTAs per SM");
    auto kern = dense_ws_kernel<TNS, NS>;
    static unsigned long long attr_set = 0;
    if (!k3_smem_attr(kern, SM::BYTES, attr_set)) return K3MOE_ERR_CUDA;
    int tiles = 0;
    for (int s = 0; s < args.nseg; ++s) tiles += args.seg[s].n_tiles * args.seg[s].splits;
    if (tiles == 0) return K3MOE_OK;
    const int grid = std::min(tiles, 2 * num_sms);
    k3_launch(kern, grid, DN_THREADS, SM::BYTES, st, a, b0, b1, args);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

int k3_dense_ws_rows(int T) { return T <= 16 ? 16 : T <= 64 ? 64 : T <= 128 ? 128 : T <= 256 ? 256 : 0; }

int k3_launch_dense_ws(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1, const DenseArgs &args,
                       int num_sms, cudaStream_t st)
{
    for (int s = 0; s < args.nseg; ++s)
        if (args.seg[s].mode != DN_OUT_F32 || args.seg[s].n_tiles * DN_BM < args.seg[s].n_out) return K3MOE_ERR_ARG;
    switch (k3_dense_ws_rows(args.M)) {
    case 16: return launch_dense_ws<16, 6>(a, b0, b1, args, num_sms, st);
    case 64: return launch_dense_ws<64, 4>(a, b0, b1, args, num_sms, st);
    case 128: return launch_dense_ws<128, 3>(a, b0, b1, args, num_sms, st);
    case 256: return launch_dense_ws<256, 2>(a, b0, b1, args, num_sms, st);
    default: return K3MOE_ERR_UNSUPPORTED;
    }
}

int k3_launch_dense_tc(int bn, const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                       const DenseArgs &args, int num_sms, cudaStream_t st)
{
    if (bn == 128) return launch_dense<128, 3>(a, b0, b1, args, num_sms, st);   // 2 CTAs per SM (decode sizes)
    if (bn == 256) return launch_dense<256, 4>(a, b0, b1, args, num_sms, st);
    return K3MOE_ERR_UNSUPPORTED;
}

int k3_launch_dense_reduce(const float *part, int splits, int M, int ldp, int c0, int n, float *out32,
                           uint16_t *out16, int ldo, cudaStream_t st)
{
    const size_t total = (size_t)M * n;
    if (total == 0) return K3MOE_OK;
    k3_launch(dense_reduce_kernel, (unsigned)((total + 255) / 256), 256, 0, st, part, splits, M, ldp, c0, n, out32, out16,
                                                                         ldo);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

int k3_launch_split_hilo(const float *w, int E, int H, uint16_t *out, cudaStream_t st)
{
    const size_t total = (size_t)E * H;
    split_hilo_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(w, E, H, out);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}
