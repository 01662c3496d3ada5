// Tensor-core path: TMA descriptors, load-time row maxima, activation prep and
// the forward orchestration around the tcgen05 grouped expert GEMMs.
#include <string.h>
#include <algorithm>
#include <vector>

#include "tc.h"
#include "tc_expert.cuh"
#include "gemv_expert.h"
#include "dense_tc.h"
#include "mx_expert.h"

using namespace k3;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// Packed MXFP4 matrix [rows, cols/2] bytes: box 128 bytes x 128 rows, 128-byte swizzle.
bool encode_packed(CUtensorMap *m, const void *base, int rows, int cols)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(cols / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols / 2)};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// f16 rows [rows, cols]: box 64 x bn rows, 128-byte swizzle (bn = 16: tiles load
// only the 16-row boxes their rows need).
bool encode_act(CUtensorMap *m, const void *base, int rows, int cols, int bn)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)bn};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_act_maps(ActMaps *m, const void *base, int rows, int cols)
{
    return encode_act(&m->big, base, rows, cols, EX_BBIG) && encode_act(&m->small, base, rows, cols, EX_BBOX);
}

// rowmax[row] = max scale byte of the row; grid over (rows, groups).
__global__ void rowmax_kernel(const uint8_t *const *tab, int groups, int rows, int kblk, uint8_t *out)
{
    const int g = blockIdx.y;
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= groups || r >= rows) return;
    const uint8_t *p = tab[g] + (size_t)r * kblk;
    uint32_t m = 0;
    for (int i = 0; i < kblk; i += 16) {
        uint4 v = *reinterpret_cast<const uint4 *>(p + i);
        m = max(m, __vmaxu4(__vmaxu4(v.x, v.y), __vmaxu4(v.z, v.w)));
    }
    m = max(max(m & 0xFF, (m >> 8) & 0xFF), max((m >> 16) & 0xFF, m >> 24));
    out[(size_t)g * rows + r] = (uint8_t)m;
}

// One CTA per token: amax of the BF16 row, power-of-two factor 2^k with
// amax * 2^k in [2^14, 2^15), f16 copies of the scaled row to each permuted row
// of the token (row_of[t*K + k]) or to row t (row_of == nullptr), and the
// inverse factor 2^-k per written row.  With `bound` (bound[0] bound[1] >= the
// largest gate row norm times the largest up row norm of the GLU this row feeds)
// it also writes ascale[row] = 2^j, the smallest power of two with
// bound ||h||^2 2^-j <= 2^15: the GLU output |silu(g) u| <= |g| |u| <= bound ||h||^2
// divided by 2^j is inside the f16 range whatever the token's scale.
__global__ void __launch_bounds__(256) prep_f16_rows_kernel(const uint16_t *__restrict__ src, int cols,
                                                           const int32_t *__restrict__ row_of, int K,
                                                           __half *__restrict__ dst,
                                                           float *__restrict__ rscale,
                                                           const float *__restrict__ bound,
                                                           float *__restrict__ ascale, int32_t *__restrict__ zero,
                                                           int zero_n)
{
    griddep_enter();
    const int t = blockIdx.x, tid = threadIdx.x;
    // block (0, 0) also clears the fused decode GEMV's counters
    if (zero && t == 0 && blockIdx.y == 0)
        for (int i = tid; i < zero_n; i += blockDim.x) zero[i] = 0;
    const uint16_t *s = src + (size_t)t * cols;
    float amax = 0.f;
    for (int i = tid * 8; i < cols; i += 256 * 8) {
        uint4 v = *reinterpret_cast<const uint4 *>(s + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            amax = fmaxf(amax, fabsf(__uint_as_float(w[q] << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(w[q] & 0xffff0000u)));
        }
    }
    __shared__ float red[8];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
    int k = 0;
    if (amax > 0.f && amax <= 3.0e38f) {
        int ex;
        frexpf(amax, &ex);                 // amax = m 2^ex, m in [0.5, 1)
        k = 15 - ex;                        // amax 2^k in [2^14, 2^15)
        k = max(-126, min(126, k));
    }
    const float up = __uint_as_float((uint32_t)(k + 127) << 23);
    const float down = __uint_as_float((uint32_t)(127 - k) << 23);
    float a_fac = 1.f;
    if (bound) {
        // S = sum (h 2^k)^2 (each term < 2^30), ||h||^2 = S 2^-2k
        float ss = 0.f;
        for (int i = tid * 8; i < cols; i += 256 * 8) {
            uint4 v = *reinterpret_cast<const uint4 *>(s + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float lo = __uint_as_float(w[q] << 16) * up, hi = __uint_as_float(w[q] & 0xffff0000u) * up;
                ss = fmaf(lo, lo, fmaf(hi, hi, ss));
            }
        }
        __syncthreads();                    // red[] is reused
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        ss = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) ss += red[w];
        const float c = bound[0] * bound[1];
        if (ss > 0.f && c > 0.f) {
            int ec, es;
            frexpf(c, &ec);
            frexpf(ss, &es);                // log2(c S 2^-2k) < ec + es - 2k
            const int j = max(0, min(126, ec + es - 2 * k - 15));
            a_fac = __uint_as_float((uint32_t)(j + 127) << 23);
        }
    }
    for (int kk = blockIdx.y; kk < K; kk += gridDim.y) {     // this CTA's copies of the row
        const int row = row_of ? row_of[(size_t)t * K + kk] : t;
        __half *d = dst + (size_t)row * cols;
        for (int i = tid * 8; i < cols; i += 256 * 8) {
            uint4 v = *reinterpret_cast<const uint4 *>(s + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint4 o;
            uint32_t *op = &o.x;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                __half2 hh = __floats2half2_rn(__uint_as_float(w[q] << 16) * up,
                                               __uint_as_float(w[q] & 0xffff0000u) * up);
                op[q] = *reinterpret_cast<uint32_t *>(&hh);
            }
            *reinterpret_cast<uint4 *>(d + i) = o;
        }
        if (tid == 0) {
            rscale[row] = down;
            if (ascale) ascale[row] = a_fac;
        }
    }
}

// Largest row L2 norm of dequantised MXFP4 matrices [rows, K] (one per group), as a
// float atomically maxed into *out (bit pattern of a non-negative float): the
// E2M1 magnitudes squared per 32-value block (exact in fp32) times 2^(2(e - 127)),
// summed in fp64.
__global__ void row_norm_max_kernel(const uint8_t *const *ptab, const uint8_t *const *stab, int rows, int K,
                                    unsigned int *out)
{
    const int g = blockIdx.y;
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    float n = 0.f;
    if (r < rows) {
        const uint8_t *p = ptab[g] + (size_t)r * (K / 2);
        const uint8_t *sc = stab[g] + (size_t)r * (K / 32);
        double acc = 0.0;
        for (int b = 0; b < K / 32; ++b) {
            const uint4 v = *reinterpret_cast<const uint4 *>(p + 16 * b);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            float sq = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float m = e2m1_to_f32((w[q] >> (4 * c)) & 0xFu, 1.f);
                    sq = fmaf(m, m, sq);
                }
            acc += ldexp((double)sq, 2 * ((int)sc[b] - 127));
        }
        n = (float)fmin(sqrt(acc), 3.0e38);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) n = fmaxf(n, __shfl_xor_sync(0xffffffffu, n, off));
    if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(n));
}

// CTAs per token for prep_f16_rows_kernel: the K copies of a row are spread
// over up to K CTAs while the grid is below two CTAs per SM.
static unsigned prep_split(int T, int K, int num_sms)
{
    int p = 1;
    while (p < K && (long)T * p * 2 <= 2L * num_sms) p *= 2;
    return (unsigned)std::min(p, K);
}

// Token tiles of a dense (all-token) GEMM: (0, row0, rows) with at most bn rows.
__global__ void dense_tiles_kernel(int T, int bn, int4 *tiles, int32_t *count)
{
    griddep_enter();
    const int n = (T + bn - 1) / bn;
    for (int i = threadIdx.x; i < n; i += blockDim.x) tiles[i] = make_int4(0, i * bn, min(bn, T - i * bn), 0);
    if (threadIdx.x == 0) *count = n;
}

template <int NMAT, int BN, int NS, int NB, int NA, int NACC, int MODE, bool ATMEM = false, int EPI = EPI_SILU>
int launch_expert(const ActMaps &bmap, const ExpertGemmArgs &a, int max_tiles, int num_sms, cudaStream_t st)
{
    using SM = ExpertSmem<NMAT, BN, NS, NB, NA, ATMEM>;
    static_assert(SM::BYTES <= 227 * 1024, "shared memory");
    auto kern = expert_gemm_kernel<NMAT, BN, NS, NB, NA, NACC, MODE, ATMEM, EPI>;
    static unsigned long long attr_set = 0;
    if (!k3_smem_attr(kern, SM::BYTES, attr_set)) return K3MOE_ERR_CUDA;
    const int grid = max(1, min(num_sms, max_tiles));
    k3_launch(kern, grid, ex_threads(NMAT, ex_nepi(BN, MODE, EPI)), SM::BYTES, st, bmap, a);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

// Tile shape by rows per expert: decode batches (<= 24 on average) take the
// GEMV; up to 192 on average (partly filled tiles) take 192-token tiles with the
// decoded weights in TMEM, which keeps shared memory below its bandwidth limit;
// more take 256-token tiles, which amortise the dequantisation and the epilogue
// over more tokens.
int pick_bn(int T, int K, int E)
{
    const size_t R = (size_t)T * K;
    if (R <= (size_t)E * 24) return 32;
    return R <= (size_t)E * 192 ? 192 : 256;
}

}  // namespace

bool k3_tc_available() { return encode_fn() != nullptr; }

// [w1, w3, w2] per expert, the shared experts' three; with the A8 option also the
// block-scaled GEMMs' FP4 weight maps [w1, w3, w2] per expert, then their scale maps.
size_t k3_tc_tmap_count(const k3moe_config &c) { return (size_t)3 * c.n_experts + 3 + (c.a8 ? (size_t)6 * c.n_experts : 0); }

namespace k3 {
bool k3_encode_mx_weight(CUtensorMap *m, const void *packed, int rows, int cols);
bool k3_encode_mx_scale(CUtensorMap *m, const void *scale, int rows, int cols);
}

size_t k3_tc_hilo_bytes(const k3moe_config &c)
{
    return c.router_dtype == K3MOE_ROUTER_F32 ? (size_t)c.n_experts * 2 * c.hidden * 2 : 0;
}

size_t k3_tc_rowmax_bytes(const k3moe_config &c)
{
    return (size_t)c.n_experts * (2 * c.inter + c.latent) + (size_t)2 * c.shared_inter +
           (c.shared_inter ? c.hidden : 0) + 64;
}

int k3_tc_prepare(k3moe_handle *h, const uint8_t *const *const tabs[6], cudaStream_t st)
{
    const k3moe_config &c = h->cfg;
    const int E = c.n_experts, L = c.latent, I = c.inter, H = c.hidden, S = c.shared_inter;
    if (!encode_fn()) return K3MOE_OK;          // tensor path unavailable; generic path serves
    std::vector<CUtensorMap> maps(k3_tc_tmap_count(c));
    memset(maps.data(), 0, maps.size() * sizeof(CUtensorMap));
    for (int e = 0; e < E; ++e) {
        if (!encode_packed(&maps[3 * e + 0], tabs[0][e], I, L)) return K3MOE_ERR_CUDA;
        if (!encode_packed(&maps[3 * e + 1], tabs[2][e], I, L)) return K3MOE_ERR_CUDA;
        if (!encode_packed(&maps[3 * e + 2], tabs[4][e], L, I)) return K3MOE_ERR_CUDA;
    }
    if (S > 0) {
        if (!encode_packed(&maps[3 * E + 0], h->shared[0], S, H)) return K3MOE_ERR_CUDA;
        if (!encode_packed(&maps[3 * E + 1], h->shared[2], S, H)) return K3MOE_ERR_CUDA;
        if (!encode_packed(&maps[3 * E + 2], h->shared[4], H, S)) return K3MOE_ERR_CUDA;
    }
    if (c.a8) {
        // block-scaled expert GEMMs: FP4 weights unpacked by TMA, and their scale bytes
        CUtensorMap *mw = maps.data() + 3 * E + 3, *ms = mw + 3 * E;
        for (int e = 0; e < E; ++e) {
            if (!k3_encode_mx_weight(&mw[3 * e + 0], tabs[0][e], I, L) ||
                !k3_encode_mx_weight(&mw[3 * e + 1], tabs[2][e], I, L) ||
                !k3_encode_mx_weight(&mw[3 * e + 2], tabs[4][e], L, I) ||
                !k3_encode_mx_scale(&ms[3 * e + 0], tabs[1][e], I, L) ||
                !k3_encode_mx_scale(&ms[3 * e + 1], tabs[3][e], I, L) ||
                !k3_encode_mx_scale(&ms[3 * e + 2], tabs[5][e], L, I))
                return K3MOE_ERR_CUDA;
        }
    }
    K3_CUDA_TRY(cudaMemcpyAsync(h->d_tmaps, maps.data(), maps.size() * sizeof(CUtensorMap),
                                cudaMemcpyHostToDevice, st));
    // per-row maximum exponent: [w1 E*I][w3 E*I][w2 E*L][ws1 S][ws3 S][ws2 H]
    uint8_t *rm = h->d_rowmax;
    rowmax_kernel<<<dim3((I + 127) / 128, E), 128, 0, st>>>(h->d_eptr[1], E, I, L / 32, rm);
    rowmax_kernel<<<dim3((I + 127) / 128, E), 128, 0, st>>>(h->d_eptr[3], E, I, L / 32, rm + (size_t)E * I);
    rowmax_kernel<<<dim3((L + 127) / 128, E), 128, 0, st>>>(h->d_eptr[5], E, L, I / 32, rm + (size_t)2 * E * I);
    if (S > 0) {
        uint8_t *rs = rm + (size_t)E * (2 * I + L);
        rowmax_kernel<<<dim3((S + 127) / 128, 1), 128, 0, st>>>(k3_shared_tab(h, 1), 1, S, H / 32, rs);
        rowmax_kernel<<<dim3((S + 127) / 128, 1), 128, 0, st>>>(k3_shared_tab(h, 3), 1, S, H / 32, rs + S);
        rowmax_kernel<<<dim3((H + 127) / 128, 1), 128, 0, st>>>(k3_shared_tab(h, 5), 1, H, S / 32, rs + 2 * S);
    }
    if (c.router_dtype == K3MOE_ROUTER_F32) {
        int rc = k3_launch_split_hilo((const float *)h->w_router, E, H, h->d_router_hilo, st);
        if (rc) return rc;
    }
    // bounds of the GLU outputs: largest gate and up row norms [routed w1, w3, shared ws1, ws3]
    unsigned int *nb = (unsigned int *)h->d_glu_bound;
    K3_CUDA_TRY(cudaMemsetAsync(nb, 0, 4 * sizeof(float), st));
    row_norm_max_kernel<<<dim3((I + 127) / 128, E), 128, 0, st>>>(h->d_eptr[0], h->d_eptr[1], I, L, nb);
    row_norm_max_kernel<<<dim3((I + 127) / 128, E), 128, 0, st>>>(h->d_eptr[2], h->d_eptr[3], I, L, nb + 1);
    if (S > 0) {
        row_norm_max_kernel<<<dim3((S + 127) / 128, 1), 128, 0, st>>>(k3_shared_tab(h, 0), k3_shared_tab(h, 1), S, H,
                                                                       nb + 2);
        row_norm_max_kernel<<<dim3((S + 127) / 128, 1), 128, 0, st>>>(k3_shared_tab(h, 2), k3_shared_tab(h, 3), S, H,
                                                                       nb + 3);
    }
    K3_CUDA_TRY(cudaGetLastError());
    return K3MOE_OK;
}

// Split-K factors for one launch of a decode-size dense GEMM (128 weight rows per
// tile): the weight-stationary kernel (ws: all T tokens in one MMA N) or the
// token-major one (ceil(T / 128) token tiles).  The kernel takes its units
// (segment 0's tiles first; per tile its splits in order, the split sizes
// differing by at most one K step) round-robin over `grid_max` CTAs.  Costs are
// in K steps (16 KB of weights): a unit costs its K steps plus its fp32 partial
// tile (rows x 128 x 4 bytes = rows / 32 K steps), and the reduction reads every
// partial once (counted as spread over the whole GPU; in the weight-stationary
// kernel the last split of each tile reads its tile's partials).  The plan
// minimises the busiest CTA's load plus the reduction; ties go to fewer units.
static void plan_splits(DenseSeg *seg, int nseg, int T, int grid_max, bool ws)
{
    const int mt = ws ? 1 : (T + 127) / 128;
    int ks_total[2], maxsp[2];
    for (int s = 0; s < nseg; ++s) {
        ks_total[s] = seg[s].K / 64;
        maxsp[s] = std::min(K3_DENSE_MAX_SPLITS, ks_total[s]);
    }
    std::vector<double> load;
    double best = 1e30;
    int best_units = 0, best_sp[2] = {1, 1};
    for (int s0 = 1; s0 <= maxsp[0]; ++s0)
        for (int s1 = 1; s1 <= (nseg > 1 ? maxsp[1] : 1); ++s1) {
            const int sp[2] = {s0, s1};
            int units = 0;
            double reduce = 0;
            for (int s = 0; s < nseg; ++s) {
                units += seg[s].n_tiles * mt * sp[s];
                reduce += (double)sp[s] * T * seg[s].n_out * 4.0;
            }
            const int grid = std::min(units, grid_max);
            load.assign(grid, 0.0);
            int u = 0;
            for (int s = 0; s < nseg; ++s)
                for (int t = 0; t < seg[s].n_tiles * mt * sp[s]; ++t, ++u) {
                    const int k = t % sp[s], m = (t / sp[s]) % mt;
                    const int rows = ws ? T : std::min(128, T - 128 * m);
                    load[u % grid] += (k + 1) * ks_total[s] / sp[s] - k * ks_total[s] / sp[s] + rows / 32.0;
                }
            const double cost = *std::max_element(load.begin(), load.end()) + reduce / (16384.0 * grid_max);
            if (cost < best - 1e-9 || (cost < best + 1e-9 && units < best_units)) {
                best = cost;
                best_units = units;
                best_sp[0] = s0;
                best_sp[1] = s1;
            }
        }
    for (int s = 0; s < nseg; ++s) seg[s].splits = best_sp[s];
}

// Cached per token count in the handle (the plan depends only on T and the shapes).
static void dense_splits(k3moe_handle *h, DenseSeg *seg, int nseg, int T, int slot, bool ws)
{
    unsigned char *c = h->dense_splits[T] + slot;
    if (!c[0]) {
        plan_splits(seg, nseg, T, 2 * h->num_sms, ws);
        for (int s = 0; s < nseg; ++s) c[s] = (unsigned char)seg[s].splits;
    }
    for (int s = 0; s < nseg; ++s) seg[s].splits = c[s];
}

// Up to 64 tokens the decode-size dense GEMMs run weight-stationary: the token
// tile of the token-major kernel would be mostly padding, and the smaller stage
// allows a deeper ring (measured at T = 16: router + down_proj 22.7 -> 21.2 us,
// up_proj 24.2 -> 19.4 us with stage events; at T = 256 the token-major kernel
// is faster).
static bool dense_ws(int T) { return T <= 64; }

// Decode-size token counts use BN = 128 tiles and split-K into fp32 partials
// (two CTAs per SM); larger counts use BN = 256 tiles writing outputs directly.
static bool dense_small(const k3_ws &ws, int T, size_t width)
{
    return T <= 256 && ws.part_floats >= (size_t)K3_DENSE_MAX_SPLITS * T * width;
}

// Token tiles per group of the token-major dense GEMM: about 32 MiB of activation rows
// (K columns of BF16), which with the weights (at most 51 MB here) stays inside the
// 129 MB L2 while every weight tile passes over the group.  Without groups each wave of
// tiles re-reads all the activation rows from HBM once T x K no longer fits in L2
// (T=32768: router + down_proj 2.15 -> 1.94 ms, up_proj 1.57 -> 1.38 ms; 64 and 16 MiB
// groups measured within 2% of 32).
static int dense_m_group(int K) { return max(1, (32 << 20) / (128 * K * 2)); }

// Router logits (fp32) and the latent h (BF16) in one tcgen05 launch.
static int dense_router_down(k3moe_handle *h, const void *x, int T, const k3_ws &ws, cudaStream_t st)
{
    const k3moe_config &c = h->cfg;
    const int H = c.hidden, L = c.latent, E = c.n_experts;
    const int Ep = (E + 15) & ~15;
    const bool small = dense_small(ws, T, (size_t)Ep + L);
    const int bn = small ? 128 : 256;
    const bool hilo = c.router_dtype == K3MOE_ROUTER_F32;
    CUtensorMap ax, br, bd;
    // decode sizes run the weight-stationary kernel, whose x tile holds only T rows (rounded up)
    const bool ws_k = small && dense_ws(T);
    if (!k3_encode_bf16_rows(&ax, x, T, H, ws_k ? k3_dense_ws_rows(T) : 128) ||
        !k3_encode_bf16_rows(&br, hilo ? (const void *)h->d_router_hilo : h->w_router, E, hilo ? 2 * H : H, bn) ||
        !k3_encode_bf16_rows(&bd, h->w_down, L, H, bn))
        return K3MOE_ERR_CUDA;
    DenseArgs a = {};
    a.nseg = 2;
    a.M = T;
    a.status = h->d_status;
    DenseSeg &r = a.seg[0], &d = a.seg[1];
    r.n_out = E;
    r.n_tiles = (E + bn - 1) / bn;
    r.K = hilo ? 2 * H : H;
    r.a_kmod = H;
    d.n_out = L;
    d.n_tiles = (L + bn - 1) / bn;
    d.K = H;
    d.a_kmod = H;
    if (small) {
        // split both segments so that the busiest CTA streams as few weight bytes as possible
        dense_splits(h, a.seg, 2, T, 0, dense_ws(T));
        // partial columns: router [0, Ep), down [Ep, Ep + L); Ep rounds E to 16 floats
        r.mode = d.mode = DN_OUT_F32;
        r.out = d.out = ws.part;
        r.ldo = d.ldo = Ep + L;
        r.col0 = 0;
        d.col0 = Ep;
        if (ws_k) {
            // the last split of each tile writes the logits (fp32) and h (BF16) itself
            a.tile_cnt = h->d_dense_cnt;
            r.red_out = ws.logits;
            r.red_mode = DN_OUT_F32;
            r.red_ldo = E;
            d.red_out = ws.h;
            d.red_mode = DN_OUT_BF16;
            d.red_ldo = L;
        }
    } else {
        r.splits = d.splits = 1;
        r.m_group = d.m_group = dense_m_group(H);
        r.mode = DN_OUT_F32;
        r.out = ws.logits;
        r.ldo = E;
        r.col0 = 0;
        d.mode = DN_OUT_BF16;
        d.out = ws.h;
        d.ldo = L;
        d.col0 = 0;
    }
    int rc;
    {
        k3_stage sg(h, K3MOE_STAGE_ROUTER, st);
        if ((rc = ws_k ? k3_launch_dense_ws(ax, br, bd, a, h->num_sms, st)
                       : k3_launch_dense_tc(small ? 128 : 256, ax, br, bd, a, h->num_sms, st)))
            return rc;
    }
    if (small && !ws_k) {
        k3_stage sg(h, K3MOE_STAGE_DOWN, st);
        if ((rc = k3_launch_dense_reduce(ws.part, r.splits, T, Ep + L, 0, E, ws.logits, nullptr, E, st))) return rc;
        if ((rc = k3_launch_dense_reduce(ws.part, d.splits, T, Ep + L, Ep, L, nullptr, ws.h, L, st))) return rc;
    }
    return K3MOE_OK;
}

// o32 = nrm W_up^T (fp32) on tcgen05; with out16 (no shared experts) the BF16
// output is written directly and o32 is not touched.
static int dense_up(k3moe_handle *h, int T, const k3_ws &ws, uint16_t *out16, cudaStream_t st)
{
    const k3moe_config &c = h->cfg;
    const int H = c.hidden, L = c.latent;
    const bool small = dense_small(ws, T, (size_t)H);
    const int bn = small ? 128 : 256;
    CUtensorMap an, bu;
    const bool ws_k = small && dense_ws(T);
    if (!k3_encode_bf16_rows(&an, ws.nrm, T, L, ws_k ? k3_dense_ws_rows(T) : 128) ||
        !k3_encode_bf16_rows(&bu, h->w_up, H, L, bn))
        return K3MOE_ERR_CUDA;
    DenseArgs a = {};
    a.nseg = 1;
    a.M = T;
    a.status = h->d_status;
    DenseSeg &u = a.seg[0];
    u.n_out = H;
    u.n_tiles = (H + bn - 1) / bn;
    u.K = L;
    u.a_kmod = L;
    u.mode = (!small && out16) ? DN_OUT_BF16 : DN_OUT_F32;
    u.col0 = 0;
    u.ldo = H;
    u.splits = 1;
    u.m_group = dense_m_group(L);
    if (small) dense_splits(h, a.seg, 1, T, 2, dense_ws(T));
    u.out = small ? (void *)ws.part : (out16 ? (void *)out16 : (void *)ws.o32);
    if (ws_k) {
        // the last split of each tile writes the output itself
        a.tile_cnt = h->d_dense_cnt + h->dense_cnt_up;
        u.red_out = out16 ? (void *)out16 : (void *)ws.o32;
        u.red_mode = out16 ? DN_OUT_BF16 : DN_OUT_F32;
        u.red_ldo = H;
    }
    int rc = ws_k ? k3_launch_dense_ws(an, bu, bu, a, h->num_sms, st) : k3_launch_dense_tc(bn, an, bu, bu, a, h->num_sms, st);
    if (rc) return rc;
    if (small && !ws_k)
        rc = k3_launch_dense_reduce(ws.part, u.splits, T, H, 0, H, out16 ? nullptr : ws.o32, out16, H, st);
    return rc;
}

// Ring depths per tile shape: (packed stages NS, activation slots NB, f16 A slots NA,
// accumulator sets NACC).  N <= 32 (shared experts at small T): gate/up 3/4/2/2
// (176 KB smem), down 4/4/4/2 (144 KB).  N <= 192: both 4/4/2/1 with the A slots
// in TMEM (2 x 192 accumulator + 2 x 2 x 32 A columns = 512; 227 KB smem): their
// dequant warps hold a packed stage until its last sub-step, so a fourth stage
// beats a fifth activation slot (T=8192: gate/up 4.88 vs 4.91 ms with 3/5).
// N <= 256: both 2/3/2/1 (224 KB; 512 TMEM columns).  The down projection takes
// 256 weight rows per job (two 128-row blocks against one activation tile,
// halving activation traffic).
// The gate/up GEMM of tile shape bn with GLU variant EPI.
template <int EPI>
static int launch_glu(int bn, const ActMaps &b1, const ExpertGemmArgs &a1, int max_tiles1, int ns, cudaStream_t st)
{
    return bn == 32    ? launch_expert<2, 32, 3, 4, 2, 2, OUT_GLU_F16, false, EPI>(b1, a1, max_tiles1, ns, st)
           : bn == 192 ? launch_expert<2, 192, 4, 4, 2, 1, OUT_GLU_F16, true, EPI>(b1, a1, max_tiles1, ns, st)
                       : launch_expert<2, 256, 2, 3, 2, 1, OUT_GLU_F16, false, EPI>(b1, a1, max_tiles1, ns, st);
}

static int expert_pair(k3moe_handle *h, int bn, const ActMaps &b1, const ActMaps &b2,
                       ExpertGemmArgs a1, ExpertGemmArgs a2, int max_tiles1, int max_tiles2,
                       cudaStream_t st, int stage1, int stage2, bool add)
{
    int rc;
    const int ns = h->num_sms;
    {
        k3_stage sg(h, stage1, st);
        const int epi = a1.a8 ? EPI_A8 : a1.act.kind == K3MOE_ACT_SITU ? EPI_SITU : EPI_SILU;
        rc = epi == EPI_A8     ? launch_glu<EPI_A8>(bn, b1, a1, max_tiles1, ns, st)
             : epi == EPI_SITU ? launch_glu<EPI_SITU>(bn, b1, a1, max_tiles1, ns, st)
                               : launch_glu<EPI_SILU>(bn, b1, a1, max_tiles1, ns, st);
        if (rc) return rc;
    }
    {
        k3_stage sg(h, stage2, st);
        // the tile list was cut at bn rows: the kernel's BN must equal bn
        // shared-expert down projections (add) always run at 256 tokens or at 32
        if (add)
            rc = bn == 32 ? launch_expert<1, 32, 4, 4, 4, 2, OUT_BF16_ADD>(b2, a2, max_tiles2, ns, st)
                          : launch_expert<2, 256, 2, 3, 2, 1, OUT_BF16_ADD>(b2, a2, max_tiles2, ns, st);
        else
            rc = bn == 32    ? launch_expert<1, 32, 4, 4, 4, 2, OUT_BF16>(b2, a2, max_tiles2, ns, st)
                 : bn == 192 ? launch_expert<2, 192, 4, 4, 2, 1, OUT_BF16, true>(b2, a2, max_tiles2, ns, st)
                             : launch_expert<2, 256, 2, 3, 2, 1, OUT_BF16>(b2, a2, max_tiles2, ns, st);
    }
    return rc;
}

// Combine + RMSNorm, the up-projection and the shared experts (after the routed
// experts have written y [R, L] BF16).
static int finish_tc(k3moe_handle *h, const void *x, int T, void *out, const k3_ws &ws, cudaStream_t st)
{
    const k3moe_config &c = h->cfg;
    const int H = c.hidden, L = c.latent, E = c.n_experts, K = c.top_k, I = c.inter, S = c.shared_inter;
    const uint8_t *rm = h->d_rowmax;
    int rc;
    {
        k3_stage sg(h, K3MOE_STAGE_COMBINE, st);
        if ((rc = k3_launch_combine_norm(ws.y, 1, ws.row_of, ws.wts, h->gamma, T, K, L, c.rms_eps, ws.nrm, st)))
            return rc;
    }
    {
        k3_stage sg(h, K3MOE_STAGE_UP, st);
        if ((rc = dense_up(h, T, ws, S > 0 ? nullptr : (uint16_t *)out, st))) return rc;
    }
    if (S == 0) return K3MOE_OK;                 // the up-projection wrote the BF16 output
    if (S > 0) {
        const int sbn = T <= 64 ? 32 : 256;
        int4 *stiles = (int4 *)ws.tiles;            // the routed tile list is no longer needed
        {
            k3_stage sg(h, K3MOE_STAGE_PREP, st);
            k3_launch(prep_f16_rows_kernel, T, 256, 0, st, (const uint16_t *)x, H, nullptr, 1, (__half *)ws.xs,
                      ws.xscale, c.act == K3MOE_ACT_SITU ? nullptr : (const float *)h->d_glu_bound + 2, ws.xascale,
                      (int32_t *)nullptr, 0);
            k3_note_launch();
            k3_launch(dense_tiles_kernel, 1, 256, 0, st, T, sbn, stiles, ws.meta + 2);
            k3_note_launch();
            K3_CUDA_TRY(cudaGetLastError());
        }
        ActMaps sb1, sb2;
        if (!encode_act_maps(&sb1, ws.xs, T, H) || !encode_act_maps(&sb2, ws.sact, T, S)) return K3MOE_ERR_CUDA;
        const uint8_t *rs = rm + (size_t)E * (2 * I + L);
        ExpertGemmArgs s1 = {};
        s1.a8 = 0;                                   // the shared experts stay A16
        s1.amaps = (const CUtensorMap *)h->d_tmaps + (size_t)3 * E;
        s1.amap_stride = 3;
        s1.amap_off[0] = 0;
        s1.amap_off[1] = 1;
        s1.status = h->d_status;
        s1.spin_limit = 0xFFFFFFFFu;
        s1.scales[0] = k3_shared_tab(h, 1);
        s1.scales[1] = k3_shared_tab(h, 3);
        s1.rowmax[0] = rs;
        s1.rowmax[1] = rs + S;
        s1.rows = S;
        s1.K = H;
        s1.tiles = stiles;
        s1.n_tiles = ws.meta + 2;
        s1.rscale = ws.xscale;
        s1.ascale = ws.xascale;
        s1.act = k3_act_of(c);
        s1.out = ws.sact;
        ExpertGemmArgs s2 = s1;
        s2.amap_off[0] = s2.amap_off[1] = 2;
        s2.scales[0] = s2.scales[1] = k3_shared_tab(h, 5);
        s2.rowmax[0] = s2.rowmax[1] = rs + 2 * S;
        s2.rows = H;
        s2.K = S;
        s2.rscale = ws.xascale;
        s2.ascale = nullptr;
        s2.addend = ws.o32;                          // the up-projection's fp32 output
        s2.out = out;                                // BF16 layer output = up + shared, rounded once
        const int nt = (T + sbn - 1) / sbn;
        if ((rc = expert_pair(h, sbn, sb1, sb2, s1, s2, nt * (S / EX_BM), nt * (H / EX_BM), st,
                              K3MOE_STAGE_SHARED, K3MOE_STAGE_SHARED_DOWN, true)))
            return rc;
    }
    return K3MOE_OK;
}

int k3_forward_tc(k3moe_handle *h, const void *x, int T, void *out, const k3_ws &ws, cudaStream_t st)
{
    const k3moe_config &c = h->cfg;
    const int L = c.latent, E = c.n_experts, K = c.top_k, I = c.inter;
    const int R = T * K;
    const bool gemv = pick_bn(T, K, E) == 32;   // routed experts at decode sizes: the streaming GEMV
    // With at most two tokens per expert on average the GEMV takes tiles of at most 8 tokens
    // (an expert with more gets several tiles, each streaming its weights): its kernel for
    // 8-token tiles keeps more registers for the one K loop and runs faster.
    const int gv_nb = (size_t)T * K <= 2 * (size_t)E ? 1 : 2;
    // Then (without A8, whose GLU output is rounded by a kernel of its own) the gate/up and
    // down GEMVs run as one persistent launch, so that neither ends in a partly idle round.
    const bool gv_fused = gemv && gv_nb == 1 && !c.a8 && L % 256 == 0;
    const bool mx = c.a8 && !gemv;              // A8 at tile sizes: block-scaled MXFP4 x MXFP8 MMAs
    const int bn = mx ? MX_BN : pick_bn(T, K, E);
    int rc;
    if ((rc = dense_router_down(h, x, T, ws, st))) return rc;
    // A8 through the decode GEMV: the routed experts read h as MXFP8 (rounded in place
    // from its BF16 value); the block-scaled path quantises h in its own prep
    if (c.a8 && gemv && (rc = k3_launch_mx8_rows(ws.h, 0, ws.h, 0, (size_t)T * L, h->d_status, h->num_sms, st)))
        return rc;
    // top-K and the permutation; token tiles: <= 16 rows for the decode GEMV, bn for the tcgen05 GEMMs
    if ((rc = k3_launch_route(h, ws, T, gemv ? 8 * gv_nb : bn, st))) return rc;
    const int max_ntiles = (R + 7) / 8 + (E < R ? E : R);     // tiles of 8 rows or more
    if (mx) {
        // h as MXFP8 in expert order [R, L] (+ scales), the GLU output as MXFP8 [R, I] (+ scales)
        uint8_t *hq8 = (uint8_t *)ws.hperm, *aq8 = hq8 + (size_t)R * L;
        uint8_t *hs8 = ws.mxs, *as8 = hs8 + (size_t)R * (L / 32);
        {
            k3_stage sg(h, K3MOE_STAGE_PREP, st);
            if ((rc = k3_launch_prep_mx8(ws.h, T, L, ws.row_of, K, hq8, hs8, h->num_sms, st))) return rc;
        }
        MxActMaps mb1, mb2;
        if (!k3_encode_mx_act(&mb1, hq8, hs8, R, L) || !k3_encode_mx_act(&mb2, aq8, as8, R, I)) return K3MOE_ERR_CUDA;
        MxGemmArgs m1 = {};
        m1.wmaps = (const CUtensorMap *)h->d_tmaps + 3 * E + 3;
        m1.smaps = m1.wmaps + 3 * E;
        m1.map_stride = 3;
        m1.map_off[0] = 0;
        m1.map_off[1] = 1;
        m1.rows = I;
        m1.K = L;
        m1.tiles = (const int4 *)ws.tiles;
        m1.n_tiles = ws.meta + 1;
        m1.out_q = aq8;
        m1.out_s = as8;
        m1.status = h->d_status;
        m1.spin_limit = 0xFFFFFFFFu;
        m1.act = k3_act_of(c);
        MxGemmArgs m2 = m1;
        m2.map_off[0] = m2.map_off[1] = 2;
        m2.rows = L;
        m2.K = I;
        m2.out_q = nullptr;
        m2.out_s = nullptr;
        m2.out_bf16 = (uint16_t *)ws.y;
        {
            k3_stage sg(h, K3MOE_STAGE_GATE_UP, st);
            if ((rc = k3_launch_mx_expert(MX_GLU, mb1, m1, max_ntiles * (I / 64), h->num_sms, st))) return rc;
        }
        {
            k3_stage sg(h, K3MOE_STAGE_EXPERT_DOWN, st);
            if ((rc = k3_launch_mx_expert(MX_DOWN, mb2, m2, max_ntiles * (L / 128), h->num_sms, st))) return rc;
        }
        return finish_tc(h, x, T, out, ws, st);
    }
    {
        k3_stage sg(h, K3MOE_STAGE_PREP, st);
        // the GLU output's power-of-two divisor (SiTU outputs are bounded by 100 and need none); A8
        // through the GEMV keeps the GLU output in fp32 until its MXFP8 rounding, which applies it
        k3_launch(prep_f16_rows_kernel, dim3(T, prep_split(T, K, h->num_sms)), 256, 0, st, ws.h, L, ws.row_of, K,
                  (__half *)ws.hperm, ws.hscale, c.act == K3MOE_ACT_SITU ? nullptr : (const float *)h->d_glu_bound,
                  ws.ascale, gv_fused ? ws.gv_sync : (int32_t *)nullptr, 2 + R + E);
        k3_note_launch();
        K3_CUDA_TRY(cudaGetLastError());
    }
    ActMaps bm1, bm2;
    // the down projection's f16 input: the GLU output (MXFP8-rounded in the tcgen05 epilogue
    // with A8), or for the decode GEMV with A8 its rounding from fp32 (in hperm)
    void *act16 = (c.a8 && gemv) ? (void *)ws.hperm : (void *)ws.act;
    if (!encode_act_maps(&bm1, ws.hperm, R, L) || !encode_act_maps(&bm2, act16, R, I)) return K3MOE_ERR_CUDA;
    const uint8_t *rm = h->d_rowmax;
    ExpertGemmArgs a1 = {};
    a1.amaps = (const CUtensorMap *)h->d_tmaps;
    a1.amap_stride = 3;
    a1.amap_off[0] = 0;
    a1.amap_off[1] = 1;
    a1.scales[0] = h->d_eptr[1];
    a1.scales[1] = h->d_eptr[3];
    a1.rowmax[0] = rm;
    a1.rowmax[1] = rm + (size_t)E * I;
    a1.rows = I;
    a1.K = L;
    a1.tiles = (const int4 *)ws.tiles;
    a1.n_tiles = ws.meta + 1;
    a1.rscale = ws.hscale;
    a1.ascale = ws.ascale;                       // GLU output divided by 2^k ...
    a1.act = k3_act_of(c);
    a1.out = ws.act;
    a1.a8 = c.a8;                                // MXFP8 rounding fused in the GLU epilogue
    a1.status = h->d_status;
    a1.spin_limit = 0xFFFFFFFFu;
    ExpertGemmArgs a2 = a1;
    a2.a8 = 0;
    a2.amap_off[0] = a2.amap_off[1] = 2;
    a2.scales[0] = a2.scales[1] = h->d_eptr[5];
    a2.rowmax[0] = a2.rowmax[1] = rm + (size_t)2 * E * I;
    a2.rows = L;
    a2.K = I;
    a2.rscale = ws.ascale;                       // ... and the down projection's output multiplied by it
    a2.ascale = nullptr;
    a2.out = ws.y;
    if (gemv) {
        // few tokens per expert: streaming GEMV, FP4 decoded in registers
        GemvArgs g1 = {};
        g1.amaps = (const CUtensorMap *)h->d_tmaps;
        g1.amap_stride = 3;
        g1.amap_off[0] = 0;
        g1.amap_off[1] = 1;
        g1.scales[0] = h->d_eptr[1];
        g1.scales[1] = h->d_eptr[3];
        g1.rows = I;
        g1.K = L;
        g1.tiles = (const int4 *)ws.tiles;
        g1.n_tiles = ws.meta + 1;
        g1.rscale = ws.hscale;
        g1.ascale = c.a8 ? nullptr : ws.ascale;  // A8: fp32 GLU output, the factor applied in its rounding
        g1.act = k3_act_of(c);
        g1.out = ws.act;
        g1.out_f32 = c.a8;
        g1.status = h->d_status;
        GemvArgs g2 = g1;
        g2.out_f32 = 0;
        g2.amap_off[0] = g2.amap_off[1] = 2;
        g2.scales[0] = g2.scales[1] = h->d_eptr[5];
        g2.rows = L;
        g2.K = I;
        g2.rscale = nullptr;
        g2.ascale = ws.ascale;
        g2.out = ws.y;
        if (gv_fused) {
            // both projections in one launch (stage timing: all of it under gate/up)
            k3_stage sg(h, K3MOE_STAGE_GATE_UP, st);
            CUtensorMap gb1, gb2;
            if (!encode_act(&gb1, ws.hperm, R, L, 16) || !encode_act(&gb2, act16, R, I, 16)) return K3MOE_ERR_CUDA;
            const int items = max_ntiles * std::max(I / 128, L / 128);
            if ((rc = k3_launch_gemv_fused(gb1, gb2, g1, g2, ws.gv_sync, items, h->num_sms, st))) return rc;
            return finish_tc(h, x, T, out, ws, st);
        }
        {
            k3_stage sg(h, K3MOE_STAGE_GATE_UP, st);
            CUtensorMap gb1;
            if (!encode_act(&gb1, ws.hperm, R, L, 16)) return K3MOE_ERR_CUDA;
            if ((rc = k3_launch_gemv_expert(1, GV_GLU_F16, gv_nb, gb1, g1, max_ntiles * (I / 128), h->num_sms, st)))
                return rc;
            // A8: the GLU output (fp32) rounded to MXFP8, as the down projection's f16 input
            if (c.a8 && (rc = k3_launch_mx8_rows(ws.act, 1, ws.hperm, 2, (size_t)R * I, h->d_status, h->num_sms,
                                                 st, ws.ascale, I)))
                return rc;
        }
        {
            k3_stage sg(h, K3MOE_STAGE_EXPERT_DOWN, st);
            CUtensorMap gb2;
            if (!encode_act(&gb2, act16, R, I, 16)) return K3MOE_ERR_CUDA;
            if ((rc = k3_launch_gemv_expert(0, GV_BF16, gv_nb, gb2, g2, max_ntiles * (L / 128), h->num_sms, st)))
                return rc;
        }
    } else if ((rc = expert_pair(h, bn, bm1, bm2, a1, a2, max_ntiles * (I / EX_BM), max_ntiles * (L / EX_BM),
                                 st, K3MOE_STAGE_GATE_UP, K3MOE_STAGE_EXPERT_DOWN, false))) {
        return rc;
    }
    return finish_tc(h, x, T, out, ws, st);
}
