// Quantile-Balancing (QB) selection-bias update ("the K3 report review",
// Quantile Balancing section): each expert's next-step bias is the quantile of
// its margins that lets q = T K / E tokens cross their thresholds, estimated
// from an nbins-bin histogram (error bounded by the bin width).
//
//   s_tj     = sigmoid(l_tj)                         router score
//   alpha_t  = (K+1)-th largest of s_tj + b_j        token threshold (current bias)
//   m_tj     = alpha_t - s_tj                        margin: token t picks j iff b_j > m_tj
//   r        = round(T K / E), kept in [1, T - 1]
//   b'_j     = upper edge of the bin (of nbins equal bins over [min m, max m])
//              holding expert j's r-th smallest margin
//
// Four launches: init (counts, range), thresholds (warp per token, pruned K+1
// extractions, range folded in with order-preserving integer atomics),
// histogram (CTA per expert group x token slice, shared-memory bins), select
// (warp per expert, cumulative counts).  Integer counts make the result
// independent of atomic order.
#include "k3moe_internal.h"

namespace k3 {

// float -> uint32 with the same order (for atomicMin / atomicMax)
__device__ __forceinline__ uint32_t qb_ord(float f)
{
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float qb_unord(uint32_t u)
{
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// sigmoid with the hardware exponential: the estimate is only resolved to a
// histogram bin (about 1e-3 of the margin range), far above its error
__device__ __forceinline__ float qb_score(float l) { return 1.0f / (1.0f + __expf(-l)); }

__global__ void qb_init_kernel(int32_t *counts, size_t n, uint32_t *range)
{
    const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (size_t i = i0; i < n; i += (size_t)gridDim.x * blockDim.x) counts[i] = 0;
    if (i0 == 0) {
        range[0] = qb_ord(INFINITY);     // running minimum
        range[1] = qb_ord(-INFINITY);    // running maximum
    }
}

// Warp-wide maximum of v and the lowest lane holding it.
__device__ __forceinline__ float qb_warp_max(float v, int lane, int *who)
{
    float m = v;
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    *who = __ffs(__ballot_sync(0xffffffffu, v == m)) - 1;
    return m;
}

// Bitonic sort of one value per lane, descending over the lanes (lane 0 the largest).
__device__ __forceinline__ float qb_sort32_desc(float v, int lane)
{
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool desc = (lane & k) == 0, low = (lane & j) == 0;
            v = (low == desc) ? fmaxf(v, o) : fminf(v, o);
        }
    return v;
}

// Bitonic sort of 64 values (element i = lane + 32 h in c[h]), descending in i.
__device__ __forceinline__ void qb_sort64_desc(float (&c)[2], int lane)
{
#pragma unroll
    for (int k = 2; k <= 64; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j == 32) {                   // partners in the same lane (k = 64: descending)
                const float hi = fmaxf(c[0], c[1]), lo = fminf(c[0], c[1]);
                c[0] = hi;
                c[1] = lo;
                continue;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = lane + 32 * h;
                const float o = __shfl_xor_sync(0xffffffffu, c[h], j);
                const bool desc = (i & k) == 0, low = (i & j) == 0;
                c[h] = (low == desc) ? fmaxf(c[h], o) : fminf(c[h], o);
            }
        }
}

// One warp per token (QB_TPW tokens per warp in turn).  The (K+1)-th largest
// key is found among the keys not below L, the (K+1)-th largest of the 32
// per-lane maxima (at least K+1 keys reach L, so alpha >= L; a bitonic sort
// of the lane maxima gives L): usually a few dozen candidates, at most two per
// lane after compaction, sorted by a 64-element bitonic network.  More than 64 candidates (heavy ties) or K + 1 >
// 32 fall back to rounds over every key.  The margin range is reduced over the
// CTA and folded into the global range with one atomic pair per CTA.
constexpr int QB_TPW = 1;
template <int MAXP>
__global__ void __launch_bounds__(256) qb_alpha_kernel(const float *__restrict__ logits,
                                                       const float *__restrict__ bias, int T, int E, int K,
                                                       float *__restrict__ alpha, uint32_t *range)
{
    __shared__ float skey[8][MAXP][32];
    __shared__ float cand[8][64];
    __shared__ float rlo[8], rhi[8];
    const int wl = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float wlo = INFINITY, whi = -INFINITY;
    for (int tt = 0; tt < QB_TPW; ++tt) {
        const int t = (blockIdx.x * QB_TPW + tt) * 8 + wl;
        if (t >= T) break;
        const float *lr = logits + (size_t)t * E;
        float smax = -INFINITY, smin = INFINITY, lmax = -INFINITY;
        float lv[MAXP];                                  // all of the row's loads in flight at once
#pragma unroll
        for (int p = 0; p < MAXP; ++p) lv[p] = p * 32 + lane < E ? lr[p * 32 + lane] : 0.f;
#pragma unroll
        for (int p = 0; p < MAXP; ++p) {
            const int j = p * 32 + lane;
            float key = -INFINITY;
            if (j < E) {
                const float s = qb_score(lv[p]);
                smax = fmaxf(smax, s);
                smin = fminf(smin, s);
                key = s + (bias ? bias[j] : 0.f);
                if (key != key) key = -INFINITY;         // a NaN logit never selects
            }
            skey[wl][p][lane] = key;
            lmax = fmaxf(lmax, key);
        }
        __syncwarp();
        float a = -INFINITY;
        int who;
        bool done = false;
        if (K + 1 <= 32) {
            // L: the (K+1)-th largest lane maximum
            const float L = __shfl_sync(0xffffffffu, qb_sort32_desc(lmax, lane), K);
            // compact the keys >= L
            int c = 0;
            for (int p = 0; p < MAXP; ++p) c += skey[wl][p][lane] >= L;
            int pre = c;
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, pre, o);
                if (lane >= o) pre += u;
            }
            const int total = __shfl_sync(0xffffffffu, pre, 31);
            if (total <= 64) {
                int pos = pre - c;
                for (int p = 0; p < MAXP; ++p) {
                    const float k = skey[wl][p][lane];
                    if (k >= L) cand[wl][pos++] = k;
                }
                __syncwarp();
                float cv[2] = {lane < total ? cand[wl][lane] : -INFINITY,
                               lane + 32 < total ? cand[wl][lane + 32] : -INFINITY};
                qb_sort64_desc(cv, lane);
                a = __shfl_sync(0xffffffffu, cv[K >> 5], K & 31);   // K < 32 here
                __syncwarp();
                done = true;
            }
        }
        if (!done) {
            // every key: K + 1 rounds, the winning lane's column rescanned
            float best = -INFINITY;
            int bp = 0;
            for (int p = 0; p < MAXP; ++p) {
                const float k = skey[wl][p][lane];
                if (k > best) {
                    best = k;
                    bp = p;
                }
            }
            for (int round = 0; round <= K; ++round) {
                a = qb_warp_max(best, lane, &who);
                if (lane == who) {
                    skey[wl][bp][lane] = -INFINITY;
                    best = -INFINITY;
                    for (int p = 0; p < MAXP; ++p) {
                        const float k = skey[wl][p][lane];
                        if (k > best) {
                            best = k;
                            bp = p;
                        }
                    }
                }
                __syncwarp();
            }
        }
        for (int o = 16; o; o >>= 1) {
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
            smin = fminf(smin, __shfl_xor_sync(0xffffffffu, smin, o));
        }
        if (lane == 0) alpha[t] = a;
        wlo = fminf(wlo, a - smax);
        whi = fmaxf(whi, a - smin);
        __syncwarp();
    }
    if (lane == 0) {
        rlo[wl] = wlo;
        rhi[wl] = whi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float lo = rlo[0], hi = rhi[0];
        for (int i = 1; i < 8; ++i) {
            lo = fminf(lo, rlo[i]);
            hi = fmaxf(hi, rhi[i]);
        }
        if (lo <= hi) {
            atomicMin(range, qb_ord(lo));
            atomicMax(range + 1, qb_ord(hi));
        }
    }
}

// Histogram of margins for experts [e0, e0 + 2^lg_eg) over tokens [t0, t1):
// thread (token row, expert) = (tid >> lg_eg, tid & (2^lg_eg - 1)).
__global__ void __launch_bounds__(256) qb_hist_kernel(const float *__restrict__ logits,
                                                      const float *__restrict__ alpha, int T, int E, int lg_eg,
                                                      int tslice, int nbins, const uint32_t *range,
                                                      int32_t *__restrict__ counts)
{
    extern __shared__ int hist[];                    // [EG][nbins]
    const int EG = 1 << lg_eg;
    const int e0 = blockIdx.x * EG, t0 = blockIdx.y * tslice, t1 = min(T, t0 + tslice);
    const int eg = min(EG, E - e0);
    for (int i = threadIdx.x; i < EG * nbins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const float lo = qb_unord(range[0]), hi = qb_unord(range[1]);
    const float w = hi > lo ? (hi - lo) / nbins : 1.0f;
    const float inv_w = 1.0f / w;
    const int jj = threadIdx.x & (EG - 1), rows = blockDim.x >> lg_eg;
    if (jj < eg) {
        const float *lp = logits + e0 + jj;
        constexpr int U = 8;                             // loads in flight per thread
        int t = t0 + (threadIdx.x >> lg_eg);
        for (; t + (U - 1) * rows < t1; t += U * rows) {
            float lv[U], av[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                lv[u] = lp[(size_t)(t + u * rows) * E];
                av[u] = alpha[t + u * rows];
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float m = av[u] - qb_score(lv[u]);
                const int b = min(nbins - 1, max(0, (int)floorf((m - lo) * inv_w)));
                atomicAdd(&hist[jj * nbins + b], 1);
            }
        }
        for (; t < t1; t += rows) {
            const float m = alpha[t] - qb_score(lp[(size_t)t * E]);
            const int b = min(nbins - 1, max(0, (int)floorf((m - lo) * inv_w)));
            atomicAdd(&hist[jj * nbins + b], 1);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < eg * nbins; i += blockDim.x)
        if (hist[i]) atomicAdd(counts + (size_t)(e0 + i / nbins) * nbins + i % nbins, hist[i]);
}

// One warp per expert: first bin whose cumulative count reaches r.
__global__ void qb_select_kernel(const int32_t *__restrict__ counts, int E, int nbins, int r,
                                 const uint32_t *range, float *__restrict__ bias_out)
{
    const int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (e >= E) return;
    const float lo = qb_unord(range[0]), hi = qb_unord(range[1]);
    const float w = hi > lo ? (hi - lo) / nbins : 1.0f;
    const int32_t *c = counts + (size_t)e * nbins;
    int base = 0, found = nbins - 1;
    for (int b0 = 0; b0 < nbins; b0 += 32) {
        const int b = b0 + lane;
        int v = b < nbins ? c[b] : 0;
        for (int o = 1; o < 32; o <<= 1) {           // inclusive warp scan
            const int u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, base + v >= r && b < nbins);
        if (hit) {
            found = b0 + __ffs(hit) - 1;
            break;
        }
        base += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) bias_out[e] = lo + (float)(found + 1) * w;
}

}  // namespace k3

using namespace k3;

// workspace: alpha [T] floats, range [2] (padded to 256 B), counts [E][nbins]
static size_t qb_layout(int T, int E, int nbins, size_t *off_range, size_t *off_counts)
{
    const size_t a = ((size_t)T * 4 + 255) & ~(size_t)255;
    *off_range = a;
    *off_counts = a + 256;
    return a + 256 + (((size_t)E * nbins * 4 + 255) & ~(size_t)255);
}

size_t k3_qb_workspace_bytes(int T, int E, int nbins)
{
    size_t r, c;
    return qb_layout(T > 0 ? T : 1, E, nbins > 0 ? nbins : 1, &r, &c);
}

int k3_qb_bias(const k3moe_handle *h, const float *logits, int T, const float *bias_in, float *bias_out,
               int nbins, void *ws, size_t ws_bytes, cudaStream_t st)
{
    const int E = h->cfg.n_experts, K = h->cfg.top_k;
    int num_sms = 0;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess || num_sms < 1)
        return K3MOE_ERR_CUDA;
    size_t off_r, off_c;
    if (ws_bytes < qb_layout(T, E, nbins, &off_r, &off_c)) return K3MOE_ERR_WORKSPACE;
    float *alpha = (float *)ws;
    uint32_t *range = (uint32_t *)((uint8_t *)ws + off_r);
    int32_t *counts = (int32_t *)((uint8_t *)ws + off_c);
    const size_t nc = (size_t)E * nbins;
    qb_init_kernel<<<(unsigned)std::min<size_t>((nc + 255) / 256, 1024), 256, 0, st>>>(counts, nc, range);
    k3_note_launch();
    const dim3 ga((T + 8 * QB_TPW - 1) / (8 * QB_TPW));
    if (E <= 128) qb_alpha_kernel<4><<<ga, 256, 0, st>>>(logits, bias_in, T, E, K, alpha, range);
    else if (E <= 256) qb_alpha_kernel<8><<<ga, 256, 0, st>>>(logits, bias_in, T, E, K, alpha, range);
    else if (E <= 512) qb_alpha_kernel<16><<<ga, 256, 0, st>>>(logits, bias_in, T, E, K, alpha, range);
    else qb_alpha_kernel<32><<<ga, 256, 0, st>>>(logits, bias_in, T, E, K, alpha, range);
    k3_note_launch();
    // expert groups (a power of two up to 256) whose bins fit 32 KB of shared
    // memory; token slices for parallelism
    int lg_eg = 0;
    while (lg_eg < 8 && (2 << lg_eg) * nbins <= 8192 && (1 << lg_eg) < E) ++lg_eg;
    const int EG = 1 << lg_eg;
    const int ngroups = (E + EG - 1) / EG;
    const long cta_target = 8L * num_sms;                  // about 8 CTAs per SM over all groups
    const int tslice = (int)std::max<long>(256, ((long)T * ngroups + cta_target - 1) / cta_target);
    const dim3 gh(ngroups, (T + tslice - 1) / tslice);
    qb_hist_kernel<<<gh, 256, (size_t)EG * nbins * 4, st>>>(logits, alpha, T, E, lg_eg, tslice, nbins, range,
                                                          counts);
    k3_note_launch();
    const long r0 = ((long)T * K * 2 + E) / (2L * E);   // round(T K / E)
    const int r = (int)std::min<long>(std::max<long>(r0, 1), T - 1);
    qb_select_kernel<<<(E * 32 + 255) / 256, 256, 0, st>>>(counts, E, nbins, r, range, bias_out);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}
