// Balanced expert-parallel plan and dispatch ("the K3 report review", section
// "3T pre-training: turning irregular MoE into a static execution plan", the
// MoonEP paragraph): with E experts on R ranks and at most E/R redundant
// expert slots per rank, every rank can receive exactly C = S*K routed pairs.
//
// Plan: one CTA; all state in shared memory.  The CTA sums the count matrix;
// then one warp runs R rounds.  Each takes the unplanned rank with the
// smallest remaining home load H (warp minimum over the ranks), gives it its
// home experts' remaining pairs (ballot + scan for the segment slots and
// receive rows), then fills its C - H remaining rows from the largest
// remaining experts, one warp maximum over the lanes' block maxima per take.
// At most E/R takes per rank (the other ranks' E/R largest experts hold at
// least C - H), at most E takes in all, at most 2E segments.
//
// Dispatch of one source rank's pairs: expert e's pairs are numbered in
// (source rank, token) order, so this rank's continue from the counts of the
// lower ranks.  The routing's chunked stable numbering (the same kernels as
// the permutation) gives each pair its number j; a binary search over the
// expert's segments (increasing src, staged in shared memory) finds the one
// holding j.
#include "k3moe_internal.h"

namespace k3 {

constexpr int EP_SEG_INTS = 5;   // expert, rank, src, count, dst

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w < v ? w : v;
    }
    return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    return v;
}

// Shared memory: rem, taken, nseg_of [E]; seg_expert, seg_ord [2E]; H [R].
// All EP_PLAN_THREADS threads sum the counts (a thread per expert, reads
// coalesced over the experts) and the home loads; warp 0 then runs the rounds.
// Lane l owns experts [l*B, l*B + B) and keeps the largest (count, -index) key
// of its block, refreshed only when a count in the block changes.
constexpr int EP_PLAN_THREADS = 1024;

__global__ void __launch_bounds__(EP_PLAN_THREADS) ep_plan_kernel(const int32_t *__restrict__ counts, int R, int E,
                                                                  int C, int32_t *__restrict__ seg,
                                                                  int32_t *__restrict__ rank_seg,
                                                                  int32_t *__restrict__ exp_off,
                                                                  int32_t *__restrict__ exp_seg,
                                                                  int32_t *__restrict__ info, int *status)
{
    griddep_enter();
    extern __shared__ int ep_sm[];
    __shared__ long long part[EP_PLAN_THREADS / 32];
    int *rem = ep_sm, *taken = rem + E, *nseg_of = taken + E;
    int *seg_expert = nseg_of + E, *seg_ord = seg_expert + 2 * E, *H = seg_ord + 2 * E;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, m = E / R;
    const long long cap = (long long)R * C;

    // per-expert totals over the source ranks
    long long s = 0;
    bool bad = false;
    if (tid < E) {
#pragma unroll 8
        for (int q = 0; q < R; ++q) {
            const int v = counts[(size_t)q * E + tid];
            bad |= v < 0;
            s += v;
        }
        bad |= s > cap;
        rem[tid] = (int)(s > cap ? 0 : s);
        taken[tid] = 0;
        nseg_of[tid] = 0;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) part[warp] = s;
    bad = __syncthreads_or(bad);
    long long tot = 0;
    for (int w = 0; w < EP_PLAN_THREADS / 32; ++w) tot += part[w];
    if (bad || tot != cap) {
        if (tid == 0) {
            set_status(status, K3MOE_ERR_RANGE, -1);
            info[0] = 0;
            info[1] = -1;
        }
        return;
    }
    if (tid < R) {
        int h = 0;
        for (int i = 0; i < m; ++i) h += rem[tid * m + i];
        H[tid] = h;                                   // -1 once planned
    }
    __syncthreads();
    if (warp != 0) return;

    const int B = (E + 31) / 32, blo = min(E, lane * B), bhi = min(E, blo + B);
    auto block_top = [&]() {
        unsigned long long k = 0;
        for (int e = blo; e < bhi; ++e) {
            const int v = rem[e];
            if (v > 0) {
                const unsigned long long kk = ((unsigned long long)(unsigned)v << 32) | (unsigned)(E - 1 - e);
                k = kk > k ? kk : k;
            }
        }
        return k;
    };
    unsigned long long mine = block_top();

    int nseg = 0, max_red = 0;
    for (int round = 0; round < R; ++round) {
        unsigned long long best = ~0ull;
        for (int r = lane; r < R; r += 32)
            if (H[r] >= 0) {
                const unsigned long long k = ((unsigned long long)(unsigned)H[r] << 32) | (unsigned)r;
                best = k < best ? k : best;
            }
        best = warp_min_u64(best);
        const int r = (int)(best & 0xffffffffu);
        int need = C - (int)(best >> 32);
        const int first = nseg;
        int dst = 0;
        // the rank's home experts, in index order
        for (int i0 = 0; i0 < m; i0 += 32) {
            const int i = i0 + lane, e = r * m + i;
            const int v = i < m ? rem[e] : 0;
            const unsigned has = __ballot_sync(0xffffffffu, v > 0);
            const int incl = warp_incl_scan(v, lane);
            if (v > 0) {
                const int sl = nseg + __popc(has & ((1u << lane) - 1u));
                int32_t *o = seg + (size_t)sl * EP_SEG_INTS;
                o[0] = e;
                o[1] = r;
                o[2] = taken[e];
                o[3] = v;
                o[4] = dst + incl - v;
                seg_expert[sl] = e;
                seg_ord[sl] = nseg_of[e]++;
                taken[e] += v;
                rem[e] = 0;
            }
            nseg += __popc(has);
            dst += __shfl_sync(0xffffffffu, incl, 31);
        }
        __syncwarp();
        if (blo < (r + 1) * m && bhi > r * m) mine = block_top();
        if (lane == 0) H[r] = -1;
        int takes = 0;
        while (need > 0) {
            // the largest remaining expert; equal counts: the lower index
            const unsigned long long top = warp_max_u64(mine);
            if (top == 0 || takes == m) {             // excluded by the bound; kept as a guard
                if (lane == 0) {
                    set_status(status, K3MOE_ERR_RANGE, -2);
                    info[0] = 0;
                    info[1] = -1;
                }
                return;
            }
            const int e = E - 1 - (int)(top & 0xffffffffu), v = (int)(top >> 32), t = min(v, need);
            if (e >= blo && e < bhi) {               // the owner lane updates the expert
                int32_t *o = seg + (size_t)nseg * EP_SEG_INTS;
                o[0] = e;
                o[1] = r;
                o[2] = taken[e];
                o[3] = t;
                o[4] = dst;
                seg_expert[nseg] = e;
                seg_ord[nseg] = nseg_of[e]++;
                taken[e] += t;
                rem[e] = v - t;
                H[e / m] -= t;
                mine = block_top();
            }
            __syncwarp();
            ++nseg;
            ++takes;
            dst += t;
            need -= t;
        }
        max_red = max(max_red, takes);
        if (lane == 0) {
            rank_seg[2 * r] = first;
            rank_seg[2 * r + 1] = nseg - first;
        }
        __syncwarp();
    }

    // segments grouped by expert: nseg_of becomes each expert's first slot
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int v = e < E ? nseg_of[e] : 0;
        const int incl = warp_incl_scan(v, lane);
        if (e < E) {
            exp_off[e] = carry + incl - v;
            nseg_of[e] = carry + incl - v;
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncwarp();
    for (int i = lane; i < nseg; i += 32) exp_seg[nseg_of[seg_expert[i]] + seg_ord[i]] = i;
    if (lane == 0) {
        exp_off[E] = carry;
        info[0] = nseg;
        info[1] = max_red;
    }
}

// base[e]: pairs of expert e on the source ranks below src; totals zeroed for
// the chunk counts that follow.
__global__ void ep_base_kernel(const int32_t *__restrict__ counts, int E, int src, int32_t *__restrict__ base,
                               int32_t *__restrict__ totals)
{
    griddep_enter();
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    int s = 0;
    for (int q = 0; q < src; ++q) s += counts[(size_t)q * E + e];
    base[e] = s;
    totals[e] = 0;
}

// EP_DISPATCH_WARPS chunks of 32 tokens per CTA, one warp each, in token
// order; lane k numbers pair (t, k).  The plan's segments, in expert order,
// are staged in shared memory (src, rank, dst) beside each expert's first
// slot; every index read from the plan is checked before use, so a plan that
// failed on the device yields -1 destinations and a status, not stray reads.
// Block 0 also checks the routing's totals against counts[src].
constexpr int EP_DISPATCH_WARPS = 4;

__global__ void __launch_bounds__(32 * EP_DISPATCH_WARPS)
    ep_dispatch_kernel(const int32_t *__restrict__ idx, int T, int K, int E, int R, int nch,
                       const int32_t *__restrict__ chunk_base, const int32_t *__restrict__ totals,
                       const int32_t *__restrict__ own_counts, const int32_t *__restrict__ seg,
                       const int32_t *__restrict__ exp_off, const int32_t *__restrict__ exp_seg,
                       const int32_t *__restrict__ info, int32_t *__restrict__ dest_rank,
                       int32_t *__restrict__ dest_row, int *status)
{
    griddep_enter();
    extern __shared__ int ep_dsm[];
    int *toff = ep_dsm;                              // [E + 1]
    int *tsrc = toff + E + 1, *tend = tsrc + 2 * E, *trank = tend + 2 * E, *tdst = trank + 2 * E;   // [2E] each
    int *next = tdst + 2 * E;                        // [EP_DISPATCH_WARPS][E]
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int C = T * K;
    int n = info[0];
    const bool plan_ok = n >= 1 && n <= 2 * E;
    n = plan_ok ? n : 0;
    for (int e = tid; e <= E; e += blockDim.x) {
        int o = plan_ok ? exp_off[e] : 0;
        toff[e] = (o < 0 || o > n) ? 0 : o;
    }
    for (int i = tid; i < n; i += blockDim.x) {
        const int sid = exp_seg[i];
        int src = 0, end = 0, rk = -1, dst = 0;
        if (sid >= 0 && sid < n) {
            const int32_t *g = seg + (size_t)sid * EP_SEG_INTS;
            src = g[2];
            end = g[2] + g[3];
            rk = g[1];
            dst = g[4];
            if (rk < 0 || rk >= R || g[3] <= 0 || dst < 0 || dst > C - g[3]) rk = -1;
        }
        tsrc[i] = src;
        tend[i] = end;
        trank[i] = rk;
        tdst[i] = dst;
    }
    const int ch = blockIdx.x * EP_DISPATCH_WARPS + w;
    int *nx = next + w * E;
    for (int e = lane; e < E; e += 32) {
        if (ch < nch) nx[e] = chunk_base[(size_t)e * nch + ch];
        if (blockIdx.x == 0 && w == 0 && totals[e] != own_counts[e]) set_status(status, K3MOE_ERR_RANGE, -3);
    }
    __syncthreads();
    if (ch >= nch) return;
    // the chunk's expert ids first (independent loads), then the numbering in
    // token order from registers
    const int t0 = ch * K3_PERM_CHUNK, nt = min(T, t0 + K3_PERM_CHUNK) - t0;
    int ids[K3_PERM_CHUNK];
#pragma unroll
    for (int i = 0; i < K3_PERM_CHUNK; ++i) ids[i] = (lane < K && i < nt) ? idx[(size_t)(t0 + i) * K + lane] : -1;
#pragma unroll
    for (int i = 0; i < K3_PERM_CHUNK; ++i) {
        if (i < nt && lane < K) {
            const int p = (t0 + i) * K + lane;
            const int e = ids[i];
            int rk = -1, row = -1;
            if (e >= 0 && e < E) {
                const int j = atomicAdd(&nx[e], 1);     // distinct experts per token: token order
                int lo = toff[e], hi = toff[e + 1];
                if (lo < hi) {
                    while (hi - lo > 1) {               // last segment with src <= j
                        const int mid = (lo + hi) >> 1;
                        if (tsrc[mid] <= j) lo = mid;
                        else hi = mid;
                    }
                    if (j >= tsrc[lo] && j < tend[lo] && trank[lo] >= 0) {
                        rk = trank[lo];
                        row = tdst[lo] + (j - tsrc[lo]);
                    }
                }
            }
            if (rk < 0) set_status(status, K3MOE_ERR_RANGE, p);
            dest_rank[p] = rk;
            dest_row[p] = row;
        }
        __syncwarp();
    }
}

}  // namespace k3

using namespace k3;

static size_t ep_align(size_t n) { return (n + 255) & ~(size_t)255; }

int k3_ep_plan(const k3moe_handle *h, const int32_t *counts, int R, int C, const k3moe_ep_plan *plan,
               cudaStream_t st)
{
    const int E = h->cfg.n_experts;
    const size_t smem = sizeof(int) * (size_t)(7 * E + R);
    k3_launch(ep_plan_kernel, 1, EP_PLAN_THREADS, smem, st, counts, R, E, C, plan->seg, plan->rank_seg,
              plan->exp_off, plan->exp_seg, plan->info, h->d_status);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

size_t k3_ep_dispatch_workspace_bytes(int T, int E)
{
    const size_t nch = (size_t)(T + K3_PERM_CHUNK - 1) / K3_PERM_CHUNK;
    return ep_align(sizeof(int32_t) * nch * E) + 2 * ep_align(sizeof(int32_t) * E);
}

int k3_ep_dispatch(const k3moe_handle *h, const int32_t *idx, int T, int src, const int32_t *counts, int R,
                   const k3moe_ep_plan *plan, int32_t *dest_rank, int32_t *dest_row, void *ws, cudaStream_t st)
{
    const int E = h->cfg.n_experts, K = h->cfg.top_k;
    const int nch = (T + K3_PERM_CHUNK - 1) / K3_PERM_CHUNK;
    uint8_t *p = static_cast<uint8_t *>(ws);
    int32_t *chunk_cnt = reinterpret_cast<int32_t *>(p);
    p += ep_align(sizeof(int32_t) * (size_t)nch * E);
    int32_t *base = reinterpret_cast<int32_t *>(p);
    p += ep_align(sizeof(int32_t) * E);
    int32_t *totals = reinterpret_cast<int32_t *>(p);
    k3_launch(ep_base_kernel, (E + 255) / 256, 256, 0, st, counts, E, src, base, totals);
    k3_note_launch();
    k3_launch_chunk_count(idx, T, K, E, chunk_cnt, totals, h->d_status, st);
    k3_launch_chunk_base(T, E, base, chunk_cnt, st);
    // the segment table (E + 1 offsets, 4 x 2E fields) and a counter row per warp: 53 KB at E = 1024
    const size_t smem = sizeof(int) * ((size_t)E + 1 + 8 * (size_t)E + (size_t)EP_DISPATCH_WARPS * E);
    // the limit is set once per device, so to the size of the largest E (1024)
    static unsigned long long attr_set = 0;
    const int smem_max = (int)sizeof(int) * (1024 + 1 + 8 * 1024 + EP_DISPATCH_WARPS * 1024);
    if (!k3_smem_attr(ep_dispatch_kernel, smem_max, attr_set)) return K3MOE_ERR_CUDA;
    k3_launch(ep_dispatch_kernel, (nch + EP_DISPATCH_WARPS - 1) / EP_DISPATCH_WARPS, 32 * EP_DISPATCH_WARPS, smem, st,
              idx, T, K, E, R, nch, chunk_cnt, totals, counts + (size_t)src * E, plan->seg, plan->exp_off,
              plan->exp_seg, plan->info, dest_rank, dest_row, h->d_status);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}
