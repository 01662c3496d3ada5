// Router top-K selection and the counting-sort token permutation.
//
// Selection ("Kimi K3, as released", table "Shape": sigmoid router, 1 group,
// routed_scaling_factor 1.0; section "Against the technical report":
// e_score_correction_bias for selection only, weights renormalised over the
// selected top-k, then routed_scaling_factor).  Permutation: rows grouped per
// expert so the gate/up and down GEMMs read the same per-expert row ranges
// ("quants.md", the moe_align_block_size fix: one layout shared by both GEMMs,
// expert ids >= 256 kept; indices here are int32).
#include "k3moe_internal.h"

namespace k3 {

// Order-preserving image of a key in uint32: a larger float gives a larger integer
// (-0 is first turned into +0, so that equal keys stay equal).  Every key, -inf
// included, maps to at least 0x007FFFFF; 0 marks "no key".
__device__ __forceinline__ uint32_t key_bits(float k)
{
    if (k == 0.f) k = 0.f;
    const uint32_t u = __float_as_uint(k);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-K of one token, one warp.  Lane l owns keys j = l + 32 i (row l of a
// [32][MAXP + 1] tile of key images in shared memory) and keeps the best untaken
// key of its row.  Each of the K rounds takes the warp-wide maximum of the lane
// bests (equal keys: lower index) with two warp reductions (max of the key, then
// min of the index among the lanes holding it), marks it taken, and the warp
// rescans only the winning lane's row the same way.  NaN keys rank below every
// number.  Writes idx in selection order (and to sidx when given) and the weights
// sigmoid(l_k) / sum_sel sigmoid(l) * scaling.
template <int MAXP>
__device__ __forceinline__ void topk_warp(const float *__restrict__ lrow, const float *__restrict__ bias, int E,
                                          int K, float scaling, uint32_t (*row)[MAXP + 1], int lane,
                                          int32_t *__restrict__ idx_row, float *__restrict__ w_row, int *sidx)
{
    constexpr uint32_t ALL = 0xffffffffu, NONE = 0xffffffffu;
    uint32_t bk = 0, bj = NONE;
#pragma unroll
    for (int i = 0; i < MAXP; ++i) {
        const int j = lane + 32 * i;
        uint32_t u = 0;
        if (j < E) {
            const float l = lrow[j];
            float k = bias ? 1.0f / (1.0f + expf(-l)) + bias[j] : l;
            if (k != k) k = -INFINITY;
            u = key_bits(k);
            if (u > bk) {                        // strictly larger: the lower index keeps equal keys
                bk = u;
                bj = j;
            }
        }
        row[lane][i] = u;
    }
    __syncwarp();
    uint32_t taken = 0;          // bit i: key lane + 32 i taken (owner lane's view)
    int sel_j = 0;
    for (int s = 0; s < K; ++s) {
        const uint32_t wk = __reduce_max_sync(ALL, bk);
        const uint32_t wj = __reduce_min_sync(ALL, bk == wk ? bj : NONE);
        const int owner = wj & 31;
        if (lane == owner) taken |= 1u << (wj >> 5);
        const uint32_t otaken = __shfl_sync(ALL, taken, owner);
        // rescan the owner's row: lane i looks at key owner + 32 i
        uint32_t ck = 0, cj = NONE;
        if (lane < MAXP) {
            const int j = owner + 32 * lane;
            if (j < E && !((otaken >> lane) & 1u)) {
                ck = row[owner][lane];
                cj = j;
            }
        }
        const uint32_t nk = __reduce_max_sync(ALL, ck);
        const uint32_t nj = __reduce_min_sync(ALL, ck == nk ? cj : NONE);
        if (lane == owner) {
            bk = nk;
            bj = nj;
        }
        if (lane == s) sel_j = (int)wj;
    }
    // weights: sigma(l) of the selected experts over their sum (a butterfly sum: every
    // lane adds the same operand pairs, so all lanes hold the same total)
    const float sg = lane < K ? 1.0f / (1.0f + expf(-lrow[sel_j])) : 0.f;
    float ssum = sg;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ssum += __shfl_xor_sync(ALL, ssum, off);
    if (lane < K) {
        idx_row[lane] = sel_j;
        w_row[lane] = sg / ssum * scaling;
        if (sidx) sidx[lane] = sel_j;
    }
}

// One warp per token (8 tokens per CTA).
template <int MAXP>
__global__ void __launch_bounds__(256) topk_kernel(const float *__restrict__ logits,
                                                   const float *__restrict__ bias, int T, int E,
                                                   int K, float scaling, int32_t *__restrict__ idx,
                                                   float *__restrict__ wts, int32_t *__restrict__ counts_zero)
{
    griddep_enter();
    // the permutation's expert histogram starts from zero (the next kernel counts into it)
    if (counts_zero && blockIdx.x == 0)
        for (int i = threadIdx.x; i < E; i += blockDim.x) counts_zero[i] = 0;
    __shared__ uint32_t skey[8][32][MAXP + 1];
    const int wl = threadIdx.x >> 5;
    const int warp = blockIdx.x * 8 + wl;
    const int lane = threadIdx.x & 31;
    if (warp >= T) return;
    topk_warp<MAXP>(logits + (size_t)warp * E, bias, E, K, scaling, skey[wl], lane, idx + (size_t)warp * K,
                    wts + (size_t)warp * K, nullptr);
}

// counts[e] = number of (t, k) selecting e; flags an index outside [0, E).
__global__ void perm_count_kernel(const int32_t *__restrict__ idx, int n, int E,
                                  int32_t *__restrict__ counts, int *status)
{
    griddep_enter();
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    int e = idx[i];
    if (e < 0 || e >= E) {
        set_status(status, K3MOE_ERR_RANGE, e);
        return;
    }
    atomicAdd(counts + e, 1);
}

// Inclusive scan over a warp (shuffles).
__device__ __forceinline__ int warp_scan_incl(int v, int lane)
{
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += t;
    }
    return v;
}

// One CTA of 1024 threads: offsets = exclusive scan of counts; active-expert
// list; tile list for the tensor path (expert, first row, rows) with at most
// tile_n rows each.  Ends with the CTA synchronised and its writes visible to it.
// Each 1024-expert chunk is scanned per warp, then over the 32 warp totals.
__device__ __forceinline__ void perm_scan_block(const int32_t *counts, int E, int tile_n,
                                                int32_t *__restrict__ offsets, int32_t *__restrict__ active,
                                                int4 *__restrict__ tiles, int32_t *__restrict__ meta)
{
    __shared__ int s_w[3][32];
    __shared__ int base_rows, base_act, base_til;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) base_rows = base_act = base_til = 0;
    __syncthreads();
    for (int e0 = 0; e0 < E; e0 += 1024) {
        const int e = e0 + tid;
        const int c = e < E ? counts[e] : 0;
        const int nt = (tile_n > 0) ? (c + tile_n - 1) / tile_n : 0;
        int sc = warp_scan_incl(c, lane), sa = warp_scan_incl(c > 0, lane), st = warp_scan_incl(nt, lane);
        if (lane == 31) {
            s_w[0][w] = sc;
            s_w[1][w] = sa;
            s_w[2][w] = st;
        }
        __syncthreads();
        if (w == 0) {
            s_w[0][lane] = warp_scan_incl(s_w[0][lane], lane);
            s_w[1][lane] = warp_scan_incl(s_w[1][lane], lane);
            s_w[2][lane] = warp_scan_incl(s_w[2][lane], lane);
        }
        __syncthreads();
        if (w > 0) {
            sc += s_w[0][w - 1];
            sa += s_w[1][w - 1];
            st += s_w[2][w - 1];
        }
        if (e < E) {
            int row0 = base_rows + sc - c;
            offsets[e] = row0;
            if (c > 0) active[base_act + sa - 1] = e;
            int t0 = base_til + st - nt;
            for (int q = 0; q < nt; ++q) {
                int r = q * tile_n;
                tiles[t0 + q] = make_int4(e, row0 + r, min(tile_n, c - r), 0);
            }
        }
        __syncthreads();
        if (tid == 1023) {
            base_rows += sc;
            base_act += sa;
            base_til += st;
        }
        __syncthreads();
    }
    if (tid == 0) {
        offsets[E] = base_rows;
        meta[0] = base_act;
        meta[1] = base_til;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(1024) perm_scan_kernel(const int32_t *__restrict__ counts, int E,
                                                         int tile_n, int32_t *__restrict__ offsets,
                                                         int32_t *__restrict__ active,
                                                         int4 *__restrict__ tiles,
                                                         int32_t *__restrict__ meta)
{
    griddep_enter();
    perm_scan_block(counts, E, tile_n, offsets, active, tiles, meta);
}

// Decode-size routing in one CTA (T <= 32 tokens, T K <= 1024 pairs, E <= 1024):
// top-K per token (warp t), the expert histogram in shared memory, the scan and
// tile list, and the stable scatter (a pair's row within its expert is the
// number of earlier pairs, in (t, k) order, that chose the same expert: the
// number of earlier tokens in the expert's token bit mask).
template <int MAXP>
__global__ void __launch_bounds__(1024) route_small_kernel(
    const float *__restrict__ logits, const float *__restrict__ bias, int T, int E, int K, float scaling,
    int32_t *__restrict__ idx, float *__restrict__ wts, int tile_n, int32_t *__restrict__ offsets,
    int32_t *__restrict__ active, int4 *__restrict__ tiles, int32_t *__restrict__ meta,
    int32_t *__restrict__ tok_of, int32_t *__restrict__ row_of, int *status)
{
    griddep_enter();
    extern __shared__ uint32_t rs_keys[];             // [32 warps][32][MAXP + 1]
    __shared__ int s_idx[1024], s_hist[1024];
    __shared__ uint32_t s_tok[1024];                 // bit t: token t selected expert e (T <= 32)
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31, n = T * K;
    s_hist[tid] = 0;
    s_tok[tid] = 0;
    __syncthreads();
    if (w < T)
        topk_warp<MAXP>(logits + (size_t)w * E, bias, E, K, scaling,
                        reinterpret_cast<uint32_t(*)[MAXP + 1]>(rs_keys + (size_t)w * 32 * (MAXP + 1)), lane,
                        idx + (size_t)w * K, wts + (size_t)w * K, s_idx + w * K);
    __syncthreads();
    if (tid < n) {
        const int e = s_idx[tid];
        if (e < 0 || e >= E) set_status(status, K3MOE_ERR_RANGE, e);
        else {
            atomicAdd(&s_hist[e], 1);
            atomicOr(&s_tok[e], 1u << (tid / K));
        }
    }
    __syncthreads();
    perm_scan_block(s_hist, E, tile_n, offsets, active, tiles, meta);
    if (tid < n) {
        const int e = s_idx[tid];
        if (e >= 0 && e < E) {
            // a token selects an expert at most once: the earlier pairs on e are its earlier tokens
            const int row = offsets[e] + __popc(s_tok[e] & ((1u << (tid / K)) - 1u));
            tok_of[row] = tid / K;
            row_of[tid] = row;
        }
    }
}

// One CTA per expert: stable scatter of its (t, k) pairs in (t, k) order.
__global__ void __launch_bounds__(256) perm_scatter_kernel(const int32_t *__restrict__ idx, int n,
                                                           int K, const int32_t *__restrict__ counts,
                                                           const int32_t *__restrict__ offsets,
                                                           int32_t *__restrict__ tok_of,
                                                           int32_t *__restrict__ row_of)
{
    griddep_enter();
    const int e = blockIdx.x;
    if (counts[e] == 0) return;
    __shared__ int warp_tot[8];
    __shared__ int base;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) base = offsets[e];
    __syncthreads();
    for (int p0 = 0; p0 < n; p0 += 256) {
        int p = p0 + tid;
        bool hit = p < n && idx[p] == e;
        uint32_t bal = __ballot_sync(0xffffffffu, hit);
        if (lane == 0) warp_tot[w] = __popc(bal);
        __syncthreads();
        int before = 0, total = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            before += q < w ? warp_tot[q] : 0;
            total += warp_tot[q];
        }
        if (hit) {
            int row = base + before + __popc(bal & ((1u << lane) - 1u));
            tok_of[row] = p / K;
            row_of[p] = row;
        }
        __syncthreads();
        if (tid == 0) base += total;
        __syncthreads();
    }
}

// ---- chunked stable permutation (large T).  A token selects an expert at most
// once, so the stable (t, k) order within an expert's segment is token order:
// a row's position is the expert's offset, plus the expert's count in earlier
// chunks, plus its count at earlier tokens of the same chunk.

// Per-chunk expert counts, expert-major [E][nch], and the totals.
__global__ void __launch_bounds__(256) perm_chunk_count_kernel(const int32_t *__restrict__ idx, int T, int K,
                                                               int E, int nch, int32_t *__restrict__ chunk_cnt,
                                                               int32_t *__restrict__ counts, int *status)
{
    griddep_enter();
    extern __shared__ int cnt[];                     // [E]
    const int ch = blockIdx.x;
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int p0 = ch * K3_PERM_CHUNK * K, p1 = min(T, (ch + 1) * K3_PERM_CHUNK) * K;
    for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
        const int e = idx[p];
        if (e < 0 || e >= E) {
            set_status(status, K3MOE_ERR_RANGE, e);
            continue;
        }
        atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int v = cnt[e];
        chunk_cnt[(size_t)e * nch + ch] = v;
        if (v) atomicAdd(counts + e, v);
    }
}

// One CTA per expert: chunk counts -> chunk bases (offset + exclusive scan over chunks).
__global__ void __launch_bounds__(1024) perm_chunk_base_kernel(int nch, const int32_t *__restrict__ offsets,
                                                               int32_t *__restrict__ chunk_cnt)
{
    griddep_enter();
    __shared__ int s[1024];
    __shared__ int carry;
    const int e = blockIdx.x, tid = threadIdx.x;
    int32_t *row = chunk_cnt + (size_t)e * nch;
    if (tid == 0) carry = offsets[e];
    __syncthreads();
    for (int c0 = 0; c0 < nch; c0 += 1024) {
        const int c = c0 + tid;
        const int v = c < nch ? row[c] : 0;
        s[tid] = v;
        __syncthreads();
        for (int off = 1; off < 1024; off <<= 1) {     // inclusive Hillis-Steele scan
            const int a = tid >= off ? s[tid - off] : 0;
            __syncthreads();
            s[tid] += a;
            __syncthreads();
        }
        if (c < nch) row[c] = carry + s[tid] - v;
        __syncthreads();
        if (tid == 1023) carry += s[1023];
        __syncthreads();
    }
}

// One warp per chunk: the chunk's tokens in order, lane k placing (t, k).
__global__ void __launch_bounds__(32) perm_chunk_scatter_kernel(const int32_t *__restrict__ idx, int T, int K,
                                                                int E, int nch,
                                                                const int32_t *__restrict__ chunk_base,
                                                                int32_t *__restrict__ tok_of,
                                                                int32_t *__restrict__ row_of)
{
    griddep_enter();
    extern __shared__ int next[];                    // [E] next free row per expert
    const int ch = blockIdx.x, lane = threadIdx.x;
    for (int e = lane; e < E; e += 32) next[e] = chunk_base[(size_t)e * nch + ch];
    __syncwarp();
    // the chunk's expert ids first (independent loads), then the placement in
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
            if (e >= 0 && e < E) {                   // the experts of one token are distinct
                const int row = next[e];
                next[e] = row + 1;
                tok_of[row] = t0 + i;
                row_of[p] = row;
            }
        }
        __syncwarp();
    }
}

}  // namespace k3

using namespace k3;

int k3_launch_topk(const k3moe_handle *h, const float *logits, int T, int32_t *idx, float *wts,
                   int32_t *counts_zero, cudaStream_t st)
{
    const k3moe_config &c = h->cfg;
    const float *bias = c.has_select_bias ? h->bias : nullptr;
    dim3 grid((T + 7) / 8), block(256);
    int E = c.n_experts;
    if (E <= 128) k3_launch(topk_kernel<4>, grid, block, 0, st, logits, bias, T, E, c.top_k, c.routed_scaling, idx, wts, counts_zero);
    else if (E <= 256) k3_launch(topk_kernel<8>, grid, block, 0, st, logits, bias, T, E, c.top_k, c.routed_scaling, idx, wts, counts_zero);
    else if (E <= 512) k3_launch(topk_kernel<16>, grid, block, 0, st, logits, bias, T, E, c.top_k, c.routed_scaling, idx, wts, counts_zero);
    else if (E <= 1024) k3_launch(topk_kernel<32>, grid, block, 0, st, logits, bias, T, E, c.top_k, c.routed_scaling, idx, wts, counts_zero);
    else return K3MOE_ERR_UNSUPPORTED;
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

template <int MAXP>
static int launch_route_small(const k3moe_handle *h, const k3_ws &ws, int T, int tile_n, cudaStream_t st)
{
    const k3moe_config &c = h->cfg;
    auto kern = route_small_kernel<MAXP>;
    const size_t smem = sizeof(uint32_t) * 32 * 32 * (MAXP + 1);
    static unsigned long long attr_set = 0;
    if (!k3_smem_attr(kern, (int)smem, attr_set)) return K3MOE_ERR_CUDA;
    const float *bias = c.has_select_bias ? h->bias : nullptr;
    k3_launch(kern, 1, 1024, smem, st, ws.logits, bias, T, c.n_experts, c.top_k, c.routed_scaling, ws.idx, ws.wts,
              tile_n, ws.offsets, ws.active, reinterpret_cast<int4 *>(ws.tiles), ws.meta, ws.tok_of, ws.row_of,
              h->d_status);
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}

int k3_launch_route(k3moe_handle *h, const k3_ws &ws, int T, int tile_n, cudaStream_t st)
{
    const int E = h->cfg.n_experts, K = h->cfg.top_k;
    int rc;
    if (T <= 32 && T * K <= 1024 && E <= 1024) {
        // one launch for top-K and the permutation
        k3_stage sg(h, K3MOE_STAGE_TOPK, st);
        if (E <= 128) return launch_route_small<4>(h, ws, T, tile_n, st);
        if (E <= 256) return launch_route_small<8>(h, ws, T, tile_n, st);
        if (E <= 512) return launch_route_small<16>(h, ws, T, tile_n, st);
        return launch_route_small<32>(h, ws, T, tile_n, st);
    }
    {
        k3_stage sg(h, K3MOE_STAGE_TOPK, st);
        if ((rc = k3_launch_topk(h, ws.logits, T, ws.idx, ws.wts, ws.counts, st))) return rc;
    }
    k3_stage sg(h, K3MOE_STAGE_PERMUTE, st);
    return k3_launch_permute(h, ws, T, tile_n, st);
}

// The chunked stable numbering of a routing's pairs on its own: per-chunk
// expert counts (and totals added into `totals`), then each chunk's first
// number of each expert counted from base[e].  Used by the expert-parallel
// dispatch, whose numbers continue those of the lower source ranks.
void k3_launch_chunk_count(const int32_t *idx, int T, int K, int E, int32_t *chunk_cnt, int32_t *totals,
                           int *status, cudaStream_t st)
{
    const int nch = (T + K3_PERM_CHUNK - 1) / K3_PERM_CHUNK;
    k3_launch(perm_chunk_count_kernel, nch, 256, sizeof(int) * E, st, idx, T, K, E, nch, chunk_cnt, totals, status);
    k3_note_launch();
}

void k3_launch_chunk_base(int T, int E, const int32_t *base, int32_t *chunk_cnt, cudaStream_t st)
{
    const int nch = (T + K3_PERM_CHUNK - 1) / K3_PERM_CHUNK;
    k3_launch(perm_chunk_base_kernel, E, 1024, 0, st, nch, base, chunk_cnt);
    k3_note_launch();
}

int k3_launch_permute(const k3moe_handle *h, const k3_ws &ws, int T, int tile_n, cudaStream_t st)
{
    const int E = h->cfg.n_experts, K = h->cfg.top_k, n = T * K;
    // ws.counts was zeroed by the top-k kernel
    const bool chunked = T >= K3_PERM_CHUNKED_T;
    const int nch = (T + K3_PERM_CHUNK - 1) / K3_PERM_CHUNK;
    const size_t esm = sizeof(int) * E;              // E <= 1024: 4 KB of shared memory
    if (chunked) {
        k3_launch(perm_chunk_count_kernel, nch, 256, esm, st, ws.idx, T, K, E, nch, ws.chunk_cnt, ws.counts,
                                                       h->d_status);
    } else {
        k3_launch(perm_count_kernel, (n + 255) / 256, 256, 0, st, ws.idx, n, E, ws.counts, h->d_status);
    }
    k3_note_launch();
    k3_launch(perm_scan_kernel, 1, 1024, 0, st, ws.counts, E, tile_n, ws.offsets, ws.active,
                                         reinterpret_cast<int4 *>(ws.tiles), ws.meta);
    k3_note_launch();
    if (chunked) {
        k3_launch(perm_chunk_base_kernel, E, 1024, 0, st, nch, ws.offsets, ws.chunk_cnt);
        k3_note_launch();
        k3_launch(perm_chunk_scatter_kernel, nch, 32, esm, st, ws.idx, T, K, E, nch, ws.chunk_cnt, ws.tok_of,
                                                        ws.row_of);
    } else {
        k3_launch(perm_scatter_kernel, E, 256, 0, st, ws.idx, n, K, ws.counts, ws.offsets, ws.tok_of, ws.row_of);
    }
    k3_note_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA;
}
