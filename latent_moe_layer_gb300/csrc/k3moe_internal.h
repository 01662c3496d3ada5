// Internal declarations shared by the translation units of libk3moe.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stddef.h>

#include <utility>

#include "k3moe.h"

#define K3_CUDA_TRY(expr)                                   \
    do {                                                    \
        cudaError_t e_ = (expr);                            \
        if (e_ != cudaSuccess) return K3MOE_ERR_CUDA;       \
    } while (0)

namespace k3 {

// Device status word layout (int32 slots in the persistent buffer).
enum StatusSlot { ST_CODE = 0, ST_DETAIL = 1, ST_COUNT = 4 };

// Shared-memory budget of one CTA on sm_103a (opt-in maximum).
constexpr int kMaxSmem = 227 * 1024;

// Record the first device-side error (atomicCAS from OK).
__device__ __forceinline__ void set_status(int *status, int code, int detail)
{
    if (atomicCAS(status + ST_CODE, K3MOE_OK, code) == K3MOE_OK)
        status[ST_DETAIL] = detail;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b)
{
    return __uint_as_float((uint32_t)b << 16);
}

// fp32 -> BF16 round to nearest even (finite inputs; NaN stays NaN).
__device__ __forceinline__ uint16_t f32_to_bf16(float f)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// GLU activation a(g, u) of one gate/up pair (K3MOE_ACT_*): SiLU g sigmoid(g) u,
// or the SiTU reading sigmoid(g) beta tanh(g / beta) linear_beta tanh(u / linear_beta)
// (the K3 report review, "SiTU-GLU is a soft fuse" section; constants from the
// released config).  inv_* are the reciprocals of the betas.
struct K3Act {
    int kind;
    float beta, linear_beta, inv_beta, inv_linear_beta;
};

__device__ __forceinline__ float k3_glu(float g, float u, const K3Act &a)
{
    const float sg = 1.0f / (1.0f + expf(-g));
    if (a.kind == K3MOE_ACT_SITU)
        return sg * a.beta * tanhf(g * a.inv_beta) * (a.linear_beta * tanhf(u * a.inv_linear_beta));
    return g * sg * u;
}

// OCP E4M3 rounding of v (nearest even, saturating at +-448) with the hardware conversion.
__device__ __forceinline__ float e4m3_rne_sat(float v)
{
    uint16_t p;
    uint32_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(p) : "f"(v), "f"(v));   // both bytes: no order question
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(p));
    return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// MXFP8 value of v in a block of 32 whose largest magnitude is amax (OCP MX v1.0):
// scale 2^X with X = floor(log2 amax) - 8 (from amax's exponent field, kept >= -127),
// element E4M3(v / 2^X).
// The same from the block scale exponent X (-127 <= X <= 119).
__device__ __forceinline__ float mx8_round_x(float v, int X)
{
    const float down = __uint_as_float((uint32_t)(127 - X) << 23);     // 2^-X (X >= -127: at most 2^127)
    const float up = X > -127 ? __uint_as_float((uint32_t)(X + 127) << 23) : __uint_as_float(0x00400000u);
    return e4m3_rne_sat(v * down) * up;
}

// X from the block's largest exponent field (floor(log2 amax) = field - 127 for
// normal amax; zero and subnormal blocks take the clamp, -127).
__device__ __forceinline__ int mx8_scale_exp(uint32_t max_exp_field) { return max((int)max_exp_field - 135, -127); }

__device__ __forceinline__ float mx8_round(float v, float amax)
{
    return mx8_round_x(v, mx8_scale_exp((__float_as_uint(amax) >> 23) & 0xFF));
}

// 2^-k for a power of two 2^k with 0 <= k <= 126 (exact: exponent arithmetic).
__device__ __forceinline__ float pow2_inverse(float p2)
{
    return __uint_as_float(0x7F000000u - (__float_as_uint(p2) & 0x7F800000u));
}

// 2^(e-127) for an E8M0 byte e in [0, 254] (e = 0 gives the fp32 subnormal 2^-127).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e)
{
    return e ? __uint_as_float(e << 23) : __uint_as_float(0x00400000u);
}

// One E2M1 code -> fp32 value times `scale`.  The three magnitude bits placed
// at fp32 bits 22..24 give exactly E2M1 x 2^-126 (exponent field 0 yields the
// subnormal 0 / 0.5 cases), which 2^126 brings back to the E2M1 value.
__device__ __forceinline__ float e2m1_to_f32(uint32_t code, float scale)
{
    float mag = __uint_as_float((code & 7u) << 22) * 0x1p126f;
    float v = mag * scale;
    return (code & 8u) ? -v : v;
}

}  // namespace k3

// Kernel-launch counter (per host thread), read around each forward stage.
extern thread_local long g_k3_launches;
inline void k3_note_launch(int n = 1) { g_k3_launches += n; }

// Raise a kernel's dynamic shared-memory limit once per device (the attribute is
// per device; `done` is the launcher's own bitmask of devices already set).
template <typename F>
inline bool k3_smem_attr(F kern, int bytes, unsigned long long &done)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done & bit)) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    done |= bit;
    return true;
}

// Largest token count of one call (K3MOE_MAX_TOKENS of the public header).
constexpr int K3_MAX_TOKENS = K3MOE_MAX_TOKENS;

// Forward-path launches use programmatic dependent launch: a kernel may be
// scheduled while the previous kernel of the stream drains, and every such
// kernel begins with griddep_wait() (all threads) before it reads anything
// the previous kernels wrote, then lets its own dependent start launching.
template <typename... KArgs, typename... Args>
inline cudaError_t k3_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args &&...args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

#ifdef __CUDACC__
// Wait until the previous kernel in the stream has completed and its writes are
// visible, then allow the next kernel to be scheduled.
__device__ __forceinline__ void griddep_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

// Stage timing ring (k3moe_profile_enable / k3moe_profile_read).
struct k3_prof {
    static constexpr int RING = 256;
    bool on = false;
    cudaEvent_t ev[RING][K3MOE_NUM_STAGES][2];
    bool used[RING][K3MOE_NUM_STAGES];
    int pos = 0;
    long launches[K3MOE_NUM_STAGES];
};

// --------------------------------------------------------------- host handle
inline k3::K3Act k3_act_of(const k3moe_config &c)
{
    k3::K3Act a;
    a.kind = c.act;
    a.beta = c.situ_beta;
    a.linear_beta = c.situ_linear_beta;
    a.inv_beta = 1.0f / c.situ_beta;
    a.inv_linear_beta = 1.0f / c.situ_linear_beta;
    return a;
}

struct k3moe_handle {
    k3moe_config cfg;
    bool loaded = false;
    bool aligned16 = false;            // all packed/scale rows 16-byte aligned (tensor path eligible)
    int num_sms = 0;
    int device = 0;
    // borrowed weights
    const void *w_router = nullptr;
    const float *bias = nullptr;
    const uint16_t *w_down = nullptr, *w_up = nullptr, *gamma = nullptr;
    const uint8_t *shared[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    // persistent (caller-owned) device buffer
    uint8_t *persist = nullptr;
    size_t persist_bytes = 0;
    int *d_status = nullptr;                   // int[ST_COUNT]
    const uint8_t **d_eptr[6] = {};            // device tables [E] for w1p,w1s,w3p,w3s,w2p,w2s
    const uint8_t **d_shtab = nullptr;         // device table [6]: shared ws1p,ws1s,ws3p,ws3s,ws2p,ws2s
    void *d_tmaps = nullptr;                   // tensor-path TMA descriptors (CUtensorMap[])
    uint8_t *d_rowmax = nullptr;               // tensor-path per-row max exponent bytes
    uint16_t *d_router_hilo = nullptr;         // tensor-path router weights as BF16 [E, 2H] (hi | lo)
    float *d_glu_bound = nullptr;              // largest gate / up row L2 norms: routed w1, w3, shared ws1, ws3
    int *d_dense_cnt = nullptr;                // split-K arrival counters of the weight-stationary dense
                                               // GEMMs: router + down_proj tiles, then up_proj tiles
    int dense_cnt_up = 0;                      // first up_proj counter
    int dense_cnt_n = 0;                       // counters in all
    size_t tmap_count = 0;
    k3_prof *prof = nullptr;                   // stage timing, when enabled
    // split-K plans of the decode-size dense GEMMs per token count (0 = not planned yet):
    // [T][0] router, [T][1] down-projection, [T][2] up-projection
    unsigned char dense_splits[257][3] = {};
};

// Stage bracket used by the forward orchestration.
struct k3_stage {
    k3moe_handle *h;
    int s;
    cudaStream_t st;
    long l0;
    k3_stage(k3moe_handle *h_, int s_, cudaStream_t st_) : h(h_), s(s_), st(st_), l0(g_k3_launches)
    {
        if (h->prof && h->prof->on && h->prof->pos < k3_prof::RING) {
            cudaEventRecord(h->prof->ev[h->prof->pos][s][0], st);
            h->prof->used[h->prof->pos][s] = true;
        }
    }
    ~k3_stage()
    {
        if (h->prof && h->prof->on) {
            if (h->prof->pos < k3_prof::RING) cudaEventRecord(h->prof->ev[h->prof->pos][s][1], st);
            h->prof->launches[s] += g_k3_launches - l0;
        }
    }
};

// --------------------------------------------------------------- workspace
struct k3_ws {
    float *logits;        // [T, E] fp32
    uint16_t *h;          // [T, L] BF16 latent
    int32_t *idx;         // [T, K]
    float *wts;           // [T, K]
    int32_t *counts;      // [E]
    int32_t *offsets;     // [E + 1]
    int32_t *tok_of;      // [T*K] permuted row -> token
    int32_t *row_of;      // [T*K] (t, k) -> permuted row
    int32_t *meta;        // small scalars: [0] = number of active experts, [1] = number of tiles
    int32_t *active;      // [E] active expert list
    int32_t *tiles;       // tensor-path tile list (int4 per tile)
    int32_t *gv_sync;     // [2 + T*K + E] fused decode GEMV: ticket counter, then per-tile finished gate/up item-warps
    void *act;            // [T*K, I] fp32 (generic) or f16 (tensor path)
    void *y;              // [T*K, L] fp32 (generic) or BF16 (tensor path)
    void *hperm;          // [T*K, L] f16 (tensor path) activation rows in expert order
    float *hscale;        // [T*K] per-row power-of-two factor of hperm
    float *ascale;        // [T*K] per-row power of two 2^k the f16 GLU output is divided by (the down projection multiplies it back)
    float *xascale;       // [T] the same for the shared experts' GLU output
    uint16_t *nrm;        // [T, L] BF16 normalised latent
    float *o32;           // [T, H] fp32 up_proj output (generic path: + shared; tensor path: the shared down's addend)
    float *part;          // split-K partials of the dense tensor-core GEMMs (small T only)
    size_t part_floats;
    void *sact;           // [T, S] shared-expert activation (fp32 generic / f16 tensor)
    void *xs;             // [T, H] f16 scaled copy of x for the shared GLU (tensor path)
    float *xscale;        // [T]
    uint16_t *stage_x;    // [T, H] BF16 staging for k3moe_forward_host
    uint16_t *stage_out;  // [T, H]
    int32_t *stage_idx;   // [T, K]
    float *stage_w;       // [T, K]
    int32_t *chunk_cnt;   // [E, ceil(T / K3_PERM_CHUNK)] per-chunk counts, then bases (large T)
    uint8_t *mxs;         // A8: E8M0 scales of the MXFP8 expert inputs, [T*K, L/32] then [T*K, I/32]
    size_t bytes;
};

// Token permutation: from K3_PERM_CHUNKED_T tokens on, a chunked stable scatter
// (tokens in chunks of K3_PERM_CHUNK) replaces the one-CTA-per-expert scan.
constexpr int K3_PERM_CHUNK = 32;
// Largest split-K factor of the decode-size dense GEMMs (partials buffer sizing).
constexpr int K3_DENSE_MAX_SPLITS = 16;
constexpr int K3_PERM_CHUNKED_T = 512;

int k3_ws_layout(const k3moe_handle *h, int T, void *base, k3_ws *ws);  // base may be NULL (sizing)

// --------------------------------------------------------------- launchers
// routing and permutation (route.cu)
int k3_launch_topk(const k3moe_handle *h, const float *logits, int T, int32_t *idx, float *wts,
                   int32_t *counts_zero, cudaStream_t st);   // counts_zero: [E] set to 0, or NULL
void k3_launch_chunk_count(const int32_t *idx, int T, int K, int E, int32_t *chunk_cnt, int32_t *totals,
                           int *status, cudaStream_t st);
void k3_launch_chunk_base(int T, int E, const int32_t *base, int32_t *chunk_cnt, cudaStream_t st);
size_t k3_ep_dispatch_workspace_bytes(int T, int E);
int k3_ep_plan(const k3moe_handle *h, const int32_t *counts, int R, int C, const k3moe_ep_plan *plan,
               cudaStream_t st);
int k3_ep_dispatch(const k3moe_handle *h, const int32_t *idx, int T, int src, const int32_t *counts, int R,
                   const k3moe_ep_plan *plan, int32_t *dest_rank, int32_t *dest_row, void *ws, cudaStream_t st);
size_t k3_qb_workspace_bytes(int T, int E, int nbins);
int k3_qb_bias(const k3moe_handle *h, const float *logits, int T, const float *bias_in, float *bias_out,
               int nbins, void *ws, size_t ws_bytes, cudaStream_t st);
int k3_launch_permute(const k3moe_handle *h, const k3_ws &ws, int T, int tile_n, cudaStream_t st);   // after top-k zeroed ws.counts
// Top-K then the permutation (one fused launch at decode sizes), with their profiling stages.
int k3_launch_route(k3moe_handle *h, const k3_ws &ws, int T, int tile_n, cudaStream_t st);

// generic CUDA-core kernels (generic.cu)
int k3_launch_rows_gemm(const void *A, int a_bf16, int M, int K, const void *W, int w_bf16, int N,
                        float *out_f32, uint16_t *out_bf16, int accumulate, cudaStream_t st);
// A8: n values (n a multiple of 32; blocks of 32 along rows) rounded to OCP MXFP8;
// in BF16 (in_fp32 = 0) or fp32; out_kind 0 BF16, 1 fp32, 2 f16 (divided by the power
// of two row_div[i / row_len] of its row when row_div is given).  in may equal out
// when the element sizes match.
int k3_launch_mx8_rows(const void *in, int in_fp32, void *out, int out_kind, size_t n, int *status, int num_sms,
                       cudaStream_t st, const float *row_div = nullptr, int row_len = 1);
int k3_launch_glu_generic(const k3::K3Act &act_fn, const uint16_t *in, int din, const int32_t *row_token, int rows,
                          const uint8_t *const *w1p, const uint8_t *const *w1s,
                          const uint8_t *const *w3p, const uint8_t *const *w3s,
                          const int32_t *offsets, int n_groups, int dint, float *act,
                          int *status, cudaStream_t st);
int k3_launch_down_generic(const float *act, int dint, int rows, const uint8_t *const *w2p,
                           const uint8_t *const *w2s, const int32_t *offsets, int n_groups,
                           int dout, float *y, int accumulate, cudaStream_t st);
int k3_launch_combine_norm(const void *y, int y_bf16, const int32_t *row_of, const float *wts,
                           const uint16_t *gamma, int T, int K, int L, float eps, uint16_t *nrm,
                           cudaStream_t st);
int k3_launch_finish(const float *o32, int n, uint16_t *out, cudaStream_t st);
int k3_launch_dequant_debug(const uint8_t *packed, const uint8_t *scale, int rows, int cols,
                            float *out, cudaStream_t st);
int k3_launch_wait_debug(int *status, int spin_limit, cudaStream_t st);
