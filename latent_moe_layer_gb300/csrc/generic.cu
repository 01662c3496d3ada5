// Generic CUDA-core kernels: any shape whose widths are multiples of 32.
//
//   rows_gemm     out[m, n] (+)= sum_k A[m, k] W[n, k]        (router, down/up projections)
//   glu_generic   act[r, i] = a(W1_e[i] . in[tok(r)], W3_e[i] . in[tok(r)])  (SiLU or SiTU GLU)
//   down_generic  y[r, o] (+)= W2_e[o] . act[r]
//   combine_norm  n[t] = rmsnorm(sum_k w[t, k] y[row(t, k)]) * gamma
//
// MXFP4 decoding: "Kimi K3, as released", Gate 3 section (two E2M1 codes per
// byte, low nibble first; one E8M0 exponent per 32 weights, value 2^(e-127)).
#include "k3moe_internal.h"

#include <algorithm>
#include "ptx.cuh"

namespace k3 {

// ------------------------------------------------------------------ dense rows GEMM
// CTA: 8 warps x 2 W-rows = 16 output columns; TM tokens per CTA; A staged in
// shared memory as fp32 in K-chunks of KC.
constexpr int RG_TM = 16, RG_KC = 512, RG_ROWS = 16;

template <bool A_BF16, bool W_BF16>
__global__ void __launch_bounds__(256) rows_gemm_kernel(const void *__restrict__ Av, int M, int K,
                                                        const void *__restrict__ Wv, int N,
                                                        float *__restrict__ out32,
                                                        uint16_t *__restrict__ out16, int accumulate)
{
    griddep_enter();
    __shared__ __align__(16) float sA[RG_TM][RG_KC];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m0 = blockIdx.y * RG_TM;
    const int n0 = blockIdx.x * RG_ROWS + warp * 2;
    float acc[2][RG_TM];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int t = 0; t < RG_TM; ++t) acc[r][t] = 0.f;

    for (int k0 = 0; k0 < K; k0 += RG_KC) {
        __syncthreads();
        for (int i = tid; i < RG_TM * RG_KC; i += 256) {
            int t = i / RG_KC, k = i % RG_KC;
            float v = 0.f;
            if (m0 + t < M && k0 + k < K) {
                size_t o = (size_t)(m0 + t) * K + k0 + k;
                v = A_BF16 ? bf16_to_f32(reinterpret_cast<const uint16_t *>(Av)[o])
                           : reinterpret_cast<const float *>(Av)[o];
            }
            sA[t][k] = v;
        }
        __syncthreads();
        float wv[2][4][4];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                int k = k0 + s * 128 + lane * 4;
                int n = n0 + r;
#pragma unroll
                for (int q = 0; q < 4; ++q) wv[r][s][q] = 0.f;
                if (n < N && k < K) {   // K is a multiple of 32, so k..k+3 are in range together
                    size_t o = (size_t)n * K + k;
                    if (W_BF16) {
                        uint2 p = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(Wv) + o);
                        wv[r][s][0] = __uint_as_float(p.x << 16);
                        wv[r][s][1] = __uint_as_float(p.x & 0xffff0000u);
                        wv[r][s][2] = __uint_as_float(p.y << 16);
                        wv[r][s][3] = __uint_as_float(p.y & 0xffff0000u);
                    } else {
                        float4 p = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(Wv) + o);
                        wv[r][s][0] = p.x; wv[r][s][1] = p.y; wv[r][s][2] = p.z; wv[r][s][3] = p.w;
                    }
                }
            }
#pragma unroll
        for (int s = 0; s < 4; ++s) {
#pragma unroll
            for (int t = 0; t < RG_TM; ++t) {
                float4 a = *reinterpret_cast<const float4 *>(&sA[t][s * 128 + lane * 4]);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    acc[r][t] = fmaf(wv[r][s][0], a.x, acc[r][t]);
                    acc[r][t] = fmaf(wv[r][s][1], a.y, acc[r][t]);
                    acc[r][t] = fmaf(wv[r][s][2], a.z, acc[r][t]);
                    acc[r][t] = fmaf(wv[r][s][3], a.w, acc[r][t]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int t = 0; t < RG_TM; ++t) {
            float v = acc[r][t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            acc[r][t] = v;
        }
    // lane t writes token t of both rows
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int t = 0; t < RG_TM; ++t)
            if (lane == t && m0 + t < M && n0 + r < N) {
                size_t o = (size_t)(m0 + t) * N + n0 + r;
                float v = acc[r][t];
                if (out32) out32[o] = accumulate ? out32[o] + v : v;
                if (out16) out16[o] = f32_to_bf16(v);
            }
}

// ------------------------------------------------------------------ MXFP4 GLU (generic)
constexpr int GX_TOK = 8;

// Decode the 32 values of one MX block (16 packed bytes at p, E8M0 byte e).
__device__ __forceinline__ void decode_block(const uint8_t *p, uint32_t e, float (&v)[32])
{
    float s = e8m0_to_f32(e);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w = p[4 * q] | (p[4 * q + 1] << 8) | (p[4 * q + 2] << 16) | ((uint32_t)p[4 * q + 3] << 24);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[8 * q + j] = e2m1_to_f32((w >> (4 * j)) & 0xFu, s);
    }
}

// Grid (dint / 8, n_groups); warp w computes output row i = 8 * blockIdx.x + w for
// every row r of the group, GX_TOK rows at a time; lanes split the K blocks.
__global__ void __launch_bounds__(256) glu_generic_kernel(
    const K3Act act_fn, const uint16_t *__restrict__ in, int din, const int32_t *__restrict__ row_token, int rows,
    const uint8_t *const *__restrict__ w1p, const uint8_t *const *__restrict__ w1s,
    const uint8_t *const *__restrict__ w3p, const uint8_t *const *__restrict__ w3s,
    const int32_t *__restrict__ offsets, int dint, float *__restrict__ act)
{
    griddep_enter();
    const int g = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i = blockIdx.x * 8 + warp;
    const int r0 = offsets ? offsets[g] : 0;
    const int r1 = offsets ? offsets[g + 1] : rows;
    if (r0 >= r1 || i >= dint) return;
    const uint8_t *p1 = w1p[g] + (size_t)i * (din / 2), *s1 = w1s[g] + (size_t)i * (din / 32);
    const uint8_t *p3 = w3p[g] + (size_t)i * (din / 2), *s3 = w3s[g] + (size_t)i * (din / 32);
    const int nblk = din / 32;
    for (int rb = r0; rb < r1; rb += GX_TOK) {
        const int nt = min(GX_TOK, r1 - rb);
        float gacc[GX_TOK], uacc[GX_TOK];
#pragma unroll
        for (int t = 0; t < GX_TOK; ++t) gacc[t] = uacc[t] = 0.f;
        for (int b = lane; b < nblk; b += 32) {
            float v1[32], v3[32];
            decode_block(p1 + 16 * b, s1[b], v1);
            decode_block(p3 + 16 * b, s3[b], v3);
#pragma unroll
            for (int t = 0; t < GX_TOK; ++t) {
                if (t < nt) {
                    int tok = row_token ? row_token[rb + t] : rb + t;
                    const uint16_t *hv = in + (size_t)tok * din + 32 * b;
                    float ga = 0.f, ua = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        float x = bf16_to_f32(hv[j]);
                        ga = fmaf(v1[j], x, ga);
                        ua = fmaf(v3[j], x, ua);
                    }
                    gacc[t] += ga;
                    uacc[t] += ua;
                }
            }
        }
#pragma unroll
        for (int t = 0; t < GX_TOK; ++t) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                gacc[t] += __shfl_xor_sync(0xffffffffu, gacc[t], off);
                uacc[t] += __shfl_xor_sync(0xffffffffu, uacc[t], off);
            }
        }
        if (lane < nt) {
            float gv = 0.f, uv = 0.f;
#pragma unroll
            for (int t = 0; t < GX_TOK; ++t)
                if (t == lane) { gv = gacc[t]; uv = uacc[t]; }
            act[(size_t)(rb + lane) * dint + i] = k3_glu(gv, uv, act_fn);
        }
    }
}

__global__ void __launch_bounds__(256) down_generic_kernel(
    const float *__restrict__ act, int dint, int rows, const uint8_t *const *__restrict__ w2p,
    const uint8_t *const *__restrict__ w2s, const int32_t *__restrict__ offsets, int dout,
    float *__restrict__ y, int accumulate)
{
    griddep_enter();
    const int g = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int o = blockIdx.x * 8 + warp;
    const int r0 = offsets ? offsets[g] : 0;
    const int r1 = offsets ? offsets[g + 1] : rows;
    if (r0 >= r1 || o >= dout) return;
    const uint8_t *p2 = w2p[g] + (size_t)o * (dint / 2), *s2 = w2s[g] + (size_t)o * (dint / 32);
    const int nblk = dint / 32;
    for (int rb = r0; rb < r1; rb += GX_TOK) {
        const int nt = min(GX_TOK, r1 - rb);
        float acc[GX_TOK];
#pragma unroll
        for (int t = 0; t < GX_TOK; ++t) acc[t] = 0.f;
        for (int b = lane; b < nblk; b += 32) {
            float v[32];
            decode_block(p2 + 16 * b, s2[b], v);
#pragma unroll
            for (int t = 0; t < GX_TOK; ++t) {
                if (t < nt) {
                    const float *av = act + (size_t)(rb + t) * dint + 32 * b;
                    float a = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) a = fmaf(v[j], av[j], a);
                    acc[t] += a;
                }
            }
        }
#pragma unroll
        for (int t = 0; t < GX_TOK; ++t)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
        if (lane < nt) {
            float v = 0.f;
#pragma unroll
            for (int t = 0; t < GX_TOK; ++t)
                if (t == lane) v = acc[t];
            size_t off = (size_t)(rb + lane) * dout + o;
            y[off] = accumulate ? y[off] + v : v;
        }
    }
}

// ------------------------------------------------------------------ combine + RMSNorm
// One CTA per token; fixed k order (deterministic, no atomics).
constexpr int CN_MAXV = 32;   // L <= 256 * 32

__global__ void __launch_bounds__(256) combine_norm_kernel(
    const void *__restrict__ yv, int y_bf16, const int32_t *__restrict__ row_of,
    const float *__restrict__ wts, const uint16_t *__restrict__ gamma, int K, int L, float eps,
    uint16_t *__restrict__ nrm)
{
    griddep_enter();
    const int t = blockIdx.x, tid = threadIdx.x;
    __shared__ float red[8];
    __shared__ int rows[64];
    __shared__ float ws_[64];
    if (tid < K) {
        rows[tid] = row_of[(size_t)t * K + tid];
        ws_[tid] = wts[(size_t)t * K + tid];
    }
    __syncthreads();
    float z[CN_MAXV];
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < CN_MAXV; ++q) {
        int i = tid + 256 * q;
        float acc = 0.f;
        if (i < L) {
            for (int k = 0; k < K; ++k) {
                size_t o = (size_t)rows[k] * L + i;
                float yv_ = y_bf16 ? bf16_to_f32(reinterpret_cast<const uint16_t *>(yv)[o])
                                   : reinterpret_cast<const float *>(yv)[o];
                acc = fmaf(ws_[k], yv_, acc);
            }
        }
        z[q] = acc;
        ss = fmaf(acc, acc, ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)L + eps);
#pragma unroll
    for (int q = 0; q < CN_MAXV; ++q) {
        int i = tid + 256 * q;
        if (i < L) nrm[(size_t)t * L + i] = f32_to_bf16(z[q] * inv * bf16_to_f32(gamma[i]));
    }
}

// Vectorised combine + RMSNorm for BF16 y: one thread per 8 latent elements (L / 8 threads).
__global__ void __launch_bounds__(1024) combine_norm_v8_kernel(
    const uint16_t *__restrict__ y, const int32_t *__restrict__ row_of, const float *__restrict__ wts,
    const uint16_t *__restrict__ gamma, int K, int L, float eps, uint16_t *__restrict__ nrm)
{
    griddep_enter();
    const int t = blockIdx.x, tid = threadIdx.x;
    __shared__ float red[32];
    __shared__ int rows[64];
    __shared__ float ws_[64];
    if (tid < K) {
        rows[tid] = row_of[(size_t)t * K + tid];
        ws_[tid] = wts[(size_t)t * K + tid];
    }
    __syncthreads();
    const int i = tid * 8;
    float z[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) z[q] = 0.f;
    if (i < L) {
        // fixed k order; the rows of a group of 8 are loaded before they are summed
        for (int k0 = 0; k0 < K; k0 += 8) {
            uint4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k0 + k < K) v[k] = *reinterpret_cast<const uint4 *>(y + (size_t)rows[k0 + k] * L + i);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (k0 + k >= K) break;
                const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                const float wk = ws_[k0 + k];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    z[2 * q] = fmaf(wk, __uint_as_float(w[q] << 16), z[2 * q]);
                    z[2 * q + 1] = fmaf(wk, __uint_as_float(w[q] & 0xffff0000u), z[2 * q + 1]);
                }
            }
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) ss = fmaf(z[q], z[q], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    const int nw = (blockDim.x + 31) >> 5;
    for (int w = 0; w < nw; ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)L + eps);
    if (i < L) {
        const uint4 g = *reinterpret_cast<const uint4 *>(gamma + i);
        const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            o[q] = (uint32_t)f32_to_bf16(z[2 * q] * inv * __uint_as_float(gw[q] << 16)) |
                   ((uint32_t)f32_to_bf16(z[2 * q + 1] * inv * __uint_as_float(gw[q] & 0xffff0000u)) << 16);
        *reinterpret_cast<uint4 *>(nrm + (size_t)t * L + i) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__global__ void finish_kernel(const float *__restrict__ o32, size_t n, uint16_t *__restrict__ out)
{
    griddep_enter();
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = f32_to_bf16(o32[i]);
}

__global__ void dequant_debug_kernel(const uint8_t *__restrict__ packed,
                                     const uint8_t *__restrict__ scale, int rows, int cols,
                                     float *__restrict__ out)
{
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)rows * cols) return;
    int r = (int)(i / cols), k = (int)(i % cols);
    uint8_t byte = packed[(size_t)r * (cols / 2) + k / 2];
    uint32_t code = (k & 1) ? (byte >> 4) : (byte & 0xF);
    out[i] = e2m1_to_f32(code, e8m0_to_f32(scale[(size_t)r * (cols / 32) + k / 32]));
}

// One CTA; thread 0 waits on a barrier nothing arrives on.
__global__ void wait_debug_kernel(int *status, int spin_limit)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mbar_wait(smem_u32(&bar), 0, (uint32_t)spin_limit))
            set_status(status, K3MOE_ERR_TIMEOUT, 1);
        else  // cannot complete; kept so the wait is not optimised away
            set_status(status, K3MOE_ERR_STATE, 1);
    }
}

// ---- A8: OCP MXFP8 rounding of activation rows (blocks of 32 along a row).
// One warp per block: lane j holds element j; X = floor(log2 amax) - 8 from the
// exponent field of amax (kept >= -127); each value becomes E4M3(v / 2^X) 2^X
// with the hardware's round-to-nearest-even, saturating E4M3 conversion.
template <typename T> __device__ __forceinline__ float mx8_load(const T *p);
template <> __device__ __forceinline__ float mx8_load<uint16_t>(const uint16_t *p) { return bf16_to_f32(*p); }
template <> __device__ __forceinline__ float mx8_load<float>(const float *p) { return *p; }


// out_kind: 0 BF16, 1 fp32, 2 f16 (|q| > 65504 is reported as K3MOE_ERR_RANGE)
template <typename TI>
__global__ void __launch_bounds__(256) mx8_rows_kernel(const TI *__restrict__ in, void *__restrict__ out,
                                                       int out_kind, size_t nblk, int *status,
                                                       const float *__restrict__ row_div, int row_len)
{
    griddep_enter();
    const int lane = threadIdx.x & 31;
    const size_t w0 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const size_t nw = ((size_t)gridDim.x * blockDim.x) >> 5;
    for (size_t b = w0; b < nblk; b += nw) {
        const size_t i = b * 32 + lane;
        const float v = mx8_load<TI>(in + i);
        float amax = fabsf(v);
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float q = mx8_round(v, amax);
        if (out_kind == 0) reinterpret_cast<uint16_t *>(out)[i] = f32_to_bf16(q);
        else if (out_kind == 1) reinterpret_cast<float *>(out)[i] = q;
        else {
            // f16 output: divided by its row's power of two (exact) to stay inside the f16 range
            const float qs = row_div ? q * pow2_inverse(row_div[i / row_len]) : q;
            if (!(fabsf(qs) <= 65504.f)) set_status(status, K3MOE_ERR_RANGE, 4);
            reinterpret_cast<__half *>(out)[i] = __float2half_rn(qs);
        }
    }
}

}  // namespace k3

using namespace k3;

#define K3_LAUNCH_OK() (cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ERR_CUDA)

int k3_launch_rows_gemm(const void *A, int a_bf16, int M, int K, const void *W, int w_bf16, int N,
                        float *out_f32, uint16_t *out_bf16, int accumulate, cudaStream_t st)
{
    if (M == 0) return K3MOE_OK;
    dim3 grid((N + RG_ROWS - 1) / RG_ROWS, (M + RG_TM - 1) / RG_TM);
    if (grid.y > 65535) return K3MOE_ERR_UNSUPPORTED;
    if (a_bf16 && w_bf16) k3_launch(rows_gemm_kernel<true, true>, grid, 256, 0, st, A, M, K, W, N, out_f32, out_bf16, accumulate);
    else if (a_bf16) k3_launch(rows_gemm_kernel<true, false>, grid, 256, 0, st, A, M, K, W, N, out_f32, out_bf16, accumulate);
    else if (w_bf16) k3_launch(rows_gemm_kernel<false, true>, grid, 256, 0, st, A, M, K, W, N, out_f32, out_bf16, accumulate);
    else k3_launch(rows_gemm_kernel<false, false>, grid, 256, 0, st, A, M, K, W, N, out_f32, out_bf16, accumulate);
    k3_note_launch();
    return K3_LAUNCH_OK();
}

int k3_launch_glu_generic(const K3Act &act_fn, const uint16_t *in, int din, const int32_t *row_token, int rows,
                          const uint8_t *const *w1p, const uint8_t *const *w1s,
                          const uint8_t *const *w3p, const uint8_t *const *w3s,
                          const int32_t *offsets, int n_groups, int dint, float *act, int *status,
                          cudaStream_t st)
{
    (void)status;
    if (n_groups > 65535) return K3MOE_ERR_UNSUPPORTED;
    dim3 grid((dint + 7) / 8, n_groups);
    k3_launch(glu_generic_kernel, grid, 256, 0, st, act_fn, in, din, row_token, rows, w1p, w1s, w3p, w3s, offsets,
              dint, act);
    k3_note_launch();
    return K3_LAUNCH_OK();
}

int k3_launch_down_generic(const float *act, int dint, int rows, const uint8_t *const *w2p,
                           const uint8_t *const *w2s, const int32_t *offsets, int n_groups,
                           int dout, float *y, int accumulate, cudaStream_t st)
{
    if (n_groups > 65535) return K3MOE_ERR_UNSUPPORTED;
    dim3 grid((dout + 7) / 8, n_groups);
    k3_launch(down_generic_kernel, grid, 256, 0, st, act, dint, rows, w2p, w2s, offsets, dout, y, accumulate);
    k3_note_launch();
    return K3_LAUNCH_OK();
}

int k3_launch_combine_norm(const void *y, int y_bf16, const int32_t *row_of, const float *wts,
                           const uint16_t *gamma, int T, int K, int L, float eps, uint16_t *nrm,
                           cudaStream_t st)
{
    if (T == 0) return K3MOE_OK;
    if (L > 256 * CN_MAXV || K > 64) return K3MOE_ERR_UNSUPPORTED;
    if (y_bf16 && L % 8 == 0 && L / 8 <= 1024) {
        const int threads = ((L / 8) + 31) / 32 * 32;
        k3_launch(combine_norm_v8_kernel, T, threads, 0, st, (const uint16_t *)y, row_of, wts, gamma, K, L, eps, nrm);
        k3_note_launch();
        return K3_LAUNCH_OK();
    }
    k3_launch(combine_norm_kernel, T, 256, 0, st, y, y_bf16, row_of, wts, gamma, K, L, eps, nrm);
    k3_note_launch();
    return K3_LAUNCH_OK();
}

int k3_launch_finish(const float *o32, int n, uint16_t *out, cudaStream_t st)
{
    if (n == 0) return K3MOE_OK;
    k3_launch(finish_kernel, (unsigned)(((size_t)n + 255) / 256), 256, 0, st, o32, (size_t)n, out);
    k3_note_launch();
    return K3_LAUNCH_OK();
}

int k3_launch_dequant_debug(const uint8_t *packed, const uint8_t *scale, int rows, int cols,
                            float *out, cudaStream_t st)
{
    size_t n = (size_t)rows * cols;
    if (n == 0) return K3MOE_OK;
    dequant_debug_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(packed, scale, rows, cols, out);
    k3_note_launch();
    return K3_LAUNCH_OK();
}

int k3_launch_wait_debug(int *status, int spin_limit, cudaStream_t st)
{
    wait_debug_kernel<<<1, 32, 0, st>>>(status, spin_limit < 1 ? 1 : spin_limit);
    k3_note_launch();
    return K3_LAUNCH_OK();
}

int k3_launch_mx8_rows(const void *in, int in_fp32, void *out, int out_kind, size_t n, int *status, int num_sms,
                       cudaStream_t st, const float *row_div, int row_len)
{
    if (n == 0) return K3MOE_OK;
    if (n % 32) return K3MOE_ERR_SHAPE;
    const size_t nblk = n / 32;
    const unsigned grid = (unsigned)std::min<size_t>((nblk + 7) / 8, (size_t)8 * (num_sms > 0 ? num_sms : 148));
    if (in_fp32)
        k3_launch(mx8_rows_kernel<float>, grid, 256, 0, st, (const float *)in, out, out_kind, nblk, status, row_div,
                  row_len);
    else
        k3_launch(mx8_rows_kernel<uint16_t>, grid, 256, 0, st, (const uint16_t *)in, out, out_kind, nblk, status,
                  row_div, row_len);
    k3_note_launch();
    return K3_LAUNCH_OK();
}
