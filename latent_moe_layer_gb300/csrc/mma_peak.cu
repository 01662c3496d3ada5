// Tensor-core peak microbenchmark: back-to-back tcgen05.mma on operands resident
// in shared memory, one CTA per SM, accumulators in tensor memory.  It measures
// the rate each MMA kind reaches with no data movement, the denominator of the
// expert GEMMs' roofline (kind::f16 for the A16 path, kind::mxf8f6f4 for the
// block-scaled A8 path).
#include "k3moe_internal.h"
#include "ptx.cuh"

namespace k3 {
namespace {

// kind: 0 = f16 (M 128, K 16 per MMA); 1 = mxf8f6f4 E4M3 x E4M3 (K 32); 2 = mxf8f6f4
// E2M1 (unpacked) x E4M3 (K 32).  Every MMA reads a 128 x 128-byte A tile and an
// n x 128-byte B tile (all zero: the data do not change the rate) and accumulates
// into one of two TMEM accumulator sets.
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int kind, int n, int iters, int *status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *a = smem, *b = smem + 128 * 128;
    uint64_t *bar = (uint64_t *)(b + 256 * 128);
    uint32_t *holder = (uint32_t *)(bar + 1);
    const int warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < (128 + 256) * 128 / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bar), 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(holder), 512);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    // unit scale factors (E8M0 127) in columns 448.. (A: 4 columns, B: 8 columns)
    {
        const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
        const uint32_t one = 0x7F7F7F7Fu;
        const uint32_t v[8] = {one, one, one, one, one, one, one, one};
        tmem_st8(lane_base + 448, v);
        tmem_st8(lane_base + 456, v);
        tc_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        const uint64_t ad = smem_desc_sw128(smem_u32(a)), bd = smem_desc_sw128(smem_u32(b));
        const int nacc = n <= 224 ? 2 : 1;
        if (kind == 0) {
            const uint32_t id = idesc_f16(128, n, 0);
            for (int it = 0; it < iters; ++it) {
                const uint32_t d = tmem + (uint32_t)((it % nacc) * n);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)   // K 128 = 8 x 16 over the tile's 64-value rows twice
                    tc_mma_f16(d, ad + 2 * (kk & 3), bd + 2 * (kk & 3), id, kk > 0 ? 1u : 0u);
            }
        } else {
            const uint32_t at = kind == 2 ? MX_E2M1 : MX_E4M3;
            uint32_t id[4];
            for (int kk = 0; kk < 4; ++kk) id[kk] = idesc_mx(128, n, at, MX_E4M3, kk, kk);
            for (int it = 0; it < iters; ++it) {
                const uint32_t d = tmem + (uint32_t)((it % nacc) * n);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_mx(d, ad + 2 * kk, bd + 2 * kk, id[kk], tmem + 448, tmem + 452, kk > 0 ? 1u : 0u);
            }
        }
        tc_commit(smem_u32(bar));
        if (!mbar_wait(smem_u32(bar), 0, 0xFFFFFFFFu)) set_status(status, K3MOE_ERR_TIMEOUT, 50);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace
}  // namespace k3

using namespace k3;

// Flops of one launch: grid x iters x 2 M N K with K = 128 per iteration.
extern "C" int k3moe_mma_peak(int kind, int n, int iters, int *status, float *ms, cudaStream_t st)
{
    if (kind < 0 || kind > 2 || n < 16 || n > 256 || n % 16 || iters < 1 || !status || !ms) return K3MOE_ERR_ARG;
    int dev = 0, sms = 0;
    K3_CUDA_TRY(cudaGetDevice(&dev));
    K3_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int smem = (128 + 256) * 128 + 64 + 1024;
    static unsigned long long attr = 0;
    if (!k3_smem_attr(mma_peak_kernel, smem, attr)) return K3MOE_ERR_CUDA;
    cudaEvent_t e0, e1;
    K3_CUDA_TRY(cudaEventCreate(&e0));
    K3_CUDA_TRY(cudaEventCreate(&e1));
    mma_peak_kernel<<<sms, 128, smem, st>>>(kind, n, iters / 8 + 1, status);   // warm-up
    K3_CUDA_TRY(cudaEventRecord(e0, st));
    mma_peak_kernel<<<sms, 128, smem, st>>>(kind, n, iters, status);
    K3_CUDA_TRY(cudaEventRecord(e1, st));
    K3_CUDA_TRY(cudaEventSynchronize(e1));
    K3_CUDA_TRY(cudaGetLastError());
    K3_CUDA_TRY(cudaEventElapsedTime(ms, e0, e1));
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return K3MOE_OK;
}
