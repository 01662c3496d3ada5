// Allocation-free routing entry point: router logits + top-K selection with the
// logits scratch in a file-scope device array instead of caller workspace.
//
// For callers that cannot allocate device memory at all -- for example a
// plugin host that hands each operator only its input and output buffers and
// forbids device allocation while it runs (cudaMalloc may block and
// synchronise the device, and a caching allocator may already own all free
// memory).  Such a caller still passes x and the idx/w outputs; the scratch
// comes from g_route_scratch below, which every GPU that loads this library
// holds until the process exits.
#include <mutex>

#include "k3moe_internal.h"

namespace {

// Capacity of the logits scratch: T * n_experts fp32 values (1 MiB).
constexpr size_t kRouteScratchFloats = K3MOE_ROUTE_STATIC_MAX_LOGITS;

static __device__ __align__(256) float g_route_scratch[kRouteScratchFloats];

// Device address of g_route_scratch per device, resolved once with that device current.
constexpr int kMaxDevices = 64;
float *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

int scratch_for_current_device(float **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return K3MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return K3MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return K3MOE_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_scratch_ptr[dev];
    return K3MOE_OK;
}

}  // namespace

extern "C" int k3moe_route_static(k3moe_handle *h, const void *x, int T, int32_t *idx_out, float *w_out,
                                  cudaStream_t stream)
{
    if (!h) return K3MOE_ERR_ARG;
    if (!h->loaded) return K3MOE_ERR_STATE;
    if (T < 0 || T > K3_MAX_TOKENS) return K3MOE_ERR_ARG;
    if (T == 0) return K3MOE_OK;
    if (!x || !idx_out || !w_out) return K3MOE_ERR_ARG;
    if ((uintptr_t)x % 16) return K3MOE_ERR_ALIGN;
    const k3moe_config &c = h->cfg;
    if ((size_t)T * (size_t)c.n_experts > kRouteScratchFloats) return K3MOE_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return K3MOE_ERR_CUDA;
    if (dev != h->device) return K3MOE_ERR_STATE;
    float *logits = nullptr;
    int rc = scratch_for_current_device(&logits);
    if (rc) return rc;
    // Every one of the T * n_experts logits is written before top-K reads it,
    // so nothing left in the array by an earlier call is ever read.
    rc = k3_launch_rows_gemm(x, 1, T, c.hidden, h->w_router, c.router_dtype == K3MOE_ROUTER_BF16,
                             c.n_experts, logits, nullptr, 0, stream);
    if (rc) return rc;
    return k3_launch_topk(h, logits, T, idx_out, w_out, nullptr, stream);
}
