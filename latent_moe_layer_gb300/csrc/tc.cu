// Tensor-core path (tcgen05 + TMA).  Filled in by the grouped expert GEMMs.
#include "tc.h"

size_t k3_tc_tmap_count(const k3moe_config &c) { (void)c; return 0; }

int k3_tc_prepare(k3moe_handle *h, const uint8_t *const *const tabs[6], cudaStream_t st)
{
    (void)h; (void)tabs; (void)st;
    return K3MOE_OK;
}

int k3_forward_tc(k3moe_handle *h, const void *x, int T, void *out, const k3_ws &ws, cudaStream_t st)
{
    (void)h; (void)x; (void)T; (void)out; (void)ws; (void)st;
    return K3MOE_ERR_UNSUPPORTED;
}
