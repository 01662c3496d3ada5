// Tensor-core (tcgen05 / TMA) path: interface used by the C ABI.
#pragma once
#include "k3moe_internal.h"

// Whether the tensor path is compiled in and usable.
bool k3_tc_available();
// Number of TMA descriptors the tensor path keeps in the persistent buffer.
size_t k3_tc_tmap_count(const k3moe_config &c);
// Bytes of per-row maximum-exponent data kept in the persistent buffer.
size_t k3_tc_rowmax_bytes(const k3moe_config &c);
// Bytes of the router's BF16 hi/lo copy (0 when the router is stored BF16).
size_t k3_tc_hilo_bytes(const k3moe_config &c);
// Build the descriptors and per-row scale data after the weights are recorded.
int k3_tc_prepare(k3moe_handle *h, const uint8_t *const *const tabs[6], cudaStream_t st);
// Full forward on the tensor path.
int k3_forward_tc(k3moe_handle *h, const void *x, int T, void *out, const k3_ws &ws, cudaStream_t st);
// Device pointer to a one-entry table holding shared matrix i (0..5: ws1p, ws1s, ws3p, ws3s, ws2p, ws2s).
inline const uint8_t *const *k3_shared_tab(const k3moe_handle *h, int i) { return h->d_shtab + i; }
