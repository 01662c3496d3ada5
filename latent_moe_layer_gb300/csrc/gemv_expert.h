// Decode-batch streaming MXFP4 expert GEMV (gemv_expert.cu): arguments and launcher.
#pragma once
#include <cudaTypedefs.h>

#include "k3moe_internal.h"

namespace k3 {

enum GemvOut { GV_GLU_F16 = 0, GV_BF16 = 1 };

struct GemvArgs {
    const CUtensorMap *amaps;          // global: packed map of group g, matrix m at amaps[g * amap_stride + amap_off[m]]
    int amap_stride;
    int amap_off[2];
    const uint8_t *const *scales[2];   // [groups] of scale matrices [rows, K/32]
    int rows, K;                       // rows: multiple of 128; K: multiple of 512
    const int4 *tiles;                 // (group, first B row, B rows <= 16) per token tile
    const int *n_tiles;                // device count of tiles
    const float *rscale;               // [R] per-row factor applied to the GLU inputs, or nullptr
    const float *ascale;               // [R] per-row power of two 2^k: the f16 GLU output is divided by it,
                                       // the down projection's output multiplied by it; or nullptr
    K3Act act;                         // GLU activation
    int out_f32;                       // GLU: 1 writes fp32 [R, rows] (the A8 path rounds it afterwards)
    void *out;                         // GLU: f16 (or fp32) [R, rows]; BF16: BF16 [R, rows]
    int *status;
};

}  // namespace k3

// bmap: f16 activation rows [R, K], box 64 x 16, 128-byte swizzle.  max_nb: 2 for tiles of up
// to 16 tokens; 1 for tiles of at most 8 (a kernel with fewer live registers).
int k3_launch_gemv_expert(int glu, int mode, int max_nb, const CUtensorMap &bmap, const k3::GemvArgs &args,
                          int max_items, int num_sms, cudaStream_t st);
// The gate/up (a1, GLU) and down (a2, BF16) GEMVs of one routing in one persistent launch,
// 8-token tiles only: bmap1 over the f16 expert inputs [R, L], bmap2 over the GLU output
// [R, I] (a1.out), both with 16-row boxes; a2.rows a multiple of 256 (down items are 256
// rows).  sync: 1 + tiles ints, zero before the launch.  max_items bounds the grid.
int k3_launch_gemv_fused(const CUtensorMap &bmap1, const CUtensorMap &bmap2, const k3::GemvArgs &a1,
                         const k3::GemvArgs &a2, int32_t *sync, int max_items, int num_sms, cudaStream_t st);
