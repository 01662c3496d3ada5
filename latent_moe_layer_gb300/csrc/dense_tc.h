// Dense BF16 GEMMs on tcgen05 (dense_tc.cu): arguments and launchers.
#pragma once
#include <cudaTypedefs.h>

#include "k3moe_internal.h"

namespace k3 {

enum DenseOut { DN_OUT_F32 = 0, DN_OUT_BF16 = 1 };

// One N segment: weight rows [0, n_out) of its tensor map (n_tiles tiles of BN rows).
struct DenseSeg {
    int n_tiles;     // ceil(n_out / BN)
    int n_out;       // valid weight rows
    int splits;      // split-K factor, 1 .. K / 64 (split s takes K steps [s KS / splits, (s + 1) KS / splits))
    int K;           // reduction length (multiple of 64)
    int a_kmod;      // X column = k % a_kmod (router hi/lo: H; otherwise K)
    int mode;        // DN_OUT_F32: out[(split * M + m) * ldo + col0 + n]; DN_OUT_BF16: out[m * ldo + col0 + n]
    int m_group;     // token-major kernel: the tiles of m_group token tiles (all n tiles) run before the next
                     // group's, so the group's activation rows and the weights stay in L2; 0 = all token tiles
    void *out;
    int ldo;
    int col0;
    // weight-stationary kernel with DenseArgs::tile_cnt: where the last split of a tile
    // writes the tile's sum over splits (red_mode DN_OUT_F32 or DN_OUT_BF16, [m * red_ldo + n])
    void *red_out;
    int red_mode;
    int red_ldo;
};

struct DenseArgs {
    DenseSeg seg[2];
    int nseg;
    int M;           // token rows
    int *status;
    // weight-stationary kernel: one arrival counter per output tile (segment 0's tiles
    // first), zero before the launch and left zero by it; nullptr = partials only
    int *tile_cnt;
};

}  // namespace k3

// X rows [rows, cols] BF16 (or weights): box 64 x box_rows, 128-byte swizzle.
bool k3_encode_bf16_rows(CUtensorMap *m, const void *base, int rows, int cols, int box_rows);
// Decode sizes (T <= 256): the weight-stationary kernel (MMA M = 128 weight rows, N =
// tokens), split-K fp32 partials; with args.tile_cnt the last split of each tile to
// finish also sums the tile's partials in split order into red_out.  a: x rows [T, K]
// with box rows k3_dense_ws_rows(T).
int k3_dense_ws_rows(int T);
int k3_launch_dense_ws(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1, const k3::DenseArgs &args,
                       int num_sms, cudaStream_t st);
int k3_launch_dense_tc(int bn, const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                       const k3::DenseArgs &args, int num_sms, cudaStream_t st);
// out = sum over splits of part[s][m][c0 + j], j < n (fp32 and/or BF16 outputs, row stride ldo).
int k3_launch_dense_reduce(const float *part, int splits, int M, int ldp, int c0, int n, float *out32,
                           uint16_t *out16, int ldo, cudaStream_t st);
int k3_launch_split_hilo(const float *w, int E, int H, uint16_t *out, cudaStream_t st);
