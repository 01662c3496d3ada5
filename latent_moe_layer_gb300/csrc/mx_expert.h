// Block-scaled grouped expert GEMMs of the A8 option (MXFP4 weights x MXFP8
// activations on tcgen05.mma kind::mxf8f6f4) and the MXFP8 activation prep.
#pragma once
#include <cudaTypedefs.h>

#include "k3moe_internal.h"

namespace k3 {

enum MxMode { MX_GLU = 0, MX_DOWN = 1 };

constexpr int MX_BN = 224;          // token rows per tile (MMA N <= 224)
constexpr int MX_KS = 128;          // K per pipeline stage: 128-byte rows of E4M3 / unpacked E2M1
constexpr int MX_GK = 512;          // K per scale group: 16 scale bytes per row
constexpr int MX_WBOX = 64;         // weight rows per TMA box

// Activation operand of one GEMM: E4M3 rows [R, K] (boxes of 128 bytes x 64 / 16
// rows, 128-byte swizzle) and their E8M0 scales [R, K / 32] (boxes of 16 bytes x
// 64 / 16 rows).
struct MxActMaps {
    CUtensorMap big, small, sbig, ssmall;
};

struct MxGemmArgs {
    const CUtensorMap *wmaps;       // FP4 weights (16U4_ALIGN16B, boxes 128 x 64 rows): group g, matrix m at
    const CUtensorMap *smaps;       //   wmaps[g * map_stride + map_off[m]]; E8M0 weight scales alike (16 B x 64 rows)
    int map_stride;
    int map_off[2];                 // MX_GLU: gate (w1), up (w3); MX_DOWN: w2 for both
    int rows;                       // weight rows per matrix (MX_GLU: multiple of 64; MX_DOWN: of 128)
    int K;                          // reduction length, multiple of 512
    const int4 *tiles;              // (group, row0, nrows, -) per token tile of at most MX_BN rows
    const int *n_tiles;             // device count of tiles
    uint8_t *out_q;                 // MX_GLU: E4M3 GLU output [R, rows]
    uint8_t *out_s;                 // MX_GLU: its E8M0 scales [R, rows / 32]
    uint16_t *out_bf16;             // MX_DOWN: BF16 [R, rows]
    int *status;
    uint32_t spin_limit;
    K3Act act;
};

bool k3_encode_mx_act(MxActMaps *m, const uint8_t *q, const uint8_t *s, int rows, int K);
int k3_launch_mx_expert(int mode, const MxActMaps &b, const MxGemmArgs &a, int max_jobs, int num_sms,
                        cudaStream_t st);
// MXFP8 of the BF16 rows h [T, L] (OCP MX: E4M3 elements, one E8M0 scale per 32),
// written as K copies in expert order: row row_of[t K + k] of q [R, L] and s [R, L / 32].
int k3_launch_prep_mx8(const uint16_t *h, int T, int L, const int32_t *row_of, int K, uint8_t *q, uint8_t *s,
                       int num_sms, cudaStream_t st);

}  // namespace k3
