// H-tiled implicit-GEMM convolution for sm_103a (declarations).
//
// An NCHW convolution with OIHW weights is, per image and per output H-tile
// of rows [o0, o1), a GEMM with
//     M = c_out,  N = (o1 - o0) * OW,  K = c * kh * kw,
//     A = W viewed as [c_out][c*kh*kw]  (already the K-major operand),
//     B = the tile's im2col matrix, gathered from the input slice
//         [in_start, min(in_end, H)) with the sub-operator pads pt', pb'
//         (tiling tutorial, "H/W 维切分的通用公式"),
//     C = y[n][c_out][o0:o1][:], row pitch OH*OW.
#pragma once

#include <cstdint>

#include "gemm_sm103a.cuh"
#include "tiles_internal.h"

namespace tiles {

// Rows of one output H-tile as the kernel consumes them (computed on the
// host by htile_rows).
struct ConvHTile {
    int32_t o0;         // first output row
    int16_t rows;       // o1 - o0
    int16_t pt;         // top pad of the sub-operator, pt'
    int32_t in_start;   // first input row of the slice
    int32_t real_rows;  // min(in_end, H) - in_start: rows of the slice inside the image
};
static_assert(sizeof(ConvHTile) == 16, "H-tile record");

// Columns of one output W-tile: the same slicing formulas as the rows
// (computed on the host by htile_rows with the width's sizes).
struct ConvWTile {
    int32_t o0;         // first output column
    int16_t cols;       // q1 - q0
    int16_t pl;         // left pad of the sub-operator, pl'
    int32_t in_start;   // first input column of the slice
    int32_t unused;
};
static_assert(sizeof(ConvWTile) == 16, "W-tile record");

// H-tiles and W-tiles handled by one launch (the tables travel in the
// kernel parameters).
constexpr int kConvMaxHTiles = 128;
constexpr int kConvMaxWTiles = 64;
// Threads of the convolution block: the GEMM's six warps plus four warps
// that gather the im2col operand.
constexpr int kConvThreads = 320;
constexpr int kConvGatherThreads = 128;

// Geometry of the TMA convolution (conv_tma_sm103a.cu).
struct ConvTmaGeometry {
    int owc, nr, bn;              // tile: nr output rows x owc columns (MMA M = 128),
                                  // bn output channels (MMA N)
    int ch_blocks, cp;            // 64-channel blocks, channels padded to them
    int64_t weights_bytes, x_bytes;
    int64_t weights_offset, x_offset, ws_bytes;   // workspace layout
};

// tile_ow: output columns per W-tile (the full width when >= ow).
bool conv_tma_geometry(const tiles_conv_desc* d, int64_t oh, int64_t ow, int tile_oh, int tile_ow,
                       ConvTmaGeometry* g);
// cfg (may be NULL): conv_weights picks the filter's place, acc_bufs the
// TMEM accumulator count of the weights-in-TMEM form (0 = planned).
// tile_ow >= 1 and tile_n >= 1 (W-tile width, images per launch group).
int conv2d_tma(const tiles_conv_desc* d, const tiles_config* cfg, int tile_oh, int tile_ow,
               int tile_n, int64_t oh, int64_t ow, const ConvTmaGeometry& g, void* ws,
               size_t ws_bytes, void* stream);
int64_t conv_workspace_bytes(const tiles_conv_desc* d, int tile_oh);

struct ConvArgs {
    const void* x;
    void* y;
    int32_t n, c, h, w, c_out, kh, kw, sh, sw, pw, dh, dw;
    int32_t oh, ow;
    int32_t k;                  // c * kh * kw
    int32_t n_htiles;           // H-tiles in this launch
    int32_t m_blocks, n_blocks, k_blocks;
    int32_t tiles;              // n * n_htiles * m_blocks * n_blocks
    int32_t out_dtype;
    uint32_t idesc;
    int32_t vec_ok;             // 16-byte vector stores are aligned for every tile
    int32_t* err;
    uint64_t wait_limit_ns;
    ConvHTile ht[kConvMaxHTiles];
};

}  // namespace tiles
