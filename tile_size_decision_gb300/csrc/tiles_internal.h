// Internal declarations shared by the planner, the C ABI and the kernels.
#pragma once

#include <cstdint>
#include <vector>

#include "../../include/tiles.h"

namespace tiles {

// Threads of the warp-specialised GEMM block: warp 0 TMA producer, warp 1
// MMA issuer and TMEM owner, warps 2-5 epilogue.
constexpr int kGemmThreads = 192;
// Registers per thread of the GEMM kernels as built (ptxas reports up to
// 164, which the per-warp granule of 256 rounds to 168); the planner's
// occupancy uses this figure.
constexpr int kGemmRegsPerThread = 168;
// Shared memory beyond the operand stages: mbarriers, the TMEM address slot,
// an abort flag (kSmemBarrierBytes) and the slack that lets the operand
// tiles start on a 1024-byte boundary, as the 128-byte swizzle requires.
constexpr int kSmemBarrierBytes = 256;
constexpr int kSmemAlignSlack = 1024;
// The epilogue's staging boxes: one 32-row x 128-byte box per epilogue warp,
// from which TMA stores copy the output tile to C.
constexpr int kSmemEpilogueBytes = 4 * 32 * 128;
constexpr int kMaxStages = 8;
// Default L2 -> shared-memory fill rate per SM per clock used by the GB300
// time model (bytes).  A model parameter calibrated on the 128x256 one-CTA
// kernel at 4096^3, whose TMA loads averaged 58 B/clk/SM over the launch
// (ncu: 1.61 GB in 96.9 us at 1.877 GHz on 152 SMs).
constexpr int kDefaultFillBytesPerClk = 64;

// A compiled kernel variant: tile rows and columns, SMs per MMA, and the
// pipeline depth it was built with.
struct KernelVariant { int bm, bn, cta_group, stages; };
extern const KernelVariant kGemmVariants[];
extern const int kNumGemmVariants;

int evaluate(const tiles_device& dev, const tiles_config& cfg, int elem_bytes, int accum_bytes,
             tiles_verdict* v);
void finish_parallelism(const tiles_device& dev, int64_t b, int64_t m, int64_t n,
                        tiles_verdict* v);
double c0_bytes(int64_t b, int64_t m, int64_t n, int64_t k, int bm, int bn, int in_bytes,
                int out_bytes);
int plan(const tiles_device& dev, const tiles_problem& p, std::vector<tiles_verdict>* out);
int64_t gb300_smem_bytes(const tiles_config& cfg, int in_bytes, int64_t* per_stage);
int64_t gb300_est_clocks(const tiles_device& dev, tiles_verdict* v, int64_t k);
// Whether the last round of `tiles` over `resident` CTA groups runs as
// N-half tiles (it would otherwise fill at most half of the groups).
bool tail_split_applies(int bn, int cta_group, int64_t tiles, int64_t resident);
int64_t gb300_resident_groups(const tiles_device& dev, const tiles_verdict& v);
// Clocks per K block of one tile (max of MMA and operand fill) and of
// reading back one partial tile per CTA.
int64_t gb300_unit_clocks(const tiles_device& dev, const tiles_config& cfg, int64_t smem_per_stage);
int64_t gb300_reduce_clocks(const tiles_device& dev, const tiles_config& cfg);
// Schedule of a last round that leaves resident groups idle: the cheapest
// (or the forced) of whole tiles (K blocks * unit), N-halves (K blocks *
// half-tile unit) and K parts s in 2 .. min(resident / rest, kMaxTailParts,
// K blocks) (ceil(K blocks / s) * unit + (s - 1) * reduce).
struct TailChoice { int mode; int parts; int64_t clocks; };
TailChoice gb300_tail_choice(const tiles_device& dev, const tiles_config& cfg, int64_t tiles,
                             int64_t resident, int64_t k_blocks, int in_bytes, int forced);
// Fixed clocks of a K-part hand-off (flag release, acquire, copy latency).
constexpr int64_t kTailHandoffClocks = 2048;
// Bytes per clock per SM at which a K part writes or reads its fp32
// partial tile.  Measured on the 4096^3 GEMM after an L2-flushing write:
// a CTA's 128 KB partial took ~5,300 clocks out (~25 B/clk) whether written
// as 4-byte or 16-byte lane stores.
constexpr int64_t kPartialBytesPerClk = 32;
constexpr int kMaxTailParts = 8;
void device_preset_h100(tiles_device* d);
void device_preset_gb300(tiles_device* d);
int htile_rows(int H, int kh, int sh, int pt, int d, int o0, int o1, tiles_htile* t);
int conv2d_tiled(const tiles_conv_desc* desc, int tile_oh, int tile_ow, int tile_n,
                 const tiles_config* cfg, void* ws, size_t ws_bytes, void* stream);
int conv2d_htiled(const tiles_conv_desc* desc, int tile_oh, const tiles_config* cfg, void* ws,
                  size_t ws_bytes, void* stream);

// Per-thread error text (tiles_last_error).
int fail(int status, const char* fmt, ...);

}  // namespace tiles
