// Internal declarations shared by the planner, the C ABI and the kernels.
#pragma once

#include <cstdint>
#include <vector>

#include "../../include/tiles.h"

namespace tiles {

// Threads of the warp-specialised GEMM block: warp 0 TMA producer, warp 1
// MMA issuer and TMEM owner, warps 2-5 epilogue.
constexpr int kGemmThreads = 192;
// Registers per thread of the GEMM kernels in the GB300 preset (the
// device model used without a GPU).  On a GPU, tiles_device_query replaces
// it with the largest register count the runtime reports for a compiled
// variant, rounded up to the per-warp allocation granule.
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
// GB300 preset values of the time model's K-split hand-off (the device
// record's handoff_clocks and partial_bytes_per_clk): fixed clocks of one
// hand-off (flag release, acquire, copy latency), and the bytes per clock
// per SM at which a K part writes or reads its fp32 partial tile.  The rate
// was measured on the 4096^3 GEMM after an L2-flushing write: a CTA's
// 128 KB partial took ~5,300 clocks out (~25 B/clk) whether written as
// 4-byte or 16-byte lane stores.
constexpr int64_t kTailHandoffClocks = 2048;
constexpr int64_t kPartialBytesPerClk = 32;
// GB300 preset of the extra fixed clocks of a CTA-pair launch over a one-CTA
// launch (the device record's pair_launch_clocks): the cluster launch, the
// pair's prologue and its last epilogue.  Measured on 512^3 GEMMs, where
// both run 8 fill-bound K blocks per unit: the 256x256 pair took 11.1 us
// against 8.6 us for 128x128 tiles, the 256x128 pair 10.9 us against 8.7 us
// for 128x64, about 2.3 us, ~4,500 clocks at the 1.93 GHz of those runs.
constexpr int64_t kPairLaunchClocks = 4500;
constexpr int kMaxTailParts = 8;
void device_preset_h100(tiles_device* d);
void device_preset_gb300(tiles_device* d);
int htile_rows(int H, int kh, int sh, int pt, int d, int o0, int o1, tiles_htile* t);
int conv2d_tiled(const tiles_conv_desc* desc, int tile_oh, int tile_ow, int tile_n,
                 const tiles_config* cfg, void* ws, size_t ws_bytes, void* stream);
int conv2d_htiled(const tiles_conv_desc* desc, int tile_oh, const tiles_config* cfg, void* ws,
                  size_t ws_bytes, void* stream);
// Output height and width of a convolution descriptor (INVALID_ARG when a
// size is out of range or no window fits).
int conv_out_hw(const tiles_conv_desc* d, int64_t* oh, int64_t* ow);

// Smallest workspace a kernel call accepts: the 256-byte header whose first
// word records a bounded wait's expiry (tiles_workspace_bytes).
constexpr int kConvMinWorkspaceBytes = 256;

// A fault planted for the bounded-wait tests (tiles_selftest_drop_stage):
// the first CTA (group) of the next GEMM or convolution launch from this
// thread skips the loads and the arrival of its `stage`-th pipeline stage,
// and every wait of that launch gives up after limit_ns.  stage < 0: none.
struct PlantedFault { int32_t stage; uint64_t limit_ns; };
// Takes the calling thread's armed fault, leaving none armed.
PlantedFault take_planted_fault();

// Per-thread error text (tiles_last_error).
int fail(int status, const char* fmt, ...);

}  // namespace tiles
