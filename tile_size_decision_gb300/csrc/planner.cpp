// Tile-size planner: constraints C0-C4, the sweep and the H-tile rows.
//
// The constraints are those of the page "04-tile-size-decision" (README,
// "目的" and the four checks it names; the script tile_decision.py fixes the
// numbers): C3 the MMA instruction shape, C1 on-chip capacity, C2 register
// pressure, the resident blocks they leave, C4 waves and last-wave fill, C0
// cache-less DRAM traffic.  Page mode reproduces the page's sweep and ranking
// bit for bit.  GB300 mode applies the same constraints to the sm_103a
// kernels of this library: C3 becomes the tcgen05 kind::f16 shape and the
// kernels' tile layout, C2 becomes the tensor-memory (TMEM) column budget of
// the accumulators, C4 counts rounds of persistent CTA groups, and the
// ranking puts a wave-quantised time estimate before C0.
//
// Host-only C++; no CUDA here.

#include "tiles_internal.h"

#include <algorithm>
#include <cfenv>
#include <climits>
#include <cmath>
#include <cstring>
#include <vector>

namespace tiles {

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The page's instruction-shape table: an MMA family fixes the multiples of
// the tile's M, N and K edges and of the block's thread count (mma
// m16n8k16 is issued per warp, wgmma m64nNk16 per warpgroup, scalar code
// per thread).
struct ShapeRule { int edge[3]; int threads; };

bool shape_rule(int instr, ShapeRule* out) {
    switch (instr) {
        case TILES_INSTR_MMA:   *out = {{16, 8, 16}, 32}; return true;
        case TILES_INSTR_WGMMA: *out = {{64, 8, 16}, 128}; return true;
        case TILES_INSTR_SIMT:  *out = {{1, 1, 1}, 32}; return true;
        default: return false;
    }
}

// Residency: for every per-SM resource, how many blocks of this demand the
// SM can hold; the scarcest resource binds.  The list order settles ties
// (registers, shared memory, threads, then tensor memory in GB300 mode), and
// the SM's block limit caps the count without ever being named as binding.
void settle_residency(const tiles_device& dev, tiles_verdict* v, bool tensor_memory) {
    struct Resource { int32_t* blocks; int64_t supply, demand; int32_t tag; };
    const Resource table[] = {
        {&v->blocks_by_regs, dev.regs_per_sm, v->regs_per_block, TILES_BIND_REGS},
        {&v->blocks_by_smem, dev.smem_per_sm, v->smem_total, TILES_BIND_SMEM},
        {&v->blocks_by_threads, dev.max_threads_per_sm, v->cfg.threads, TILES_BIND_THREADS},
        {&v->blocks_by_tmem, dev.tmem_cols, v->tmem_cols_alloc, TILES_BIND_TMEM},
    };
    const int used = tensor_memory ? 4 : 3;
    int64_t scarcest = INT64_MAX;
    int32_t tag = TILES_BIND_NONE;
    for (int i = 0; i < used; ++i) {
        const int64_t fit = table[i].supply / std::max<int64_t>(table[i].demand, 1);
        *table[i].blocks = static_cast<int32_t>(fit);
        if (fit < scarcest) { scarcest = fit; tag = table[i].tag; }
    }
    v->blocks_per_sm = static_cast<int32_t>(
        std::max<int64_t>(std::min<int64_t>(scarcest, dev.max_blocks_per_sm), 0));
    if (v->blocks_per_sm == 0) {
        v->failures |= TILES_FAIL_OCC;
        v->binding = TILES_BIND_NONE;
    } else {
        v->binding = tag;
    }
}

// Page mode, one configuration of the MMA family whose shape rule is `rule`.
void evaluate_page(const tiles_device& dev, const tiles_config& cfg, const ShapeRule& rule,
                   int elem_bytes, int accum_bytes, tiles_verdict* v) {
    // C3: each tile edge and the thread count is a whole multiple of the
    // family's shape, and the block stays within the per-block thread limit;
    // every broken condition counts once.
    const int edges[3] = {cfg.bm, cfg.bn, cfg.bk};
    int broken = cfg.threads % rule.threads != 0;
    for (int i = 0; i < 3; ++i) broken += edges[i] % rule.edge[i] != 0;
    broken += cfg.threads > dev.max_threads_per_block;
    v->c3_violations = broken;
    if (broken) v->failures |= TILES_FAIL_C3;
    // C1: a stage holds the A slice (bm x bk) and the B slice (bk x bn); the
    // pipeline holds `stages` of them, within one block's shared memory.
    v->smem_per_stage = (int64_t)(cfg.bm + cfg.bn) * cfg.bk * elem_bytes;
    v->smem_total = v->smem_per_stage * cfg.stages;
    if (v->smem_total > dev.smem_per_block_max) v->failures |= TILES_FAIL_C1;
    // C2: the bm x bn accumulator tile spread over the block's threads, in
    // 32-bit registers; a warp's registers come in whole allocation granules.
    v->accum_per_thread = (int32_t)ceil_div((int64_t)cfg.bm * cfg.bn, cfg.threads);
    const int64_t lane_words = (int64_t)v->accum_per_thread * accum_bytes / 4;
    const int64_t granules = ceil_div(lane_words * dev.warp_size, dev.reg_granularity_per_warp);
    v->regs_per_thread = (int32_t)(granules * dev.reg_granularity_per_warp / dev.warp_size);
    if (v->regs_per_thread > dev.regs_per_thread_max) v->failures |= TILES_FAIL_C2;
    v->regs_per_block = v->regs_per_thread * cfg.threads;
    settle_residency(dev, v, false);
}

}  // namespace

// GB300 kernel variants compiled into this library (bm, bn, cta_group,
// stages), in enumeration order.  bk is one 128-byte swizzle atom of the
// input type; the stage count is the deepest pipeline that fits 227 KB next
// to the epilogue's staging boxes (at most kMaxStages).
const KernelVariant kGemmVariants[] = {
    {128, 64, 1, 8}, {128, 128, 1, 6}, {128, 192, 1, 5}, {128, 256, 1, 4},
    {256, 128, 2, 8}, {256, 256, 2, 6},
};
const int kNumGemmVariants = sizeof(kGemmVariants) / sizeof(kGemmVariants[0]);

int64_t gb300_smem_bytes(const tiles_config& cfg, int in_bytes, int64_t* per_stage) {
    const int cg = std::max(cfg.cta_group, 1);
    // Each CTA of a group stages its own bm/cg rows of A and bn/cg columns of B.
    int64_t stage = (int64_t)(cfg.bm / cg + cfg.bn / cg) * cfg.bk * in_bytes;
    if (per_stage) *per_stage = stage;
    return stage * cfg.stages + kSmemEpilogueBytes + kSmemBarrierBytes + kSmemAlignSlack;
}

static int pow2_at_least(int x) {
    int p = 32;
    while (p < x) p <<= 1;
    return p;
}

void evaluate_gb300(const tiles_device& dev, const tiles_config& cfg, int in_bytes,
                    tiles_verdict* v) {
    const int cg = cfg.cta_group;
    const bool cg_ok = cg == 1 || cg == 2;
    const int cgs = cg_ok ? cg : 1;
    // C3: tcgen05.mma kind::f16 takes M = 128 rows per CTA (cta_group::1:
    // M 128; ::2: M 256 over the pair), N a multiple of 16 in [16, 256], K 16
    // per instruction.  The kernels add their tile layout: a K block is one
    // 128-byte swizzle atom, B arrives in 64-column atoms per CTA, threads
    // are the 6 warps of the warp-specialised block.
    const bool conditions[] = {
        cg_ok,
        cfg.bm == 128 * cgs,
        cfg.bn % 16 == 0 && cfg.bn >= 16 && cfg.bn <= 256,
        cfg.bk % 16 == 0 && cfg.bk * in_bytes == 128,
        (cfg.bn / cgs) % 64 == 0,
        cfg.threads == kGemmThreads,
        cfg.acc_bufs >= 1 && cfg.acc_bufs <= 2,
        cfg.stages >= 1 && cfg.stages <= kMaxStages,
    };
    int broken = 0;
    for (bool ok : conditions) broken += !ok;
    v->c3_violations = broken;
    if (broken) v->failures |= TILES_FAIL_C3;
    // C1: pipeline stages plus the epilogue's staging boxes, the barriers
    // and the 1 KB alignment slack of the swizzled operand tiles, within the
    // opt-in per-block limit.
    tiles_config c = cfg;
    c.cta_group = cgs;
    v->smem_total = gb300_smem_bytes(c, in_bytes, &v->smem_per_stage);
    if (v->smem_total > dev.smem_per_block_max) v->failures |= TILES_FAIL_C1;
    // C2: the fp32 accumulators live in TMEM, 128 lanes x bn columns per
    // buffer per CTA; the allocation is a power of two of at least 32.
    const int cols = std::max(cfg.acc_bufs, 0) * cfg.bn;
    v->tmem_cols_alloc = pow2_at_least(std::max(cols, 1));
    if (v->tmem_cols_alloc > dev.tmem_cols) v->failures |= TILES_FAIL_C2;
    // The kernels' own register figure (not an accumulator count).
    v->accum_per_thread = 0;
    v->regs_per_thread = dev.kernel_regs_per_thread;
    v->regs_per_block = dev.kernel_regs_per_thread * cfg.threads;
    settle_residency(dev, v, true);
}

int evaluate(const tiles_device& dev, const tiles_config& cfg, int elem_bytes, int accum_bytes,
             tiles_verdict* v) {
    std::memset(v, 0, sizeof(*v));
    v->cfg = cfg;
    if (cfg.instr == TILES_INSTR_TCGEN05) {
        evaluate_gb300(dev, cfg, elem_bytes, v);
        return TILES_OK;
    }
    ShapeRule rule;
    if (!shape_rule(cfg.instr, &rule)) return TILES_ERR_INVALID_ARG;
    evaluate_page(dev, cfg, rule, elem_bytes, accum_bytes, v);
    return TILES_OK;
}

void finish_parallelism(const tiles_device& dev, int64_t b, int64_t m, int64_t n,
                        tiles_verdict* v) {
    const tiles_config& cfg = v->cfg;
    // C4: one block per output tile; the tiles run in waves of the blocks
    // resident at once (never fewer than one, even when none fits).
    v->grid = b * ceil_div(m, cfg.bm) * ceil_div(n, cfg.bn);
    const int64_t resident =
        cfg.instr == TILES_INSTR_TCGEN05
            ? gb300_resident_groups(dev, *v)
            : std::max<int64_t>((int64_t)v->blocks_per_sm * dev.sm_count, 1);
    v->waves = ceil_div(v->grid, resident);
    const int64_t last = v->grid % resident;
    v->last_wave_fill = last ? (double)last / (double)resident : 1.0;
    v->warnings = 0;
    if (v->waves > 1 && v->last_wave_fill < 0.5) v->warnings |= TILES_WARN_TAIL;
    if (v->grid < dev.sm_count) v->warnings |= TILES_WARN_IDLE;
}

double c0_bytes(int64_t b, int64_t m, int64_t n, int64_t k, int bm, int bn, int in_bytes,
                int out_bytes) {
    // Every tile streams a bm x K panel of A and a K x bn panel of B, so A is
    // read N/bn times and B M/bm times; C is written once.  The sum is
    // formed left to right in double, as the page writes it: the integer
    // product (exact in 128 bits, like Python's integers) converts once and
    // multiplies (1/bn + 1/bm); the output term adds.
    const __int128 operand = (__int128)in_bytes * b * m * n * k;
    const __int128 output = (__int128)out_bytes * b * m * n;
    return (double)operand * (1.0 / bn + 1.0 / bm) + (double)output;
}

// Round half to even, as Python's round() on a float.
static int64_t round_even(double x) {
    const int saved = std::fegetround();
    std::fesetround(FE_TONEAREST);
    double r = std::nearbyint(x);
    std::fesetround(saved);
    return (int64_t)r;
}

int64_t gb300_resident_groups(const tiles_device& dev, const tiles_verdict& v) {
    // Persistent CTA groups at once: blocks_per_sm per SM, or per CTA pair
    // (the device's count of co-resident 2-CTA clusters when known).
    const int cg = std::max(v.cfg.cta_group, 1);
    const int64_t slots = (cg == 2 && dev.cta_pairs > 0) ? dev.cta_pairs : dev.sm_count / cg;
    return std::max<int64_t>((int64_t)v.blocks_per_sm * slots, 1);
}

bool tail_split_applies(int bn, int cta_group, int64_t tiles, int64_t resident) {
    const int cg = std::max(cta_group, 1);
    if ((bn / 2) % cg || ((bn / 2) / cg) % 64) return false;   // a half must be whole B atoms
    if (resident < 1) return false;
    const int64_t rem = tiles % resident;
    return rem > 0 && 2 * rem <= resident;
}

int64_t gb300_unit_clocks(const tiles_device& dev, const tiles_config& cfg, int64_t smem_per_stage) {
    const int cg = std::max(cfg.cta_group, 1);
    const int64_t mma =
        (int64_t)(cfg.bm / cg) * cfg.bn * cfg.bk * 2 / std::max(dev.mma_flops_per_clk, 1);
    const int64_t fill = ceil_div(smem_per_stage, std::max(dev.fill_bytes_per_clk, 1));
    return std::max(mma, fill);
}

int64_t gb300_reduce_clocks(const tiles_device& dev, const tiles_config& cfg) {
    // One fp32 partial tile per CTA written by a leading part and read back
    // by the last part, plus the hand-off's fixed latency.  The partials
    // move at the device's partial rate, not at the operand fill rate: they
    // are written while every SM stores at once into an L2 full of dirty
    // lines.
    const int cg = std::max(cfg.cta_group, 1);
    return 2 * ceil_div((int64_t)(cfg.bm / cg) * cfg.bn * 4, std::max(dev.partial_bytes_per_clk, 1)) +
           dev.handoff_clocks;
}

TailChoice gb300_tail_choice(const tiles_device& dev, const tiles_config& cfg, int64_t tiles,
                             int64_t resident, int64_t k_blocks, int in_bytes, int forced) {
    TailChoice tc{TILES_TAIL_WHOLE, 0, 0};
    int64_t stage = 0;
    gb300_smem_bytes(cfg, in_bytes, &stage);
    const int64_t unit = gb300_unit_clocks(dev, cfg, stage);
    tc.clocks = k_blocks * unit;
    const int64_t rest = resident > 0 ? tiles % resident : 0;
    if (rest == 0) return tc;
    const int cg = std::max(cfg.cta_group, 1);
    // N-halves: each half loads all of A and half of B per K block.
    if ((forced == TILES_TAIL_AUTO || forced == TILES_TAIL_NHALF) &&
        tail_split_applies(cfg.bn, cg, tiles, resident)) {
        tiles_config h = cfg;
        h.bn = cfg.bn / 2;
        int64_t half_stage = 0;
        gb300_smem_bytes(h, in_bytes, &half_stage);
        const int64_t t = k_blocks * gb300_unit_clocks(dev, h, half_stage);
        if (forced == TILES_TAIL_NHALF || t < tc.clocks) tc = TailChoice{TILES_TAIL_NHALF, 0, t};
    }
    // K parts: each part runs ceil(K blocks / s) K blocks; the last reads
    // back s - 1 partial tiles.
    if (forced == TILES_TAIL_AUTO || forced == TILES_TAIL_KSPLIT) {
        const int64_t smax = std::min<int64_t>(std::min<int64_t>(resident / rest, kMaxTailParts),
                                               k_blocks);
        const int64_t reduce = gb300_reduce_clocks(dev, cfg);
        bool first = forced == TILES_TAIL_KSPLIT;
        for (int64_t s = 2; s <= smax; ++s) {
            const int64_t t = ceil_div(k_blocks, s) * unit + (s - 1) * reduce;
            if (first || t < tc.clocks) { tc = TailChoice{TILES_TAIL_KSPLIT, (int)s, t}; first = false; }
        }
    }
    return tc;
}

int64_t gb300_est_clocks(const tiles_device& dev, tiles_verdict* v, int64_t k) {
    const tiles_config& cfg = v->cfg;
    const int64_t kblocks = ceil_div(k, cfg.bk);
    int64_t stage = 0;
    gb300_smem_bytes(cfg, 2, &stage);
    const int64_t unit = gb300_unit_clocks(dev, cfg, stage);
    const int64_t resident = gb300_resident_groups(dev, *v);
    const int64_t rest = v->grid % resident;
    const TailChoice tc = gb300_tail_choice(dev, cfg, v->grid, resident, kblocks, 2, TILES_TAIL_AUTO);
    v->tail_split = tc.mode == TILES_TAIL_KSPLIT ? tc.parts : tc.mode == TILES_TAIL_NHALF ? -1 : 0;
    const int64_t launch = cfg.cta_group == 2 ? dev.pair_launch_clocks : 0;
    return (v->grid / resident) * kblocks * unit + (rest ? tc.clocks : 0) + launch;
}

static int bytes_of(int dtype) {
    switch (dtype) {
        case TILES_F16: case TILES_BF16: return 2;
        case TILES_F32: return 4;
        default: return 0;
    }
}

namespace {

// A feasible verdict with its rank key: the rounded C0 and its place in the
// enumeration (ties keep that order).
struct Ranked { tiles_verdict v; int64_t c0r; };

// Page mode: the candidate grid of the page's sweep (bm, bn over 16..256,
// bk over 16..128 but not beyond K, 2-4 stages, 128/256/512 threads, the
// innermost varying fastest), feasible ones only.
void sweep_page(const tiles_device& dev, const tiles_problem& p, int in_b, int out_b,
                const ShapeRule& rule, std::vector<Ranked>* kept) {
    static const int kEdges[] = {16, 32, 64, 128, 256};
    static const int kDepths[] = {16, 32, 64, 128};
    static const int kStages[] = {2, 3, 4};
    static const int kThreads[] = {128, 256, 512};
    for (int bm : kEdges) for (int bn : kEdges) for (int bk : kDepths) {
        if (bk > p.k) continue;
        for (int st : kStages) for (int th : kThreads) {
            if (th % rule.threads) continue;
            tiles_config c{};
            c.bm = bm; c.bn = bn; c.bk = bk; c.stages = st; c.threads = th; c.instr = p.instr;
            tiles_verdict v;
            evaluate(dev, c, in_b, 4, &v);
            if (v.failures) continue;
            finish_parallelism(dev, p.b, p.m, p.n, &v);
            v.c0_bytes = c0_bytes(p.b, p.m, p.n, p.k, bm, bn, in_b, out_b);
            kept->push_back({v, round_even(v.c0_bytes)});
        }
    }
}

// GB300 mode: the compiled kernel variants, feasible ones only.
void sweep_gb300(const tiles_device& dev, const tiles_problem& p, int in_b, int out_b,
                 std::vector<Ranked>* kept) {
    for (int i = 0; i < kNumGemmVariants; ++i) {
        const KernelVariant& kv = kGemmVariants[i];
        tiles_config c{};
        c.bm = kv.bm; c.bn = kv.bn; c.bk = 128 / in_b; c.threads = kGemmThreads;
        c.instr = TILES_INSTR_TCGEN05; c.acc_bufs = 2; c.cta_group = kv.cta_group;
        c.stages = kv.stages;
        tiles_verdict v;
        evaluate(dev, c, in_b, 4, &v);
        if (v.failures) continue;
        finish_parallelism(dev, p.b, p.m, p.n, &v);
        v.c0_bytes = c0_bytes(p.b, p.m, p.n, p.k, c.bm, c.bn, in_b, out_b);
        v.est_clocks = gb300_est_clocks(dev, &v, p.k);
        kept->push_back({v, round_even(v.c0_bytes)});
    }
}

}  // namespace

int plan(const tiles_device& dev, const tiles_problem& p, std::vector<tiles_verdict>* out) {
    const int in_b = bytes_of(p.in_dtype), out_b = bytes_of(p.out_dtype);
    if (!in_b || !out_b) return TILES_ERR_UNSUPPORTED_DTYPE;
    std::vector<Ranked> kept;
    // The page's design order: least traffic first, then more resident
    // blocks, then less shared memory.  GB300 mode puts the time estimate
    // in front.
    auto traffic_first = [](const Ranked& a, const Ranked& b) {
        if (a.c0r != b.c0r) return a.c0r < b.c0r;
        if (a.v.blocks_per_sm != b.v.blocks_per_sm) return a.v.blocks_per_sm > b.v.blocks_per_sm;
        return a.v.smem_total < b.v.smem_total;
    };
    if (p.mode == TILES_MODE_PAGES) {
        ShapeRule rule;
        if (!shape_rule(p.instr, &rule)) return TILES_ERR_INVALID_ARG;
        sweep_page(dev, p, in_b, out_b, rule, &kept);
        std::stable_sort(kept.begin(), kept.end(), traffic_first);
    } else if (p.mode == TILES_MODE_GB300) {
        if (in_b != 2) return TILES_ERR_UNSUPPORTED_DTYPE;
        sweep_gb300(dev, p, in_b, out_b, &kept);
        std::stable_sort(kept.begin(), kept.end(), [&](const Ranked& a, const Ranked& b) {
            if (a.v.est_clocks != b.v.est_clocks) return a.v.est_clocks < b.v.est_clocks;
            return traffic_first(a, b);
        });
    } else {
        return TILES_ERR_INVALID_ARG;
    }
    out->clear();
    for (auto& r : kept) out->push_back(r.v);
    return TILES_OK;
}

void device_preset_h100(tiles_device* d) {
    std::memset(d, 0, sizeof(*d));
    d->smem_per_sm = 228 * 1024;
    d->smem_per_block_max = 227 * 1024;
    d->regs_per_sm = 65536;
    d->max_threads_per_sm = 2048;
    d->max_threads_per_block = 1024;
    d->max_blocks_per_sm = 32;
    d->regs_per_thread_max = 255;
    d->reg_granularity_per_warp = 256;
    d->warp_size = 32;
    d->sm_count = 132;
}

void device_preset_gb300(tiles_device* d) {
    device_preset_h100(d);
    d->sm_count = 148;
    d->tmem_cols = 512;
    d->mma_flops_per_clk = 8192;
    d->fill_bytes_per_clk = kDefaultFillBytesPerClk;
    d->kernel_regs_per_thread = kGemmRegsPerThread;
    d->partial_bytes_per_clk = kPartialBytesPerClk;
    d->handoff_clocks = kTailHandoffClocks;
    d->pair_launch_clocks = kPairLaunchClocks;
}

int htile_rows(int H, int kh, int sh, int pt, int d, int o0, int o1, tiles_htile* t) {
    if (H <= 0 || kh <= 0 || sh <= 0 || d <= 0 || pt < 0 || o0 < 0 || o1 <= o0)
        return TILES_ERR_INVALID_ARG;
    t->in_start = std::max(0, o0 * sh - pt);
    t->in_end = (o1 - 1) * sh - pt + (kh - 1) * d + 1;
    t->in_span = t->in_end - t->in_start;
    t->pt = std::max(0, pt - o0 * sh);
    t->pb = std::max(0, t->in_end - H);
    t->halo = (kh - 1) * d + 1 - sh;
    return TILES_OK;
}

}  // namespace tiles
