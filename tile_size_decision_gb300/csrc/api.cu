// C ABI of libtiles (declarations and contracts in include/tiles.h).
//
// Host side of the kernels: argument validation, the memoised GB300 plan,
// TMA tensor-map encoding (through the runtime's driver entry point, so the
// library loads without a GPU) and the launch on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "conv_sm103a.cuh"
#include "gemm_sm103a.cuh"
#include "tiles_internal.h"

namespace tiles {

namespace {

thread_local std::string g_last_error;

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;   // 2 s per wait
// Grouped tile order: A panels of up to kTileGroupBytes (a third of the
// 129 MB L2) keep plain M-fastest order; beyond it tiles go in groups of
// kTileGroupM M blocks (8 + 76/8 panels in flight for 76 CTA pairs).
constexpr int64_t kTileGroupBytes = 43ll << 20;
constexpr int32_t kTileGroupM = 8;
constexpr size_t kWorkspaceBytes = 256;
static_assert(kWorkspaceBytes == static_cast<size_t>(kConvMinWorkspaceBytes),
              "one workspace minimum for every kernel call");

int bytes_of(int dtype) {
    switch (dtype) {
        case TILES_F16: case TILES_BF16: return 2;
        case TILES_F32: return 4;
        default: return 0;
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The tensor map through which the GEMM epilogue's TMA stores write C: a
// row-major [batch][m][n] array of the output type with row pitch `ldc` and
// item pitch `sc` (elements), box {128 bytes of columns, 32 rows, 1}, the
// 128-byte swizzle of the staging boxes.  False when C cannot take TMA
// stores (base or pitches not 16-byte multiples, or the encoder refuses);
// the epilogue then writes C from registers.
bool encode_c_store(CUtensorMap* map, int dtype, void* base, uint64_t n, uint64_t m,
                    uint64_t batch, uint64_t ldc, uint64_t sc) {
    auto fn = encode_fn();
    const uint64_t eb = dtype == TILES_F32 ? 4 : 2;
    if (!fn || !aligned16(base) || (ldc * eb) % 16 != 0 || (sc * eb) % 16 != 0) return false;
    const CUtensorMapDataType t = dtype == TILES_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                  : dtype == TILES_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[3] = {n, m, batch};
    cuuint64_t strides[2] = {ldc * eb, sc * eb};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / eb), 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, t, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 3-D tensor map over a row-major [d2][d1][d0] array of 16-bit elements
// with row pitch `pitch1` and item pitch `pitch2` (elements), box
// {box0, box1, 1}, 128-byte swizzle, zero fill out of range.
int encode_3d(CUtensorMap* map, int dtype, const void* base, uint64_t d0, uint64_t d1,
              uint64_t d2, uint64_t pitch1, uint64_t pitch2, uint32_t box0, uint32_t box1) {
    auto fn = encode_fn();
    if (!fn) return fail(TILES_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (no CUDA driver?)");
    const CUtensorMapDataType t =
        dtype == TILES_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {pitch1 * 2, pitch2 * 2};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, t, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TILES_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return TILES_OK;
}

struct DeviceInfo { int ordinal; tiles_device dev; };

int current_device(tiles_device* dev, int* ordinal) {
    static std::mutex mu;
    static std::map<int, tiles_device> cache;
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(d);
    if (it == cache.end()) {
        tiles_device q;
        int s = tiles_device_query(d, &q);
        if (s != TILES_OK) return s;
        it = cache.emplace(d, q).first;
    }
    *dev = it->second;
    if (ordinal) *ordinal = d;
    return TILES_OK;
}

using PlanKey = std::tuple<int, int64_t, int64_t, int64_t, int64_t, int, int>;

int planned_config(const tiles_device& dev, int ordinal, int64_t b, int64_t m, int64_t n,
                   int64_t k, int in_dtype, int out_dtype, tiles_config* cfg) {
    static std::mutex mu;
    static std::map<PlanKey, tiles_config> cache;
    PlanKey key{ordinal, b, m, n, k, in_dtype, out_dtype};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) { *cfg = it->second; return TILES_OK; }
    }
    tiles_problem p{};
    p.b = b; p.m = m; p.n = n; p.k = k;
    p.in_dtype = in_dtype; p.out_dtype = out_dtype;
    p.instr = TILES_INSTR_TCGEN05; p.mode = TILES_MODE_GB300;
    std::vector<tiles_verdict> ranked;
    int s = plan(dev, p, &ranked);
    if (s != TILES_OK) return s;
    if (ranked.empty()) return fail(TILES_ERR_INFEASIBLE, "no GB300 configuration passes C1-C4");
    *cfg = ranked.front().cfg;
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = *cfg;
    return TILES_OK;
}

// A given configuration must be one of the compiled variants and pass C1-C4
// on this device.
int check_config(const tiles_device& dev, const tiles_config& cfg, int in_bytes) {
    bool compiled = false;
    for (int i = 0; i < kNumGemmVariants; ++i) {
        const KernelVariant& kv = kGemmVariants[i];
        if (kv.bm == cfg.bm && kv.bn == cfg.bn && kv.cta_group == cfg.cta_group &&
            kv.stages == cfg.stages)
            compiled = true;
    }
    tiles_verdict v;
    evaluate(dev, cfg, in_bytes, 4, &v);
    if (v.failures)
        return fail(TILES_ERR_INFEASIBLE, "configuration %dx%dx%d/%d fails constraints (bits 0x%x)",
                    cfg.bm, cfg.bn, cfg.bk, cfg.stages, v.failures);
    if (!compiled || cfg.instr != TILES_INSTR_TCGEN05 || cfg.acc_bufs != 2)
        return fail(TILES_ERR_INFEASIBLE, "configuration %dx%dx%d/%d is not a compiled variant",
                    cfg.bm, cfg.bn, cfg.bk, cfg.stages);
    return TILES_OK;
}

// Persistent CTA groups that fit at once for a compiled variant (cached per
// device and variant).
int max_groups(int ordinal, int bn, int cg, int sm_count) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_tuple(ordinal, bn, cg);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int g = sm_count / cg;
    if (cg == 2 && bn == 256) g = gemm_variant_max_groups<256, 2>(sm_count);
    if (cg == 2 && bn == 128) g = gemm_variant_max_groups<128, 2>(sm_count);
    cache[key] = g;
    return g;
}

int variant_attributes(int bn, int cg, int sm_count, VariantAttributes* out) {
    if (cg == 1) {
        switch (bn) {
            case 64: return gemm_variant_attributes<64, 1>(sm_count, out);
            case 128: return gemm_variant_attributes<128, 1>(sm_count, out);
            case 192: return gemm_variant_attributes<192, 1>(sm_count, out);
            case 256: return gemm_variant_attributes<256, 1>(sm_count, out);
            default: break;
        }
    } else if (cg == 2) {
        switch (bn) {
            case 128: return gemm_variant_attributes<128, 2>(sm_count, out);
            case 256: return gemm_variant_attributes<256, 2>(sm_count, out);
            default: break;
        }
    }
    return static_cast<int>(cudaErrorInvalidValue);
}

// The configuration of compiled variant i.
tiles_config variant_config(int i) {
    const KernelVariant& kv = kGemmVariants[i];
    tiles_config c{};
    c.bm = kv.bm; c.bn = kv.bn; c.bk = 64; c.stages = kv.stages; c.threads = kGemmThreads;
    c.instr = TILES_INSTR_TCGEN05; c.acc_bufs = 2; c.cta_group = kv.cta_group;
    return c;
}

int launch_variant(int bn, int cg, const CUtensorMap& ta, const CUtensorMap& tb,
                   const CUtensorMap& tc, const GemmArgs& args, int groups, cudaStream_t st) {
    if (cg == 1) {
        switch (bn) {
            case 64: return launch_gemm_variant<64, 1>(ta, tb, tc, args, groups, st);
            case 128: return launch_gemm_variant<128, 1>(ta, tb, tc, args, groups, st);
            case 192: return launch_gemm_variant<192, 1>(ta, tb, tc, args, groups, st);
            case 256: return launch_gemm_variant<256, 1>(ta, tb, tc, args, groups, st);
            default: break;
        }
    } else if (cg == 2) {
        switch (bn) {
            case 128: return launch_gemm_variant<128, 2>(ta, tb, tc, args, groups, st);
            case 256: return launch_gemm_variant<256, 2>(ta, tb, tc, args, groups, st);
            default: break;
        }
    }
    return static_cast<int>(cudaErrorInvalidValue);
}

// Tuned configurations: the winners of measured shortlists
// (tiles_gemm_autotune or a loaded file), keyed by the problem and the SM
// count, consulted before the planner when no configuration is given.
using TunedKey = std::tuple<int, int64_t, int64_t, int64_t, int64_t, int, int>;
struct TunedEntry { tiles_config cfg; float us; };
std::mutex g_tuned_mu;
std::map<TunedKey, TunedEntry> g_tuned;

bool tuned_config(const TunedKey& key, tiles_config* cfg) {
    std::lock_guard<std::mutex> lock(g_tuned_mu);
    auto it = g_tuned.find(key);
    if (it == g_tuned.end()) return false;
    *cfg = it->second.cfg;
    return true;
}

// Everything a GEMM launch decides before touching the GPU's queues:
// validated arguments, the configuration and the wave-aware schedule.
struct GemmPlan {
    tiles_device dev;
    int ordinal;
    tiles_config cfg;
    int64_t tiles, resident, full_units, units, groups;
    int tail_mode, ksplit;
    int64_t flags_offset, partials_offset, ws_needed;   // bytes, K-split layout
};

constexpr size_t kHeaderBytes = 256;

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// Workspace layout of a K-split tail: the 256-byte header (error word),
// the readiness flags, then the fp32 partial tiles.
void ksplit_layout(GemmPlan* gp, int64_t rest) {
    const int64_t flags = rest * gp->cfg.cta_group * (gp->ksplit - 1) * 4;
    gp->flags_offset = kHeaderBytes;
    gp->partials_offset = align256(gp->flags_offset + flags * 4);
    gp->ws_needed = gp->partials_offset +
                    rest * (gp->ksplit - 1) * (int64_t)gp->cfg.bm * gp->cfg.bn * 4;
}

int gemm_prepare(const tiles_gemm_desc* d, const tiles_config* user_cfg, bool batched,
                 size_t ws_bytes, GemmPlan* gp) {
    if (!d) return fail(TILES_ERR_INVALID_ARG, "null descriptor");
    if (!d->a || !d->b || !d->c) return fail(TILES_ERR_INVALID_ARG, "null matrix pointer");
    if (d->m < 1 || d->n < 1 || d->k < 1 || d->batch < 1)
        return fail(TILES_ERR_INVALID_ARG, "sizes must be >= 1 (m=%lld n=%lld k=%lld batch=%lld)",
                    (long long)d->m, (long long)d->n, (long long)d->k, (long long)d->batch);
    if (!batched && d->batch != 1)
        return fail(TILES_ERR_INVALID_ARG, "tiles_gemm takes batch == 1; use tiles_gemm_batched");
    if (d->m > INT32_MAX / 2 || d->n > INT32_MAX / 2 || d->k > INT32_MAX / 2 ||
        d->batch > INT32_MAX / 2)
        return fail(TILES_ERR_TOO_LARGE, "a size exceeds 2^30");
    if ((d->a_dtype != TILES_F16 && d->a_dtype != TILES_BF16) || d->b_dtype != d->a_dtype)
        return fail(TILES_ERR_UNSUPPORTED_DTYPE, "A and B must both be f16 or both bf16");
    const int cb = bytes_of(d->c_dtype);
    if (!cb) return fail(TILES_ERR_UNSUPPORTED_DTYPE, "C must be f32, f16 or bf16");
    if (d->lda < d->k || d->ldb < d->n || d->ldc < d->n)
        return fail(TILES_ERR_INVALID_ARG, "leading dimension smaller than the row length");
    if (d->lda % 8 || d->ldb % 8 || (d->ldc * cb) % 16)
        return fail(TILES_ERR_MISALIGNED, "row pitches must be multiples of 16 bytes");
    if (!aligned16(d->a) || !aligned16(d->b) || !aligned16(d->c))
        return fail(TILES_ERR_MISALIGNED, "matrix base pointers must be 16-byte aligned");
    if (batched && d->batch > 1) {
        if (d->stride_a % 8 || d->stride_b % 8 || (d->stride_c * cb) % 16)
            return fail(TILES_ERR_MISALIGNED, "batch strides must be multiples of 16 bytes");
        if (d->stride_a < d->m * d->lda || d->stride_b < d->k * d->ldb ||
            d->stride_c < d->m * d->ldc)
            return fail(TILES_ERR_INVALID_ARG, "batch strides overlap the items");
    }
    int s = current_device(&gp->dev, &gp->ordinal);
    if (s != TILES_OK) return s;
    // The configuration: the caller's, else a tuned one for this problem,
    // else the planner's first choice.  A tuned last-round schedule is a
    // preference: without the workspace for a K split it yields to the
    // planner's choice instead of failing.
    tiles_config tuned;
    const tiles_config* eff = user_cfg;
    if (user_cfg) {
        gp->cfg = *user_cfg;
        s = check_config(gp->dev, gp->cfg, 2);
        if (s != TILES_OK) return s;
    } else if (tuned_config(TunedKey{gp->dev.sm_count, d->batch, d->m, d->n, d->k, d->a_dtype,
                                     d->c_dtype}, &tuned) &&
               check_config(gp->dev, tuned, 2) == TILES_OK) {
        gp->cfg = tuned;
        eff = &tuned;
    } else {
        s = planned_config(gp->dev, gp->ordinal, d->batch, d->m, d->n, d->k, d->a_dtype,
                           d->c_dtype, &gp->cfg);
        if (s != TILES_OK) return s;
    }
    const tiles_config& cfg = gp->cfg;
    gp->tiles = d->batch * ((d->m + cfg.bm - 1) / cfg.bm) * ((d->n + cfg.bn - 1) / cfg.bn);
    if (gp->tiles > INT32_MAX / 2) return fail(TILES_ERR_TOO_LARGE, "too many output tiles");
    // Wave-aware schedule (C4): rounds of the resident groups.  A partial
    // last round runs as whole tiles, as N-halves (when it fills at most half
    // of the groups and the halves are whole B atoms) or split along K
    // (when the workspace holds the partial tiles): the cheapest under the
    // planner's time model (gb300_tail_choice), or the one the configuration
    // forces.
    gp->resident = max_groups(gp->ordinal, cfg.bn, cfg.cta_group, gp->dev.sm_count);
    gp->full_units = gp->units = gp->tiles;
    gp->tail_mode = kTailNone;
    gp->ksplit = 1;
    gp->flags_offset = gp->partials_offset = 0;
    gp->ws_needed = kHeaderBytes;
    const int64_t k_blocks = (d->k + cfg.bk - 1) / cfg.bk;
    const int64_t rest = gp->tiles % gp->resident;
    const int64_t full = gp->tiles - rest;
    int forced = eff ? eff->tail : TILES_TAIL_AUTO;
    if (forced < TILES_TAIL_AUTO || forced > TILES_TAIL_KSPLIT)
        return fail(TILES_ERR_INVALID_ARG, "unknown tail schedule %d", forced);
    TailChoice tc = gb300_tail_choice(gp->dev, cfg, gp->tiles, gp->resident, k_blocks, 2, forced);
    if (rest && tc.mode == TILES_TAIL_KSPLIT) {
        GemmPlan k = *gp;
        k.ksplit = tc.parts;
        ksplit_layout(&k, rest);
        if (static_cast<uint64_t>(ws_bytes) >= static_cast<uint64_t>(k.ws_needed)) {
            *gp = k;
            gp->tail_mode = kTailKSplit;
            gp->full_units = full;
            gp->units = full + rest * tc.parts;
        } else if (forced == TILES_TAIL_KSPLIT && user_cfg) {
            return fail(TILES_ERR_INVALID_ARG, "a K-split last round needs %lld workspace bytes",
                        (long long)k.ws_needed);
        } else {
            // Not enough workspace: the cheaper of whole tiles and N-halves.
            const TailChoice nh = gb300_tail_choice(gp->dev, cfg, gp->tiles, gp->resident,
                                                    k_blocks, 2, TILES_TAIL_NHALF);
            const TailChoice wh = gb300_tail_choice(gp->dev, cfg, gp->tiles, gp->resident,
                                                    k_blocks, 2, TILES_TAIL_WHOLE);
            tc = (nh.mode == TILES_TAIL_NHALF && nh.clocks < wh.clocks) ? nh : wh;
        }
    }
    if (rest && gp->tail_mode == kTailNone && tc.mode == TILES_TAIL_NHALF) {
        if (!tail_split_applies(cfg.bn, cfg.cta_group, gp->tiles, gp->resident))
            return fail(TILES_ERR_INVALID_ARG, "this tile cannot split into N-halves");
        gp->tail_mode = kTailNHalf;
        gp->full_units = full;
        gp->units = full + 2 * rest;
    }
    gp->groups = std::min<int64_t>(gp->units, gp->resident);
    return TILES_OK;
}

// Bytes of workspace a K-split tail of this GEMM would use (the header alone
// when its last round needs no split).
int64_t gemm_ws_bytes(const tiles_gemm_desc* d, const tiles_config* user_cfg, int* status) {
    GemmPlan gp;
    *status = gemm_prepare(d, user_cfg, true, SIZE_MAX, &gp);
    return *status == TILES_OK ? gp.ws_needed : 0;
}

std::atomic<uint32_t> g_epoch{0};

int gemm_common(const tiles_gemm_desc* d, const tiles_config* user_cfg, void* ws, size_t ws_bytes,
                void* stream, bool batched) {
    GemmPlan gp;
    int s = gemm_prepare(d, user_cfg, batched, ws ? ws_bytes : 0, &gp);
    if (s != TILES_OK) return s;
    // The workspace carries the kernel's timeout report: without one an
    // expired wait would go unreported.
    if (!ws || ws_bytes < kWorkspaceBytes)
        return fail(TILES_ERR_INVALID_ARG, "a workspace of at least %zu bytes is required",
                    kWorkspaceBytes);
    const tiles_config& cfg = gp.cfg;
    const int64_t batch = d->batch;
    const int64_t sa = batch > 1 ? d->stride_a : d->m * d->lda;
    const int64_t sb = batch > 1 ? d->stride_b : d->k * d->ldb;
    CUtensorMap ta, tb;
    // Each CTA loads 128 rows of A and 64-column atoms of B per K block.
    s = encode_3d(&ta, d->a_dtype, d->a, d->k, d->m, batch, d->lda, sa, 64, 128);
    if (s != TILES_OK) return s;
    s = encode_3d(&tb, d->b_dtype, d->b, d->n, d->k, batch, d->ldb, sb, 64, 64);
    if (s != TILES_OK) return s;
    CUtensorMap tc{};
    const int64_t sc = batch > 1 ? d->stride_c : d->m * d->ldc;
    const bool tma_c = encode_c_store(&tc, d->c_dtype, d->c, d->n, d->m, batch, d->ldc, sc);

    GemmArgs args{};
    args.m = (int32_t)d->m; args.n = (int32_t)d->n; args.k = (int32_t)d->k;
    args.batch = (int32_t)batch;
    args.m_blocks = (int32_t)((d->m + cfg.bm - 1) / cfg.bm);
    // Grouped tile order (the persistent scheduler's rasterisation): when the
    // A panels of every M block of an item would not stay in L2 while the
    // concurrent CTAs sweep N, the tiles go in groups of kTileGroupM M blocks.
    // A window of resident groups then covers kTileGroupM M blocks by about
    // resident / kTileGroupM N blocks of panels.
    const int64_t a_panels = static_cast<int64_t>(args.m_blocks) * cfg.bm * d->k * 2;
    args.group_m = a_panels <= kTileGroupBytes ? args.m_blocks
                                               : std::min<int32_t>(args.m_blocks, kTileGroupM);
    args.n_blocks = (int32_t)((d->n + cfg.bn - 1) / cfg.bn);
    args.k_blocks = (int32_t)((d->k + cfg.bk - 1) / cfg.bk);
    args.tiles = (int32_t)gp.tiles;
    args.full_units = (int32_t)gp.full_units;
    args.units = (int32_t)gp.units;
    args.tail_mode = gp.tail_mode;
    args.ksplit = gp.ksplit;
    if (gp.tail_mode == kTailKSplit) {
        char* base = static_cast<char*>(ws);
        args.flags = reinterpret_cast<uint32_t*>(base + gp.flags_offset);
        args.partials = reinterpret_cast<float*>(base + gp.partials_offset);
        uint32_t e = g_epoch.fetch_add(1) + 1;
        if (e == 0) e = g_epoch.fetch_add(1) + 1;      // 0 marks "never written"
        args.epoch = e;
    }
    args.c = d->c;
    args.ldc = d->ldc;
    args.stride_c = batch > 1 ? d->stride_c : 0;
    args.c_dtype = d->c_dtype;
    args.tma_store = tma_c ? 1 : 0;
    args.idesc = ptx::idesc_f16_f32acc(d->a_dtype == TILES_BF16, true, cfg.bm, cfg.bn);
    args.idesc_half = ptx::idesc_f16_f32acc(d->a_dtype == TILES_BF16, true, cfg.bm, cfg.bn / 2);
    args.err = static_cast<int32_t*>(ws);
    args.wait_limit_ns = kDefaultWaitLimitNs;
    const PlantedFault planted = take_planted_fault();
    args.drop_stage = planted.stage;
    if (planted.stage >= 0) args.wait_limit_ns = planted.limit_ns;
    int e = launch_variant(cfg.bn, cfg.cta_group, ta, tb, tc, args, (int)gp.groups,
                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(TILES_ERR_CUDA, "GEMM launch failed: %s",
                    cudaGetErrorString(static_cast<cudaError_t>(e)));
    return TILES_OK;
}

}  // namespace

namespace {
thread_local PlantedFault g_planted{-1, 0};
}  // namespace

PlantedFault take_planted_fault() {
    const PlantedFault f = g_planted;
    g_planted = PlantedFault{-1, 0};
    return f;
}

int fail(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

__global__ void selftest_wait_kernel(int32_t* err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // Nothing ever arrives on `bar`: its phase 0 never completes, so the
    // bounded wait must give up after limit_ns and report it.
    if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, &abort_flag, limit_ns) && err)
        atomicOr(err, kErrSelftest);
}

}  // namespace tiles

// ---- GEMM without caller-allocated memory ----------------------------------
//
// Callers that cannot call cudaMalloc (code running where device allocation
// is forbidden or unavailable: inside an allocator or driver callback, under
// a runtime that owns all device memory, or in a real-time path that must
// not allocate) cannot provide the workspace that tiles_gemm takes.  For
// them tiles_gemm_noalloc uses this file-scope device array instead.  It is
// exactly the kernels' workspace (the error word a bounded wait writes on
// expiry), 256 bytes, and every GPU that loads the library holds it until the
// process exits.  It starts at zero when the module loads; the error word is
// cleared each time a waiting call reads it.
static __device__ __align__(256) unsigned char tiles_noalloc_scratch[256];

namespace tiles {
namespace {

constexpr size_t kNoAllocScratchBytes = sizeof(tiles_noalloc_scratch);
// The device address of the scratch array on the current device.  In host
// code the array's name is only a host-side stand-in, so the address is
// asked of the runtime, with the device current, on every call (after a
// device reset the module, and the array, load anew at another address).
int noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, tiles_noalloc_scratch);
    if (e != cudaSuccess || !p)
        return fail(TILES_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    *out = p;
    return TILES_OK;
}

}  // namespace
}  // namespace tiles

using namespace tiles;

extern "C" {

const char* tiles_status_string(int status) {
    switch (status) {
        case TILES_OK: return "TILES_OK";
        case TILES_ERR_INVALID_ARG: return "TILES_ERR_INVALID_ARG";
        case TILES_ERR_UNSUPPORTED_DTYPE: return "TILES_ERR_UNSUPPORTED_DTYPE";
        case TILES_ERR_MISALIGNED: return "TILES_ERR_MISALIGNED";
        case TILES_ERR_INFEASIBLE: return "TILES_ERR_INFEASIBLE";
        case TILES_ERR_CUDA: return "TILES_ERR_CUDA";
        case TILES_ERR_TIMEOUT: return "TILES_ERR_TIMEOUT";
        case TILES_ERR_TOO_LARGE: return "TILES_ERR_TOO_LARGE";
        default: return "TILES_ERR_UNKNOWN";
    }
}

const char* tiles_last_error(void) { return g_last_error.c_str(); }

const char* tiles_version(void) { return "tiles 0.1 (sm_103a)"; }

int tiles_device_preset(int preset, tiles_device* out) {
    if (!out) return fail(TILES_ERR_INVALID_ARG, "null output");
    if (preset == TILES_DEV_H100_PAGES) { device_preset_h100(out); return TILES_OK; }
    if (preset == TILES_DEV_GB300) { device_preset_gb300(out); return TILES_OK; }
    return fail(TILES_ERR_INVALID_ARG, "unknown device preset %d", preset);
}

int tiles_device_query(int ordinal, tiles_device* out) {
    if (!out) return fail(TILES_ERR_INVALID_ARG, "null output");
    tiles_device d;
    device_preset_gb300(&d);
    struct { cudaDeviceAttr attr; int32_t* field; } q[] = {
        {cudaDevAttrMultiProcessorCount, &d.sm_count},
        {cudaDevAttrMaxSharedMemoryPerMultiprocessor, &d.smem_per_sm},
        {cudaDevAttrMaxSharedMemoryPerBlockOptin, &d.smem_per_block_max},
        {cudaDevAttrMaxRegistersPerMultiprocessor, &d.regs_per_sm},
        {cudaDevAttrMaxThreadsPerMultiProcessor, &d.max_threads_per_sm},
        {cudaDevAttrMaxThreadsPerBlock, &d.max_threads_per_block},
        {cudaDevAttrMaxBlocksPerMultiprocessor, &d.max_blocks_per_sm},
        {cudaDevAttrWarpSize, &d.warp_size},
    };
    for (auto& e : q) {
        int v = 0;
        cudaError_t r = cudaDeviceGetAttribute(&v, e.attr, ordinal);
        if (r != cudaSuccess)
            return fail(TILES_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(r));
        *e.field = v;
    }
    int major = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, ordinal);
    d.tmem_cols = major == 10 ? 512 : 0;
    if (major == 10) {
        int current = 0;
        cudaGetDevice(&current);
        if (current == ordinal) {
            d.cta_pairs = max_groups(ordinal, 256, 2, d.sm_count);
            // The kernels' register figure as the runtime reports it: the
            // largest count of any compiled variant, rounded up to the
            // per-warp allocation granule as the page's C2 rounds.
            int regs = 0;
            for (int i = 0; i < kNumGemmVariants; ++i) {
                VariantAttributes va{};
                if (variant_attributes(kGemmVariants[i].bn, kGemmVariants[i].cta_group, d.sm_count,
                                       &va) == cudaSuccess)
                    regs = std::max(regs, va.regs);
                else
                    cudaGetLastError();
            }
            if (regs > 0 && d.warp_size > 0 && d.reg_granularity_per_warp > 0) {
                const int per_warp = (regs * d.warp_size + d.reg_granularity_per_warp - 1) /
                                     d.reg_granularity_per_warp * d.reg_granularity_per_warp;
                d.kernel_regs_per_thread = per_warp / d.warp_size;
            }
        }
    }
    *out = d;
    return TILES_OK;
}

int tiles_gemm_variant_count(void) { return kNumGemmVariants; }

int tiles_gemm_variant(int index, tiles_config* out) {
    if (!out || index < 0 || index >= kNumGemmVariants)
        return fail(TILES_ERR_INVALID_ARG, "variant index %d outside [0, %d)", index,
                    kNumGemmVariants);
    *out = variant_config(index);
    return TILES_OK;
}

int tiles_gemm_variant_info(int index, tiles_variant_info* out) {
    if (!out || index < 0 || index >= kNumGemmVariants)
        return fail(TILES_ERR_INVALID_ARG, "variant index %d outside [0, %d)", index,
                    kNumGemmVariants);
    int ordinal = 0;
    cudaError_t e = cudaGetDevice(&ordinal);
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ordinal);
    if (e != cudaSuccess)
        return fail(TILES_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    std::memset(out, 0, sizeof(*out));
    out->cfg = variant_config(index);
    VariantAttributes va{};
    const int r = variant_attributes(out->cfg.bn, out->cfg.cta_group, sms, &va);
    if (r != cudaSuccess) {
        cudaGetLastError();
        return fail(TILES_ERR_CUDA, "variant %d: %s", index,
                    cudaGetErrorString(static_cast<cudaError_t>(r)));
    }
    out->regs_per_thread = va.regs;
    out->local_bytes_per_thread = va.local_bytes;
    out->static_smem_bytes = va.static_smem;
    out->dynamic_smem_bytes = va.dynamic_smem;
    out->max_dynamic_smem_bytes = va.max_dynamic_smem;
    out->blocks_per_sm = va.blocks_per_sm;
    out->resident_groups = va.groups;
    return TILES_OK;
}

int tiles_evaluate(const tiles_device* dev, const tiles_config* cfg, int elem_bytes,
                   int accum_bytes, tiles_verdict* out) {
    if (!dev || !cfg || !out) return fail(TILES_ERR_INVALID_ARG, "null argument");
    if (elem_bytes <= 0 || accum_bytes <= 0 || cfg->bm <= 0 || cfg->bn <= 0 || cfg->bk <= 0 ||
        cfg->stages <= 0 || cfg->threads <= 0)
        return fail(TILES_ERR_INVALID_ARG, "sizes must be positive");
    return evaluate(*dev, *cfg, elem_bytes, accum_bytes, out);
}

int tiles_finish_parallelism(const tiles_device* dev, int64_t b, int64_t m, int64_t n,
                             tiles_verdict* inout) {
    if (!dev || !inout) return fail(TILES_ERR_INVALID_ARG, "null argument");
    if (b < 1 || m < 1 || n < 1) return fail(TILES_ERR_INVALID_ARG, "sizes must be >= 1");
    finish_parallelism(*dev, b, m, n, inout);
    return TILES_OK;
}

double tiles_c0_bytes(int64_t b, int64_t m, int64_t n, int64_t k, int bm, int bn, int in_bytes,
                      int out_bytes) {
    if (bm <= 0 || bn <= 0) return 0.0;
    return c0_bytes(b, m, n, k, bm, bn, in_bytes, out_bytes);
}

int tiles_plan(const tiles_device* dev, const tiles_problem* prob, tiles_verdict* out,
               int capacity, int* n_feasible) {
    if (!dev || !prob || !n_feasible || capacity < 0 || (capacity > 0 && !out))
        return fail(TILES_ERR_INVALID_ARG, "null argument or negative capacity");
    *n_feasible = 0;
    if (prob->b < 1 || prob->m < 1 || prob->n < 1 || prob->k < 1)
        return fail(TILES_ERR_INVALID_ARG, "sizes must be >= 1");
    std::vector<tiles_verdict> ranked;
    int s = plan(*dev, *prob, &ranked);
    if (s != TILES_OK) return fail(s, "planning failed");
    *n_feasible = (int)ranked.size();
    for (int i = 0; i < capacity && i < (int)ranked.size(); ++i) out[i] = ranked[i];
    return TILES_OK;
}

int tiles_htile_rows(int H, int kh, int sh, int pt, int d, int o0, int o1, tiles_htile* out) {
    if (!out) return fail(TILES_ERR_INVALID_ARG, "null output");
    int s = htile_rows(H, kh, sh, pt, d, o0, o1, out);
    if (s != TILES_OK) return fail(s, "invalid H-tile arguments");
    return TILES_OK;
}

size_t tiles_workspace_bytes(void) { return kWorkspaceBytes; }

int tiles_gemm(const tiles_gemm_desc* desc, const tiles_config* cfg, void* ws, size_t ws_bytes,
               void* stream) {
    return gemm_common(desc, cfg, ws, ws_bytes, stream, false);
}

int tiles_gemm_batched(const tiles_gemm_desc* desc, const tiles_config* cfg, void* ws,
                       size_t ws_bytes, void* stream) {
    return gemm_common(desc, cfg, ws, ws_bytes, stream, true);
}

size_t tiles_gemm_workspace_bytes(const tiles_gemm_desc* desc, const tiles_config* cfg) {
    int status = TILES_OK;
    const int64_t n = gemm_ws_bytes(desc, cfg, &status);
    return status == TILES_OK ? (size_t)n : 0;
}

int tiles_gemm_schedule(const tiles_gemm_desc* desc, const tiles_config* cfg, size_t ws_bytes,
                        tiles_schedule* out) {
    if (!out) return fail(TILES_ERR_INVALID_ARG, "null output");
    GemmPlan gp;
    int s = gemm_prepare(desc, cfg, true, ws_bytes, &gp);
    if (s != TILES_OK) return s;
    out->tail_mode = gp.tail_mode;
    out->ksplit = gp.ksplit;
    out->workspace_bytes = gp.ws_needed;
    out->cfg = gp.cfg;
    out->tiles = gp.tiles;
    out->resident_groups = gp.resident;
    out->full_units = gp.full_units;
    out->units = gp.units;
    out->groups = gp.groups;
    return TILES_OK;
}

int tiles_gemm_autotune(const tiles_gemm_desc* desc, int top_k, int reps, void* ws,
                        size_t ws_bytes, void* stream, tiles_tune_result* results,
                        int capacity, int* n_results, tiles_config* best) {
    if (n_results) *n_results = 0;
    if (!desc || !best) return fail(TILES_ERR_INVALID_ARG, "null descriptor or output");
    if (top_k < 1 || top_k > 16 || reps < 1 || reps > 100)
        return fail(TILES_ERR_INVALID_ARG, "top_k must be in [1, 16] and reps in [1, 100]");
    if (capacity < 0 || (capacity > 0 && !results))
        return fail(TILES_ERR_INVALID_ARG, "results must hold capacity entries");
    // Validates the problem (shapes, pitches, dtypes) and finds the device.
    GemmPlan gp0;
    int s = gemm_prepare(desc, nullptr, true, ws ? ws_bytes : 0, &gp0);
    if (s != TILES_OK) return s;
    // Steps 1-2: the feasible configurations in the planner's rank order.
    tiles_problem p{};
    p.b = desc->batch; p.m = desc->m; p.n = desc->n; p.k = desc->k;
    p.in_dtype = desc->a_dtype; p.out_dtype = desc->c_dtype;
    p.instr = TILES_INSTR_TCGEN05; p.mode = TILES_MODE_GB300;
    std::vector<tiles_verdict> ranked;
    s = plan(gp0.dev, p, &ranked);
    if (s != TILES_OK) return s;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Two passes of reps launches back to back, each between one pair of
    // events: launches overlap their neighbours' set-up (programmatic
    // serialization), so a launch's own time is the pass's time over reps.
    std::vector<cudaEvent_t> ev(4);
    for (auto& e : ev) {
        cudaError_t ce = cudaEventCreate(&e);
        if (ce != cudaSuccess) {
            for (auto& x : ev) if (x) cudaEventDestroy(x);
            return fail(TILES_ERR_CUDA, "cudaEventCreate: %s", cudaGetErrorString(ce));
        }
    }
    int count = 0;
    float best_us = 0.0f;
    bool have_best = false;
    tiles_config winner{};
    auto record = [&](const tiles_tune_result& r) {
        if (count < capacity) results[count] = r;
        ++count;
    };
    const int n_cfg = std::min<int>(top_k, static_cast<int>(ranked.size()));
    for (int i = 0; i < n_cfg; ++i) {
        // Step 3: each schedule the configuration admits for the last round,
        // the planner's own choice first (so that it wins ties).
        std::vector<std::pair<int, int>> seen;   // (tail_mode, ksplit) already timed
        const int tails[4] = {TILES_TAIL_AUTO, TILES_TAIL_WHOLE, TILES_TAIL_NHALF,
                              TILES_TAIL_KSPLIT};
        for (int t : tails) {
            tiles_tune_result r{};
            r.cfg = ranked[i].cfg;
            r.cfg.tail = t;
            r.ksplit = 1;
            GemmPlan gp;
            r.status = gemm_prepare(desc, &r.cfg, true, ws ? ws_bytes : 0, &gp);
            if (r.status == TILES_OK) {
                r.tail_mode = gp.tail_mode;
                r.ksplit = static_cast<int32_t>(gp.ksplit);
                const std::pair<int, int> sched{gp.tail_mode, r.ksplit};
                if (std::find(seen.begin(), seen.end(), sched) != seen.end()) continue;
                seen.push_back(sched);
                r.status = gemm_common(desc, &r.cfg, ws, ws_bytes, stream, true);   // untimed
                for (int pass = 0; pass < 2 && r.status == TILES_OK; ++pass) {
                    cudaEventRecord(ev[2 * pass], st);
                    for (int k = 0; k < reps && r.status == TILES_OK; ++k)
                        r.status = gemm_common(desc, &r.cfg, ws, ws_bytes, stream, true);
                    cudaEventRecord(ev[2 * pass + 1], st);
                }
                if (r.status == TILES_OK) r.status = tiles_check(ws, stream);
                if (r.status == TILES_OK) {
                    float ms[2] = {0.0f, 0.0f};
                    for (int pass = 0; pass < 2 && r.status == TILES_OK; ++pass)
                        if (cudaEventElapsedTime(&ms[pass], ev[2 * pass], ev[2 * pass + 1]) != cudaSuccess)
                            r.status = fail(TILES_ERR_CUDA, "cudaEventElapsedTime failed");
                    if (r.status == TILES_OK) {
                        r.us = 1000.0f * std::min(ms[0], ms[1]) / static_cast<float>(reps);
                        // Step 4: keep the fastest.
                        if (!have_best || r.us < best_us) {
                            have_best = true;
                            best_us = r.us;
                            winner = r.cfg;
                        }
                    }
                }
            }
            record(r);
        }
    }
    for (auto& e : ev) cudaEventDestroy(e);
    if (n_results) *n_results = count;
    if (!have_best) return fail(TILES_ERR_INFEASIBLE, "no candidate configuration ran");
    *best = winner;
    std::lock_guard<std::mutex> lock(g_tuned_mu);
    g_tuned[TunedKey{gp0.dev.sm_count, desc->batch, desc->m, desc->n, desc->k, desc->a_dtype,
                     desc->c_dtype}] = TunedEntry{winner, best_us};
    return TILES_OK;
}

int tiles_tuned_lookup(int sm_count, int64_t batch, int64_t m, int64_t n, int64_t k, int in_dtype,
                       int out_dtype, tiles_config* out) {
    if (!out) return fail(TILES_ERR_INVALID_ARG, "null output");
    if (!tuned_config(TunedKey{sm_count, batch, m, n, k, in_dtype, out_dtype}, out))
        return fail(TILES_ERR_INFEASIBLE, "no tuned configuration for this problem");
    return TILES_OK;
}

static const char kTunedHeader[] = "tiles-tuned 1";

int tiles_tuned_save(const char* path) {
    if (!path) return fail(TILES_ERR_INVALID_ARG, "null path");
    FILE* f = std::fopen(path, "w");
    if (!f) return fail(TILES_ERR_INVALID_ARG, "cannot write %s", path);
    std::lock_guard<std::mutex> lock(g_tuned_mu);
    std::fprintf(f, "%s\n", kTunedHeader);
    for (const auto& kv : g_tuned) {
        const TunedKey& key = kv.first;
        const tiles_config& c = kv.second.cfg;
        std::fprintf(f, "%d %lld %lld %lld %lld %d %d %d %d %d %d %d %d %d %d %d %.3f\n",
                     std::get<0>(key), (long long)std::get<1>(key), (long long)std::get<2>(key),
                     (long long)std::get<3>(key), (long long)std::get<4>(key), std::get<5>(key),
                     std::get<6>(key), c.bm, c.bn, c.bk, c.stages, c.threads, c.instr, c.acc_bufs,
                     c.cta_group, c.tail, kv.second.us);
    }
    const bool ok = std::fflush(f) == 0;
    std::fclose(f);
    return ok ? TILES_OK : fail(TILES_ERR_INVALID_ARG, "write to %s failed", path);
}

int tiles_tuned_load(const char* path) {
    if (!path) return fail(TILES_ERR_INVALID_ARG, "null path");
    FILE* f = std::fopen(path, "r");
    if (!f) return fail(TILES_ERR_INVALID_ARG, "cannot read %s", path);
    std::map<TunedKey, TunedEntry> loaded;
    char line[512];
    int lineno = 0;
    int status = TILES_OK;
    while (std::fgets(line, sizeof line, f)) {
        ++lineno;
        size_t len = std::strlen(line);
        if (len == sizeof line - 1 && line[len - 1] != '\n') {
            status = fail(TILES_ERR_INVALID_ARG, "%s:%d: line too long", path, lineno);
            break;
        }
        while (len && (line[len - 1] == '\n' || line[len - 1] == '\r')) line[--len] = 0;
        if (lineno == 1) {
            if (std::strcmp(line, kTunedHeader) != 0) {
                status = fail(TILES_ERR_INVALID_ARG, "%s: not a tuned-configuration file", path);
                break;
            }
            continue;
        }
        if (len == 0) continue;
        int sm, in_dt, out_dt;
        long long b, m, n, k;
        tiles_config c{};
        float us = 0.0f;
        int used = 0;
        const int got = std::sscanf(line, "%d %lld %lld %lld %lld %d %d %d %d %d %d %d %d %d %d %d %f %n",
                                    &sm, &b, &m, &n, &k, &in_dt, &out_dt, &c.bm, &c.bn, &c.bk,
                                    &c.stages, &c.threads, &c.instr, &c.acc_bufs, &c.cta_group,
                                    &c.tail, &us, &used);
        const bool sizes_ok = sm > 0 && b >= 1 && m >= 1 && n >= 1 && k >= 1;
        const bool dtypes_ok = (in_dt == TILES_F16 || in_dt == TILES_BF16) && bytes_of(out_dt) > 0;
        const bool cfg_ok = c.bm > 0 && c.bn > 0 && c.bk > 0 && c.stages > 0 && c.threads > 0 &&
                            c.tail >= TILES_TAIL_AUTO && c.tail <= TILES_TAIL_KSPLIT &&
                            c.cta_group >= 1 && c.cta_group <= 2 && us >= 0.0f;
        if (got != 17 || line[used] != 0 || !sizes_ok || !dtypes_ok || !cfg_ok) {
            status = fail(TILES_ERR_INVALID_ARG, "%s:%d: malformed entry", path, lineno);
            break;
        }
        loaded[TunedKey{sm, b, m, n, k, in_dt, out_dt}] = TunedEntry{c, us};
    }
    if (status == TILES_OK && lineno == 0)
        status = fail(TILES_ERR_INVALID_ARG, "%s: empty file", path);
    std::fclose(f);
    if (status != TILES_OK) return status;
    std::lock_guard<std::mutex> lock(g_tuned_mu);
    for (const auto& kv : loaded) g_tuned[kv.first] = kv.second;
    return TILES_OK;
}

int tiles_tuned_clear(void) {
    std::lock_guard<std::mutex> lock(g_tuned_mu);
    g_tuned.clear();
    return TILES_OK;
}

int tiles_check(void* ws, void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
    if (!ws) return TILES_OK;
    int32_t word = 0;
    e = cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "read workspace: %s", cudaGetErrorString(e));
    if (word == 0) return TILES_OK;
    e = cudaMemset(ws, 0, sizeof(word));
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "clear workspace: %s", cudaGetErrorString(e));
    return fail(TILES_ERR_TIMEOUT, "a bounded device wait expired (error bits 0x%x)", word);
}

int tiles_selftest_wait_timeout(void* ws, int64_t limit_ns, void* stream) {
    if (limit_ns <= 0 || limit_ns > 10000000000ll)
        return fail(TILES_ERR_INVALID_ARG, "limit_ns must be in (0, 1e10]");
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<int32_t*>(ws), (uint64_t)limit_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    return TILES_OK;
}

int tiles_selftest_drop_stage(int stage, int64_t limit_ns) {
    if (stage < 0) {
        take_planted_fault();
        return TILES_OK;
    }
    if (limit_ns <= 0 || limit_ns > 10000000000ll)
        return fail(TILES_ERR_INVALID_ARG, "limit_ns must be in (0, 1e10]");
    g_planted = PlantedFault{stage, static_cast<uint64_t>(limit_ns)};
    return TILES_OK;
}

int tiles_conv2d_htiled(const tiles_conv_desc* desc, int tile_oh, const tiles_config* cfg,
                        void* ws, size_t ws_bytes, void* stream) {
    return conv2d_htiled(desc, tile_oh, cfg, ws, ws_bytes, stream);
}

int tiles_conv2d_tiled(const tiles_conv_desc* desc, int tile_oh, int tile_ow, int tile_n,
                       const tiles_config* cfg, void* ws, size_t ws_bytes, void* stream) {
    return conv2d_tiled(desc, tile_oh, tile_ow, tile_n, cfg, ws, ws_bytes, stream);
}

int tiles_conv_out_hw(const tiles_conv_desc* desc, int32_t* oh, int32_t* ow) {
    if (!oh || !ow) return fail(TILES_ERR_INVALID_ARG, "null output");
    int64_t h = 0, w = 0;
    const int s = conv_out_hw(desc, &h, &w);
    if (s != TILES_OK) return s;
    if (h > INT32_MAX || w > INT32_MAX) return fail(TILES_ERR_TOO_LARGE, "output too large");
    *oh = static_cast<int32_t>(h);
    *ow = static_cast<int32_t>(w);
    return TILES_OK;
}

size_t tiles_conv_workspace_bytes(const tiles_conv_desc* desc, int tile_oh) {
    return static_cast<size_t>(conv_workspace_bytes(desc, tile_oh));
}

int tiles_gemm_noalloc(const tiles_gemm_desc* desc, const tiles_config* cfg, void* stream,
                       int wait) {
    static_assert(kWorkspaceBytes <= kNoAllocScratchBytes,
                  "the static scratch holds the kernels' error word");
    // Every schedule but a K-split last round needs the error word alone; a
    // configuration that forces a K split needs room for its partial tiles.
    if (cfg && cfg->tail == TILES_TAIL_KSPLIT) {
        int st = TILES_OK;
        const int64_t need = gemm_ws_bytes(desc, cfg, &st);
        if (st != TILES_OK) return st;
        if (need > static_cast<int64_t>(kNoAllocScratchBytes))
            return fail(TILES_ERR_TOO_LARGE, "a K-split last round needs %lld bytes of scratch; "
                        "the static array holds %zu", (long long)need, kNoAllocScratchBytes);
    }
    void* scratch = nullptr;
    int s = noalloc_scratch(&scratch);
    if (s != TILES_OK) return s;
    s = gemm_common(desc, cfg, scratch, kNoAllocScratchBytes, stream, true);
    if (s != TILES_OK || !wait) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
    int32_t word = 0;
    e = cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "read scratch: %s", cudaGetErrorString(e));
    if (word == 0) return TILES_OK;
    e = cudaMemset(scratch, 0, sizeof(word));
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "clear scratch: %s", cudaGetErrorString(e));
    return fail(TILES_ERR_TIMEOUT, "a bounded device wait expired (error bits 0x%x)", word);
}

}  // extern "C"
