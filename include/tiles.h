/*
 * tiles.h — C ABI of libtiles: a tile-size planner (constraints C0-C4) and
 * the GB300 (sm_103a) kernels it drives: a tiled dense GEMM C = A x B with
 * fp16/bf16 inputs and fp32 accumulation, optionally batched, and an NCHW
 * conv2d run as an implicit GEMM tiled over the output height.
 *
 * Sources of the operations (pages of the tile-size-decision material):
 *   - constraint procedure: page "04-tile-size-decision/tile_decision.py"
 *     (records Device/Config/Verdict; functions evaluate, finish_parallelism,
 *     dram_traffic, sweep) and its README ("目的": C0 with the batch term b);
 *   - GEMM problem statement C = A x B: tiling tutorial (m.nlpx.cn/news/214310),
 *     "案例解释 / 前提" and "Tiled 方法分块复用数据";
 *   - H-tile rows (in_start, in_end, in_span, pt', pb', halo): the tutorial's
 *     "H/W 维切分的通用公式" and its worked example "详细数值例子".
 *
 * Conventions for every call:
 *   - Plain C types only.  Device pointers are CUDA device addresses the
 *     caller allocated; the library allocates no device memory and never
 *     frees caller memory.  `stream` is a cudaStream_t passed as void*
 *     (NULL = the legacy default stream).  Launches are asynchronous.
 *   - Every call returns TILES_OK (0) or a negative tiles_status; nothing is
 *     printed and nothing is thrown across the ABI.  tiles_last_error()
 *     returns a human-readable message for the calling thread's last failure.
 *   - Matrices are row-major.  Leading dimensions (ld*) and batch strides
 *     (stride_*) are in elements; row pitches must be multiples of 16 bytes
 *     and base pointers 16-byte aligned (TMA requirement), else
 *     TILES_ERR_MISALIGNED.  There is no fallback path.
 *   - Workspace: a caller-owned device buffer, zeroed once before first
 *     use, of at least tiles_workspace_bytes() bytes.  Kernels record a
 *     bounded-wait timeout in its first word; tiles_check() reads and clears
 *     it.  A GEMM given tiles_gemm_workspace_bytes() bytes also uses it for
 *     the partial tiles of a last round split along K.  The kernel calls
 *     (GEMM, convolution, and their host-buffer forms) reject a NULL or
 *     smaller workspace with TILES_ERR_INVALID_ARG, so that no expired wait
 *     goes unreported; tiles_gemm_noalloc is the one kernel call that takes
 *     none (it has its own).  One workspace serves one launch at a time.
 */
#ifndef TILES_H
#define TILES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TILES_OK = 0,
    TILES_ERR_INVALID_ARG = -1,      /* null pointer, non-positive size, bad enum */
    TILES_ERR_UNSUPPORTED_DTYPE = -2,
    TILES_ERR_MISALIGNED = -3,       /* pointer or row pitch not 16-byte aligned */
    TILES_ERR_INFEASIBLE = -4,       /* no config passes C1-C4, or the given one fails */
    TILES_ERR_CUDA = -5,             /* a CUDA runtime/driver call failed */
    TILES_ERR_TIMEOUT = -6,          /* a bounded device wait expired (tiles_check) */
    TILES_ERR_TOO_LARGE = -7         /* size beyond a documented maximum */
} tiles_status;

typedef enum { TILES_F16 = 0, TILES_BF16 = 1, TILES_F32 = 2 } tiles_dtype;

/* MMA families of the constraint C3.  MMA, WGMMA and SIMT are the page's
 * instruction-shape table; TCGEN05 is the sm_100/sm_103 tensor-core MMA
 * (kind::f16) that the GB300 kernels issue. */
typedef enum {
    TILES_INSTR_MMA = 0,
    TILES_INSTR_WGMMA = 1,
    TILES_INSTR_SIMT = 2,
    TILES_INSTR_TCGEN05 = 3
} tiles_instr;

typedef enum { TILES_DEV_H100_PAGES = 0, TILES_DEV_GB300 = 1 } tiles_device_preset_id;

/* Planner modes: PAGES reproduces the page's sweep and ranking bit for bit;
 * GB300 ranks the configurations the sm_103a kernels implement. */
typedef enum { TILES_MODE_PAGES = 0, TILES_MODE_GB300 = 1 } tiles_mode;

/* Failure bits of a verdict (the page reports them as message prefixes). */
#define TILES_FAIL_C3   0x1u   /* instruction shape / thread multiple / kernel layout */
#define TILES_FAIL_C1   0x2u   /* shared-memory capacity per block */
#define TILES_FAIL_C2   0x4u   /* registers (page) or tensor-memory columns (GB300) */
#define TILES_FAIL_OCC  0x8u   /* no resident block fits: blocks_per_sm == 0 */
/* Warning bits (constraint C4). */
#define TILES_WARN_TAIL 0x1u   /* more than one wave and the last is < 50% full */
#define TILES_WARN_IDLE 0x2u   /* fewer tiles than SMs */

/* Binding resource of the occupancy computation. */
typedef enum {
    TILES_BIND_NONE = 0, TILES_BIND_REGS = 1, TILES_BIND_SMEM = 2,
    TILES_BIND_THREADS = 3, TILES_BIND_TMEM = 4
} tiles_binding;

/* Hardware model (the page's Device record plus GB300 fields). */
typedef struct {
    int32_t smem_per_sm;              /* bytes */
    int32_t smem_per_block_max;       /* bytes, opt-in limit of one block */
    int32_t regs_per_sm;
    int32_t max_threads_per_sm;
    int32_t max_threads_per_block;
    int32_t max_blocks_per_sm;
    int32_t regs_per_thread_max;
    int32_t reg_granularity_per_warp;
    int32_t warp_size;
    int32_t sm_count;
    /* GB300 additions (zero on the page's device) */
    int32_t tmem_cols;                /* tensor-memory columns per SM (512) */
    int32_t mma_flops_per_clk;        /* dense f16/bf16 FLOP per clock per SM */
    int32_t fill_bytes_per_clk;       /* L2 -> shared bytes per clock per SM (time model) */
    int32_t kernel_regs_per_thread;   /* register budget of the GB300 kernels */
    int32_t cta_pairs;                /* GB300: CTA pairs (2-CTA clusters) resident at once;
                                         0 = sm_count / 2 */
    int32_t partial_bytes_per_clk;    /* GB300 time model: bytes per clock per SM at which a
                                         K part of a split last round writes or reads its
                                         fp32 partial tile (0 counts as 1) */
    int32_t handoff_clocks;           /* GB300 time model: fixed clocks of one K-part
                                         hand-off (flag release, acquire, latency) */
    int32_t pair_launch_clocks;       /* GB300 time model: the extra fixed clocks of a launch
                                         of the CTA-pair kernels (cluster launch, the pair's
                                         prologue and last epilogue) over one-CTA kernels */
} tiles_device;

/* One tile configuration (the page's Config record plus GB300 fields). */
typedef struct {
    int32_t bm, bn, bk;      /* output tile rows/cols and K step (elements) */
    int32_t stages;          /* shared-memory pipeline depth */
    int32_t threads;         /* threads per block */
    int32_t instr;           /* tiles_instr */
    int32_t acc_bufs;        /* GB300: TMEM accumulator buffers (0 on the page) */
    int32_t cta_group;       /* GB300: 1 or 2 SMs per MMA (0 on the page) */
    int32_t tail;            /* GB300 last-round schedule, tiles_tail (0 = planner's choice) */
    int32_t conv_weights;    /* convolution with the TMA producer: where the weights sit,
                                tiles_conv_weights (0 = tensor memory when they fit) */
    int32_t reserved[2];
} tiles_config;

/* Where the TMA convolution keeps the filter (tiles_config.conv_weights).
 * TMEM: the weights are the MMA's A operand in tensor memory (M = 128
 * output channels, N = a tile of output pixels); it applies when c_out <=
 * 128 and the K columns plus one accumulator fit the 512 columns; each
 * (filter tap, 64 channels) is one pixel box.  TMEM_ROWS: the same filter
 * placement with one output row per tile, whose input rows are loaded once
 * per (kernel row, 64 channels) as stride phases and shared by all the
 * row's taps through shifted descriptors (kw <= 8, the row's input span
 * within one TMA box).  SMEM: the weights are the B operand in shared
 * memory (M = 128 output pixels, N = a block of output channels); it
 * applies to every TMA convolution.  TMEM_ROWS_DIRECT: the rows form over
 * an NCHW input read in place (W a multiple of 8, a stage's input span at
 * most 249 columns): warps of the kernel transpose each stage's input rows
 * into the stride-phase planes, so no NHWC copy is made.  AUTO takes the
 * first of TMEM_ROWS_DIRECT, TMEM_ROWS, TMEM, SMEM that applies. */
typedef enum {
    TILES_CONV_W_AUTO = 0, TILES_CONV_W_SMEM = 1, TILES_CONV_W_TMEM = 2,
    TILES_CONV_W_TMEM_ROWS = 3, TILES_CONV_W_TMEM_ROWS_DIRECT = 4
} tiles_conv_weights;

/* Schedules of a last round of tiles that would leave resident CTA groups
 * idle (constraint C4): as whole tiles, as N-half tiles, or split along K
 * into parts whose fp32 partials the last part adds (needs workspace). */
typedef enum {
    TILES_TAIL_AUTO = 0, TILES_TAIL_WHOLE = 1, TILES_TAIL_NHALF = 2, TILES_TAIL_KSPLIT = 3
} tiles_tail;

/* Result of checking one configuration (the page's Verdict record). */
typedef struct {
    tiles_config cfg;
    int64_t smem_per_stage;      /* bytes */
    int64_t smem_total;          /* bytes (GB300: + barriers and alignment) */
    int32_t accum_per_thread;    /* C2 accumulators per thread */
    int32_t regs_per_thread;     /* C2, warp-rounded */
    int32_t regs_per_block;
    int32_t blocks_by_regs;
    int32_t blocks_by_smem;
    int32_t blocks_by_threads;
    int32_t blocks_by_tmem;      /* GB300 */
    int32_t blocks_per_sm;
    int32_t tmem_cols_alloc;     /* GB300: power-of-two TMEM allocation */
    int32_t binding;             /* tiles_binding */
    uint32_t failures;           /* TILES_FAIL_* bits */
    int32_t c3_violations;       /* how many C3 conditions failed */
    uint32_t warnings;           /* TILES_WARN_* bits */
    int32_t tail_split;          /* GB300 last round: K parts (>= 2), -1 N-halves, 0 whole */
    int64_t grid;                /* C4: output tiles (times the batch) */
    int64_t waves;               /* C4 */
    double last_wave_fill;       /* C4, in [0, 1] */
    double c0_bytes;             /* C0, float64 as on the page */
    int64_t est_clocks;          /* GB300 time model (0 in page mode): whole rounds of
                                    ceil(K/bk) K blocks of max(MMA, fill) clocks,
                                    then the last round in its cheapest schedule, plus
                                    pair_launch_clocks for a CTA-pair kernel */
} tiles_verdict;

/* A planning request. */
typedef struct {
    int64_t b, m, n, k;          /* batch and GEMM sizes, all >= 1 */
    int32_t in_dtype;            /* tiles_dtype of A and B */
    int32_t out_dtype;           /* tiles_dtype of C */
    int32_t instr;               /* PAGES mode: the MMA family swept */
    int32_t mode;                /* tiles_mode */
} tiles_problem;

/* Rows of one H-tile of a convolution (tutorial, "H/W 维切分的通用公式"). */
typedef struct {
    int32_t in_start;   /* max(0, o0*sh - pt) */
    int32_t in_end;     /* (o1-1)*sh - pt + (kh-1)*d + 1, exclusive */
    int32_t in_span;    /* in_end - in_start (counts pb' virtual rows) */
    int32_t pt;         /* top pad of the sub-operator: max(0, pt - o0*sh) */
    int32_t pb;         /* bottom pad of the sub-operator: max(0, in_end - H) */
    int32_t halo;       /* (kh-1)*d + 1 - sh, signed */
} tiles_htile;

/* One GEMM (or a batch of equally shaped GEMMs):
 * C[t] = A[t] x B[t] for t < batch, A[t] at a + t*stride_a, etc. */
typedef struct {
    int64_t m, n, k;
    int64_t batch;                    /* >= 1; tiles_gemm requires 1 */
    const void* a;                    /* device, M x K, row pitch lda */
    const void* b;                    /* device, K x N, row pitch ldb */
    void* c;                          /* device, M x N, row pitch ldc */
    int64_t lda, ldb, ldc;            /* elements */
    int64_t stride_a, stride_b, stride_c;   /* elements between batch items */
    int32_t a_dtype, b_dtype, c_dtype;      /* a == b in {F16, BF16}; c in {F32, F16, BF16} */
    int32_t pad0;
} tiles_gemm_desc;

/* Memory order of the convolution input. */
typedef enum { TILES_LAYOUT_NCHW = 0, TILES_LAYOUT_NHWC = 1 } tiles_layout;

/* A convolution with OIHW weights and NCHW output, fully packed; the input
 * is NCHW or NHWC (x_layout). */
typedef struct {
    int32_t n, c, h, w;               /* input */
    int32_t c_out, kh, kw;            /* weights */
    int32_t sh, sw, ph, pw, dh, dw;   /* stride, symmetric pad, dilation */
    int32_t in_dtype, out_dtype;      /* in: F16/BF16 (x and w); out: F16/BF16/F32 */
    int32_t x_layout;                 /* tiles_layout of x */
    const void* x;                    /* device, [n][c][h][w] or [n][h][w][c] */
    const void* wt;                   /* device, [c_out][c][kh][kw] */
    void* y;                          /* device, [n][c_out][oh][ow] */
} tiles_conv_desc;

/* The launch geometry tiles_gemm would use for a descriptor. */
typedef struct {
    tiles_config cfg;            /* the configuration (planned or given) */
    int64_t tiles;               /* output tiles, b * ceil(M/bm) * ceil(N/bn) */
    int64_t resident_groups;     /* CTA groups (CTAs or CTA pairs) resident at once */
    int64_t full_units;          /* units run as whole tiles */
    int64_t units;               /* whole tiles plus the last round's split units */
    int64_t groups;              /* persistent CTA groups launched */
    int32_t tail_mode;           /* 0: last round as whole tiles; 1: as N-halves;
                                    2: split along K into ksplit parts */
    int32_t ksplit;              /* K parts per last-round tile (tail_mode 2) */
    int64_t workspace_bytes;     /* workspace this schedule uses (>= 256) */
} tiles_schedule;

/* ---- status and diagnostics -------------------------------------------- */

/* Static name of a status code. */
const char* tiles_status_string(int status);
/* Message for the calling thread's last non-OK return ("" if none). */
const char* tiles_last_error(void);
/* Library version string. */
const char* tiles_version(void);

/* ---- hardware model ----------------------------------------------------- */

/* Fill *out with a preset: TILES_DEV_H100_PAGES is the page's Device record
 * (132 SMs, 228 KB per SM, 227 KB per block, 65536 registers ...);
 * TILES_DEV_GB300 is the GB300 model (148 SMs until queried, 228 KB per SM,
 * 227 KB per block, 512 TMEM columns).  INVALID_ARG on a bad id or NULL. */
int tiles_device_preset(int preset, tiles_device* out);

/* The GB300 preset with the runtime's values for CUDA device `ordinal`
 * (SM count, shared memory per SM and per block, registers, threads).  When
 * `ordinal` is the current device it also takes the compiled kernels' facts
 * from the runtime: kernel_regs_per_thread is the largest register count of
 * a compiled variant rounded up to the per-warp granule, and cta_pairs the
 * co-resident 2-CTA clusters of the 256-wide pair kernel.  CUDA error if no
 * such device. */
int tiles_device_query(int ordinal, tiles_device* out);

/* ---- constraint procedure ---------------------------------------------- */

/* C3, C1, C2 and occupancy for one configuration (the page's evaluate):
 * cfg->instr selects the page's rules (MMA/WGMMA/SIMT) or the GB300 rules
 * (TCGEN05).  elem_bytes is the input width, accum_bytes the accumulator
 * width.  Writes *out entirely; the grid/wave/C0 fields are left zero. */
int tiles_evaluate(const tiles_device* dev, const tiles_config* cfg, int elem_bytes,
                   int accum_bytes, tiles_verdict* out);

/* C4 (the page's finish_parallelism) for a batch of b GEMMs of M x N:
 * grid = b*ceil(M/bm)*ceil(N/bn); waves and last-wave fill over
 * max(blocks_per_sm * sm_count, 1) resident blocks (GB300: over resident
 * CTA groups); sets the warning bits.  Updates *inout in place. */
int tiles_finish_parallelism(const tiles_device* dev, int64_t b, int64_t m, int64_t n,
                             tiles_verdict* inout);

/* C0: in_bytes*b*M*N*K*(1/bn + 1/bm) + out_bytes*b*M*N, evaluated left to
 * right in IEEE double (README "目的"; the page's dram_traffic at b=1). */
double tiles_c0_bytes(int64_t b, int64_t m, int64_t n, int64_t k, int bm, int bn,
                      int in_bytes, int out_bytes);

/* The sweep: enumerate, keep the feasible, rank best first.  PAGES mode
 * enumerates bm,bn in {16..256}, bk in {16..128} (<= K), stages 2..4,
 * threads 128/256/512 and ranks by (round(C0), -blocks_per_sm, smem_total);
 * GB300 mode enumerates the compiled sm_103a kernel variants and ranks by
 * (est_clocks, round(C0), -blocks_per_sm, smem_total).  Ties keep the
 * enumeration order.  Writes min(capacity, n) verdicts to out (out may be
 * NULL when capacity is 0) and always writes *n_feasible. */
int tiles_plan(const tiles_device* dev, const tiles_problem* prob, tiles_verdict* out,
               int capacity, int* n_feasible);

/* The H-tile rows of output rows [o0, o1) (formulas above).  INVALID_ARG if
 * a size is non-positive, o1 <= o0 or pt < 0. */
int tiles_htile_rows(int H, int kh, int sh, int pt, int d, int o0, int o1, tiles_htile* out);

/* ---- kernels (sm_103a) --------------------------------------------------- */

/* Bytes of workspace a kernel call needs (a small constant). */
size_t tiles_workspace_bytes(void);

/* C = A x B on one GPU: fp16/bf16 inputs, fp32 accumulation in tensor
 * memory, output cast to c_dtype with round-to-nearest-even.  cfg == NULL
 * lets the GB300 planner choose (memoised per shape); a given cfg must be a
 * compiled variant (bm = 128*cta_group, bk = 64, acc_bufs = 2, threads 192)
 * and pass C1-C4, else INFEASIBLE.  desc->batch must be 1.  M, N, K >= 1;
 * ragged edges are handled (zero fill on loads, clipped stores). */
int tiles_gemm(const tiles_gemm_desc* desc, const tiles_config* cfg, void* workspace,
               size_t ws_bytes, void* stream);

/* The schedule a tiles_gemm_batched call with these arguments and a
 * workspace of ws_bytes would launch: the planned (or given, checked)
 * configuration and rounds of the resident CTA groups.  A last round that
 * would fill at most half of them (constraint C4, last-wave fill) is split:
 * along K into resident/rest parts (at most 8) when the workspace holds the
 * fp32 partial tiles -- the leading parts hand their partials to the last
 * part, which adds them in part order (deterministic) and stores C -- else
 * into N-halves when a half is whole 64-column B atoms.  Validates like
 * tiles_gemm_batched; launches nothing. */
int tiles_gemm_schedule(const tiles_gemm_desc* desc, const tiles_config* cfg, size_t ws_bytes,
                        tiles_schedule* out);

/* ---- The compiled GEMM kernels as the hardware sees them ----------------
 * The GB300 planner's C1, C2 and occupancy figures (README of
 * tile_decision.py, "已知局限": the constraints are bounds that the real
 * kernel has to confirm) restated as what the CUDA runtime reports for each
 * compiled kernel variant. */
typedef struct {
    tiles_config cfg;                 /* bm, bn, bk, stages, threads, instr, acc_bufs,
                                         cta_group of the variant (tail 0) */
    int32_t regs_per_thread;          /* cudaFuncAttributes::numRegs */
    int32_t local_bytes_per_thread;   /* cudaFuncAttributes::localSizeBytes (spills) */
    int32_t static_smem_bytes;        /* cudaFuncAttributes::sharedSizeBytes */
    int32_t dynamic_smem_bytes;       /* dynamic shared memory every launch requests */
    int32_t max_dynamic_smem_bytes;   /* cudaFuncAttributes::maxDynamicSharedSizeBytes once
                                         the library has opted the kernel in */
    int32_t blocks_per_sm;            /* cudaOccupancyMaxActiveBlocksPerMultiprocessor at
                                         that dynamic shared memory */
    int32_t resident_groups;          /* CTA groups resident at once: blocks_per_sm * SMs
                                         for one CTA per tile, cudaOccupancyMaxActiveClusters
                                         for CTA pairs */
    int32_t reserved[5];
} tiles_variant_info;

/* Number of compiled GEMM kernel variants.  Host only. */
int tiles_gemm_variant_count(void);

/* The configuration of compiled variant `index` (0 <= index < count), in
 * the planner's enumeration order.  Host only: no GPU needed.
 * INVALID_ARG for a bad index or NULL. */
int tiles_gemm_variant(int index, tiles_config* out);

/* What the CUDA runtime reports for compiled variant `index` on the current
 * device (register count, shared memory, occupancy).  Opts the kernel into
 * its dynamic shared memory as a launch would; launches nothing.
 * INVALID_ARG for a bad index, CUDA when a runtime query fails. */
int tiles_gemm_variant_info(int index, tiles_variant_info* out);

/* Workspace bytes that let this GEMM split its last round along K (256 when
 * it needs no split; 0 on invalid arguments, see tiles_last_error).  A
 * smaller workspace is accepted by the GEMM calls and changes only the
 * schedule.  A workspace serves one launch at a time. */
size_t tiles_gemm_workspace_bytes(const tiles_gemm_desc* desc, const tiles_config* cfg);

/* The batched form: desc->batch >= 1 equally shaped GEMMs with element
 * strides stride_a/b/c between items (each a multiple of 8 elements). */
int tiles_gemm_batched(const tiles_gemm_desc* desc, const tiles_config* cfg, void* workspace,
                       size_t ws_bytes, void* stream);

/* y = conv2d(x, w) as an implicit GEMM per output H-tile of tile_oh rows:
 * per image and tile, M = c_out, N = the tile's output pixels, K =
 * c*kh*kw, and each tile reads only its input slice [in_start, min(in_end,
 * H)) with the sub-operator pads pt'/pb' from tiles_htile_rows.
 *
 * Two producers build the im2col operand:
 *  - TMA (default when it applies: c % 8 == 0 and strides <= 8; needs
 *    tiles_conv_workspace_bytes() of workspace): TMA boxes of the input
 *    rows feed the MMA, the pads arriving as zero fill.  An NCHW input is
 *    read in place by the direct rows form (TILES_CONV_W_TMEM_ROWS_DIRECT:
 *    warps of the kernel transpose each stage's box into the operand); the
 *    forms that need NHWC rows transpose an NCHW input into the workspace
 *    first.  The filter is reordered to [c_out][r][s][c padded to 64] in the
 *    workspace, except a 3x3 filter over 64 channels bound for tensor
 *    memory, which the kernel builds from its OIHW rows;
 *  - gather (NCHW input only; c*kh*kw a multiple of 8): four warps gather
 *    the operand from global memory into shared memory.
 * With the TMA producer the filter sits in tensor memory as the MMA's A
 * operand when it fits (tiles_conv_weights), else in shared memory.
 * cfg == NULL picks the TMA producer when the workspace allows; a cfg with
 * threads 192 forces it (cfg->conv_weights then picks the filter's place:
 * TILES_ERR_INFEASIBLE when TMEM is asked for and it does not fit), threads
 * 320 forces the gather.  tile_oh >= 1. */
int tiles_conv2d_htiled(const tiles_conv_desc* desc, int tile_oh, const tiles_config* cfg,
                        void* workspace, size_t ws_bytes, void* stream);

/* The same convolution tiled over the batch, the output height and the
 * output width: output tiles of tile_n images x tile_oh rows x tile_ow
 * columns, each an independent sub-convolution of its input slice.  The
 * width's slices follow the same formulas as the rows (tutorial, "H/W 维切
 * 分的通用公式", applied to W, kw, sw, pw, dw); images need no halo, so a
 * batch tile is just fewer images (tutorial, "为什么教学工程先切 batch 维").
 * tile_ow <= 0 or >= the output width means one W-tile, tile_n <= 0 or >=
 * n one batch tile; tiles_conv2d_htiled(desc, t, ...) is
 * tiles_conv2d_tiled(desc, t, 0, 0, ...).  W-tiles narrower than the
 * output need the TMA producer (TILES_ERR_INFEASIBLE otherwise); tile_ow
 * and the pads must be below 32768.  For a given producer the tiling
 * changes no output bit: each output's K sum runs in the same order. */
int tiles_conv2d_tiled(const tiles_conv_desc* desc, int tile_oh, int tile_ow, int tile_n,
                       const tiles_config* cfg, void* workspace, size_t ws_bytes, void* stream);

/* ---- End to end from host memory ---------------------------------------
 * The same operations with their operands starting, and their results
 * ending, in host memory: the call a user with host data makes.  The source
 * pages have no counterpart (they state the operation on resident operands);
 * these calls add only the copies around the kernels above.
 *
 * The descriptor describes the caller's device buffers as for the device
 * calls; each host buffer mirrors its device buffer (the same layout, pitches
 * and batch strides).  Host buffers should be page-locked (cudaHostAlloc,
 * cudaHostRegister): pageable memory still works, but its copies do not
 * overlap anything.  The call enqueues, ordered after earlier work on
 * `stream`:
 *   - the operands that every piece needs (B of a single GEMM, the filter),
 *   - then, piece by piece (chunks pieces: runs of batch items or images, or
 *     for a single GEMM runs of rows of A and C rounded to whole tiles), the
 *     piece's inputs, its kernels as soon as they have landed, and its
 *     results back to the host as soon as the kernels are done.
 * Host-to-device and device-to-host copies run on two copy streams the
 * library creates on a host thread's first call on a device and releases
 * when that thread exits; the kernels run on `stream`, and work enqueued on
 * `stream` after the call starts once every result is in host memory.  No
 * device memory is allocated.  chunks is in 1 .. 16.  Calls that share
 * device buffers and overlap (different streams) race.  On an error some
 * pieces may already be enqueued, on the copy streams as well, and `stream`
 * is then not ordered after them: synchronize the device before reusing or
 * freeing the buffers.  The status is that of the first failing step
 * (tiles_last_error). */

/* tiles_gemm_batched from host buffers a_host, b_host to c_host. */
int tiles_gemm_host(const tiles_gemm_desc* desc, const tiles_config* cfg, const void* a_host,
                    const void* b_host, void* c_host, int chunks, void* workspace,
                    size_t ws_bytes, void* stream);

/* tiles_conv2d_htiled from host buffers x_host, w_host to y_host; the pieces
 * are runs of images.  The workspace must serve the whole batch (it then
 * serves every piece). */
int tiles_conv2d_host(const tiles_conv_desc* desc, int tile_oh, const tiles_config* cfg,
                      const void* x_host, const void* w_host, void* y_host, int chunks,
                      void* workspace, size_t ws_bytes, void* stream);

/* Output height and width of the convolution `desc` describes (only its
 * n/c/h/w, kernel, stride, pad and dilation fields are read):
 * oh = (h + 2*ph - (kh-1)*dh - 1) / sh + 1, and ow likewise, the output of
 * the direct convolution the H-tiles partition.  INVALID_ARG when a size is
 * out of range or no window fits. */
int tiles_conv_out_hw(const tiles_conv_desc* desc, int32_t* oh, int32_t* ow);

/* Workspace bytes the TMA producer needs for this convolution (256 when it
 * does not apply; 0 on invalid arguments). */
size_t tiles_conv_workspace_bytes(const tiles_conv_desc* desc, int tile_oh);

/* The GEMM of tiles_gemm_batched (batch >= 1) for callers that cannot
 * allocate device memory and so cannot pass a workspace.  The source pages
 * have no counterpart: it exists for code that runs where cudaMalloc is not
 * allowed (allocator or driver callbacks, runtimes that own all device
 * memory, paths that must not allocate).  Its scratch is a 256-byte static
 * device array in the library, held by every GPU that loads the library until
 * the process exits; the call allocates nothing and calls no allocating
 * routine.  The GEMM needs exactly that much (its timeout error word): the
 * last round of tiles never splits along K here (it runs as whole tiles or
 * N-halves), and a cfg that forces a K split, whose partial tiles would need
 * more, is rejected with TILES_ERR_TOO_LARGE.  Every call looks up the
 * array's device address (cudaGetSymbolAddress) on the current device, so
 * that it follows a device reset, after which the array loads at a new
 * address.  All calls share the array: a
 * timeout recorded by a call stays until a call with wait != 0 reads and
 * clears it, and calls that overlap on the GPU race on it.
 * wait == 0: asynchronous on `stream`, returns the launch status.
 * wait != 0: also synchronises `stream` and returns TILES_ERR_TIMEOUT if a
 * bounded wait expired in a call since the last read. */
int tiles_gemm_noalloc(const tiles_gemm_desc* desc, const tiles_config* cfg, void* stream,
                       int wait);

/* ---- Measured shortlist (tutorial, "自动调优": enumerate the tile
 * configurations, drop those that break a hardware constraint, time each
 * survivor on the target GPU, keep the fastest) ---------------------------- */

/* One timed candidate. */
typedef struct {
    tiles_config cfg;        /* the configuration; cfg.tail is the last-round schedule asked for */
    int32_t status;          /* TILES_OK, or why the candidate could not run (us is then 0) */
    int32_t tail_mode;       /* the schedule the launches used: 0 none needed, 1 N-halves, 2 K split */
    int32_t ksplit;          /* K parts of a split last round (1 otherwise) */
    float us;                /* time per launch, microseconds: the faster of two passes of
                                reps launches back to back, each pass's time over reps */
} tiles_tune_result;

/* Time the planner's top_k configurations (GB300 mode, in rank order) for
 * this GEMM, each with every last-round schedule it admits (the planner's
 * own choice first, then whole tiles, N-halves, a K split when the
 * workspace holds its partials; ties keep the earlier): one untimed
 * launch, then two passes of reps launches back to back, each between one
 * pair of CUDA events on `stream`; the faster pass's time over reps counts
 * (launches overlap their neighbours' set-up, so a launch has no time of
 * its own between events).  The fastest becomes the tuned configuration of the
 * problem (batch, m, n, k, dtypes, SM count), which tiles_gemm and
 * tiles_gemm_batched use when called with cfg == NULL; *best receives it.
 *
 * Runs the caller's GEMM (desc->c is overwritten) and synchronises
 * `stream`.  results (capacity entries, may be NULL) receives the
 * candidates in the order tried and *n_results their number.  1 <= top_k <=
 * 16, 1 <= reps <= 100.  TILES_ERR_INFEASIBLE when no candidate ran. */
int tiles_gemm_autotune(const tiles_gemm_desc* desc, int top_k, int reps, void* workspace,
                        size_t ws_bytes, void* stream, tiles_tune_result* results,
                        int capacity, int* n_results, tiles_config* best);

/* The tuned configuration of a problem: TILES_OK and *out filled when one
 * is recorded, TILES_ERR_INFEASIBLE when none is.  Host only. */
int tiles_tuned_lookup(int sm_count, int64_t batch, int64_t m, int64_t n, int64_t k, int in_dtype,
                       int out_dtype, tiles_config* out);

/* Write every tuned configuration to a text file: a header line, then one
 * line per problem with sm_count batch m n k in_dtype out_dtype bm bn bk
 * stages threads instr acc_bufs cta_group tail us.  Host only. */
int tiles_tuned_save(const char* path);

/* Merge the entries of a file written by tiles_tuned_save into the table.
 * A missing file or a malformed line returns TILES_ERR_INVALID_ARG and
 * merges nothing.  Host only. */
int tiles_tuned_load(const char* path);

/* Forget every tuned configuration.  Host only. */
int tiles_tuned_clear(void);

/* Synchronise `stream`, read and clear the workspace's error word:
 * TILES_OK, or TILES_ERR_TIMEOUT if a kernel's bounded wait expired. */
int tiles_check(void* workspace, void* stream);

/* Test hook for the timeout path: launches one block whose thread waits on
 * an mbarrier that nothing arrives at, bounded by limit_ns nanoseconds; the
 * wait expires and records a timeout in the workspace.  Returns the launch
 * status; tiles_check then reports TILES_ERR_TIMEOUT. */
int tiles_selftest_wait_timeout(void* workspace, int64_t limit_ns, void* stream);

/* Test hook for the kernels' own bounded waits (the production kernels,
 * not a separate one).  Arms, for the calling thread's next GEMM launch
 * (tiles_gemm, tiles_gemm_batched, tiles_gemm_noalloc) or next TMA
 * convolution launch (tiles_conv2d_htiled / _tiled with the TMA producer), a
 * planted fault: the first CTA group's TMA producer skips the loads and the
 * arrival of its `stage`-th pipeline stage (counted from 0 over the loads it
 * issues), so the stage's consumer waits on a barrier that never completes;
 * every wait of that launch gives up after limit_ns nanoseconds.  The
 * kernel then records the expiry in the workspace's error word (or the
 * no-alloc scratch), lets its other roles stop, waits for its own copies
 * and MMAs in flight, frees its tensor memory and returns; tiles_check
 * reports TILES_ERR_TIMEOUT and the context stays usable.  The other CTA
 * groups of the launch run normally.  The launch consumes the fault; stage
 * < 0 disarms it.  INVALID_ARG unless 0 < limit_ns <= 1e10. */
int tiles_selftest_drop_stage(int stage, int64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* TILES_H */
