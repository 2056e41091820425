// Persistent warp-specialised tcgen05 GEMM for sm_103a:
//   C[b] = A[b] x B[b],  A row-major M x K (K-major operand),
//                        B row-major K x N (MN-major operand),
//   fp16/bf16 inputs, fp32 accumulation in tensor memory, fp32/fp16/bf16 out.
//
// This is the tutorial's block-tiled GEMM ("Tiled 方法分块复用数据": one
// output tile per block, A and B slices staged on chip and reused by the
// whole tile) with its multi-stage pipeline ("Double Buffering /
// Multi-Stage Pipelining") and 128-byte swizzle ("Bank Conflict 与
// Swizzling"), rebuilt on Blackwell's TMA, mbarriers and tensor memory.
//
// CG = 1: one CTA per 128 x BN output tile.
// CG = 2: a CTA pair (cluster of 2) per 256 x BN tile.  Each CTA loads its
//         own 128 rows of A and BN/2 columns of B; both CTAs' loads complete
//         on the leader's (rank 0) full barrier; one thread of the leader
//         issues tcgen05.mma.cta_group::2 (M = 256), whose commits multicast
//         to both CTAs; each CTA's TMEM holds its 128 rows of the tile.
//         Per SM this halves B's share of the L2 -> shared traffic.
//
// Roles in each CTA (192 threads):
//   warp 0      TMA producer.
//   warp 1      TMEM owner; in the leader it issues the MMAs: 4 per stage
//               (K = 16 each), commits the stage back to the producers, and
//               commits a finished tile to the epilogues.
//   Both loops run on the whole warp, which keeps the loop state
//   warp-uniform, and one lane chosen by elect.sync issues the TMA, MMA and
//   commit instructions.  (The same loops run by a single lane made the
//   4096^3 GEMM 2.4% slower with a CTA pair and 6% slower with one CTA.)
//   warps 2-5   epilogue: warp w owns TMEM lanes 32*(w%4)..+31, i.e. 32
//               rows of the tile.  It reads them with tcgen05.ld, casts to
//               the output type and writes each 128-byte-wide column box
//               (32 fp32 or 64 16-bit columns) into its own swizzled 4 KB
//               staging box in shared memory, which one TMA store copies
//               to C, clipped at M and N.  Each lane's 16-byte writes land
//               in distinct banks, and the store leaves the L1 path free;
//               a C whose rows are not 16-byte multiples is written from
//               the registers instead.
//
// Work is scheduled persistently: CTA group g takes units g, g+groups, ...
// The units are the output tiles, except that when the last round would
// leave more than half the groups idle, its tiles are split into two
// N-halves each (the planner's C4 last-wave fill), which all run in that
// round.  Two TMEM accumulators let one unit's epilogue overlap the next
// unit's mainloop.  Every wait is bounded (mbar_wait); on expiry the kernel records
// the role in the workspace error word, lets the other roles stop, waits
// for its own asynchronous work and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"
#include "tiles_internal.h"

namespace tiles {

// Error bits written to the workspace's first word.
constexpr int kErrProducer = 1;
constexpr int kErrMma = 2;
constexpr int kErrEpilogue = 4;
constexpr int kErrSelftest = 8;
constexpr int kErrConvGather = 16;

struct GemmArgs {
    int32_t m, n, k, batch;
    int32_t m_blocks, n_blocks, k_blocks;
    int32_t tiles;             // batch * m_blocks * n_blocks
    int32_t group_m;           // tile order: groups of group_m M blocks (1 .. m_blocks)
    // Work units: units [0, full_units) are whole tiles.  The tiles after
    // them (the last, partly filled round) run by tail_mode:
    //   kTailNone   as whole tiles (units = tiles);
    //   kTailNHalf  as two N-halves each (units = full + 2 * rest);
    //   kTailKSplit as ksplit parts along K each (units = full + ksplit *
    //               rest): parts 0..ksplit-2 write fp32 partial tiles to
    //               `partials` and raise their flags; the last part adds them
    //               to its own accumulator in part order and stores C.
    int32_t full_units, units;
    int32_t tail_mode, ksplit;
    float* partials;           // kTailKSplit: [rest * (ksplit-1)][BN][BM] fp32
    uint32_t* flags;           // kTailKSplit: one per (tail tile, CTA, part, warp)
    uint32_t epoch;            // kTailKSplit: the flag value that means "ready"
    void* c;
    int64_t ldc, stride_c;     // elements
    int32_t c_dtype;           // tiles_dtype
    int32_t tma_store;         // 1: C leaves through TMA stores of staged boxes
    uint32_t idesc;            // tcgen05 instruction descriptor, N = BN
    uint32_t idesc_half;       // the same with N = BN / 2
    int32_t* err;              // workspace error word
    uint64_t wait_limit_ns;
    int32_t drop_stage;        // test hook: the first group skips this stage's loads (-1: none)
};

struct PipeBarriers {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(PipeBarriers) <= kSmemBarrierBytes, "barrier block too large");

template <int BN_, int STAGES_, int CG_>
struct GemmLayout {
    static constexpr int CG = CG_;
    static constexpr int BM = 128 * CG;                // output rows per tile
    static constexpr int BN = BN_, BK = 64, STAGES = STAGES_;
    static constexpr int B_COLS = BN / CG;            // B columns each CTA loads
    static constexpr int A_BYTES = 128 * BK * 2;       // 16 KB: 128 rows x 128 B
    static constexpr int B_CHUNK = BK * 64 * 2;        // 8 KB: 64 K-rows x 64 columns
    static constexpr int B_BYTES = B_CHUNK * (B_COLS / 64);
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;          // per CTA
    static constexpr int TX_BYTES = STAGE_BYTES * CG;              // on the leader's barrier
    static constexpr int OPERAND_BYTES = STAGES * STAGE_BYTES;
    // One staging box per epilogue warp: 32 rows x 128 bytes.
    static constexpr int EPI_BOX_BYTES = 32 * 128;
    static constexpr int STAGING_BYTES = 4 * EPI_BOX_BYTES;
    static constexpr int SMEM_BYTES =
        OPERAND_BYTES + STAGING_BYTES + kSmemBarrierBytes + kSmemAlignSlack;
    static constexpr int ACC_COLS = 2 * BN;
    static constexpr int TMEM_COLS = ACC_COLS <= 32 ? 32 : ACC_COLS <= 64 ? 64
                                   : ACC_COLS <= 128 ? 128 : ACC_COLS <= 256 ? 256 : 512;
    static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair");
    static_assert(B_COLS % 64 == 0 && BN <= 256, "B columns per CTA must be whole 64-column atoms");
    static_assert(STAGES >= 2 && STAGES <= kMaxStages, "stage count");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per block");
    // The last K part of a split tile stages one partial per epilogue warp
    // (32 rows x BN fp32) in the idle operand stages.
    static_assert(4 * 32 * BN * 4 <= OPERAND_BYTES, "partial staging must fit the stages");
    static_assert(STAGING_BYTES == kSmemEpilogueBytes, "the planner counts this staging");
    static_assert(OPERAND_BYTES % 1024 == 0, "staging boxes sit on the 128-byte swizzle's 1 KB atoms");
};

struct TileCoord { int b, mi, ni; };

__device__ __forceinline__ TileCoord decode_tile(int t, int m_blocks, int n_blocks, int group_m) {
    // Within a batch item the tiles go in groups of group_m M blocks: M
    // fastest inside a group (concurrent CTAs share B panels), then N, then
    // the next group (the groups keep the A panels of concurrent CTAs few
    // enough to stay in L2).  group_m == m_blocks is plain M-fastest order.
    const int per_batch = m_blocks * n_blocks;
    TileCoord c;
    c.b = t / per_batch;
    const int r = t - c.b * per_batch;
    const int span = group_m * n_blocks;
    const int g = r / span;
    const int first = g * group_m;
    const int rows = min(group_m, m_blocks - first);
    const int q = r - g * span;
    c.mi = first + q % rows;
    c.ni = q / rows;
    return c;
}

constexpr int kTailNone = 0;
constexpr int kTailNHalf = 1;
constexpr int kTailKSplit = 2;

// One work unit: a whole tile, one N-half of a last-round tile, or one K
// part of a last-round tile.
struct UnitCoord {
    int b, mi;
    int n0;        // first output column
    int width;     // columns: BN or BN / 2
    int kb0, kb1;  // K blocks [kb0, kb1)
    int part;      // K part (-1 unless split along K)
    int tail;      // index of the tile among the last round's tiles
};

template <int BN>
__device__ __forceinline__ UnitCoord decode_unit(int u, const GemmArgs& a) {
    int t = u, off = 0, width = BN, kb0 = 0, kb1 = a.k_blocks, part = -1, tail = -1;
    if (u >= a.full_units) {
        const int h = u - a.full_units;
        if (a.tail_mode == kTailNHalf) {
            t = a.full_units + (h >> 1);
            off = (h & 1) * (BN / 2);
            width = BN / 2;
        } else if (a.tail_mode == kTailKSplit) {
            tail = h / a.ksplit;
            part = h - tail * a.ksplit;
            t = a.full_units + tail;
            kb0 = part * a.k_blocks / a.ksplit;
            kb1 = (part + 1) * a.k_blocks / a.ksplit;
        }
    }
    const TileCoord tc = decode_tile(t, a.m_blocks, a.n_blocks, a.group_m);
    return UnitCoord{tc.b, tc.mi, tc.ni * BN + off, width, kb0, kb1, part, tail};
}

__device__ __forceinline__ void store_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t load_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait (bounded) until *flag == epoch; every lane polls with acquire
// semantics, and the warp agrees on the outcome.
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, uint32_t epoch,
                                          const volatile int* abort, uint64_t limit_ns) {
    bool ok = load_acquire_gpu(flag) == epoch;
    if (!__all_sync(0xffffffffu, ok)) {
        const uint64_t t0 = ptx::globaltimer_ns();
        for (;;) {
            ok = load_acquire_gpu(flag) == epoch;
            if (__all_sync(0xffffffffu, ok)) break;
            if (__any_sync(0xffffffffu, *abort != 0 || ptx::globaltimer_ns() - t0 > limit_ns))
                return false;
            __nanosleep(256);
        }
    }
    return true;
}

__device__ __forceinline__ void raise_error(int32_t* err, volatile int* abort, int bit) {
    *abort = 1;
    if (err) atomicOr(err, bit);
}

// After an abort, loads or commits this CTA issued may still be in flight:
// hold the block for a fixed, short interval before it may exit.
__device__ __forceinline__ void settle_after_abort() {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < 100000ull) {
    }
}

// Store 32 consecutive fp32 accumulators of one row, cast to the output type,
// clipped at column n.  `row` points at the row's first element.  With
// vec, full chunks use 16-byte stores (the caller guarantees alignment).
__device__ __forceinline__ void store_row_chunk(void* row, int64_t col0, int64_t n,
                                                const uint32_t (&v)[32], int dtype,
                                                bool vec = true) {
    if (dtype == TILES_F32) {
        float* p = static_cast<float*>(row) + col0;
        if (vec && col0 + 32 <= n) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                float4 q = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                       __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                *reinterpret_cast<float4*>(p + i) = q;
            }
        } else {
            for (int i = 0; i < 32; ++i)
                if (col0 + i < n) p[i] = __uint_as_float(v[i]);
        }
    } else if (dtype == TILES_F16) {
        __half* p = static_cast<__half*>(row) + col0;
        uint32_t h[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            __half2 t = __floats2half2_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            h[i] = *reinterpret_cast<uint32_t*>(&t);
        }
        if (vec && col0 + 32 <= n) {
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<uint4*>(p + 2 * i) = make_uint4(h[i], h[i + 1], h[i + 2], h[i + 3]);
        } else {
            for (int i = 0; i < 32; ++i)
                if (col0 + i < n)
                    p[i] = __ushort_as_half(static_cast<unsigned short>(h[i >> 1] >> ((i & 1) * 16)));
        }
    } else {
        __nv_bfloat16* p = static_cast<__nv_bfloat16*>(row) + col0;
        uint32_t h[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 t =
                __floats2bfloat162_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            h[i] = *reinterpret_cast<uint32_t*>(&t);
        }
        if (vec && col0 + 32 <= n) {
#pragma unroll
            for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<uint4*>(p + 2 * i) = make_uint4(h[i], h[i + 1], h[i + 2], h[i + 3]);
        } else {
            for (int i = 0; i < 32; ++i)
                if (col0 + i < n)
                    p[i] = __ushort_as_bfloat16(static_cast<unsigned short>(h[i >> 1] >> ((i & 1) * 16)));
        }
    }
}

// Two fp32 accumulators as one packed pair of the 16-bit output type.
__device__ __forceinline__ uint32_t pack_f16x2(uint32_t lo, uint32_t hi) {
    __half2 t = __floats2half2_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<uint32_t*>(&t);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<uint32_t*>(&t);
}

__device__ __forceinline__ uint32_t pack_pair(float lo, float hi, bool f16) {
    if (f16) {
        __half2 t = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&t);
    }
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}

// Write one 128-byte row (w[0..31]) of a 32-row staging box in the 128-byte
// swizzled layout a SWIZZLE_128B tensor map reads: 16-byte piece q of row r
// sits at piece position q ^ (r % 8).  With one row per lane, the eight
// lanes of each quarter-warp store phase hit eight different bank groups.
__device__ __forceinline__ void stage_box_row(uint32_t box, int row, const uint32_t (&w)[32]) {
    const uint32_t r = box + static_cast<uint32_t>(row) * 128u;
#pragma unroll
    for (int q = 0; q < 8; ++q)
        ptx::st_shared_v4(r + (static_cast<uint32_t>(q ^ (row & 7)) << 4), w[4 * q], w[4 * q + 1],
                          w[4 * q + 2], w[4 * q + 3]);
}

template <int BN, int STAGES, int CG>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
    using L = GemmLayout<BN, STAGES, CG>;
    extern __shared__ uint8_t smem_raw[];
    // Operand tiles start on a 1024-byte boundary: the 128-byte swizzle is a
    // function of address bits 4-9 and the descriptors assume base offset 0.
    // The offset is the same in both CTAs of a pair (same kernel, same
    // dynamic shared memory), as the pair MMA requires.
    const uint32_t raw = ptx::smem_addr(smem_raw);
    uint8_t* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* smA = base;
    uint8_t* smB = base + STAGES * L::A_BYTES;
    uint8_t* staging = base + L::OPERAND_BYTES;
    PipeBarriers* bar = reinterpret_cast<PipeBarriers*>(staging + L::STAGING_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = CG == 2 ? ptx::cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int group = CG == 2 ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
    const int groups = CG == 2 ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&bar->full[s], 1);
            ptx::mbar_init(&bar->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&bar->acc_full[a], 1);
            ptx::mbar_init(&bar->acc_empty[a], 4 * CG);   // every epilogue warp of the group
        }
        ptx::mbar_init(&bar->drain, 1);
        bar->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&tmA);
        ptx::tma_prefetch_desc(&tmB);
        if (args.tma_store) ptx::tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(&bar->tmem_base, L::TMEM_COLS);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before();
    if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after();
    // The previous kernel on the stream may still be draining (programmatic
    // serialization): nothing global is read or written before it has
    // completed.  Every block of this grid is resident from here on, so the
    // next kernel on the stream may start its own set-up on SMs as they free.
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    const uint32_t tmem = bar->tmem_base;
    volatile int* abort = &bar->abort;
    const uint64_t limit = args.wait_limit_ns;

    if (warp == 0) {
        {
            // ---------------- TMA producer (whole warp; one elected lane issues) ----------------
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool aborted = false;
            for (int u = group; u < args.units && !aborted; u += groups) {
                const UnitCoord uc = decode_unit<BN>(u, args);
                const int row0 = uc.mi * L::BM + static_cast<int>(rank) * 128;
                const int bcols = uc.width / CG;             // B columns this CTA loads
                const int col0 = uc.n0 + static_cast<int>(rank) * bcols;
                const int atoms = bcols / 64;
                const uint32_t tx = static_cast<uint32_t>(L::A_BYTES + atoms * L::B_CHUNK) * CG;
                for (int kb = uc.kb0; kb < uc.kb1; ++kb) {
                    const bool ok = __all_sync(0xffffffffu,
                        ptx::mbar_wait(&bar->empty[stage], phase ^ 1u, abort, limit));
                    if (!ok) {
                        if (lane == 0) raise_error(args.err, abort, kErrProducer);
                        aborted = true;
                        break;
                    }
                    uint8_t* a_dst = smA + stage * L::A_BYTES;
                    uint8_t* b_dst = smB + stage * L::B_BYTES;
                    // A planted fault (test hook): both CTAs of the first
                    // group skip the same stage, so its full barrier never
                    // completes and the MMA issuer's bounded wait expires.
                    const bool planted = group == 0 && issued == args.drop_stage;
                    if (!planted && ptx::elect_one_sync()) {
                        if (leader) ptx::mbar_arrive_expect_tx(&bar->full[stage], tx);
                        if constexpr (CG == 1) {
                            ptx::tma_load_3d(a_dst, &tmA, &bar->full[stage], kb * L::BK, row0, uc.b);
                            for (int j = 0; j < atoms; ++j)
                                ptx::tma_load_3d(b_dst + j * L::B_CHUNK, &tmB, &bar->full[stage],
                                                 col0 + j * 64, kb * L::BK, uc.b);
                        } else {
                            const uint32_t fb = ptx::map_to_cta(ptx::smem_addr(&bar->full[stage]), 0);
                            ptx::tma_load_3d_pair(a_dst, &tmA, fb, kb * L::BK, row0, uc.b);
                            for (int j = 0; j < atoms; ++j)
                                ptx::tma_load_3d_pair(b_dst + j * L::B_CHUNK, &tmB, fb, col0 + j * 64,
                                                      kb * L::BK, uc.b);
                        }
                    }
                    __syncwarp();
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (aborted) {
                settle_after_abort();
            } else if (CG == 1) {
                // Every load landed before its stage was consumed; waiting on
                // the last (up to STAGES) full barriers is then immediate.
                for (int i = 0; i < (issued < STAGES ? issued : STAGES); ++i) {
                    if (stage == 0) { stage = STAGES - 1; phase ^= 1u; } else { --stage; }
                    ptx::mbar_wait(&bar->full[stage], phase, nullptr, limit);
                }
            }
        }
    } else if (warp == 1) {
        if (leader) {
            // ---------------- MMA issuer (leader CTA; whole warp, one elected lane issues) ----------------
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            // Descriptors of stage 0's operands; a stage or K step moves the
            // start-address field (address >> 4, 14 bits: shared-memory
            // addresses stay below 256 KB, so the sums never carry out).
            //  A, K-major: 16 K elements = 32 bytes inside the 128-byte
            //  swizzle row; 8-row groups 1024 B apart.
            //  B, MN-major: 16 K rows = two 8-row groups of 1024 B; 64-column
            //  atoms B_CHUNK apart.
            const uint64_t a_desc0 = ptx::smem_desc_sw128(ptx::smem_addr(smA), 16, 1024);
            const uint64_t b_desc0 = ptx::smem_desc_sw128(ptx::smem_addr(smB), L::B_CHUNK, 1024);
            // The same lane issues every MMA and commit: a commit tracks the
            // MMAs of the thread that issues it.
            const bool issuer = ptx::elect_one_sync();
            for (int u = group; u < args.units; u += groups) {
                const UnitCoord uc = decode_unit<BN>(u, args);
                const uint32_t idesc = uc.width == BN ? args.idesc : args.idesc_half;
                if (!__all_sync(0xffffffffu,
                                ptx::mbar_wait(&bar->acc_empty[acc], acc_phase ^ 1u, abort, limit))) {
                    if (lane == 0) raise_error(args.err, abort, kErrMma);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                bool ok = true;
                for (int kb = uc.kb0; kb < uc.kb1; ++kb) {
                    if (!__all_sync(0xffffffffu,
                                    ptx::mbar_wait(&bar->full[stage], phase, abort, limit))) {
                        if (lane == 0) raise_error(args.err, abort, kErrMma);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t a_st = a_desc0 + ((stage * L::A_BYTES) >> 4);
                    const uint64_t b_st = b_desc0 + ((stage * L::B_BYTES) >> 4);
                    if (issuer) {
#pragma unroll
                        for (int kk = 0; kk < L::BK / 16; ++kk)
                            ptx::mma_f16<CG>(d, a_st + kk * (32 >> 4), b_st + kk * (2048 >> 4), idesc,
                                             (kb != uc.kb0 || kk != 0) ? 1u : 0u);
                        ptx::mma_commit<CG>(&bar->empty[stage]);
                    }
                    __syncwarp();
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (issuer) ptx::mma_commit<CG>(&bar->acc_full[acc]);
                __syncwarp();
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            // Every MMA issued here completes before the group tears down.
            if (issuer) {
                ptx::mma_commit_local<CG>(&bar->drain);
                ptx::mbar_wait(&bar->drain, 0, nullptr, limit);
            }
            __syncwarp();
        }
    } else {
        // ---------------- epilogue (warps 2-5) ----------------
        const int quarter = warp & 3;               // TMEM lanes this warp may read
        const int row_in_tile = quarter * 32 + lane;
        const int out_bytes = args.c_dtype == TILES_F32 ? 4 : 2;
        uint8_t* box_ptr = staging + quarter * L::EPI_BOX_BYTES;
        const uint32_t box = ptx::smem_addr(box_ptr);
        // One 128-byte-wide box of the warp's 32 rows (w: this lane's row)
        // goes to C at column x through the staging box.  Lane 0 issues
        // every store, so its bulk groups track them all.
        auto store_box = [&](const uint32_t (&w)[32], int x, int row0, int b) {
            // The previous box's store has finished reading the staging box.
            if (lane == 0) ptx::bulk_wait_read_all();
            __syncwarp();
            stage_box_row(box, lane, w);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && x < args.n && row0 < args.m) {
                ptx::tma_store_3d(&tmC, box_ptr, x, row0, b);
                ptx::bulk_commit_group();
            }
        };
        // Whole 128-byte boxes: 32 fp32 or 64 16-bit columns.
        const int per_box = out_bytes == 4 ? 1 : 2;
        uint32_t acc = 0, acc_phase = 0;
        for (int u = group; u < args.units; u += groups) {
            const UnitCoord uc = decode_unit<BN>(u, args);
            bool ok = ptx::mbar_wait(&bar->acc_full[acc], acc_phase, abort, limit);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) raise_error(args.err, abort, kErrEpilogue);
                break;
            }
            ptx::tc_fence_after();
            const int64_t row = static_cast<int64_t>(uc.mi) * L::BM + rank * 128 + row_in_tile;
            const int box_row0 = uc.mi * L::BM + static_cast<int>(rank) * 128 + quarter * 32;
            const bool row_ok = row < args.m;
            char* crow = static_cast<char*>(args.c) +
                         (static_cast<int64_t>(uc.b) * args.stride_c + row * args.ldc) * out_bytes;
            const uint32_t tacc = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
            // Partial tiles are column-major [BN][BM] so that a warp's 32
            // rows of one column are 128 contiguous bytes.
            const int64_t tile_elems = static_cast<int64_t>(L::BM) * BN;
            const int prow = static_cast<int>(rank) * 128 + row_in_tile;
            if (uc.part >= 0 && uc.part < args.ksplit - 1) {
                // A leading K part: hand the fp32 partial tile to the last part.
                float* dst = args.partials +
                             (static_cast<int64_t>(uc.tail) * (args.ksplit - 1) + uc.part) * tile_elems;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld_32cols(tacc + c * 32, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        dst[static_cast<int64_t>(c * 32 + i) * L::BM + prow] = __uint_as_float(v[i]);
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) {
                    uint32_t* f = args.flags +
                                  ((static_cast<int64_t>(uc.tail) * CG + rank) * (args.ksplit - 1) +
                                   uc.part) * 4 + quarter;
                    store_release_gpu(f, args.epoch);
                }
            } else if (uc.part >= 0) {
                // The last K part: wait for the leading parts, then add each
                // partial into the accumulator.  This is the group's last
                // unit, so its operand shared memory is idle: each warp
                // stages its 32 rows of one partial there (32 KB, all copies
                // in flight at once) as [column][32 rows] -- conflict-free
                // reads -- and adds them into TMEM; after the last partial it
                // casts and stores C.
                bool ready = true;
                for (int j = 0; j < args.ksplit - 1 && ready; ++j) {
                    const uint32_t* f = args.flags +
                        ((static_cast<int64_t>(uc.tail) * CG + rank) * (args.ksplit - 1) + j) * 4 +
                        quarter;
                    ready = wait_flag(f, args.epoch, abort, limit);
                }
                if (!ready && lane == 0) raise_error(args.err, abort, kErrEpilogue);
                float* stage_buf = reinterpret_cast<float*>(base) + quarter * (BN * 32);
                for (int j = 0; j < args.ksplit - 1 && ready; ++j) {
                    const float* src = args.partials +
                        (static_cast<int64_t>(uc.tail) * (args.ksplit - 1) + j) * tile_elems +
                        static_cast<int64_t>(rank) * 128 + quarter * 32;
#pragma unroll 4
                    for (int i = 0; i < BN * 8 / 32; ++i) {
                        const int piece = i * 32 + lane;          // 16-byte piece of the slice
                        const int col = piece >> 3, seg = piece & 7;
                        ptx::cp_async_16(stage_buf + col * 32 + seg * 4,
                                         src + static_cast<int64_t>(col) * L::BM + seg * 4);
                    }
                    ptx::cp_async_wait_all();
                    __syncwarp();
                    const bool last = j == args.ksplit - 2;
                    if (last && args.tma_store) {
                        // The last partial's sums leave box by box.
                        const bool f16 = args.c_dtype == TILES_F16;
#pragma unroll 1
                        for (int c = 0; c < BN / 32; c += per_box) {
                            uint32_t w[32];
                            const float* p0 = stage_buf + c * 32 * 32 + lane;   // column c*32+i at p0[32*i]
                            if (per_box == 1) {
                                ptx::tmem_ld_32cols(tacc + c * 32, w);
                                ptx::tmem_ld_wait();
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    w[i] = __float_as_uint(__uint_as_float(w[i]) + p0[32 * i]);
                            } else {
                                uint32_t v0[32], v1[32];
                                ptx::tmem_ld_32cols(tacc + c * 32, v0);
                                ptx::tmem_ld_32cols(tacc + c * 32 + 32, v1);
                                ptx::tmem_ld_wait();
                                const float* p1 = p0 + 32 * 32;
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    w[i] = pack_pair(__uint_as_float(v0[2 * i]) + p0[32 * (2 * i)],
                                                     __uint_as_float(v0[2 * i + 1]) + p0[32 * (2 * i + 1)],
                                                     f16);
                                    w[16 + i] = pack_pair(__uint_as_float(v1[2 * i]) + p1[32 * (2 * i)],
                                                          __uint_as_float(v1[2 * i + 1]) + p1[32 * (2 * i + 1)],
                                                          f16);
                                }
                            }
                            store_box(w, uc.n0 + c * 32, box_row0, uc.b);
                        }
                    } else {
#pragma unroll 1
                        for (int c = 0; c < BN / 32; ++c) {
                            uint32_t v[32];
                            ptx::tmem_ld_32cols(tacc + c * 32, v);
                            ptx::tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                v[i] = __float_as_uint(__uint_as_float(v[i]) +
                                                       stage_buf[(c * 32 + i) * 32 + lane]);
                            if (!last) {
                                ptx::tmem_st_32cols(tacc + c * 32, v);
                                ptx::tmem_st_wait();
                            } else if (row_ok) {
                                store_row_chunk(crow, static_cast<int64_t>(uc.n0) + c * 32, args.n, v,
                                                args.c_dtype);
                            }
                        }
                    }
                    __syncwarp();
                }
            } else {
                int c = 0;                                  // next 32-column TMEM chunk
                if (args.tma_store) {
                    const int boxes = uc.width / (32 * per_box);
#pragma unroll 1
                    for (int j = 0; j < boxes; ++j, c += per_box) {
                        uint32_t w[32];
                        if (per_box == 1) {
                            ptx::tmem_ld_32cols(tacc + c * 32, w);
                            ptx::tmem_ld_wait();
                        } else {
                            uint32_t v0[32], v1[32];
                            ptx::tmem_ld_32cols(tacc + c * 32, v0);
                            ptx::tmem_ld_32cols(tacc + c * 32 + 32, v1);
                            ptx::tmem_ld_wait();
                            if (args.c_dtype == TILES_F16) {
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    w[i] = pack_f16x2(v0[2 * i], v0[2 * i + 1]);
                                    w[16 + i] = pack_f16x2(v1[2 * i], v1[2 * i + 1]);
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    w[i] = pack_bf16x2(v0[2 * i], v0[2 * i + 1]);
                                    w[16 + i] = pack_bf16x2(v1[2 * i], v1[2 * i + 1]);
                                }
                            }
                        }
                        store_box(w, uc.n0 + c * 32, box_row0, uc.b);
                    }
                }
                // Register stores: the whole unit when C has no store map,
                // else the 32 columns a 16-bit box could not take (no
                // compiled unit width leaves any).
#pragma unroll 1
                for (; c < uc.width / 32; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld_32cols(tacc + c * 32, v);
                    ptx::tmem_ld_wait();
                    if (row_ok)
                        store_row_chunk(crow, static_cast<int64_t>(uc.n0) + c * 32, args.n, v,
                                        args.c_dtype);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 1)
                    ptx::mbar_arrive(&bar->acc_empty[acc]);
                else
                    ptx::mbar_arrive_cluster(ptx::map_to_cta(ptx::smem_addr(&bar->acc_empty[acc]), 0));
            }
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        // The staging boxes are free once the stores have read them; their
        // writes to C complete with the grid, before anything that waits
        // for it (a later kernel, or griddepcontrol.wait) reads C.
        if (lane == 0) ptx::bulk_wait_read_all();
        __syncwarp();
    }

    ptx::tc_fence_before();
    if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc<CG>(tmem, L::TMEM_COLS);
    }
}

// Host-side launch of one compiled variant (defined per (BN, CG) in
// gemm_sm103a.cu).  `groups` is the number of persistent CTA groups.
// Returns a cudaError_t value.
template <int BN, int CG>
int launch_gemm_variant(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                        const GemmArgs& args, int groups, cudaStream_t stream);

// Persistent CTA groups that fit on the device at once for a variant.
template <int BN, int CG>
int gemm_variant_max_groups(int sm_count);

// What the CUDA runtime reports for one compiled variant on the current
// device (defined per (BN, CG) in gemm_sm103a.cu).
struct VariantAttributes {
    int regs;               // registers per thread
    int local_bytes;        // local memory per thread (spills)
    int static_smem;        // static shared memory per block
    int dynamic_smem;       // dynamic shared memory a launch requests
    int max_dynamic_smem;   // the opted-in dynamic shared-memory limit
    int blocks_per_sm;      // resident blocks per SM at that shared memory
    int groups;             // resident CTA groups (clusters for CTA pairs)
};

// Fills *out; returns a cudaError_t value.
template <int BN, int CG>
int gemm_variant_attributes(int sm_count, VariantAttributes* out);

// Stages compiled for each (BN, CG) (the planner's kGemmVariants agree).
template <int BN, int CG> struct GemmStages;
template <> struct GemmStages<64, 1>  { static constexpr int value = 8; };
template <> struct GemmStages<128, 1> { static constexpr int value = 6; };
template <> struct GemmStages<192, 1> { static constexpr int value = 5; };
template <> struct GemmStages<256, 1> { static constexpr int value = 4; };
template <> struct GemmStages<128, 2> { static constexpr int value = 8; };
template <> struct GemmStages<256, 2> { static constexpr int value = 6; };

__global__ void selftest_wait_kernel(int32_t* err, uint64_t limit_ns);

}  // namespace tiles
