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
//   warp 0      TMA producer (one lane).
//   warp 1      TMEM owner; in the leader one lane issues the MMAs: 4 per
//               stage (K = 16 each), commits the stage back to the
//               producers, and commits a finished tile to the epilogues.
//   warps 2-5   epilogue: tcgen05.ld 32 columns at a time, cast, store the
//               rows they own (warp w reads TMEM lanes 32*(w%4)..+31).
//
// Tiles are scheduled persistently: CTA group g takes tiles g, g+groups, ...
// Two TMEM accumulators let one tile's epilogue overlap the next tile's
// mainloop.  Every wait is bounded (mbar_wait); on expiry the kernel records
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
    void* c;
    int64_t ldc, stride_c;     // elements
    int32_t c_dtype;           // tiles_dtype
    uint32_t idesc;            // tcgen05 instruction descriptor
    int32_t* err;              // workspace error word, may be null
    uint64_t wait_limit_ns;
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
    static constexpr int SMEM_BYTES = OPERAND_BYTES + kSmemBarrierBytes + kSmemAlignSlack;
    static constexpr int ACC_COLS = 2 * BN;
    static constexpr int TMEM_COLS = ACC_COLS <= 32 ? 32 : ACC_COLS <= 64 ? 64
                                   : ACC_COLS <= 128 ? 128 : ACC_COLS <= 256 ? 256 : 512;
    static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair");
    static_assert(B_COLS % 64 == 0 && BN <= 256, "B columns per CTA must be whole 64-column atoms");
    static_assert(STAGES >= 2 && STAGES <= kMaxStages, "stage count");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per block");
};

struct TileCoord { int b, mi, ni; };

__device__ __forceinline__ TileCoord decode_tile(int t, int m_blocks, int n_blocks) {
    const int per_batch = m_blocks * n_blocks;
    TileCoord c;
    c.b = t / per_batch;
    const int r = t - c.b * per_batch;
    c.mi = r % m_blocks;        // M fastest: concurrent CTAs share B panels
    c.ni = r / m_blocks;
    return c;
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

template <int BN, int STAGES, int CG>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
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
    PipeBarriers* bar = reinterpret_cast<PipeBarriers*>(base + L::OPERAND_BYTES);

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
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(&bar->tmem_base, L::TMEM_COLS);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before();
    if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after();

    const uint32_t tmem = bar->tmem_base;
    volatile int* abort = &bar->abort;
    const uint64_t limit = args.wait_limit_ns;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool aborted = false;
            for (int t = group; t < args.tiles && !aborted; t += groups) {
                const TileCoord tc = decode_tile(t, args.m_blocks, args.n_blocks);
                const int row0 = tc.mi * L::BM + static_cast<int>(rank) * 128;
                const int col0 = tc.ni * BN + static_cast<int>(rank) * L::B_COLS;
                for (int kb = 0; kb < args.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(&bar->empty[stage], phase ^ 1u, abort, limit)) {
                        raise_error(args.err, abort, kErrProducer);
                        aborted = true;
                        break;
                    }
                    if (leader) ptx::mbar_arrive_expect_tx(&bar->full[stage], L::TX_BYTES);
                    uint8_t* a_dst = smA + stage * L::A_BYTES;
                    uint8_t* b_dst = smB + stage * L::B_BYTES;
                    if constexpr (CG == 1) {
                        ptx::tma_load_3d(a_dst, &tmA, &bar->full[stage], kb * L::BK, row0, tc.b);
#pragma unroll
                        for (int j = 0; j < L::B_COLS / 64; ++j)
                            ptx::tma_load_3d(b_dst + j * L::B_CHUNK, &tmB, &bar->full[stage],
                                             col0 + j * 64, kb * L::BK, tc.b);
                    } else {
                        const uint32_t fb = ptx::map_to_cta(ptx::smem_addr(&bar->full[stage]), 0);
                        ptx::tma_load_3d_pair(a_dst, &tmA, fb, kb * L::BK, row0, tc.b);
#pragma unroll
                        for (int j = 0; j < L::B_COLS / 64; ++j)
                            ptx::tma_load_3d_pair(b_dst + j * L::B_CHUNK, &tmB, fb, col0 + j * 64,
                                                  kb * L::BK, tc.b);
                    }
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
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (leader CTA) ----------------
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            for (int t = group; t < args.tiles; t += groups) {
                if (!ptx::mbar_wait(&bar->acc_empty[acc], acc_phase ^ 1u, abort, limit)) {
                    raise_error(args.err, abort, kErrMma);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                bool ok = true;
                for (int kb = 0; kb < args.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(&bar->full[stage], phase, abort, limit)) {
                        raise_error(args.err, abort, kErrMma);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a0 = ptx::smem_addr(smA + stage * L::A_BYTES);
                    const uint32_t b0 = ptx::smem_addr(smB + stage * L::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < L::BK / 16; ++kk) {
                        // A, K-major: 16 K elements = 32 bytes inside the
                        // 128-byte swizzle row; 8-row groups 1024 B apart.
                        const uint64_t ad = ptx::smem_desc_sw128(a0 + kk * 32, 16, 1024);
                        // B, MN-major: 16 K rows = two 8-row groups of
                        // 1024 B; 64-column atoms B_CHUNK apart.
                        const uint64_t bd = ptx::smem_desc_sw128(b0 + kk * 2048, L::B_CHUNK, 1024);
                        ptx::mma_f16<CG>(d, ad, bd, args.idesc, (kb | kk) != 0);
                    }
                    ptx::mma_commit<CG>(&bar->empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit<CG>(&bar->acc_full[acc]);
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            // Every MMA issued here completes before the group tears down.
            ptx::mma_commit_local<CG>(&bar->drain);
            ptx::mbar_wait(&bar->drain, 0, nullptr, limit);
        }
    } else {
        // ---------------- epilogue (warps 2-5) ----------------
        const int quarter = warp & 3;               // TMEM lanes this warp may read
        const int row_in_tile = quarter * 32 + lane;
        const int out_bytes = args.c_dtype == TILES_F32 ? 4 : 2;
        uint32_t acc = 0, acc_phase = 0;
        for (int t = group; t < args.tiles; t += groups) {
            const TileCoord tc = decode_tile(t, args.m_blocks, args.n_blocks);
            bool ok = ptx::mbar_wait(&bar->acc_full[acc], acc_phase, abort, limit);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) raise_error(args.err, abort, kErrEpilogue);
                break;
            }
            ptx::tc_fence_after();
            const int64_t row = static_cast<int64_t>(tc.mi) * L::BM + rank * 128 + row_in_tile;
            const bool row_ok = row < args.m;
            char* crow = static_cast<char*>(args.c) +
                         (static_cast<int64_t>(tc.b) * args.stride_c + row * args.ldc) * out_bytes;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                ptx::tmem_ld_32cols(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN + c * 32, v);
                ptx::tmem_ld_wait();
                if (row_ok)
                    store_row_chunk(crow, static_cast<int64_t>(tc.ni) * BN + c * 32, args.n, v,
                                    args.c_dtype);
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
int launch_gemm_variant(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& args,
                        int groups, cudaStream_t stream);

// Persistent CTA groups that fit on the device at once for a variant.
template <int BN, int CG>
int gemm_variant_max_groups(int sm_count);

// Stages compiled for each (BN, CG) (the planner's kGemmVariants agree).
template <int BN, int CG> struct GemmStages;
template <> struct GemmStages<64, 1>  { static constexpr int value = 8; };
template <> struct GemmStages<128, 1> { static constexpr int value = 7; };
template <> struct GemmStages<192, 1> { static constexpr int value = 5; };
template <> struct GemmStages<256, 1> { static constexpr int value = 4; };
template <> struct GemmStages<128, 2> { static constexpr int value = 8; };
template <> struct GemmStages<256, 2> { static constexpr int value = 7; };

__global__ void selftest_wait_kernel(int32_t* err, uint64_t limit_ns);

}  // namespace tiles
