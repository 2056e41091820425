// H-tiled convolution with a TMA-built im2col operand (sm_103a).
//
// With the input channels innermost (NHWC), one filter tap (r, s) and 64
// input channels of the im2col matrix are a plain 4-D tile of the input:
//     X[p][(r, s, ci)] = x[n][ih0 + rr*sh][iw0 + cc*sw][ci],  p = rr*OWc + cc,
// which a TMA box {64 channels, OWc*sw columns, nr*sh rows, 1 image} with
// element strides {1, sw, sh, 1} loads as 128-byte pixel rows: a K-major,
// 128-byte-swizzled MMA operand.  Rows and columns outside the image (the
// pads) arrive as zeros.  The row coordinate of each output H-tile comes
// from its slice, ih0 = in_start - pt' + ..., the tiling tutorial's
// "H/W 维切分的通用公式".
//
// The GEMM per tile is Y^T = X * W^T: M = 128 output pixels (nr rows x OWc
// columns of one H-tile), N = a block of output channels, K = (r, s, ci).
// With pixels on the TMEM lanes, each epilogue thread owns one pixel and
// holds consecutive output channels, so for every channel a warp stores 32
// neighbouring pixels of one NCHW output plane: coalesced stores.
//
// The weights are reordered once per call to [c_out][r][s][C padded to 64]
// (the K-major operand in the same K order) in the caller's workspace,
// except a 3x3 filter over 64 channels bound for tensor memory, which the
// kernel builds from its OIHW rows.  An NCHW input is read in place by the
// direct rows form (its warps transpose each stage's TMA box of input rows
// into the operand); the other forms read NHWC rows, so for them an NCHW
// input is first transposed to NHWC in the workspace.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <cudaTypedefs.h>

#include "conv_sm103a.cuh"
#include "gemm_sm103a.cuh"

namespace tiles {

namespace {

constexpr int kTmaConvMaxN = 256;     // output channels per tile (MMA N)
constexpr int kTmaConvPixels = 128;   // output pixels per tile (MMA M)
// Per stage: 128 pixel rows of 128 bytes (A), then the weight rows (B).
constexpr int kTmaConvA = kTmaConvPixels * 128;
constexpr int kTmaConvTmemCols = 2 * kTmaConvMaxN;

struct ConvTmaArgs {
    void* y;
    int32_t n, c, h, w, c_out, kh, kw, sh, sw, pw, dh, dw, oh, ow;
    int32_t owc, nr;                      // pixel tile: nr rows x owc columns (= 128)
    int32_t nco;                          // output channels per tile (MMA N)
    int32_t rblocks, cblocks, co_blocks, ch_blocks, k_blocks, n_htiles, units;
    int32_t n_wtiles;                     // W-tiles in this launch (cblocks column blocks each)
    int32_t img0;                         // first image of this launch's batch tile
    uint32_t tx_bytes;                    // bytes the boxes of a stage deliver
    int32_t vec_ok;                       // 16-byte output stores are aligned (OW % 8 == 0)
    int32_t w_resident;                   // weights loaded once into shared memory
    uint32_t w_bytes;                     // resident weights: all K blocks x nco rows
    int32_t out_dtype;
    uint32_t idesc;
    int32_t* err;
    uint64_t wait_limit_ns;
    int32_t drop_stage;                   // test hook: CTA 0 skips this input load (-1: none)
    // Weights in tensor memory (conv_wtmem_kernel): the reordered weights,
    // their row length kh*kw*Cp, the pixels of a tile (MMA N), the first
    // TMEM column of the weights (after the accumulators) and the shared-
    // memory layout.
    const uint16_t* wr;
    int32_t kp, npix, a_col;
    int32_t acc_bufs;                     // TMEM accumulators (1 or 2)
    int32_t stages;                       // pixel-box ring depth
    int32_t stg_off, stg_pitch;           // staging tile: offset and row pitch (bytes)
    int32_t bar_off;                      // barrier block offset (bytes)
    int32_t w_slots;                      // 16 KB filter blocks per start-up pass
    int32_t stage_b;                      // bytes of one ring stage
    // Rows form (conv_wtmem_kernel<true>): a stage is one kernel row r and
    // 64 channels; its n_planes stride phases of the input row hold pmax
    // pixels each, plane_bytes apart; tap s reads plane tap_plane[s] from
    // pixel tap_shift[s] on.  k_stages = kh * ch_blocks (else k_blocks).
    int32_t k_stages, n_planes, plane_bytes, pmax;
    int32_t tma_store;                    // rows form: the staged tile leaves by one TMA store
    int32_t raw_filter;                   // filter in TMEM read from the caller's OIHW rows (3x3)
    int32_t contig;                       // a CTA runs a contiguous run of units (not a stride)
    int32_t reuse;                        // FORM 2: units reuse the previous unit's last stage ...
    int32_t reuse_period;                 // ... except every reuse_period-th (an image's first row)
    int32_t tap_plane[8], tap_shift[8], plane_phase[8];
    // Rows form over an NCHW input read in place (FORM 2): each stage's raw
    // box, 64 channel rows of xw input columns (xw / 8 odd), lands in one of
    // raw_stages slots of raw_b bytes from raw_off; phase_planes holds the
    // plane of each stride phase (4 bits per phase, 15 = no tap reads it);
    // plane p starts plane_rows0 >> 4p & 15 rows into its plane_bytes.
    int32_t raw_off, raw_b, raw_stages, xw;
    int32_t raw_early;                    // raw slots below the filter's start-up space
    uint32_t plane_rows0;
    uint32_t phase_planes;
    // Offsets of the plane (or pixel box) ring and of the filter's start-up
    // passes in shared memory.
    int32_t ring_off, w_off;
    ConvHTile ht[kConvMaxHTiles];
    ConvWTile wt[kConvMaxWTiles];
};

struct ConvUnit { int img, ht, rb, wt, cb, mb; };

// Unit index -> (image, H-tile, row block, W-tile, column block, channel
// block), the channel and column blocks fastest.  img counts from the
// launch's first image (args.img0).
__device__ __forceinline__ ConvUnit decode_conv_unit(int u, const ConvTmaArgs& a) {
    ConvUnit c;
    c.mb = u % a.co_blocks;
    u /= a.co_blocks;
    c.cb = u % a.cblocks;
    u /= a.cblocks;
    c.wt = u % a.n_wtiles;
    u /= a.n_wtiles;
    c.rb = u % a.rblocks;
    u /= a.rblocks;
    c.ht = u % a.n_htiles;
    c.img = u / a.n_htiles;
    return c;
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(ptx::smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(ptx::smem_addr(bar)), "r"(c0), "r"(c1),
        "r"(c2), "r"(c3)
        : "memory");
}

// Transpose an 8 x 8 matrix of 16-bit values held by 8 consecutive lanes:
// lane j (= lane & 7) enters with row j as 4 words (elements 2k, 2k+1 in
// word k) and leaves with column j in the same form.  Three shfl.xor
// stages exchange 4 x 4, 2 x 2 and 1 x 1 blocks.  All 32 lanes must call.
__device__ __forceinline__ void transpose8x8_b16(uint32_t& w0, uint32_t& w1, uint32_t& w2,
                                                 uint32_t& w3, int j) {
    const unsigned all = 0xffffffffu;
    const bool low_half = j < 4;
    uint32_t s0 = low_half ? w2 : w0, s1 = low_half ? w3 : w1;
    uint32_t r0 = __shfl_xor_sync(all, s0, 4), r1 = __shfl_xor_sync(all, s1, 4);
    uint32_t u0, u1, u2, u3;
    if (low_half) { u0 = w0; u1 = w1; u2 = r0; u3 = r1; }
    else          { u0 = r0; u1 = r1; u2 = w2; u3 = w3; }
    const bool b1 = (j & 2) != 0;
    s0 = b1 ? u0 : u1;
    s1 = b1 ? u2 : u3;
    r0 = __shfl_xor_sync(all, s0, 2);
    r1 = __shfl_xor_sync(all, s1, 2);
    uint32_t v0, v1, v2, v3;
    if (!b1) { v0 = u0; v1 = r0; v2 = u2; v3 = r1; }
    else     { v0 = r0; v1 = u1; v2 = r1; v3 = u3; }
    const uint32_t q0 = __shfl_xor_sync(all, v0, 1), q1 = __shfl_xor_sync(all, v1, 1);
    const uint32_t q2 = __shfl_xor_sync(all, v2, 1), q3 = __shfl_xor_sync(all, v3, 1);
    if ((j & 1) == 0) {
        w0 = __byte_perm(v0, q0, 0x5410); w1 = __byte_perm(v1, q1, 0x5410);
        w2 = __byte_perm(v2, q2, 0x5410); w3 = __byte_perm(v3, q3, 0x5410);
    } else {
        w0 = __byte_perm(q0, v0, 0x7632); w1 = __byte_perm(q1, v1, 0x7632);
        w2 = __byte_perm(q2, v2, 0x7632); w3 = __byte_perm(q3, v3, 0x7632);
    }
}

// a / d for 0 <= a < 2^22 and d >= 1, from a float reciprocal of d: the
// rounded product is within one of the quotient (its error is below
// a * 2^-23 < 1), and one comparison each way fixes it.  The epilogue's
// chunk indices stay below 128 * 256 * 4 / 16 = 8192.
__device__ __forceinline__ int div_small(int a, int d, float inv_d) {
    int q = __float2int_rz(__int2float_rn(a) * inv_d);
    if (q * d > a) --q;
    else if ((q + 1) * d <= a) ++q;
    return q;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int k) {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b, bool bf16) {
    if (bf16) {
        __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&t);
    }
    __half2 t = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&t);
}

__device__ __forceinline__ void store_one(void* base, int64_t idx, uint32_t bits, int dtype) {
    const float f = __uint_as_float(bits);
    if (dtype == TILES_F32) static_cast<float*>(base)[idx] = f;
    else if (dtype == TILES_F16) static_cast<__half*>(base)[idx] = __float2half_rn(f);
    else static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(f);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    conv_tma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ ConvTmaArgs args, int stages, int stage_bytes) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    uint8_t* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    // With resident weights: [all weight K blocks][stages x pixel tile];
    // else each stage holds its pixel tile (A, 16 KB) then its weight tile.
    uint8_t* wres = base;
    uint8_t* ring = base + (args.w_resident ? args.w_bytes : 0u);
    PipeBarriers* bar = reinterpret_cast<PipeBarriers*>(ring + stages * stage_bytes);
    const uint32_t w_kblock_bytes = static_cast<uint32_t>(args.nco) * 128u;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            ptx::mbar_init(&bar->full[s], 1);
            ptx::mbar_init(&bar->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&bar->acc_full[a], 1);
            ptx::mbar_init(&bar->acc_empty[a], 4);
        }
        ptx::mbar_init(&bar->drain, 1);
        ptx::mbar_init(&bar->full[kMaxStages - 1], 1);   // resident weights (stages < kMaxStages)
        bar->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&tmW);
        ptx::tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        ptx::tmem_alloc<1>(&bar->tmem_base, kTmaConvTmemCols);
        ptx::tmem_relinquish<1>();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::grid_dependency_wait();     // the prepared operands are complete

    const uint32_t tmem = bar->tmem_base;
    volatile int* abort = &bar->abort;
    const uint64_t limit = args.wait_limit_ns;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: the pixel box and the weights ----------------
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool aborted = false;
            uint64_t* wbar = &bar->full[kMaxStages - 1];
            if (args.w_resident && static_cast<int>(blockIdx.x) < args.units) {
                // Every K block of the (single) output-channel block, once.
                ptx::mbar_arrive_expect_tx(wbar, args.w_bytes);
                for (int kb = 0; kb < args.k_blocks; ++kb)
                    ptx::tma_load_3d(wres + kb * w_kblock_bytes, &tmW, wbar, kb * 64, 0, 0);
            }
            for (int u = blockIdx.x; u < args.units && !aborted; u += gridDim.x) {
                const ConvUnit cu = decode_conv_unit(u, args);
                const ConvHTile ht = args.ht[cu.ht];
                // Input row and column under the unit's first output pixel,
                // placed by the H-tile's slice: in_start - pt' is the row of
                // the window over the tile's first output row.
                const ConvWTile wt = args.wt[cu.wt];
                const int row0 = ht.in_start - ht.pt + cu.rb * args.nr * args.sh;
                const int col0 = wt.in_start - wt.pl + cu.cb * args.owc * args.sw;
                for (int kb = 0; kb < args.k_blocks; ++kb) {
                    const int tap = kb / args.ch_blocks;
                    const int chb = kb - tap * args.ch_blocks;
                    const int r = tap / args.kw;
                    const int s = tap - r * args.kw;
                    if (!ptx::mbar_wait(&bar->empty[stage], phase ^ 1u, abort, limit)) {
                        raise_error(args.err, abort, kErrProducer);
                        aborted = true;
                        break;
                    }
                    uint8_t* st = ring + stage * stage_bytes;
                    ptx::mbar_arrive_expect_tx(&bar->full[stage], args.tx_bytes);
                    tma_load_4d(st, &tmX, &bar->full[stage], chb * 64, col0 + s * args.dw,
                                row0 + r * args.dh, args.img0 + cu.img);
                    if (!args.w_resident)
                        ptx::tma_load_3d(st + kTmaConvA, &tmW, &bar->full[stage], kb * 64,
                                         cu.mb * args.nco, 0);
                    ++issued;
                    if (++stage == static_cast<uint32_t>(stages)) { stage = 0; phase ^= 1u; }
                }
            }
            if (aborted) {
                settle_after_abort();
            } else {
                for (int i = 0; i < (issued < stages ? issued : stages); ++i) {
                    if (stage == 0) { stage = stages - 1; phase ^= 1u; } else { --stage; }
                    ptx::mbar_wait(&bar->full[stage], phase, nullptr, limit);
                }
                if (args.w_resident && static_cast<int>(blockIdx.x) < args.units)
                    ptx::mbar_wait(wbar, 0, nullptr, limit);
            }
        }
    } else if (warp == 1) {
        {
            // ---------------- MMA issuer ----------------
            // The loop runs on the whole warp (warp-uniform state); one lane
            // chosen by elect.sync issues the MMAs and commits.
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool weights_ready = !args.w_resident;
            // The same lane issues every MMA and commit: a commit tracks the
            // MMAs of the thread that issues it.
            const bool issuer = ptx::elect_one_sync();
            for (int u = blockIdx.x; u < args.units; u += gridDim.x) {
                if (!weights_ready) {
                    if (!__all_sync(0xffffffffu,
                                    ptx::mbar_wait(&bar->full[kMaxStages - 1], 0, abort, limit))) {
                        if (lane == 0) raise_error(args.err, abort, kErrMma);
                        break;
                    }
                    weights_ready = true;
                }
                if (!__all_sync(0xffffffffu,
                                ptx::mbar_wait(&bar->acc_empty[acc], acc_phase ^ 1u, abort, limit))) {
                    if (lane == 0) raise_error(args.err, abort, kErrMma);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem + acc * kTmaConvMaxN;
                bool ok = true;
                for (int kb = 0; kb < args.k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bar->full[stage], phase, abort, limit))) {
                        if (lane == 0) raise_error(args.err, abort, kErrMma);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a0 = ptx::smem_addr(ring + stage * stage_bytes);
                    const uint32_t b0 = args.w_resident ? ptx::smem_addr(wres + kb * w_kblock_bytes)
                                                        : a0 + kTmaConvA;
                    if (issuer) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            // Both operands K-major: 16 channels = 32 bytes of a
                            // 128-byte row; 8-row groups 1024 B apart.
                            const uint64_t ad = ptx::smem_desc_sw128(a0 + kk * 32, 16, 1024);
                            const uint64_t bd = ptx::smem_desc_sw128(b0 + kk * 32, 16, 1024);
                            ptx::mma_f16<1>(d, ad, bd, args.idesc, (kb | kk) != 0);
                        }
                        ptx::mma_commit<1>(&bar->empty[stage]);
                    }
                    __syncwarp();
                    if (++stage == static_cast<uint32_t>(stages)) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (issuer) ptx::mma_commit<1>(&bar->acc_full[acc]);
                __syncwarp();
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            // Every MMA issued here completes before the block tears down.
            if (issuer) {
                ptx::mma_commit_local<1>(&bar->drain);
                ptx::mbar_wait(&bar->drain, 0, nullptr, limit);
            }
            __syncwarp();
        }
    } else {
        // ---------------- epilogue (warps 2-5): one output pixel per thread ----------------
        const int quarter = warp & 3;
        const int p = quarter * 32 + lane;             // pixel of the tile = TMEM lane
        const int rr = p / args.owc;
        const int cc = p - rr * args.owc;
        const int64_t plane = static_cast<int64_t>(args.oh) * args.ow;
        uint32_t acc = 0, acc_phase = 0;
        for (int u = blockIdx.x; u < args.units; u += gridDim.x) {
            const ConvUnit cu = decode_conv_unit(u, args);
            bool ok = ptx::mbar_wait(&bar->acc_full[acc], acc_phase, abort, limit);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) raise_error(args.err, abort, kErrEpilogue);
                break;
            }
            ptx::tc_fence_after();
            const ConvHTile ht = args.ht[cu.ht];
            const ConvWTile wt = args.wt[cu.wt];
            const int ow_end = wt.o0 + wt.cols;               // the W-tile's last column + 1
            const int img = args.img0 + cu.img;
            const int oh = ht.o0 + cu.rb * args.nr + rr;
            const int ow = wt.o0 + cu.cb * args.owc + cc;
            const bool pix_ok = rr < args.nr && oh < ht.o0 + ht.rows && ow < ow_end;
            // Element index of (img, co = 0, oh, ow); channel co adds co * plane.
            const int64_t pix = static_cast<int64_t>(img) * args.c_out * plane +
                                static_cast<int64_t>(oh) * args.ow + ow;
            const uint32_t tacc = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kTmaConvMaxN;
            // 16-bit output: the 8 lanes of a group hold 8 consecutive pixels of
            // one output row (owc is a multiple of 8); after an 8 x 8
            // transpose each lane holds those 8 pixels of one channel and
            // writes them as one 16-byte store.
            const int g8 = lane >> 3, j8 = lane & 7;
            const int pg = quarter * 32 + g8 * 8;              // first pixel of the group
            const int rr_g = pg / args.owc;
            const int oh_g = ht.o0 + cu.rb * args.nr + rr_g;
            const int ow_g = wt.o0 + cu.cb * args.owc + (pg - rr_g * args.owc);
            const bool row_g = rr_g < args.nr && oh_g < ht.o0 + ht.rows;
            const int64_t pix_g = static_cast<int64_t>(img) * args.c_out * plane +
                                  static_cast<int64_t>(oh_g) * args.ow + ow_g;
            const bool half_out = args.out_dtype != TILES_F32;
            const bool bf16_out = args.out_dtype == TILES_BF16;
#pragma unroll 1
            for (int c = 0; c < (args.nco + 31) / 32; ++c) {
                uint32_t v[32];
                ptx::tmem_ld_32cols(tacc + c * 32, v);
                ptx::tmem_ld_wait();
                const int co0 = cu.mb * args.nco + c * 32;
                if (half_out) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint32_t w0 = pack_half2(__uint_as_float(v[8 * g + 0]), __uint_as_float(v[8 * g + 1]), bf16_out);
                        uint32_t w1 = pack_half2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]), bf16_out);
                        uint32_t w2 = pack_half2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]), bf16_out);
                        uint32_t w3 = pack_half2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]), bf16_out);
                        transpose8x8_b16(w0, w1, w2, w3, j8);
                        const int co = co0 + 8 * g + j8;
                        if (!row_g || co >= args.c_out) continue;
                        uint16_t* dst = static_cast<uint16_t*>(args.y) + pix_g +
                                        static_cast<int64_t>(co) * plane;
                        if (args.vec_ok && ow_g + 8 <= ow_end) {
                            *reinterpret_cast<uint4*>(dst) = make_uint4(w0, w1, w2, w3);
                        } else {
                            const uint32_t wv[4] = {w0, w1, w2, w3};
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                if (ow_g + e < ow_end)
                                    dst[e] = static_cast<uint16_t>(wv[e >> 1] >> ((e & 1) * 16));
                        }
                    }
                } else if (pix_ok) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (co0 + i < args.c_out)
                            store_one(args.y, pix + static_cast<int64_t>(co0 + i) * plane, v[i],
                                      args.out_dtype);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar->acc_empty[acc]);
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc<1>(tmem, kTmaConvTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Weights in tensor memory.  For c_out <= 128 and a short K the whole filter
// fits in TMEM (K/2 columns: two 16-bit values per column) beside one or two
// accumulators, so it is the MMA's A operand for the kernel's lifetime:
// M = 128 output channels on the TMEM lanes, N = npix output pixels (nr rows
// x owc columns), K = (r, s, ci).  Per K block only the pixel box crosses
// shared memory.  One tcgen05.mma costs the issuing thread a roughly fixed
// time, so wide pixel tiles (N up to 256 with a single accumulator) keep the
// tensor core busy; with two accumulators the epilogue overlaps the next
// tile's MMAs at half the width.
//
// Warps: 0 TMA producer, 1 MMA issuer, 2-9 epilogue.
//  - Start: the producer TMA-loads the reordered filter into the (still
//    unused) shared memory, in passes of as many 16 KB K blocks as fit; the
//    epilogue warps copy each block's rows into tensor memory (warp w owns
//    lanes 32*(w%4) .. +31 and every other K block) and release the space.
//  - Per tile: the epilogue warps read the accumulator (a thread = one output
//    channel, npix/2 consecutive pixels), write it as 16-bit or fp32 rows to
//    a shared staging tile whose row pitch is an odd number of 16-byte
//    chunks (no bank conflicts), then store the tile row-contiguously to the
//    NCHW output: consecutive threads write consecutive 16 bytes.
constexpr int kWtThreads = 320;
constexpr int kWtEpilogueWarps = 8;
constexpr int kWtEpilogueThreads = kWtEpilogueWarps * 32;
constexpr int kWtTmemCols = 512;
constexpr int kWtWeightBlockBytes = 128 * 128;   // 128 rows x 64 channels x 2 bytes
// Rows form read straight from an NCHW input: kTrWarps more warps, after
// the producer, the MMA issuer and the epilogue warps, build each stage's
// stride-phase planes from the input rows.  They take the warps past the
// epilogue's that do not share the MMA issuer's scheduler (warp % 4 != 1);
// the others there stay idle.
constexpr int kTrWarps = 12;
// A warp's items keep its channel half and step 8 kTrWarps / 2 columns, a
// multiple of 16 so that stride-2 rows advance by a multiple of 8.
static_assert(kTrWarps % 4 == 0, "transposer count");
constexpr int kTrFirstWarp = 2 + 8;          // after the producer, the MMA issuer, 8 epilogue warps
// Boxes of 64 elements per 64 input channels of a 3x3 filter's OIHW row.
constexpr int kRawFilterBoxes = 9;
constexpr int kWtDirectThreads =
    (kTrFirstWarp + (kTrWarps - 1) + (kTrWarps - 1) / 3 + 1) * 32;
static_assert(kTrFirstWarp % 4 == 2, "transposer warp mapping assumes warp 10 sits on scheduler 2");
// Transposer items per warp and stage: a raw box of at most 256 columns is
// 32 column groups x 2 channel halves.
constexpr int kTrItems = (64 + kTrWarps - 1) / kTrWarps;

struct WtBarriers {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint64_t wfull;      // a pass of filter blocks landed in shared memory
    uint64_t wcons;      // the epilogue warps copied that pass to tensor memory
    uint64_t wready;     // the whole filter is in tensor memory
    int32_t raw_col0[kMaxStages];   // FORM 2: span column origin of each raw slot's box
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(WtBarriers) <= kSmemBarrierBytes, "barrier block");

// Named barrier 1 over the epilogue warps, and the same barrier returning
// the AND of every thread's flag (one answer for all, so the warps take the
// same branch after it).
__device__ __forceinline__ void epilogue_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(kWtEpilogueThreads) : "memory");
}
__device__ __forceinline__ bool epilogue_bar_and(bool flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(flag ? 1u : 0u), "r"(kWtEpilogueThreads) : "memory");
    return r != 0;
}

// Four 8 x 8 blocks of 16-bit elements from shared memory, transposed: lane
// l gives the address of row l & 7 of block l >> 3 (16 bytes, 16-byte
// aligned) and receives, in d[b], elements (2(l & 3), l >> 2) and
// (2(l & 3) + 1, l >> 2) of block b, the first in the low half.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&d)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(addr)
                 : "memory");
}

// Where one stage of the rows form reads its input: image, input row,
// first channel and the first input column of the span (pmax * sw columns
// from col0).
struct RowStage { int img, ih, c0, col0; };

__device__ __forceinline__ RowStage row_stage(int u, int kb, const ConvTmaArgs& a) {
    const ConvUnit cu = decode_conv_unit(u, a);
    const ConvHTile ht = a.ht[cu.ht];
    const ConvWTile wt = a.wt[cu.wt];
    const int r = kb / a.ch_blocks;
    RowStage s;
    s.img = a.img0 + cu.img;
    s.ih = ht.in_start - ht.pt + cu.rb * a.nr * a.sh + r * a.dh;
    s.c0 = (kb - r * a.ch_blocks) * 64;
    s.col0 = wt.in_start - wt.pl + cu.cb * a.owc * a.sw;
    return s;
}

// The units of a CTA.  With args.contig a contiguous run [first, end), so
// that consecutive output rows, whose input rows overlap, stay on one CTA;
// otherwise units blockIdx.x, + gridDim.x, ... up to args.units.
struct UnitRange { int first, end, step; };

__device__ __forceinline__ UnitRange unit_range(const ConvTmaArgs& a) {
    if (a.contig) {
        const int64_t u0 = static_cast<int64_t>(blockIdx.x) * a.units / gridDim.x;
        const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * a.units / gridDim.x;
        return UnitRange{static_cast<int>(u0), static_cast<int>(u1), 1};
    }
    return UnitRange{static_cast<int>(blockIdx.x), a.units, static_cast<int>(gridDim.x)};
}

// Whether unit u's first stage reads the same input row, image, channels and
// columns as the previous unit's last stage, so that its stride-phase planes
// are still in the ring and the stage is neither loaded nor transposed again
// (stride 2 and a 3-row filter: output rows oh and oh+1 share input row
// 2 oh + 1).  The host sets reuse only where the units of an image are its
// output rows in order (one W tile, one column and output-channel block,
// whole H tiles, one channel block, (kh-1)*dh == sh): then every unit but a
// CTA's first and an image's first row qualifies.  Every role of the kernel
// takes the same decision.
__device__ __forceinline__ bool reuses_prev(int u, const UnitRange& ur, const ConvTmaArgs& a) {
    return a.reuse && u != ur.first && u % a.reuse_period != 0;
}

// FORM 0: one pixel box per (tap, 64 channels).  FORM 1 (rows form): one
// output row per tile and one stage per (kernel row, 64 channels), whose
// stride phases of the input row serve every tap of that row: tap s's B
// operand starts tap_shift[s] 128-byte rows into plane tap_plane[s] (a
// K-major 128-byte-swizzled tile read from a whole-row offset is the same
// tile shifted, the swizzle following the address bits).  FORM 2: the rows
// form over an NCHW input, its planes written by transposer warps from raw
// NCHW boxes instead of loaded by TMA from an NHWC copy.
template <int FORM>
__global__ void __launch_bounds__(FORM == 2 ? kWtDirectThreads : kWtThreads, 1)
    conv_wtmem_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmY, const __grid_constant__ ConvTmaArgs args) {
    constexpr bool ROWS = FORM != 0;
    constexpr bool DIRECT = FORM == 2;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    uint8_t* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    // FORM 0, 1: [stages x pixel box][staging tile][barriers], the filter
    // passes in [0, w_slots x 16 KB) at the start.  FORM 2: [raw ring][plane
    // ring][staging tile][barriers], the filter passes from raw slot
    // raw_early on, so the first raw_early boxes load beside them.
    uint8_t* ring = base + args.ring_off;
    uint8_t* staging = base + args.stg_off;
    WtBarriers* bar = reinterpret_cast<WtBarriers*>(base + args.bar_off);
    const int stages = args.stages;
    const uint32_t stage_bytes = static_cast<uint32_t>(args.stage_b);
    // Filter passes.  Reordered filter: w_slots K blocks per pass.  Raw
    // filter (3x3, C a multiple of 64): one pass per 64 input channels, the
    // 9 boxes of 64 elements of each OIHW row that hold them.
    const int passes = args.raw_filter ? args.ch_blocks
                                       : (args.k_blocks + args.w_slots - 1) / args.w_slots;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            // FORM 2: every transposer warp arrives once per stage.
            ptx::mbar_init(&bar->full[s], DIRECT ? kTrWarps : 1);
            ptx::mbar_init(&bar->empty[s], 1);
        }
        if (DIRECT) {
            // The raw ring's barriers follow the plane ring's.
            for (int s = 0; s < args.raw_stages; ++s) {
                ptx::mbar_init(&bar->full[stages + s], 1);
                ptx::mbar_init(&bar->empty[stages + s], kTrWarps);
            }
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&bar->acc_full[a], 1);
            ptx::mbar_init(&bar->acc_empty[a], kWtEpilogueWarps);
        }
        ptx::mbar_init(&bar->drain, 1);
        ptx::mbar_init(&bar->wfull, 1);
        ptx::mbar_init(&bar->wcons, kWtEpilogueWarps);
        ptx::mbar_init(&bar->wready, kWtEpilogueWarps);
        bar->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::tma_prefetch_desc(&tmW);
        ptx::tma_prefetch_desc(&tmX);
        if (args.tma_store) ptx::tma_prefetch_desc(&tmY);
    }
    if (warp == 1) {
        ptx::tmem_alloc<1>(&bar->tmem_base, kWtTmemCols);
        ptx::tmem_relinquish<1>();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    // Set-up above overlaps the operand preparation; its results (filter,
    // NHWC input) are read only after this point.
    ptx::grid_dependency_wait();

    const uint32_t tmem = bar->tmem_base;
    volatile int* abort = &bar->abort;
    const uint64_t limit = args.wait_limit_ns;
    const bool has_work = static_cast<int>(blockIdx.x) < args.units;
    const UnitRange ur = unit_range(args);

    if (warp == 0) {
        if (lane == 0) {
            bool aborted = false;
            // ---------------- the filter, pass by pass ----------------
            auto filter_pass = [&](int p) {
                if (p > 0 && !ptx::mbar_wait(&bar->wcons, (p - 1) & 1, abort, limit)) {
                    raise_error(args.err, abort, kErrProducer);
                    aborted = true;
                    return;
                }
                const int kb0 = args.raw_filter ? p * kRawFilterBoxes : p * args.w_slots;
                const int nkb = args.raw_filter ? kRawFilterBoxes : min(args.w_slots, args.k_blocks - kb0);
                ptx::mbar_arrive_expect_tx(&bar->wfull, static_cast<uint32_t>(nkb * kWtWeightBlockBytes));
                // Every CTA reads the same blocks at start-up; each begins at
                // a different one (blockIdx.x mod nkb) so that the L2 lines
                // in demand at any moment are spread over the whole filter.
                const int rot = static_cast<int>(blockIdx.x % static_cast<unsigned>(nkb));
                for (int j = 0; j < nkb; ++j) {
                    const int i = j + rot < nkb ? j + rot : j + rot - nkb;
                    ptx::tma_load_3d(base + args.w_off + i * kWtWeightBlockBytes, &tmW, &bar->wfull,
                                     (kb0 + i) * 64, 0, 0);
                }
            };
            if constexpr (DIRECT) {
                // ---------------- TMA producer: each stage's raw NCHW box ----------------
                // 64 channel rows of xw columns from the span's 8-column
                // group (x 16-byte aligned); rows, columns and channels
                // outside the input arrive as zeros.  The first raw_early
                // boxes go out with the filter's first pass, the rest once
                // the filter has left the slots after them.
                uint32_t rs = 0, rphase = 0;
                int issued = 0, u = ur.first, kb = 0;
                const uint32_t raw_tx = static_cast<uint32_t>(args.raw_b);
                auto issue_raw = [&]() {
                    // A stage whose planes are reused needs no box.
                    if (kb == 0 && reuses_prev(u, ur, args)) kb = 1;
                    if (!ptx::mbar_wait(&bar->empty[stages + rs], rphase ^ 1u, abort, limit)) {
                        raise_error(args.err, abort, kErrProducer);
                        aborted = true;
                        return;
                    }
                    const RowStage st = row_stage(u, kb, args);
                    uint64_t* rfull = &bar->full[stages + rs];
                    // The transposers read the box's column origin after
                    // waiting on the slot's barrier (the arrive releases it).
                    bar->raw_col0[rs] = st.col0;
                    // A planted fault (test hook) skips one box: its slot
                    // never fills and the transposers' bounded wait expires.
                    if (!(blockIdx.x == 0 && issued == args.drop_stage)) {
                        ptx::mbar_arrive_expect_tx(rfull, raw_tx);
                        tma_load_4d(base + args.raw_off + rs * args.raw_b, &tmX, rfull,
                                    st.col0 & ~7, st.ih, st.c0, st.img);
                    }
                    ++issued;
                    if (++rs == static_cast<uint32_t>(args.raw_stages)) { rs = 0; rphase ^= 1u; }
                    if (++kb == args.k_stages) { kb = 0; u += ur.step; }
                };
                // The filter's loads go first: one TMA queue serves both, and
                // a raw box from DRAM ahead of them would hold them up.
                if (has_work) filter_pass(0);
                while (!aborted && u < ur.end && issued < args.raw_early) issue_raw();
                for (int p = 1; p < passes && has_work && !aborted; ++p) filter_pass(p);
                if (!aborted && has_work && !ptx::mbar_wait(&bar->wcons, (passes - 1) & 1, abort, limit)) {
                    raise_error(args.err, abort, kErrProducer);
                    aborted = true;
                }
                while (!aborted && u < ur.end) issue_raw();
                if (aborted) {
                    settle_after_abort();
                } else {
                    for (int i = 0; i < (issued < args.raw_stages ? issued : args.raw_stages); ++i) {
                        if (rs == 0) { rs = args.raw_stages - 1; rphase ^= 1u; } else { --rs; }
                        ptx::mbar_wait(&bar->full[stages + rs], rphase, nullptr, limit);
                    }
                }
            } else {
            for (int p = 0; p < passes && has_work && !aborted; ++p) filter_pass(p);
            // The pixel boxes reuse that space once the last pass is copied.
            if (!aborted && has_work && !ptx::mbar_wait(&bar->wcons, (passes - 1) & 1, abort, limit)) {
                raise_error(args.err, abort, kErrProducer);
                aborted = true;
            }
            // ---------------- TMA producer: one pixel box per K block ----------------
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            for (int u = ur.first; u < ur.end && !aborted; u += ur.step) {
                const ConvUnit cu = decode_conv_unit(u, args);
                const ConvHTile ht = args.ht[cu.ht];
                const ConvWTile wt = args.wt[cu.wt];
                const int row0 = ht.in_start - ht.pt + cu.rb * args.nr * args.sh;
                const int col0 = wt.in_start - wt.pl + cu.cb * args.owc * args.sw;
                for (int kb = 0; kb < args.k_stages; ++kb) {
                    if (!ptx::mbar_wait(&bar->empty[stage], phase ^ 1u, abort, limit)) {
                        raise_error(args.err, abort, kErrProducer);
                        aborted = true;
                        break;
                    }
                    uint8_t* st = ring + stage * stage_bytes;
                    if (blockIdx.x == 0 && issued == args.drop_stage) {
                        // A planted fault (test hook): this stage never fills.
                        ++issued;
                        if (++stage == static_cast<uint32_t>(stages)) { stage = 0; phase ^= 1u; }
                        continue;
                    }
                    ptx::mbar_arrive_expect_tx(&bar->full[stage], args.tx_bytes);
                    if constexpr (ROWS) {
                        // Kernel row r, 64 channels: every stride phase of
                        // the input row, pmax pixels each.
                        const int r = kb / args.ch_blocks;
                        const int chb = kb - r * args.ch_blocks;
                        for (int p = 0; p < args.n_planes; ++p)
                            tma_load_4d(st + p * args.plane_bytes, &tmX, &bar->full[stage], chb * 64,
                                        col0 + args.plane_phase[p], row0 + r * args.dh,
                                        args.img0 + cu.img);
                    } else {
                        const int tap = kb / args.ch_blocks;
                        const int chb = kb - tap * args.ch_blocks;
                        const int r = tap / args.kw;
                        const int s = tap - r * args.kw;
                        tma_load_4d(st, &tmX, &bar->full[stage], chb * 64, col0 + s * args.dw,
                                    row0 + r * args.dh, args.img0 + cu.img);
                    }
                    ++issued;
                    if (++stage == static_cast<uint32_t>(stages)) { stage = 0; phase ^= 1u; }
                }
            }
            if (aborted) {
                settle_after_abort();
            } else {
                for (int i = 0; i < (issued < stages ? issued : stages); ++i) {
                    if (stage == 0) { stage = stages - 1; phase ^= 1u; } else { --stage; }
                    ptx::mbar_wait(&bar->full[stage], phase, nullptr, limit);
                }
            }
            }
        }
    } else if (warp == 1) {
        {
            // ---------------- MMA issuer ----------------
            // The loop runs on the whole warp (warp-uniform state); one lane
            // chosen by elect.sync issues the MMAs and commits.
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            // Pixel rows K-major: 16 channels = 32 bytes of each 128-byte row,
            // 8-row groups 1024 B apart; stages and K steps move the
            // descriptor's start-address field (address >> 4, no carry).
            const uint64_t b_desc0 = ptx::smem_desc_sw128(ptx::smem_addr(ring), 16, 1024);
            // Rows form: each tap's descriptor offset (plane and pixel shift,
            // in 16-byte units) and filter column stride, held in registers.
            uint32_t tap_off[8];
#pragma unroll
            for (int t = 0; t < 8; ++t)
                tap_off[t] = ROWS && t < args.kw
                                 ? static_cast<uint32_t>(
                                       (args.tap_plane[t] * args.plane_bytes +
                                        (static_cast<int>((args.plane_rows0 >> (4 * args.tap_plane[t])) & 15u) +
                                         args.tap_shift[t]) * 128) >> 4)
                                 : 0u;
            const int kw = args.kw;
            const uint32_t tap_cols = static_cast<uint32_t>(args.ch_blocks * 32);
            // The same lane issues every MMA and commit: a commit tracks the
            // MMAs of the thread that issues it.
            const bool issuer = ptx::elect_one_sync();
            bool ok = __all_sync(0xffffffffu,
                                 !has_work || ptx::mbar_wait(&bar->wready, 0, abort, limit));
            if (!ok && lane == 0) raise_error(args.err, abort, kErrMma);
            ptx::tc_fence_after();
            // A reused stage reads the previous stage's slot again; that
            // slot is released only after the second use.
            bool reuse_this = false;
            uint32_t last_slot = 0;
            for (int u = ur.first; ok && u < ur.end; u += ur.step) {
                if (!__all_sync(0xffffffffu,
                                ptx::mbar_wait(&bar->acc_empty[acc], acc_phase ^ 1u, abort, limit))) {
                    if (lane == 0) raise_error(args.err, abort, kErrMma);
                    break;
                }
                ptx::tc_fence_after();
                const bool reuse_next = u + ur.step < ur.end && reuses_prev(u + ur.step, ur, args);
                const uint32_t d = tmem + acc * static_cast<uint32_t>(args.npix);
                for (int kb = 0; kb < args.k_stages; ++kb) {
                    const bool reused = kb == 0 && reuse_this;
                    const uint32_t slot = reused ? last_slot : stage;
                    if (!reused) {
                        if (!__all_sync(0xffffffffu,
                                        ptx::mbar_wait(&bar->full[stage], phase, abort, limit))) {
                            if (lane == 0) raise_error(args.err, abort, kErrMma);
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                    }
                    const bool keep = kb == args.k_stages - 1 && reuse_next;   // reused next
                    const uint64_t b_st = b_desc0 + ((slot * stage_bytes) >> 4);
                    if (issuer) {
                        if constexpr (ROWS) {
                            const int r = kb / args.ch_blocks;
                            const int chb = kb - r * args.ch_blocks;
                            // Filter columns of tap (r, 0); tap s adds s * tap_cols.
                            const uint32_t a_r = tmem + static_cast<uint32_t>(
                                args.a_col + (r * kw * args.ch_blocks + chb) * 32);
                            const uint32_t first = kb != 0 ? 1u : 0u;   // 0: the tile's first MMA
                            if (kw == 3) {
                                // The common 3-tap row, fully unrolled: 12 MMAs
                                // with offsets in registers and no branches.
#pragma unroll
                                for (int t = 0; t < 3; ++t)
#pragma unroll
                                    for (int kk = 0; kk < 4; ++kk)
                                        ptx::mma_f16_tmem_a(d, a_r + t * tap_cols + kk * 8,
                                                            b_st + tap_off[t] + kk * (32 >> 4),
                                                            args.idesc,
                                                            (t | kk) != 0 ? 1u : first);
                            } else {
#pragma unroll
                                for (int t = 0; t < 8; ++t) {
                                    if (t >= kw) break;
                                    const uint64_t b_tap = b_st + tap_off[t];
                                    const uint32_t a0 = a_r + static_cast<uint32_t>(t) * tap_cols;
#pragma unroll
                                    for (int kk = 0; kk < 4; ++kk)
                                        ptx::mma_f16_tmem_a(d, a0 + kk * 8, b_tap + kk * (32 >> 4),
                                                            args.idesc, (kb | t | kk) != 0);
                                }
                            }
                        } else {
                            const uint32_t a0 = tmem + static_cast<uint32_t>(args.a_col + kb * 32);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)   // 16 channels: 8 TMEM columns of A
                                ptx::mma_f16_tmem_a(d, a0 + kk * 8, b_st + kk * (32 >> 4), args.idesc,
                                                    (kb | kk) != 0);
                        }
                        if (!keep) ptx::mma_commit<1>(&bar->empty[slot]);
                    }
                    __syncwarp();
                    if (!reused) {
                        last_slot = stage;
                        if (++stage == static_cast<uint32_t>(stages)) { stage = 0; phase ^= 1u; }
                    }
                }
                reuse_this = reuse_next;
                if (!ok) break;
                if (issuer) ptx::mma_commit<1>(&bar->acc_full[acc]);
                __syncwarp();
                if (args.acc_bufs == 2) acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            // Every MMA issued here completes before the block tears down.
            if (issuer) {
                ptx::mma_commit_local<1>(&bar->drain);
                ptx::mbar_wait(&bar->drain, 0, nullptr, limit);
            }
            __syncwarp();
        }
    } else if (warp < 2 + kWtEpilogueWarps) {
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int et = threadIdx.x - 64;                // 0 .. 255
        const int co = quarter * 32 + lane;             // output channel = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        // ---------------- the filter into tensor memory ----------------
        bool ok = true;
        for (int p = 0; p < passes && has_work; ++p) {
            ok = ptx::mbar_wait(&bar->wfull, p & 1, abort, limit);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) raise_error(args.err, abort, kErrEpilogue);
                ok = false;
                break;
            }
            if (args.raw_filter) {
                // Pass p holds input channels 64p .. 64p+63 of every OIHW row:
                // element e = channel * 9 + tap of the pass, box e / 64,
                // 16-byte chunk (e % 64) / 8 at chunk ^ (row & 7).  This
                // thread builds row co's 32 channels half*32 .. +31, eight at
                // a time: the 72 elements of 8 channels are 9 chunks, and each
                // TMEM column (tap t, channels 2j, 2j+1) takes two halves of
                // them (K order (tap, channel), two channels per column).
                const uint8_t* rowb = base + args.w_off + co * 128;
#pragma unroll 1
                for (int k = 0; k < 4; ++k) {
                    const int cl = half * 32 + k * 8;          // first channel of the chunk
                    uint32_t L[36];
#pragma unroll
                    for (int q = 0; q < 9; ++q) {
                        const int qq = (cl / 8) * 9 + q;
                        const uint4 v = *reinterpret_cast<const uint4*>(
                            rowb + (qq >> 3) * kWtWeightBlockBytes + (((qq & 7) ^ (co & 7)) << 4));
                        L[4 * q] = v.x; L[4 * q + 1] = v.y; L[4 * q + 2] = v.z; L[4 * q + 3] = v.w;
                    }
#pragma unroll
                    for (int t = 0; t < kRawFilterBoxes; ++t) {
                        uint32_t o[4];
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const int e0 = 18 * jj + t, e1 = e0 + 9;
                            o[jj] = __byte_perm(L[e0 >> 1], L[e1 >> 1],
                                                ((e0 & 1) ? 0x32u : 0x10u) | ((e1 & 1) ? 0x7600u : 0x5400u));
                        }
                        ptx::tmem_st_4cols(tmem + lane_base +
                                               static_cast<uint32_t>(args.a_col + (t * args.ch_blocks + p) * 32 + cl / 2),
                                           o);
                    }
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bar->wcons);
                continue;
            }
            const int kb0 = p * args.w_slots;
            const int nkb = min(args.w_slots, args.k_blocks - kb0);
            for (int i = half; i < nkb; i += 2) {
                // Row co of a 128-byte-swizzled block: 16-byte chunk j sits
                // at chunk j ^ (co & 7).
                const uint8_t* row = base + args.w_off + i * kWtWeightBlockBytes + co * 128;
                uint32_t v[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 t = *reinterpret_cast<const uint4*>(row + ((j ^ (co & 7)) << 4));
                    v[4 * j + 0] = t.x; v[4 * j + 1] = t.y; v[4 * j + 2] = t.z; v[4 * j + 3] = t.w;
                }
                ptx::tmem_st_32cols(tmem + lane_base + static_cast<uint32_t>(args.a_col + (kb0 + i) * 32), v);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar->wcons);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (has_work && ok && lane == 0) ptx::mbar_arrive(&bar->wready);
        // Every epilogue warp enters the tile loop, or none does.
        ok = epilogue_bar_and(ok);
        // ---------------- epilogue ----------------
        const int ob = args.out_dtype == TILES_F32 ? 4 : 2;
        const bool bf16_out = args.out_dtype == TILES_BF16;
        const int col_begin = half * (args.npix >> 1);
        const int col_end = col_begin + (args.npix >> 1);
        const int64_t plane = static_cast<int64_t>(args.oh) * args.ow;
        // Output chunks of 16 bytes: per (channel, pixel row) owc*ob/16.
        const int seg_chunks = args.owc * ob / 16;
        const int tile_chunks = 128 * args.nr * seg_chunks;
        const float inv_seg = 1.0f / static_cast<float>(seg_chunks);
        const float inv_nr = 1.0f / static_cast<float>(args.nr);
        const int ch_elems = 16 / ob;
        uint32_t acc = 0, acc_phase = 0;
        for (int u = ur.first; ok && u < ur.end; u += ur.step) {
            const ConvUnit cu = decode_conv_unit(u, args);
            const bool okw = ptx::mbar_wait(&bar->acc_full[acc], acc_phase, abort, limit);
            // The previous tile's TMA store has read the staging tile
            // before the barrier below lets anyone write it again.
            if (args.tma_store && et == 0) ptx::bulk_wait_read_all();
            // One decision for all epilogue warps; passing this barrier also
            // means the previous tile's stores have read the staging tile.
            if (!epilogue_bar_and(okw)) {
                if (et == 0) raise_error(args.err, abort, kErrEpilogue);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t tacc = tmem + lane_base + acc * static_cast<uint32_t>(args.npix);
            uint8_t* srow = staging + co * args.stg_pitch;
            // All of this thread's columns (npix/2 <= 128) come out of TMEM in
            // one round trip, after which the accumulator is released; the
            // conversion and the staging writes overlap the next tile's MMAs.
            const int ncols = col_end - col_begin;
            if constexpr (DIRECT) {
                // 32 columns at a time (the wider block leaves fewer
                // registers per thread); the accumulator is released after
                // the last chunk.
#pragma unroll 1
                for (int c0 = 0; c0 < ncols; c0 += 32) {
                    uint32_t w[32];
                    const int nc = min(32, ncols - c0);
                    if (nc == 32) {
                        ptx::tmem_ld_32cols(tacc + col_begin + c0, w);
                    } else {
#pragma unroll
                        for (int g = 0; g < 4; ++g)
                            if (8 * g + 8 <= nc)
                                ptx::tmem_ld_8cols(tacc + col_begin + c0 + 8 * g, w[8 * g + 0],
                                                   w[8 * g + 1], w[8 * g + 2], w[8 * g + 3],
                                                   w[8 * g + 4], w[8 * g + 5], w[8 * g + 6],
                                                   w[8 * g + 7]);
                    }
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (8 * g + 8 > nc) continue;
                        const int c = col_begin + c0 + 8 * g;
                        if (ob == 2) {
                            uint4 t;
                            t.x = pack_half2(__uint_as_float(w[8 * g + 0]), __uint_as_float(w[8 * g + 1]), bf16_out);
                            t.y = pack_half2(__uint_as_float(w[8 * g + 2]), __uint_as_float(w[8 * g + 3]), bf16_out);
                            t.z = pack_half2(__uint_as_float(w[8 * g + 4]), __uint_as_float(w[8 * g + 5]), bf16_out);
                            t.w = pack_half2(__uint_as_float(w[8 * g + 6]), __uint_as_float(w[8 * g + 7]), bf16_out);
                            *reinterpret_cast<uint4*>(srow + c * 2) = t;
                        } else {
                            uint4* dst = reinterpret_cast<uint4*>(srow + c * 4);
                            dst[0] = make_uint4(w[8 * g + 0], w[8 * g + 1], w[8 * g + 2], w[8 * g + 3]);
                            dst[1] = make_uint4(w[8 * g + 4], w[8 * g + 5], w[8 * g + 6], w[8 * g + 7]);
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bar->acc_empty[acc]);
            } else {
            uint32_t v[128];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int c0 = 32 * q;
                if (c0 + 32 <= ncols) {
                    uint32_t (&w)[32] = *reinterpret_cast<uint32_t (*)[32]>(&v[c0]);
                    ptx::tmem_ld_32cols(tacc + col_begin + c0, w);
                } else {
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        if (c0 + 8 * g + 8 <= ncols)
                            ptx::tmem_ld_8cols(tacc + col_begin + c0 + 8 * g, v[c0 + 8 * g + 0],
                                               v[c0 + 8 * g + 1], v[c0 + 8 * g + 2],
                                               v[c0 + 8 * g + 3], v[c0 + 8 * g + 4],
                                               v[c0 + 8 * g + 5], v[c0 + 8 * g + 6],
                                               v[c0 + 8 * g + 7]);
                }
            }
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar->acc_empty[acc]);
#pragma unroll
            for (int g = 0; g < 16; ++g) {
                if (8 * g + 8 > ncols) continue;
                const int c = col_begin + 8 * g;
                if (ob == 2) {
                    uint4 t;
                    t.x = pack_half2(__uint_as_float(v[8 * g + 0]), __uint_as_float(v[8 * g + 1]), bf16_out);
                    t.y = pack_half2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]), bf16_out);
                    t.z = pack_half2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]), bf16_out);
                    t.w = pack_half2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]), bf16_out);
                    *reinterpret_cast<uint4*>(srow + c * 2) = t;
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(srow + c * 4);
                    dst[0] = make_uint4(v[8 * g + 0], v[8 * g + 1], v[8 * g + 2], v[8 * g + 3]);
                    dst[1] = make_uint4(v[8 * g + 4], v[8 * g + 5], v[8 * g + 6], v[8 * g + 7]);
                }
            }
            }
            if (args.acc_bufs == 2) acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
            if (args.tma_store) {
                // One output row: [128 channels][owc pixels] leaves as one
                // box of y at (ow0, oh, 0, img); channels past c_out and
                // columns past the width fall outside the tensor.
                ptx::fence_proxy_async_smem();
                epilogue_bar_sync();
                if (et == 0) {
                    const ConvHTile ht = args.ht[cu.ht];
                    const ConvWTile wt = args.wt[cu.wt];
                    ptx::tma_store_4d(&tmY, staging, wt.o0 + cu.cb * args.owc, ht.o0 + cu.rb, 0,
                                      args.img0 + cu.img);
                    ptx::bulk_commit_group();
                }
                continue;
            }
            epilogue_bar_sync();
            // Staging tile -> NCHW output, 16 bytes per thread per step:
            // consecutive threads take consecutive chunks of a (channel,
            // row) segment, so a warp writes 512 contiguous bytes.
            const ConvHTile ht = args.ht[cu.ht];
            const ConvWTile wt = args.wt[cu.wt];
            const int oh0 = ht.o0 + cu.rb * args.nr;
            const int oh_end = ht.o0 + ht.rows;
            const int ow0 = wt.o0 + cu.cb * args.owc;
            const int ow_end = wt.o0 + wt.cols;
            const int img = args.img0 + cu.img;
            for (int i = et; i < tile_chunks; i += kWtEpilogueThreads) {
                const int seg = div_small(i, seg_chunks, inv_seg);
                const int j = i - seg * seg_chunks;
                const int c = div_small(seg, args.nr, inv_nr);
                const int rr = seg - c * args.nr;
                const int oh = oh0 + rr;
                const int ow = ow0 + j * ch_elems;
                if (c >= args.c_out || oh >= oh_end || ow >= ow_end) continue;
                const uint8_t* src = staging + c * args.stg_pitch + (rr * args.owc + j * ch_elems) * ob;
                const uint4 t = *reinterpret_cast<const uint4*>(src);
                const int64_t idx = (static_cast<int64_t>(img) * args.c_out + c) * plane +
                                    static_cast<int64_t>(oh) * args.ow + ow;
                char* dst = static_cast<char*>(args.y) + idx * ob;
                if (args.vec_ok && ow + ch_elems <= ow_end) {
                    *reinterpret_cast<uint4*>(dst) = t;
                } else {
                    const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (e >= ch_elems || ow + e >= ow_end) continue;
                        if (ob == 2)
                            reinterpret_cast<uint16_t*>(dst)[e] =
                                static_cast<uint16_t>(w4[e >> 1] >> ((e & 1) * 16));
                        else
                            reinterpret_cast<uint32_t*>(dst)[e] = w4[e & 3];
                    }
                }
            }
        }
        // The last TMA store has read the staging tile before the block
        // (and its shared memory) goes away; its writes to y complete with
        // the grid, before anything that waits for it reads y.
        if (args.tma_store && et == 0) ptx::bulk_wait_read_all();
    } else if constexpr (DIRECT) {
        // ---------------- transposer warps (FORM 2) ----------------
        // A raw box is 64 channel rows of xw input columns (row pitch 2 xw
        // bytes, an odd multiple of 16, so the 8 rows of an 8 x 8 block sit
        // in 8 bank groups).  A work item is one 8-column group and 32
        // channels: one ldmatrix .x4 .trans reads its four 8 x 8 blocks
        // transposed, leaving lane l with channels 2(l & 3), 2(l & 3) + 1 of
        // column l >> 2 in each block; four 4-byte stores put them into the
        // column's phase plane row, 16-byte chunk (channel group) ^ (row & 7)
        // under the 128-byte swizzle.
        // Transposer index: warps kTrFirstWarp + j, j % 4 == 3 idle (they
        // share the MMA issuer's scheduler).
        const int j = warp - kTrFirstWarp;
        const int tw = (j & 3) == 3 ? -1 : j - (j >> 2);
        if (tw < 0) goto transposers_done;
        {
        const int span = args.pmax * args.sw;
        const int items = args.xw >> 2;            // xw / 8 column groups x 2 channel halves
        const uint32_t pitch = 2u * static_cast<uint32_t>(args.xw);
        // Item q of this warp is it = tw + q kTrWarps: channel half tw & 1
        // and column group (tw >> 1) + q kTrWarps / 2, kColStep columns
        // after the previous one.
        constexpr int kColStep = 8 * (kTrWarps / 2);
        const int half = tw & 1, g0 = tw >> 1;
        // ldmatrix row of this lane: block l >> 3, channel row l & 7.
        const uint32_t ld_off = static_cast<uint32_t>(half * 32 + (lane >> 3) * 8 + (lane & 7)) * pitch +
                                16u * static_cast<uint32_t>(g0);
        const int px = lane >> 2;                   // column within the group after the transpose
        const int pair = (lane & 3) * 4;
        // Strides dividing kColStep into a multiple of 8 rows keep a lane's
        // phase plane and swizzle row (mod 8) across its items: rows advance
        // by kColStep / sw per item.
        const bool fast = kColStep % args.sw == 0 && (kColStep / args.sw) % 8 == 0;
        const int row_step = fast ? kColStep / args.sw : 0;
        uint32_t ps = 0, pphase = 0, rs = 0, rphase = 0;
        // The planes reuse the filter's start-up space.
        bool ok = !has_work || __all_sync(0xffffffffu, ptx::mbar_wait(&bar->wready, 0, abort, limit));
        // Per-unit lane set-up, recomputed only when a box's column origin
        // (written by the producer beside the box) changes: with one W tile
        // every unit's boxes start at the same column.
        int cached_col0 = INT32_MIN, t0 = 0, lane_off = 0, pl0 = 15, co[4] = {0, 0, 0, 0};
        for (int u = ur.first; ok && u < ur.end; u += ur.step) {
            // A stage whose planes are reused is skipped here, as by the
            // producer; the MMA warp reads the previous slot again.
            const int kb_first = reuses_prev(u, ur, args) ? 1 : 0;
            for (int kb = kb_first; kb < args.k_stages; ++kb) {
                ok = __all_sync(0xffffffffu,
                                ptx::mbar_wait(&bar->full[stages + rs], rphase, abort, limit)) &&
                     __all_sync(0xffffffffu, ptx::mbar_wait(&bar->empty[ps], pphase ^ 1u, abort, limit));
                if (!ok) break;
                if (kb == kb_first) {
                    const int col0 = static_cast<volatile int32_t*>(bar->raw_col0)[rs];
                    if (col0 != cached_col0) {
                        cached_col0 = col0;
                        // Span column of raw column 0 (the box starts at the
                        // span's 8-column group), and of this lane's first item.
                        const int x_first = -(col0 & 7);
                        t0 = x_first + 8 * g0 + px;
                        if (fast) {
                            const int phi = ((t0 % args.sw) + args.sw) % args.sw;
                            const int jr0 = (t0 - phi) / args.sw;
                            pl0 = static_cast<int>((args.phase_planes >> (4 * phi)) & 15u);
                            const int rr0 =
                                static_cast<int>((args.plane_rows0 >> (4 * pl0)) & 15u) + jr0;
                            lane_off = pl0 * args.plane_bytes + rr0 * 128 + pair;
#pragma unroll
                            for (int m = 0; m < 4; ++m) co[m] = ((half * 4 + m) ^ (rr0 & 7)) << 4;
                        }
                    }
                }
                const uint32_t raw = ptx::smem_addr(base + args.raw_off + rs * args.raw_b) + ld_off;
                uint8_t* slot = ring + ps * stage_bytes;
                // All of this warp's items (at most kTrItems: items <= 64)
                // are read first, so their loads overlap; the conditions
                // are warp-uniform and the warp converged for ldmatrix.
                uint32_t d[kTrItems][4];
                __syncwarp();
#pragma unroll
                for (int q = 0; q < kTrItems; ++q)
                    if (tw + q * kTrWarps < items)
                        ldmatrix_x4_trans(raw + 16u * static_cast<uint32_t>(q * (kTrWarps / 2)), d[q]);
#pragma unroll
                for (int q = 0; q < kTrItems; ++q) {
                    if (tw + q * kTrWarps >= items) break;
                    const int t = t0 + kColStep * q;          // span column of this lane's value
                    if (t < 0 || t >= span) continue;
                    int rr, pl;
                    uint8_t* row;
                    if (fast) {
                        if (pl0 == 15) continue;
                        pl = pl0;
                        row = slot + lane_off + q * row_step * 128;
#pragma unroll
                        for (int m = 0; m < 4; ++m)
                            *reinterpret_cast<uint32_t*>(row + co[m]) = d[q][m];
                    } else {
                        const int jr = t / args.sw, phi = t - jr * args.sw;
                        pl = static_cast<int>((args.phase_planes >> (4 * phi)) & 15u);
                        if (pl == 15) continue;
                        rr = static_cast<int>((args.plane_rows0 >> (4 * pl)) & 15u) + jr;
                        row = slot + pl * args.plane_bytes + rr * 128 + pair;
#pragma unroll
                        for (int m = 0; m < 4; ++m)
                            *reinterpret_cast<uint32_t*>(row + (((half * 4 + m) ^ (rr & 7)) << 4)) = d[q][m];
                    }
                }
                // The raw slot is read (its values are in registers) ...
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bar->empty[stages + rs]);
                // ... and the planes go to the tensor cores (the async proxy).
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bar->full[ps]);
                if (++ps == static_cast<uint32_t>(stages)) { ps = 0; pphase ^= 1u; }
                if (++rs == static_cast<uint32_t>(args.raw_stages)) { rs = 0; rphase ^= 1u; }
            }
        }
        if (!ok && lane == 0) raise_error(args.err, abort, kErrProducer);
        }
    transposers_done:;
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc<1>(tmem, kWtTmemCols);
    }
}

// Items (64 channels x 32 columns of one row) per warp: all their loads are
// in flight before the first transpose.
constexpr int kPrepItemsPerWarp = 1;

// NCHW -> NHWC for 16-bit elements with 16-byte accesses on both sides (C
// and W multiples of 8, x 16-byte aligned), fused with the weight reorder.
// A warp moves kPrepItemsPerWarp items of 64 channels x 32 columns of one
// (image, row): lane (cg, q) loads channels 8cg..8cg+7 at columns 8q..8q+7 as eight 16-byte words,
// transposes the 8 x 8 block with byte permutes and stores eight pixels of
// 8 channels.  For a fixed register a warp reads 8 runs of 64 bytes and
// writes 4 runs of 128 bytes.  Blocks past the transpose reorder the
// weights as reorder_weights_kernel does.
__global__ void __launch_bounds__(256)
    conv_prep_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ xt, int C, int H,
                     int W, int64_t items, unsigned transpose_blocks,
                     const uint16_t* __restrict__ w, uint16_t* __restrict__ wr, int Cp, int kh,
                     int kw, int64_t w_total) {
    ptx::grid_launch_dependents();
    if (blockIdx.x >= transpose_blocks) {
        const int64_t i = static_cast<int64_t>(blockIdx.x - transpose_blocks) * 256 + threadIdx.x;
        if (i >= w_total) return;
        const int ci = static_cast<int>(i % Cp);
        int64_t t = i / Cp;
        const int s = static_cast<int>(t % kw);
        t /= kw;
        const int r = static_cast<int>(t % kh);
        const int64_t co = t / kh;
        wr[i] = ci < C ? w[((co * C + ci) * kh + r) * kw + s] : static_cast<uint16_t>(0);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int wblks = (W + 31) >> 5, cblks = (C + 63) >> 6;
    const int64_t plane = static_cast<int64_t>(H) * W;
    const int64_t first =
        (static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * kPrepItemsPerWarp;
    // Item -> (image, row, channel octet, column octet) of this lane; false
    // past the end (whole octets: C and W are multiples of 8).
    auto locate = [&](int64_t item, int64_t* n, int* h, int* c, int* w0) {
        int64_t t = item;
        const int wb = static_cast<int>(t % wblks);
        t /= wblks;
        const int cb = static_cast<int>(t % cblks);
        t /= cblks;
        *h = static_cast<int>(t % H);
        *n = t / H;
        *c = cb * 64 + (lane & 7) * 8;
        *w0 = wb * 32 + (lane >> 3) * 8;
        return item < items && *c < C && *w0 < W;
    };
    uint4 r[kPrepItemsPerWarp][8];
#pragma unroll
    for (int it = 0; it < kPrepItemsPerWarp; ++it) {
        int64_t n;
        int h, c, w0;
        if (locate(first + it, &n, &h, &c, &w0)) {
            const uint16_t* src = x + ((n * C + c) * H + h) * static_cast<int64_t>(W) + w0;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                r[it][j] = __ldg(reinterpret_cast<const uint4*>(src + j * plane));
        }
    }
#pragma unroll
    for (int it = 0; it < kPrepItemsPerWarp; ++it) {
        int64_t n;
        int h, c, w0;
        if (!locate(first + it, &n, &h, &c, &w0)) continue;
        uint16_t* dst = xt + ((n * H + h) * static_cast<int64_t>(W) + w0) * C + c;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            // Pixel p: channel pairs (2i, 2i+1) from word p/2 of rows 2i, 2i+1.
            const uint32_t sel = (p & 1) ? 0x7632u : 0x5410u;
            uint4 o;
            o.x = __byte_perm(word_of(r[it][0], p >> 1), word_of(r[it][1], p >> 1), sel);
            o.y = __byte_perm(word_of(r[it][2], p >> 1), word_of(r[it][3], p >> 1), sel);
            o.z = __byte_perm(word_of(r[it][4], p >> 1), word_of(r[it][5], p >> 1), sel);
            o.w = __byte_perm(word_of(r[it][6], p >> 1), word_of(r[it][7], p >> 1), sel);
            *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(p) * C) = o;
        }
    }
}

// NCHW -> NHWC for 16-bit elements, one 64-channel x 64-column tile of one
// (image, row) per block.  PAIRS moves 32-bit pairs on both sides (W even;
// C is a multiple of 8), else single elements.
template <bool PAIRS>
__global__ void __launch_bounds__(256)
    nchw_to_nhwc_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ xt, int C, int H,
                        int W) {
    __shared__ uint16_t tile[64][66];
    const int w0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
    const int n = blockIdx.z / H, h = blockIdx.z - (blockIdx.z / H) * H;
    const int lane = threadIdx.x & 31, wrp = threadIdx.x >> 5;
    for (int cc = wrp; cc < 64; cc += 8) {
        const int c = c0 + cc;
        const uint16_t* row = x + ((static_cast<int64_t>(n) * C + c) * H + h) * W;
        if (PAIRS) {
            const int w = w0 + 2 * lane;
            uint32_t v = 0;
            if (c < C && w < W) v = *reinterpret_cast<const uint32_t*>(row + w);
            tile[cc][2 * lane] = static_cast<uint16_t>(v);
            tile[cc][2 * lane + 1] = static_cast<uint16_t>(v >> 16);
        } else {
            for (int j = lane; j < 64; j += 32) {
                const int w = w0 + j;
                tile[cc][j] = (c < C && w < W) ? row[w] : static_cast<uint16_t>(0);
            }
        }
    }
    __syncthreads();
    for (int ww = wrp; ww < 64; ww += 8) {
        const int w = w0 + ww;
        if (w >= W) continue;
        uint16_t* dst = xt + ((static_cast<int64_t>(n) * H + h) * W + w) * C;
        const int c = c0 + 2 * lane;
        if (c < C) {
            const uint32_t v = tile[2 * lane][ww] | (static_cast<uint32_t>(tile[2 * lane + 1][ww]) << 16);
            *reinterpret_cast<uint32_t*>(dst + c) = v;
        }
    }
}

// OIHW weights -> [c_out][r][s][Cp] with the channels zero-padded to Cp.
__global__ void reorder_weights_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ wr,
                                       int C, int Cp, int kh, int kw, int64_t total) {
    ptx::grid_launch_dependents();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int ci = static_cast<int>(i % Cp);
    int64_t t = i / Cp;
    const int s = static_cast<int>(t % kw);
    t /= kw;
    const int r = static_cast<int>(t % kh);
    const int64_t co = t / kh;
    wr[i] = ci < C ? w[((co * C + ci) * kh + r) * kw + s] : static_cast<uint16_t>(0);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_tma_conv() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        tried = true;
    }
    return fn;
}

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

}  // namespace

// Geometry of the TMA convolution, or false when it does not apply.  The
// pixel tile is nr rows x owc columns = 128 pixels, owc a power of two from
// 8 to 128, chosen to compute the fewest pixels over an H-tile (ties: the
// wider rows); output channels go in blocks of up to 256 (a multiple of 16).
bool conv_tma_geometry(const tiles_conv_desc* d, int64_t oh, int64_t ow, int tile_oh, int tile_ow,
                       ConvTmaGeometry* g) {
    if (d->c % 8 || d->sw > 8 || d->sh > 8 || d->dw < 1 || d->dh < 1) return false;
    const int64_t rows = std::min<int64_t>(tile_oh, oh);
    ow = std::min<int64_t>(tile_ow, ow);     // columns of one W-tile
    int64_t best_cost = -1;
    int owc = 0;
    for (int cols = 128; cols >= 8; cols /= 2) {
        const int nr = kTmaConvPixels / cols;
        if (cols * d->sw > 256 || nr * d->sh > 256) continue;
        const int64_t cost = ((ow + cols - 1) / cols) * cols * ((rows + nr - 1) / nr) * nr;
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; owc = cols; }
    }
    if (!owc) return false;
    g->owc = owc;
    g->nr = kTmaConvPixels / owc;
    g->bn = static_cast<int>(std::min<int64_t>(kTmaConvMaxN, (d->c_out + 15) / 16 * 16));
    g->ch_blocks = (d->c + 63) / 64;
    g->cp = g->ch_blocks * 64;
    g->weights_bytes = static_cast<int64_t>(d->c_out) * d->kh * d->kw * g->cp * 2;
    g->x_bytes = d->x_layout == TILES_LAYOUT_NHWC
                     ? 0 : static_cast<int64_t>(d->n) * d->c * d->h * d->w * 2;
    g->weights_offset = 256;
    g->x_offset = align256(g->weights_offset + g->weights_bytes);
    g->ws_bytes = g->x_offset + g->x_bytes;
    return true;
}

// Geometry and shared-memory layout of the weights-in-TMEM kernel.
struct WtPlan {
    int owc = 0, nr = 0, acc_bufs = 0, stages = 0;
    int raw_stages = 0;              // direct rows form: raw box slots (beside `stages` plane slots)
    int stg_pitch = 0, stg_bytes = 0, w_slots = 0, smem = 0;
};

// Pixel tile owc (a multiple of 8) x nr with npix = owc * nr a multiple of
// 16; acc_bufs accumulators of npix columns beside the k_blocks * 32 filter
// columns.  Time model per tile: each K block issues 4 MMAs of npix/2 clocks
// but no faster than ~345 issue clocks (4 MMAs + 1 commit, measured), plus,
// with one accumulator, the drain before the next tile (2 * npix + 400);
// tiles run in rounds over the SMs.  forced_acc = 1 or 2 fixes the count.
// False when the filter does not fit.
bool wtmem_plan(const tiles_conv_desc* d, int64_t oh, int64_t ow, int tile_oh, int tile_ow,
                int64_t k_blocks, int sms, int forced_acc, WtPlan* out) {
    if (d->c_out > 128) return false;
    const int64_t a_cols = k_blocks * 32;
    const int ob = d->out_dtype == TILES_F32 ? 4 : 2;
    const int budget = 227 * 1024 - kSmemBarrierBytes - kSmemAlignSlack;
    const int64_t rows = std::min<int64_t>(tile_oh, oh);
    const int64_t n_ht = (oh + tile_oh - 1) / tile_oh;
    const int64_t n_wt = (ow + tile_ow - 1) / tile_ow;
    ow = std::min<int64_t>(tile_ow, ow);     // columns of one W-tile
    int64_t best = -1;
    for (int acc = 1; acc <= 2; ++acc) {
        if (forced_acc && acc != forced_acc) continue;
        const int64_t nmax = std::min<int64_t>(256, (kWtTmemCols - a_cols) / acc) / 16 * 16;
        for (int owc = 8; owc <= nmax && owc * d->sw <= 256; owc += 8) {
            for (int nr = 1; owc * nr <= nmax && nr * d->sh <= 256; ++nr) {
                const int npix = owc * nr;
                if (npix % 16) continue;
                const int pitch = npix * ob + 16;
                const int stg = 128 * pitch;
                const int stage = npix * 128;
                const int stages = std::min(kMaxStages, (budget - stg) / stage);
                if (stages < 2) continue;
                const int64_t units = static_cast<int64_t>(d->n) * n_ht * ((rows + nr - 1) / nr) *
                                      n_wt * ((ow + owc - 1) / owc);
                const int64_t per_unit = k_blocks * std::max<int64_t>(2 * npix, 345) +
                                         (acc == 1 ? 2 * npix + 400 : 0);
                const int64_t cost = (units + sms - 1) / sms * per_unit;
                if (best < 0 || cost < best || (cost == best && owc > out->owc)) {
                    best = cost;
                    out->owc = owc;
                    out->nr = nr;
                    out->acc_bufs = acc;
                    out->stages = stages;
                    out->stg_pitch = pitch;
                    out->stg_bytes = stg;
                    out->w_slots = (stages * stage + stg) / kWtWeightBlockBytes;
                    // At least half an SM's shared memory, so that one block
                    // (and one 512-column TMEM allocation) sits on each SM.
                    out->smem = std::max(stages * stage + stg + kSmemBarrierBytes + kSmemAlignSlack,
                                         116 * 1024);
                }
            }
        }
    }
    return best >= 0;
}

// Geometry of the rows form: one output row of owc pixels per tile.  Tap s
// of a kernel row reads input columns base + s*dw + j*sw (j < owc): stride
// phase (s*dw) % sw at pixel offset (s*dw) / sw.  Each distinct phase is a
// plane of pmax = owc + max offset pixels (one TMA box, pmax*sw <= 256
// columns wide).  Cost model as in wtmem_plan, with one wait and commit per
// (kernel row, 64 channels) and kw taps of 4 MMAs each per stage.
struct RowsPlan {
    WtPlan wp;
    int n_planes = 0, plane_bytes = 0, pmax = 0;
    int raw_b = 0, xw = 0;           // direct form: raw box bytes and columns
    int tap_plane[8] = {}, tap_shift[8] = {}, plane_phase[8] = {};
};

// direct: the form over an NCHW input read in place, with a ring of raw
// boxes of 64 channel rows x xw columns (xw / 8 odd, at most 256, at least
// the span pmax * sw plus the 7 columns of its 8-column group) beside the
// plane ring: 2 plane stages and as many raw boxes as fit, up to 6.  The raw
// boxes come from DRAM, so their ring is the one whose depth hides latency;
// the plane ring only hands transposed stages to the MMA warp.
bool rows_plan(const tiles_conv_desc* d, int64_t oh, int64_t ow, int tile_oh, int tile_ow,
               int64_t k_blocks, int sms, int forced_acc, bool direct, RowsPlan* out) {
    if (d->c_out > 128 || d->kw > 8) return false;
    RowsPlan rp;
    int qmax = 0;
    for (int t = 0; t < d->kw; ++t) {
        const int c = t * d->dw;
        const int phase = c % d->sw, q = c / d->sw;
        int p = 0;
        while (p < rp.n_planes && rp.plane_phase[p] != phase) ++p;
        if (p == rp.n_planes) rp.plane_phase[rp.n_planes++] = phase;
        rp.tap_plane[t] = p;
        rp.tap_shift[t] = q;
        qmax = std::max(qmax, q);
    }
    const int64_t a_cols = k_blocks * 32;
    const int ob = d->out_dtype == TILES_F32 ? 4 : 2;
    const int budget = 227 * 1024 - kSmemBarrierBytes - kSmemAlignSlack;
    const int64_t rows = std::min<int64_t>(tile_oh, oh);
    const int64_t n_ht = (oh + tile_oh - 1) / tile_oh;
    const int64_t n_wt = (ow + tile_ow - 1) / tile_ow;
    const int64_t wcols = std::min<int64_t>(tile_ow, ow);
    const int64_t stages_k = static_cast<int64_t>(d->kh) * (k_blocks / (d->kh * d->kw));
    int64_t best = -1;
    for (int owc = 16; owc <= 256; owc += 16) {
        const int pmax = owc + qmax;
        if (static_cast<int64_t>(pmax) * d->sw > 256) break;
        int xw = 0;
        if (direct) {
            xw = (pmax * d->sw + 7 + 7) / 8 * 8;
            if ((xw / 8) % 2 == 0) xw += 8;
            if (xw > 256) break;
        }
        int acc = 2 * owc + a_cols <= kWtTmemCols ? 2 : owc + a_cols <= kWtTmemCols ? 1 : 0;
        if (forced_acc) acc = (forced_acc * owc + a_cols <= kWtTmemCols) ? forced_acc : 0;
        if (!acc) continue;
        // Direct form: a plane may start up to 7 rows into its space.
        const int plane_bytes = ((pmax + (direct ? 7 : 0)) * 128 + 1023) / 1024 * 1024;
        const int raw_b = 128 * xw;
        const int planes = rp.n_planes * plane_bytes;
        const int pitch = owc * ob + 16;
        const int stg = 128 * pitch;
        int stages = 0, raw_stages = 0;
        if (direct) {
            stages = 2;
            raw_stages = std::min(kMaxStages - stages, (budget - stg - stages * planes) / raw_b);
            if (raw_stages < 2) continue;
        } else {
            stages = std::min(kMaxStages, (budget - stg) / planes);
            if (stages < 2) continue;
        }
        const int ring_bytes = raw_stages * raw_b + stages * planes;
        const int64_t units = static_cast<int64_t>(d->n) * n_ht * rows * n_wt *
                              ((wcols + owc - 1) / owc);
        const int64_t per_unit = stages_k * (std::max<int64_t>(d->kw * 4 * (owc / 2),
                                                               d->kw * 4 * 55) + 300) +
                                 (acc == 1 ? 2 * owc + 400 : 0);
        const int64_t cost = (units + sms - 1) / sms * per_unit;
        if (best < 0 || cost < best || (cost == best && owc > rp.wp.owc)) {
            best = cost;
            rp.wp.owc = owc;
            rp.wp.nr = 1;
            rp.wp.acc_bufs = acc;
            rp.wp.stages = stages;
            rp.wp.raw_stages = raw_stages;
            rp.wp.stg_pitch = pitch;
            rp.wp.stg_bytes = stg;
            // The filter's start-up passes use everything from raw slot 1
            // on (the direct form's first raw box loads beside them; a 3x3
            // filter read from its OIHW rows starts as high as its 9 boxes
            // allow, so that more raw boxes load beside it).
            rp.wp.w_slots = (ring_bytes + stg - (direct ? raw_b : 0)) / kWtWeightBlockBytes;
            rp.wp.smem = std::max(ring_bytes + stg + kSmemBarrierBytes + kSmemAlignSlack,
                                  116 * 1024);
            rp.pmax = pmax;
            rp.plane_bytes = plane_bytes;
            rp.raw_b = raw_b;
            rp.xw = xw;
        }
    }
    if (best < 0) return false;
    *out = rp;
    return true;
}

// cudaFuncSetAttribute once per kernel and size.
cudaError_t set_smem_attr(const void* fn, std::atomic<int>* cached, int smem) {
    if (cached->load(std::memory_order_relaxed) == smem) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) cached->store(smem, std::memory_order_relaxed);
    return e;
}
std::atomic<int> g_smem_wtmem{0}, g_smem_rows{0}, g_smem_direct{0}, g_smem_tma{0};

int conv2d_tma(const tiles_conv_desc* d, const tiles_config* cfg, int tile_oh, int tile_ow,
               int tile_n, int64_t oh, int64_t ow, const ConvTmaGeometry& g, void* ws,
               size_t ws_bytes, void* stream) {
    const int weights_mode = cfg ? cfg->conv_weights : TILES_CONV_W_AUTO;
    if (!ws || static_cast<int64_t>(ws_bytes) < g.ws_bytes)
        return fail(TILES_ERR_INVALID_ARG, "the TMA convolution needs %lld workspace bytes",
                    (long long)g.ws_bytes);
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) || (reinterpret_cast<uintptr_t>(d->x) & 15u))
        return fail(TILES_ERR_MISALIGNED, "workspace must be 256-byte and x 16-byte aligned");
    if (weights_mode < TILES_CONV_W_AUTO || weights_mode > TILES_CONV_W_TMEM_ROWS_DIRECT)
        return fail(TILES_ERR_INVALID_ARG,
                    "conv_weights must be auto, smem, tmem, tmem_rows or tmem_rows_direct");
    const int forced_acc = cfg ? cfg->acc_bufs : 0;
    if ((weights_mode == TILES_CONV_W_TMEM || weights_mode == TILES_CONV_W_TMEM_ROWS ||
         weights_mode == TILES_CONV_W_TMEM_ROWS_DIRECT) &&
        (forced_acc < 0 || forced_acc > 2))
        return fail(TILES_ERR_INVALID_ARG, "acc_bufs must be 0 (auto), 1 or 2");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "device query: %s", cudaGetErrorString(e));

    // ---- the whole launch is planned before the first kernel goes out ----
    const int64_t k_blocks = static_cast<int64_t>(d->kh) * d->kw * g.ch_blocks;
    WtPlan wp;
    RowsPlan rp;
    bool use_tmem = false, use_rows = false, use_direct = false;
    // The rows form over an NCHW input read directly: 16-byte loads of 8
    // columns (W a multiple of 8), and a stage's span, from its 8-column
    // group, within the transposers' 32 groups.
    if (d->x_layout == TILES_LAYOUT_NCHW && d->w % 8 == 0 &&
        (weights_mode == TILES_CONV_W_AUTO || weights_mode == TILES_CONV_W_TMEM_ROWS_DIRECT))
        use_direct = rows_plan(d, oh, ow, tile_oh, tile_ow, k_blocks, sms,
                               weights_mode == TILES_CONV_W_TMEM_ROWS_DIRECT ? forced_acc : 0,
                               true, &rp);
    if (weights_mode == TILES_CONV_W_TMEM_ROWS_DIRECT && !use_direct)
        return fail(TILES_ERR_INFEASIBLE,
                    "the direct rows form needs an NCHW input with W a multiple of 8, the filter "
                    "in tensor memory, kw <= 8 and an input row span of at most 241 columns");
    use_rows = use_direct;
    if (!use_rows && (weights_mode == TILES_CONV_W_AUTO || weights_mode == TILES_CONV_W_TMEM_ROWS))
        use_rows = rows_plan(d, oh, ow, tile_oh, tile_ow, k_blocks, sms,
                             weights_mode == TILES_CONV_W_TMEM_ROWS ? forced_acc : 0, false, &rp);
    if (weights_mode == TILES_CONV_W_TMEM_ROWS && !use_rows)
        return fail(TILES_ERR_INFEASIBLE,
                    "the rows form needs the filter in tensor memory, kw <= 8 and an input row "
                    "span within one TMA box");
    if (use_rows) {
        wp = rp.wp;
        use_tmem = true;
    } else if (weights_mode != TILES_CONV_W_SMEM) {
        use_tmem = wtmem_plan(d, oh, ow, tile_oh, tile_ow, k_blocks, sms,
                              weights_mode == TILES_CONV_W_TMEM ? forced_acc : 0, &wp);
    }
    if (weights_mode == TILES_CONV_W_TMEM && !use_tmem)
        return fail(TILES_ERR_INFEASIBLE,
                    "the filter does not fit tensor memory (needs c_out <= 128 and kh*kw*ceil(c/64) <= 14)");
    // A 3x3 filter over whole 64-channel blocks that goes to tensor memory
    // (with no NHWC copy of the input to prepare) is read straight from the
    // caller's OIHW rows: the kernel puts it in K order, one pass of 9 boxes
    // per channel block, and there is no reorder launch.  The pass needs 9
    // blocks of start-up space; a smaller plan pads its staging area.
    const bool raw_shape = use_tmem && (d->x_layout != TILES_LAYOUT_NCHW || use_direct) &&
                           d->kh * d->kw == kRawFilterBoxes && d->c % 64 == 0 &&
                           d->c_out <= 128 && (reinterpret_cast<uintptr_t>(d->wt) & 15u) == 0;
    if (raw_shape && wp.w_slots < kRawFilterBoxes) {
        const int extra = (kRawFilterBoxes - wp.w_slots) * kWtWeightBlockBytes;
        if (wp.smem + extra <= 227 * 1024) {
            wp.stg_bytes += extra;
            wp.smem += extra;
            wp.w_slots = kRawFilterBoxes;
        }
    }
    const bool raw_filter = raw_shape && wp.w_slots >= kRawFilterBoxes;
    const int owc = use_tmem ? wp.owc : g.owc;
    const int nr = use_tmem ? wp.nr : g.nr;

    char* wsb = static_cast<char*>(ws);
    uint16_t* wr = reinterpret_cast<uint16_t*>(wsb + g.weights_offset);
    const uint16_t* x_src = static_cast<const uint16_t*>(d->x);
    uint16_t* xt = d->x_layout == TILES_LAYOUT_NCHW && !use_direct
                       ? reinterpret_cast<uint16_t*>(wsb + g.x_offset) : nullptr;
    const uint16_t* xn = xt ? xt : x_src;

    auto fn = encode_fn_tma_conv();
    if (!fn) return fail(TILES_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (no CUDA driver?)");
    const CUtensorMapDataType dt = d->in_dtype == TILES_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tw, tx;
    {
        // Weight rows [c_out][kh*kw*Cp]: K blocks of 64 channels x (the
        // output-channel block, or 128 rows with zero fill for TMEM).  The
        // raw OIHW rows have the same length (Cp = C).
        const int64_t k = static_cast<int64_t>(d->kh) * d->kw * g.cp;
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(d->c_out), 1};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(k) * 2,
                                 static_cast<cuuint64_t>(k) * 2 * static_cast<cuuint64_t>(d->c_out)};
        cuuint32_t box[3] = {64, static_cast<cuuint32_t>(use_tmem ? 128 : g.bn), 1};
        cuuint32_t estr[3] = {1, 1, 1};
        void* wbase = raw_filter ? const_cast<void*>(d->wt) : static_cast<void*>(wr);
        CUresult r = fn(&tw, dt, 3, wbase, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(TILES_ERR_CUDA, "cuTensorMapEncodeTiled(weights) failed (%d)", (int)r);
    }
    if (use_direct) {
        // NCHW input: a stage's raw box is 64 channel rows of xw columns of
        // one input row.
        cuuint64_t dims[4] = {static_cast<cuuint64_t>(d->w), static_cast<cuuint64_t>(d->h),
                              static_cast<cuuint64_t>(d->c), static_cast<cuuint64_t>(d->n)};
        cuuint64_t strides[3] = {static_cast<cuuint64_t>(d->w) * 2,
                                 static_cast<cuuint64_t>(d->h) * d->w * 2,
                                 static_cast<cuuint64_t>(d->c) * d->h * d->w * 2};
        cuuint32_t box[4] = {static_cast<cuuint32_t>(rp.xw), 1, 64, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        CUresult r = fn(&tx, dt, 4, const_cast<uint16_t*>(x_src), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(TILES_ERR_CUDA, "cuTensorMapEncodeTiled(input) failed (%d)", (int)r);
    } else {
        cuuint64_t dims[4] = {static_cast<cuuint64_t>(d->c), static_cast<cuuint64_t>(d->w),
                              static_cast<cuuint64_t>(d->h), static_cast<cuuint64_t>(d->n)};
        cuuint64_t strides[3] = {static_cast<cuuint64_t>(d->c) * 2,
                                 static_cast<cuuint64_t>(d->w) * d->c * 2,
                                 static_cast<cuuint64_t>(d->h) * d->w * d->c * 2};
        // Rows form: one input row, pmax pixels at the column stride; else
        // nr rows x owc columns at both strides.
        cuuint32_t box[4] = {64, static_cast<cuuint32_t>((use_rows ? rp.pmax : owc) * d->sw),
                             static_cast<cuuint32_t>(use_rows ? 1 : nr * d->sh), 1};
        cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(d->sw),
                              static_cast<cuuint32_t>(use_rows ? 1 : d->sh), 1};
        CUresult r = fn(&tx, dt, 4, const_cast<uint16_t*>(xn), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(TILES_ERR_CUDA, "cuTensorMapEncodeTiled(input) failed (%d)", (int)r);
    }

    // Rows form: the epilogue's tile (one output row, owc columns, 128
    // channels) leaves by one TMA store when y's rows are 16-byte multiples,
    // tiles never straddle a W-tile, and y is 16-byte aligned.
    CUtensorMap ty;
    std::memset(&ty, 0, sizeof ty);
    const int yb = d->out_dtype == TILES_F32 ? 4 : 2;
    bool tma_store = false;
    if (use_rows && (reinterpret_cast<uintptr_t>(d->y) & 15u) == 0 && (ow * yb) % 16 == 0 &&
        (std::min<int64_t>(tile_ow, ow) == ow || tile_ow % owc == 0)) {
        const CUtensorMapDataType yt = d->out_dtype == TILES_F32  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : d->out_dtype == TILES_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        cuuint64_t dims[4] = {static_cast<cuuint64_t>(ow), static_cast<cuuint64_t>(oh),
                              static_cast<cuuint64_t>(d->c_out), static_cast<cuuint64_t>(d->n)};
        cuuint64_t strides[3] = {static_cast<cuuint64_t>(ow) * yb,
                                 static_cast<cuuint64_t>(oh) * ow * yb,
                                 static_cast<cuuint64_t>(d->c_out) * oh * ow * yb};
        cuuint32_t box[4] = {static_cast<cuuint32_t>(owc), 1, 128, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        CUresult r = fn(&ty, yt, 4, d->y, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        tma_store = r == CUDA_SUCCESS;
    }

    const int budget = 227 * 1024 - kSmemBarrierBytes - kSmemAlignSlack;
    ConvTmaArgs a{};
    a.y = d->y;
    a.n = d->n; a.c = d->c; a.h = d->h; a.w = d->w; a.c_out = d->c_out; a.kh = d->kh; a.kw = d->kw;
    a.sh = d->sh; a.sw = d->sw; a.pw = d->pw; a.dh = d->dh; a.dw = d->dw;
    a.oh = static_cast<int32_t>(oh); a.ow = static_cast<int32_t>(ow);
    a.owc = owc; a.nr = nr;
    // Column blocks per W-tile (each W-tile's columns start a block).
    const int64_t wcols = std::min<int64_t>(tile_ow, ow);
    a.cblocks = static_cast<int32_t>((wcols + owc - 1) / owc);
    a.ch_blocks = g.ch_blocks;
    a.k_blocks = static_cast<int32_t>(k_blocks);
    a.out_dtype = d->out_dtype;
    a.err = static_cast<int32_t*>(ws);
    a.wait_limit_ns = 2000000000ull;
    // A fault planted by the test hook goes to the first launch (of the TMEM
    // forms, which take it) alone.
    const PlantedFault planted = take_planted_fault();
    a.drop_stage = planted.stage;
    if (planted.stage >= 0) a.wait_limit_ns = planted.limit_ns;
    a.wr = wr;
    a.kp = static_cast<int32_t>(d->kh * d->kw * g.cp);
    const bool y16 = (reinterpret_cast<uintptr_t>(d->y) & 15u) == 0;
    int stages = 0, stage_bytes = 0, smem = 0;
    if (use_tmem) {
        // M = 128 output channels (one block), N = the pixel tile; TMA
        // delivers owc x nr pixel rows of 128 bytes per K block.
        a.npix = owc * nr;
        a.acc_bufs = wp.acc_bufs;
        a.a_col = wp.acc_bufs * a.npix;
        a.nco = 128;
        a.co_blocks = 1;
        if (use_rows) {
            a.k_stages = d->kh * g.ch_blocks;
            a.n_planes = rp.n_planes;
            a.plane_bytes = rp.plane_bytes;
            a.pmax = rp.pmax;
            for (int i = 0; i < 8; ++i) {
                a.tap_plane[i] = rp.tap_plane[i];
                a.tap_shift[i] = rp.tap_shift[i];
                a.plane_phase[i] = rp.plane_phase[i];
            }
            a.stage_b = rp.n_planes * rp.plane_bytes;
            a.tx_bytes = static_cast<uint32_t>(rp.n_planes * rp.pmax * 128);
            a.raw_b = rp.raw_b;
            a.xw = rp.xw;
            a.phase_planes = 0xffffffffu;
            for (int p = 0; p < rp.n_planes; ++p)
                a.phase_planes = (a.phase_planes & ~(15u << (4 * rp.plane_phase[p]))) |
                                 (static_cast<uint32_t>(p) << (4 * rp.plane_phase[p]));
        } else {
            a.k_stages = static_cast<int32_t>(k_blocks);
            a.stage_b = a.npix * 128;
            a.tx_bytes = static_cast<uint32_t>(a.npix * 128);
        }
        {
            const int chunk = d->out_dtype == TILES_F32 ? 4 : 8;
            a.vec_ok = (y16 && ow % chunk == 0 && (wcols == ow || tile_ow % chunk == 0)) ? 1 : 0;
        }
        a.idesc = ptx::idesc_f16_f32acc(d->in_dtype == TILES_BF16, false, 128, a.npix);
        a.stages = wp.stages;
        // FORM 2: [raw ring][plane ring][staging]; else [ring][staging].
        a.raw_stages = use_direct ? wp.raw_stages : 0;
        a.raw_off = 0;
        a.ring_off = use_direct ? wp.raw_stages * a.raw_b : 0;
        a.raw_early = use_direct ? 1 : 0;
        a.w_off = a.raw_early * a.raw_b;
        // Direct form: each plane starts some rows into its space so that
        // the columns one store instruction writes (8 consecutive span
        // columns) fall in 8 different swizzle rows.  At stride 2 the two
        // phase planes' rows coincide when the span's columns start even
        // (the planes need 4 rows between them, mod 8) and are one apart
        // when odd (5 rows); the start's parity is pw's, the same for every
        // tile of the launch.  Other strides: plane p starts p rows in.
        a.plane_rows0 = 0;
        if (use_direct) {
            if (d->sw == 2 && rp.n_planes == 2) {
                const int skew = (d->pw % 2 == 0) ? 4 : 5;
                for (int p = 0; p < 2; ++p)
                    if (rp.plane_phase[p] == 1) a.plane_rows0 |= static_cast<uint32_t>(skew) << (4 * p);
            } else {
                for (int p = 0; p < rp.n_planes; ++p) a.plane_rows0 |= static_cast<uint32_t>(p) << (4 * p);
            }
        }
        a.stg_off = a.ring_off + wp.stages * a.stage_b;
        // A TMA store reads the box densely: [channel][owc pixels].
        a.tma_store = tma_store ? 1 : 0;
        a.raw_filter = raw_filter ? 1 : 0;
        // The direct form runs each CTA on a contiguous run of output rows
        // and, with one channel block per kernel row, lets a row's first
        // stage reuse the planes of the previous row's last stage when they
        // hold the same input row.
        a.contig = use_direct ? 1 : 0;
        a.stg_pitch = tma_store ? owc * yb : wp.stg_pitch;
        a.bar_off = a.stg_off + wp.stg_bytes;
        a.w_slots = wp.w_slots;
        if (use_direct && raw_filter) {
            // Every raw slot below the 9 filter boxes' start-up space loads
            // beside them.
            while (a.raw_early + 1 < a.raw_stages &&
                   a.bar_off - (a.raw_early + 1) * a.raw_b >= kRawFilterBoxes * kWtWeightBlockBytes)
                ++a.raw_early;
            a.w_off = a.raw_early * a.raw_b;
        }
        smem = wp.smem;
        e = use_direct ? set_smem_attr(reinterpret_cast<const void*>(conv_wtmem_kernel<2>),
                                       &g_smem_direct, smem)
            : use_rows ? set_smem_attr(reinterpret_cast<const void*>(conv_wtmem_kernel<1>),
                                       &g_smem_rows, smem)
                       : set_smem_attr(reinterpret_cast<const void*>(conv_wtmem_kernel<0>),
                                       &g_smem_wtmem, smem);
    } else {
        // Weights stay resident in shared memory when there is one output-
        // channel block and they leave room for at least 3 pixel stages;
        // the ring then carries 16 KB pixel tiles.  Otherwise each stage
        // holds a pixel tile and a weight tile.  At most kMaxStages - 1
        // stages (the last barrier slot marks the resident weights).
        const int64_t w_res_bytes = k_blocks * g.bn * 128;
        const bool w_resident =
            (d->c_out + g.bn - 1) / g.bn == 1 && w_res_bytes + 3 * kTmaConvA <= budget;
        stage_bytes = w_resident ? kTmaConvA : (kTmaConvA + g.bn * 128 + 1023) / 1024 * 1024;
        stages = static_cast<int>(std::min<int64_t>(
            kMaxStages - 1, (budget - (w_resident ? w_res_bytes : 0)) / stage_bytes));
        smem = static_cast<int>((w_resident ? w_res_bytes : 0) + stages * stage_bytes) +
               kSmemBarrierBytes + kSmemAlignSlack;
        a.nco = g.bn;
        a.co_blocks = (d->c_out + g.bn - 1) / g.bn;
        // TMA loads ceil(box / stride) elements per dimension: 64 channels
        // x owc x nr = 128 pixel rows of 128 bytes, and bn weight rows.
        a.vec_ok = (y16 && ow % 8 == 0 && (wcols == ow || tile_ow % 8 == 0)) ? 1 : 0;
        a.w_resident = w_resident ? 1 : 0;
        a.w_bytes = static_cast<uint32_t>(w_res_bytes);
        a.tx_bytes = static_cast<uint32_t>(kTmaConvA + (w_resident ? 0 : g.bn * 128));
        a.idesc = ptx::idesc_f16_f32acc(d->in_dtype == TILES_BF16, false, kTmaConvPixels, g.bn);
        e = set_smem_attr(reinterpret_cast<const void*>(conv_tma_kernel), &g_smem_tma, smem);
    }
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "smem attribute: %s", cudaGetErrorString(e));

    // ---- launches: operand preparation, then the convolution ----
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint16_t* wsrc = static_cast<const uint16_t*>(d->wt);
    const int64_t w_total = static_cast<int64_t>(d->c_out) * d->kh * d->kw * g.cp;
    const unsigned w_blocks = static_cast<unsigned>((w_total + 255) / 256);
    if (xt) {
        if (d->c % 8 == 0 && d->w % 8 == 0) {
            // One launch: 16-byte transpose blocks, then weight blocks.
            const int64_t items = static_cast<int64_t>(d->n) * d->h * ((d->c + 63) / 64) *
                                  ((d->w + 31) / 32);
            const int64_t t_blocks = (items + 8 * kPrepItemsPerWarp - 1) / (8 * kPrepItemsPerWarp);
            if (t_blocks + w_blocks > INT32_MAX)
                return fail(TILES_ERR_TOO_LARGE, "input too large for one transpose launch");
            conv_prep_kernel<<<static_cast<unsigned>(t_blocks + w_blocks), 256, 0, st>>>(
                x_src, xt, d->c, d->h, d->w, items, static_cast<unsigned>(t_blocks), wsrc, wr,
                g.cp, d->kh, d->kw, w_total);
        } else {
            reorder_weights_kernel<<<w_blocks, 256, 0, st>>>(wsrc, wr, d->c, g.cp, d->kh, d->kw,
                                                             w_total);
            dim3 grid((d->w + 63) / 64, (d->c + 63) / 64, static_cast<unsigned>(d->n) * d->h);
            if (d->w % 2 == 0)
                nchw_to_nhwc_kernel<true><<<grid, 256, 0, st>>>(x_src, xt, d->c, d->h, d->w);
            else
                nchw_to_nhwc_kernel<false><<<grid, 256, 0, st>>>(x_src, xt, d->c, d->h, d->w);
        }
    } else if (!raw_filter) {
        reorder_weights_kernel<<<w_blocks, 256, 0, st>>>(wsrc, wr, d->c, g.cp, d->kh, d->kw,
                                                         w_total);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "conv prep: %s", cudaGetErrorString(e));

    // Launches: batch tiles (images need no halo) x chunks of up to
    // kConvMaxHTiles H-tiles x chunks of up to kConvMaxWTiles W-tiles.
    const int64_t n_ht_total = (oh + tile_oh - 1) / tile_oh;
    const int64_t n_wt_total = (ow + tile_ow - 1) / tile_ow;
    for (int n0 = 0; n0 < d->n; n0 += tile_n) {
        const int n_imgs = std::min(tile_n, d->n - n0);
        a.img0 = n0;
        for (int64_t hfirst = 0; hfirst < n_ht_total; hfirst += kConvMaxHTiles) {
            const int hcount = static_cast<int>(std::min<int64_t>(kConvMaxHTiles, n_ht_total - hfirst));
            int max_rows = 0;
            for (int i = 0; i < hcount; ++i) {
                const int o0 = static_cast<int>((hfirst + i) * tile_oh);
                const int o1 = static_cast<int>(std::min<int64_t>(o0 + tile_oh, oh));
                tiles_htile t;
                int s = htile_rows(d->h, d->kh, d->sh, d->ph, d->dh, o0, o1, &t);
                if (s != TILES_OK) return fail(s, "htile_rows failed");
                a.ht[i].o0 = o0;
                a.ht[i].rows = static_cast<int16_t>(o1 - o0);
                a.ht[i].pt = static_cast<int16_t>(t.pt);
                a.ht[i].in_start = t.in_start;
                a.ht[i].real_rows = std::max(0, std::min(t.in_end, d->h) - t.in_start);
                max_rows = std::max(max_rows, o1 - o0);
            }
            a.n_htiles = hcount;
            a.rblocks = (max_rows + nr - 1) / nr;
            for (int64_t wfirst = 0; wfirst < n_wt_total; wfirst += kConvMaxWTiles) {
                const int wcount =
                    static_cast<int>(std::min<int64_t>(kConvMaxWTiles, n_wt_total - wfirst));
                for (int i = 0; i < wcount; ++i) {
                    // The width's tiles follow the same slicing formulas.
                    const int q0 = static_cast<int>((wfirst + i) * tile_ow);
                    const int q1 = static_cast<int>(std::min<int64_t>(q0 + tile_ow, ow));
                    tiles_htile t;
                    int s = htile_rows(d->w, d->kw, d->sw, d->pw, d->dw, q0, q1, &t);
                    if (s != TILES_OK) return fail(s, "htile_rows (width) failed");
                    a.wt[i].o0 = q0;
                    a.wt[i].cols = static_cast<int16_t>(q1 - q0);
                    a.wt[i].pl = static_cast<int16_t>(t.pt);
                    a.wt[i].in_start = t.in_start;
                    a.wt[i].unused = 0;
                }
                a.n_wtiles = wcount;
                // Stage reuse (direct form, see reuses_prev): the launch's
                // units of an image are its output rows in order.
                bool full_htiles = true;
                for (int i = 0; i < hcount; ++i) full_htiles = full_htiles && a.ht[i].rows == a.rblocks;
                a.reuse = use_direct && nr == 1 && g.ch_blocks == 1 &&
                                  (d->kh - 1) * d->dh == d->sh && wcount == 1 && a.cblocks == 1 &&
                                  a.co_blocks == 1 && full_htiles
                              ? 1 : 0;
                a.reuse_period = hcount * a.rblocks;
                const int64_t units = static_cast<int64_t>(n_imgs) * hcount * a.rblocks * wcount *
                                      a.cblocks * a.co_blocks;
                if (units > INT32_MAX) return fail(TILES_ERR_TOO_LARGE, "too many tiles");
                a.units = static_cast<int32_t>(units);
                // Programmatic serialization: the blocks launch while the
                // previous kernel on the stream drains and wait for it
                // in-kernel.
                cudaLaunchConfig_t lc{};
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                attr[0].val.programmaticStreamSerializationAllowed = 1;
                lc.gridDim = dim3(static_cast<unsigned>(std::min<int64_t>(units, sms)));
                lc.dynamicSmemBytes = static_cast<size_t>(smem);
                lc.stream = st;
                lc.attrs = attr;
                lc.numAttrs = 1;
                if (use_direct) {
                    lc.blockDim = dim3(kWtDirectThreads);
                    e = cudaLaunchKernelEx(&lc, conv_wtmem_kernel<2>, tw, tx, ty, a);
                } else if (use_tmem) {
                    lc.blockDim = dim3(kWtThreads);
                    e = use_rows ? cudaLaunchKernelEx(&lc, conv_wtmem_kernel<1>, tw, tx, ty, a)
                                 : cudaLaunchKernelEx(&lc, conv_wtmem_kernel<0>, tw, tx, ty, a);
                } else {
                    lc.blockDim = dim3(kGemmThreads);
                    e = cudaLaunchKernelEx(&lc, conv_tma_kernel, tw, tx, a, stages, stage_bytes);
                }
                if (e == cudaSuccess) e = cudaGetLastError();
                if (e != cudaSuccess)
                    return fail(TILES_ERR_CUDA, "conv launch: %s", cudaGetErrorString(e));
                a.drop_stage = -1;
                a.wait_limit_ns = 2000000000ull;
            }
        }
    }
    return TILES_OK;
}

}  // namespace tiles
