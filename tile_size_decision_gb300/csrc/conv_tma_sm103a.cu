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
// (the K-major B operand in the same K order), and an NCHW input is first
// transposed to NHWC; both go to the caller's workspace.
#include <cuda_runtime.h>

#include <algorithm>
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
    uint32_t tx_bytes;                    // bytes the boxes of a stage deliver
    int32_t vec_ok;                       // 16-byte output stores are aligned (OW % 8 == 0)
    int32_t w_resident;                   // weights loaded once into shared memory
    uint32_t w_bytes;                     // resident weights: all K blocks x nco rows
    int32_t out_dtype;
    uint32_t idesc;
    int32_t* err;
    uint64_t wait_limit_ns;
    ConvHTile ht[kConvMaxHTiles];
};

struct ConvUnit { int img, ht, rb, cb, mb; };

__device__ __forceinline__ ConvUnit decode_conv_unit(int u, const ConvTmaArgs& a) {
    ConvUnit c;
    c.mb = u % a.co_blocks;
    u /= a.co_blocks;
    c.cb = u % a.cblocks;
    u /= a.cblocks;
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
                const int row0 = ht.in_start - ht.pt + cu.rb * args.nr * args.sh;
                const int col0 = cu.cb * args.owc * args.sw - args.pw;
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
                                row0 + r * args.dh, cu.img);
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
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool weights_ready = !args.w_resident;
            for (int u = blockIdx.x; u < args.units; u += gridDim.x) {
                if (!weights_ready) {
                    if (!ptx::mbar_wait(&bar->full[kMaxStages - 1], 0, abort, limit)) {
                        raise_error(args.err, abort, kErrMma);
                        break;
                    }
                    weights_ready = true;
                }
                if (!ptx::mbar_wait(&bar->acc_empty[acc], acc_phase ^ 1u, abort, limit)) {
                    raise_error(args.err, abort, kErrMma);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d = tmem + acc * kTmaConvMaxN;
                bool ok = true;
                for (int kb = 0; kb < args.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(&bar->full[stage], phase, abort, limit)) {
                        raise_error(args.err, abort, kErrMma);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a0 = ptx::smem_addr(ring + stage * stage_bytes);
                    const uint32_t b0 = args.w_resident ? ptx::smem_addr(wres + kb * w_kblock_bytes)
                                                        : a0 + kTmaConvA;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // Both operands K-major: 16 channels = 32 bytes of a
                        // 128-byte row; 8-row groups 1024 B apart.
                        const uint64_t ad = ptx::smem_desc_sw128(a0 + kk * 32, 16, 1024);
                        const uint64_t bd = ptx::smem_desc_sw128(b0 + kk * 32, 16, 1024);
                        ptx::mma_f16<1>(d, ad, bd, args.idesc, (kb | kk) != 0);
                    }
                    ptx::mma_commit<1>(&bar->empty[stage]);
                    if (++stage == static_cast<uint32_t>(stages)) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit<1>(&bar->acc_full[acc]);
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            ptx::mma_commit_local<1>(&bar->drain);
            ptx::mbar_wait(&bar->drain, 0, nullptr, limit);
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
            const int oh = ht.o0 + cu.rb * args.nr + rr;
            const int ow = cu.cb * args.owc + cc;
            const bool pix_ok = rr < args.nr && oh < ht.o0 + ht.rows && ow < args.ow;
            // Element index of (img, co = 0, oh, ow); channel co adds co * plane.
            const int64_t pix = static_cast<int64_t>(cu.img) * args.c_out * plane +
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
            const int ow_g = cu.cb * args.owc + (pg - rr_g * args.owc);
            const bool row_g = rr_g < args.nr && oh_g < ht.o0 + ht.rows;
            const int64_t pix_g = static_cast<int64_t>(cu.img) * args.c_out * plane +
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
                        if (args.vec_ok && ow_g + 8 <= args.ow) {
                            *reinterpret_cast<uint4*>(dst) = make_uint4(w0, w1, w2, w3);
                        } else {
                            const uint32_t wv[4] = {w0, w1, w2, w3};
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                if (ow_g + e < args.ow)
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
bool conv_tma_geometry(const tiles_conv_desc* d, int64_t oh, int64_t ow, int tile_oh,
                       ConvTmaGeometry* g) {
    if (d->c % 8 || d->sw > 8 || d->sh > 8 || d->dw < 1 || d->dh < 1) return false;
    const int64_t rows = std::min<int64_t>(tile_oh, oh);
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

int conv2d_tma(const tiles_conv_desc* d, int tile_oh, int64_t oh, int64_t ow,
               const ConvTmaGeometry& g, void* ws, size_t ws_bytes, void* stream) {
    if (!ws || static_cast<int64_t>(ws_bytes) < g.ws_bytes)
        return fail(TILES_ERR_INVALID_ARG, "the TMA convolution needs %lld workspace bytes",
                    (long long)g.ws_bytes);
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) || (reinterpret_cast<uintptr_t>(d->x) & 15u))
        return fail(TILES_ERR_MISALIGNED, "workspace must be 256-byte and x 16-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* wsb = static_cast<char*>(ws);
    uint16_t* wr = reinterpret_cast<uint16_t*>(wsb + g.weights_offset);
    const uint16_t* xn = static_cast<const uint16_t*>(d->x);
    {
        const int64_t total = static_cast<int64_t>(d->c_out) * d->kh * d->kw * g.cp;
        reorder_weights_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(
            static_cast<const uint16_t*>(d->wt), wr, d->c, g.cp, d->kh, d->kw, total);
    }
    if (d->x_layout == TILES_LAYOUT_NCHW) {
        uint16_t* xt = reinterpret_cast<uint16_t*>(wsb + g.x_offset);
        dim3 grid((d->w + 63) / 64, (d->c + 63) / 64, static_cast<unsigned>(d->n) * d->h);
        if (d->w % 2 == 0 && (reinterpret_cast<uintptr_t>(xn) & 3u) == 0)
            nchw_to_nhwc_kernel<true><<<grid, 256, 0, st>>>(xn, xt, d->c, d->h, d->w);
        else
            nchw_to_nhwc_kernel<false><<<grid, 256, 0, st>>>(xn, xt, d->c, d->h, d->w);
        xn = xt;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "conv prep: %s", cudaGetErrorString(e));

    auto fn = encode_fn_tma_conv();
    if (!fn) return fail(TILES_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (no CUDA driver?)");
    const CUtensorMapDataType dt = d->in_dtype == TILES_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tw, tx;
    {
        const int64_t k = static_cast<int64_t>(d->kh) * d->kw * g.cp;
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(d->c_out), 1};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(k) * 2,
                                 static_cast<cuuint64_t>(k) * 2 * static_cast<cuuint64_t>(d->c_out)};
        cuuint32_t box[3] = {64, static_cast<cuuint32_t>(g.bn), 1};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = fn(&tw, dt, 3, wr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(TILES_ERR_CUDA, "cuTensorMapEncodeTiled(weights) failed (%d)", (int)r);
    }
    {
        cuuint64_t dims[4] = {static_cast<cuuint64_t>(d->c), static_cast<cuuint64_t>(d->w),
                              static_cast<cuuint64_t>(d->h), static_cast<cuuint64_t>(d->n)};
        cuuint64_t strides[3] = {static_cast<cuuint64_t>(d->c) * 2,
                                 static_cast<cuuint64_t>(d->w) * d->c * 2,
                                 static_cast<cuuint64_t>(d->h) * d->w * d->c * 2};
        cuuint32_t box[4] = {64, static_cast<cuuint32_t>(g.owc * d->sw),
                             static_cast<cuuint32_t>(g.nr * d->sh), 1};
        cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(d->sw), static_cast<cuuint32_t>(d->sh), 1};
        CUresult r = fn(&tx, dt, 4, const_cast<uint16_t*>(xn), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(TILES_ERR_CUDA, "cuTensorMapEncodeTiled(input) failed (%d)", (int)r);
    }
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    // Weights stay resident in shared memory when there is one output-
    // channel block and they leave room for at least 3 pixel stages; the
    // ring then carries 16 KB pixel tiles.  Otherwise each stage holds a
    // pixel tile and a weight tile.  At most kMaxStages - 1 stages (the last
    // barrier slot marks the resident weights).
    const int budget = 227 * 1024 - kSmemBarrierBytes - kSmemAlignSlack;
    const int64_t k_blocks = static_cast<int64_t>(d->kh) * d->kw * g.ch_blocks;
    const int64_t w_res_bytes = k_blocks * g.bn * 128;
    const bool w_resident = (d->c_out + g.bn - 1) / g.bn == 1 && w_res_bytes + 3 * kTmaConvA <= budget;
    const int stage_bytes = w_resident ? kTmaConvA : (kTmaConvA + g.bn * 128 + 1023) / 1024 * 1024;
    const int stages = static_cast<int>(std::min<int64_t>(
        kMaxStages - 1, (budget - (w_resident ? w_res_bytes : 0)) / stage_bytes));
    const int smem = static_cast<int>((w_resident ? w_res_bytes : 0) + stages * stage_bytes) +
                     kSmemBarrierBytes + kSmemAlignSlack;
    e = cudaFuncSetAttribute(conv_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "smem attribute: %s", cudaGetErrorString(e));

    ConvTmaArgs a{};
    a.y = d->y;
    a.n = d->n; a.c = d->c; a.h = d->h; a.w = d->w; a.c_out = d->c_out; a.kh = d->kh; a.kw = d->kw;
    a.sh = d->sh; a.sw = d->sw; a.pw = d->pw; a.dh = d->dh; a.dw = d->dw;
    a.oh = static_cast<int32_t>(oh); a.ow = static_cast<int32_t>(ow);
    a.owc = g.owc; a.nr = g.nr; a.nco = g.bn;
    a.cblocks = static_cast<int32_t>((ow + g.owc - 1) / g.owc);
    a.co_blocks = (d->c_out + g.bn - 1) / g.bn;
    a.ch_blocks = g.ch_blocks;
    a.k_blocks = d->kh * d->kw * g.ch_blocks;
    // TMA loads ceil(box / stride) elements per dimension: 64 channels x owc
    // x nr = 128 pixel rows of 128 bytes, and bn weight rows of 128 bytes.
    a.vec_ok = ((reinterpret_cast<uintptr_t>(d->y) & 15u) == 0 && ow % 8 == 0) ? 1 : 0;
    a.w_resident = w_resident ? 1 : 0;
    a.w_bytes = static_cast<uint32_t>(w_res_bytes);
    a.tx_bytes = static_cast<uint32_t>(kTmaConvA + (w_resident ? 0 : g.bn * 128));
    a.out_dtype = d->out_dtype;
    a.idesc = ptx::idesc_f16_f32acc(d->in_dtype == TILES_BF16, false, kTmaConvPixels, g.bn);
    a.err = static_cast<int32_t*>(ws);
    a.wait_limit_ns = 2000000000ull;

    const int64_t n_ht_total = (oh + tile_oh - 1) / tile_oh;
    for (int64_t first = 0; first < n_ht_total; first += kConvMaxHTiles) {
        const int count = static_cast<int>(std::min<int64_t>(kConvMaxHTiles, n_ht_total - first));
        int max_rows = 0;
        for (int i = 0; i < count; ++i) {
            const int o0 = static_cast<int>((first + i) * tile_oh);
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
        a.n_htiles = count;
        a.rblocks = (max_rows + g.nr - 1) / g.nr;
        const int64_t units = static_cast<int64_t>(d->n) * count * a.rblocks * a.cblocks * a.co_blocks;
        if (units > INT32_MAX) return fail(TILES_ERR_TOO_LARGE, "too many tiles");
        a.units = static_cast<int32_t>(units);
        const int grid = static_cast<int>(std::min<int64_t>(units, sms));
        conv_tma_kernel<<<grid, kGemmThreads, smem, st>>>(tw, tx, a, stages, stage_bytes);
        e = cudaGetLastError();
        if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "conv launch: %s", cudaGetErrorString(e));
    }
    return TILES_OK;
}

}  // namespace tiles
