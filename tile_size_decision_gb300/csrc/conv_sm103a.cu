// H-tiled implicit-GEMM convolution for sm_103a.
//
// Per (image, output H-tile, c_out block, column block) the block computes a
// 128 x BN tile of the GEMM described in conv_sm103a.cuh:
//   warp 0      TMA producer of the weight tile (A, 128 x 64 per stage).
//   warp 1      TMEM owner; one lane issues tcgen05.mma (4 per stage).
//   warps 2-5   epilogue (as the GEMM's), rows = output channels, columns =
//               output pixels of the tile, row pitch OH*OW.
//   warps 6-9   gather the im2col operand (B, 64 x BN per stage) straight
//               into the 128-byte-swizzled MN-major layout the MMA reads:
//               element (k, p) with k = (ci, r, s) and p = (oh - o0)*OW + ow
//               is x[n][ci][in_start + l][iw] with
//                   l  = (oh - o0)*sh - pt' + r*dh,  0 <= l < real_rows,
//                   iw = ow*sw - pw + s*dw,           0 <= iw < W,
//               else zero: the sub-operator on the tile's input slice with
//               its own pads pt' (top) and pb' (bottom: l >= real_rows).
// The stage's full barrier counts the TMA's transaction bytes and one
// arrival per gather warp (after a proxy fence, so the tensor core sees the
// threads' shared-memory writes).
#include <cuda_runtime.h>

#include <algorithm>
#include <cudaTypedefs.h>

#include "conv_sm103a.cuh"
#include "gemm_sm103a.cuh"

namespace tiles {

namespace {

constexpr int kConvBN = 256;
constexpr int kConvStages = 4;
using CL = GemmLayout<kConvBN, kConvStages, 1>;

__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct ConvCoord { int img, ht, mb, nb; };

__device__ __forceinline__ ConvCoord decode_conv_tile(int t, const ConvArgs& a) {
    ConvCoord c;
    c.mb = t % a.m_blocks;
    t /= a.m_blocks;
    c.nb = t % a.n_blocks;
    t /= a.n_blocks;
    c.ht = t % a.n_htiles;
    c.img = t / a.n_htiles;
    return c;
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kConvThreads, 1)
    conv_htiled_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ ConvArgs args) {
    using L = GemmLayout<BN, STAGES, 1>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    uint8_t* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* smA = base;
    uint8_t* smB = base + STAGES * L::A_BYTES;
    PipeBarriers* bar = reinterpret_cast<PipeBarriers*>(base + L::OPERAND_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&bar->full[s], 1 + kConvGatherThreads / 32);
            ptx::mbar_init(&bar->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&bar->acc_full[a], 1);
            ptx::mbar_init(&bar->acc_empty[a], 4);
        }
        ptx::mbar_init(&bar->drain, 1);
        bar->abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) ptx::tma_prefetch_desc(&tmW);
    if (warp == 1) {
        ptx::tmem_alloc<1>(&bar->tmem_base, L::TMEM_COLS);
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
            // ---------------- weight TMA producer ----------------
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool aborted = false;
            for (int t = blockIdx.x; t < args.tiles && !aborted; t += gridDim.x) {
                const ConvCoord cc = decode_conv_tile(t, args);
                for (int kb = 0; kb < args.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(&bar->empty[stage], phase ^ 1u, abort, limit)) {
                        raise_error(args.err, abort, kErrProducer);
                        aborted = true;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&bar->full[stage], L::A_BYTES);
                    ptx::tma_load_3d(smA + stage * L::A_BYTES, &tmW, &bar->full[stage], kb * L::BK,
                                     cc.mb * 128, 0);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (aborted) {
                settle_after_abort();
            } else {
                for (int i = 0; i < (issued < STAGES ? issued : STAGES); ++i) {
                    if (stage == 0) { stage = STAGES - 1; phase ^= 1u; } else { --stage; }
                    ptx::mbar_wait(&bar->full[stage], phase, nullptr, limit);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            for (int t = blockIdx.x; t < args.tiles; t += gridDim.x) {
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
                        const uint64_t ad = ptx::smem_desc_sw128(a0 + kk * 32, 16, 1024);
                        const uint64_t bd = ptx::smem_desc_sw128(b0 + kk * 2048, L::B_CHUNK, 1024);
                        ptx::mma_f16<1>(d, ad, bd, args.idesc, (kb | kk) != 0);
                    }
                    ptx::mma_commit<1>(&bar->empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit<1>(&bar->acc_full[acc]);
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            ptx::mma_commit_local<1>(&bar->drain);
            ptx::mbar_wait(&bar->drain, 0, nullptr, limit);
        }
    } else if (warp < 6) {
        // ---------------- epilogue (warps 2-5) ----------------
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
        const int out_bytes = args.out_dtype == TILES_F32 ? 4 : 2;
        const int64_t plane = static_cast<int64_t>(args.oh) * args.ow;
        uint32_t acc = 0, acc_phase = 0;
        for (int t = blockIdx.x; t < args.tiles; t += gridDim.x) {
            const ConvCoord cc = decode_conv_tile(t, args);
            bool ok = ptx::mbar_wait(&bar->acc_full[acc], acc_phase, abort, limit);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) raise_error(args.err, abort, kErrEpilogue);
                break;
            }
            ptx::tc_fence_after();
            const ConvHTile ht = args.ht[cc.ht];
            const int64_t ntile = static_cast<int64_t>(ht.rows) * args.ow;
            const int64_t co = static_cast<int64_t>(cc.mb) * 128 + row_in_tile;
            const bool row_ok = co < args.c_out;
            char* crow = static_cast<char*>(args.y) +
                         ((static_cast<int64_t>(cc.img) * args.c_out + co) * plane +
                          static_cast<int64_t>(ht.o0) * args.ow) * out_bytes;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                ptx::tmem_ld_32cols(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN + c * 32, v);
                ptx::tmem_ld_wait();
                const int64_t col0 = static_cast<int64_t>(cc.nb) * BN + c * 32;
                if (row_ok && col0 < ntile)
                    store_row_chunk(crow, col0, ntile, v, args.out_dtype, args.vec_ok != 0);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar->acc_empty[acc]);
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
    } else {
        // ---------------- im2col gather (warps 6-9) ----------------
        const int gt = threadIdx.x - 6 * 32;                 // 0..127
        constexpr int kChunksPerRow = BN / 8;                 // 16-byte chunks per K row
        constexpr int kChunksPerThread = L::BK * kChunksPerRow / kConvGatherThreads;
        const int khw = args.kh * args.kw;
        const int64_t chw = static_cast<int64_t>(args.h) * args.w;
        const uint16_t* x = static_cast<const uint16_t*>(args.x);
        uint32_t stage = 0, phase = 0;
        bool aborted = false;
        for (int t = blockIdx.x; t < args.tiles && !aborted; t += gridDim.x) {
            const ConvCoord cc = decode_conv_tile(t, args);
            const ConvHTile ht = args.ht[cc.ht];
            const int ntile = ht.rows * args.ow;
            const uint16_t* ximg = x + static_cast<int64_t>(cc.img) * args.c * chw;
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                bool ok = ptx::mbar_wait(&bar->empty[stage], phase ^ 1u, abort, limit);
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) raise_error(args.err, abort, kErrConvGather);
                    aborted = true;
                    break;
                }
                uint8_t* bst = smB + stage * L::B_BYTES;
#pragma unroll 4
                for (int it = 0; it < kChunksPerThread; ++it) {
                    const int chunk = it * kConvGatherThreads + gt;
                    const int kr = chunk / kChunksPerRow;
                    const int c8 = chunk - kr * kChunksPerRow;
                    const int k = kb * L::BK + kr;
                    const int p0 = cc.nb * BN + c8 * 8;
                    uint32_t packed[4] = {0u, 0u, 0u, 0u};
                    if (k < args.k && p0 < ntile) {
                        const int ci = k / khw;
                        const int rs = k - ci * khw;
                        const int r = rs / args.kw;
                        const int s = rs - r * args.kw;
                        const uint16_t* xc = ximg + static_cast<int64_t>(ci) * chw +
                                             static_cast<int64_t>(ht.in_start) * args.w;
                        int ohl = p0 / args.ow;
                        int ow = p0 - ohl * args.ow;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            uint32_t val = 0;
                            if (p0 + e < ntile) {
                                const int l = ohl * args.sh - ht.pt + r * args.dh;
                                const int iw = ow * args.sw - args.pw + s * args.dw;
                                if (static_cast<unsigned>(l) < static_cast<unsigned>(ht.real_rows) &&
                                    static_cast<unsigned>(iw) < static_cast<unsigned>(args.w))
                                    val = __ldg(xc + static_cast<int64_t>(l) * args.w + iw);
                            }
                            packed[e >> 1] |= val << ((e & 1) * 16);
                            if (++ow == args.ow) { ow = 0; ++ohl; }
                        }
                    }
                    // MN-major, 128-byte swizzle: 64-column atoms of 64 K rows;
                    // the 16-byte chunk index is XORed with the row index mod 8.
                    const int atom = c8 >> 3;
                    const int phys = (c8 & 7) ^ (kr & 7);
                    *reinterpret_cast<uint4*>(bst + atom * L::B_CHUNK + kr * 128 + phys * 16) =
                        make_uint4(packed[0], packed[1], packed[2], packed[3]);
                }
                fence_async_shared();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bar->full[stage]);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc<1>(tmem, L::TMEM_COLS);
    }
}

int bytes_of(int dtype) {
    switch (dtype) {
        case TILES_F16: case TILES_BF16: return 2;
        case TILES_F32: return 4;
        default: return 0;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 conv_encode_fn() {
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

}  // namespace

int conv_out_hw(const tiles_conv_desc* d, int64_t* oh, int64_t* ow) {
    if (!d) return fail(TILES_ERR_INVALID_ARG, "null descriptor");
    if (d->h < 1 || d->w < 1 || d->kh < 1 || d->kw < 1 || d->sh < 1 || d->sw < 1 || d->dh < 1 ||
        d->dw < 1 || d->ph < 0 || d->pw < 0)
        return fail(TILES_ERR_INVALID_ARG, "sizes, strides and dilations must be >= 1, pads >= 0");
    // Output extent of a padded, dilated, strided window sweep: the windows
    // (k-1)*d+1 wide that fit in h + 2p, one every s.
    const int64_t span_h = static_cast<int64_t>(d->kh - 1) * d->dh + 1;
    const int64_t span_w = static_cast<int64_t>(d->kw - 1) * d->dw + 1;
    const int64_t in_h = static_cast<int64_t>(d->h) + 2 * d->ph;
    const int64_t in_w = static_cast<int64_t>(d->w) + 2 * d->pw;
    if (in_h < span_h || in_w < span_w) return fail(TILES_ERR_INVALID_ARG, "empty output");
    *oh = (in_h - span_h) / d->sh + 1;
    *ow = (in_w - span_w) / d->sw + 1;
    return TILES_OK;
}

int conv2d_tiled(const tiles_conv_desc* d, int tile_oh, int tile_ow, int tile_n,
                 const tiles_config* cfg, void* ws, size_t ws_bytes, void* stream) {
    if (!d) return fail(TILES_ERR_INVALID_ARG, "null descriptor");
    if (!d->x || !d->wt || !d->y) return fail(TILES_ERR_INVALID_ARG, "null tensor pointer");
    if (d->n < 1 || d->c < 1 || d->h < 1 || d->w < 1 || d->c_out < 1 || d->kh < 1 || d->kw < 1 ||
        d->sh < 1 || d->sw < 1 || d->dh < 1 || d->dw < 1 || d->ph < 0 || d->pw < 0 || tile_oh < 1)
        return fail(TILES_ERR_INVALID_ARG, "sizes, strides and dilations must be >= 1, pads >= 0");
    if (d->in_dtype != TILES_F16 && d->in_dtype != TILES_BF16)
        return fail(TILES_ERR_UNSUPPORTED_DTYPE, "x and w must be f16 or bf16");
    const int ob = bytes_of(d->out_dtype);
    if (!ob) return fail(TILES_ERR_UNSUPPORTED_DTYPE, "y must be f32, f16 or bf16");
    if (d->x_layout != TILES_LAYOUT_NCHW && d->x_layout != TILES_LAYOUT_NHWC)
        return fail(TILES_ERR_INVALID_ARG, "unknown input layout %d", d->x_layout);
    const int64_t k = static_cast<int64_t>(d->c) * d->kh * d->kw;
    if ((reinterpret_cast<uintptr_t>(d->x) & 1u) || (reinterpret_cast<uintptr_t>(d->y) & (ob - 1)) ||
        (reinterpret_cast<uintptr_t>(d->wt) & 1u))
        return fail(TILES_ERR_MISALIGNED, "x, w and y must be element aligned");
    int64_t oh = 0, ow = 0;
    const int hw = conv_out_hw(d, &oh, &ow);
    if (hw != TILES_OK) return hw;
    // tile_ow / tile_n <= 0: the whole width / batch in one tile.
    if (tile_ow <= 0 || tile_ow > ow) tile_ow = static_cast<int>(std::min<int64_t>(ow, INT32_MAX));
    if (tile_n <= 0 || tile_n > d->n) tile_n = d->n;
    const int64_t tile_cols = static_cast<int64_t>(std::min<int64_t>(tile_oh, oh)) * ow;
    if (tile_oh > 32767 || d->ph > 32767 || d->pw > 32767)
        return fail(TILES_ERR_TOO_LARGE, "tile_oh and the pads must be below 32768");
    if (tile_ow < ow && tile_ow > 32767)
        return fail(TILES_ERR_TOO_LARGE, "tile_ow must be below 32768");
    if (k > (1 << 24) || tile_cols > (1 << 30) || static_cast<int64_t>(d->n) * d->c * d->h * d->w > (1ll << 40))
        return fail(TILES_ERR_TOO_LARGE, "convolution too large");
    // The workspace carries the kernels' timeout report: without one an
    // expired wait would go unreported.
    if (!ws || ws_bytes < kConvMinWorkspaceBytes)
        return fail(TILES_ERR_INVALID_ARG, "a workspace of at least %d bytes is required",
                    kConvMinWorkspaceBytes);

    // Producer: the TMA im2col when it applies and the workspace holds its
    // prepared operands (or when forced), else the thread gather.
    const bool force_tma = cfg && cfg->threads == kGemmThreads;
    const bool force_gather = cfg && cfg->threads == kConvThreads;
    if (cfg && !force_tma && !force_gather)
        return fail(TILES_ERR_INFEASIBLE, "conv cfg: threads 192 (TMA producer) or 320 (gather)");
    ConvTmaGeometry g;
    const bool tma_ok = conv_tma_geometry(d, oh, ow, tile_oh, tile_ow, &g);
    if (force_tma && !tma_ok)
        return fail(TILES_ERR_INFEASIBLE, "the TMA producer does not apply to this convolution");
    if (!force_gather && tma_ok && (force_tma || (ws && static_cast<int64_t>(ws_bytes) >= g.ws_bytes)))
        return conv2d_tma(d, cfg, tile_oh, tile_ow, tile_n, oh, ow, g, ws, ws_bytes, stream);
    if (d->x_layout != TILES_LAYOUT_NCHW)
        return fail(TILES_ERR_INFEASIBLE, "NHWC input needs the TMA producer (and its workspace)");
    if (tile_ow < ow)
        return fail(TILES_ERR_INFEASIBLE, "W-tiles need the TMA producer (and its workspace)");
    if (tile_n < d->n) {
        // Batch tiles share no input rows: each is the same convolution on
        // its own images (pointers moved by whole images).
        for (int n0 = 0; n0 < d->n; n0 += tile_n) {
            tiles_conv_desc sub = *d;
            sub.n = std::min(tile_n, d->n - n0);
            const int ib = bytes_of(d->in_dtype);
            sub.x = static_cast<const char*>(d->x) +
                    static_cast<int64_t>(n0) * d->c * d->h * d->w * ib;
            sub.y = static_cast<char*>(d->y) + static_cast<int64_t>(n0) * d->c_out * oh * ow * ob;
            const int s = conv2d_tiled(&sub, tile_oh, tile_ow, sub.n, cfg, ws, ws_bytes, stream);
            if (s != TILES_OK) return s;
        }
        return TILES_OK;
    }
    if (k % 8) return fail(TILES_ERR_MISALIGNED, "c*kh*kw must be a multiple of 8 (weight rows)");
    if (reinterpret_cast<uintptr_t>(d->wt) & 15u)
        return fail(TILES_ERR_MISALIGNED, "w must be 16-byte aligned");

    auto fn = conv_encode_fn();
    if (!fn) return fail(TILES_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (no CUDA driver?)");
    CUtensorMap tw;
    {
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(d->c_out), 1};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(k) * 2,
                                 static_cast<cuuint64_t>(k) * 2 * static_cast<cuuint64_t>(d->c_out)};
        cuuint32_t box[3] = {64, 128, 1};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = fn(&tw, d->in_dtype == TILES_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(d->wt), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(TILES_ERR_CUDA, "cuTensorMapEncodeTiled(weights) failed (%d)", (int)r);
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "device query: %s", cudaGetErrorString(e));

    auto kernel = conv_htiled_kernel<kConvBN, kConvStages>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CL::SMEM_BYTES);
    if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "smem attribute: %s", cudaGetErrorString(e));

    ConvArgs a{};
    a.x = d->x; a.y = d->y;
    a.n = d->n; a.c = d->c; a.h = d->h; a.w = d->w; a.c_out = d->c_out; a.kh = d->kh; a.kw = d->kw;
    a.sh = d->sh; a.sw = d->sw; a.pw = d->pw; a.dh = d->dh; a.dw = d->dw;
    a.oh = static_cast<int32_t>(oh); a.ow = static_cast<int32_t>(ow);
    a.k = static_cast<int32_t>(k);
    a.m_blocks = (d->c_out + 127) / 128;
    a.n_blocks = static_cast<int32_t>((tile_cols + kConvBN - 1) / kConvBN);
    a.k_blocks = static_cast<int32_t>((k + 63) / 64);
    a.out_dtype = d->out_dtype;
    a.idesc = ptx::idesc_f16_f32acc(d->in_dtype == TILES_BF16, true, 128, kConvBN);
    a.err = (ws && ws_bytes >= sizeof(int32_t)) ? static_cast<int32_t*>(ws) : nullptr;
    a.wait_limit_ns = 2000000000ull;
    // 16-byte stores need every row and tile start on a 16-byte boundary.
    const int64_t plane_bytes = oh * ow * ob;
    const int64_t tile_bytes = static_cast<int64_t>(tile_oh) * ow * ob;
    a.vec_ok = ((reinterpret_cast<uintptr_t>(d->y) & 15u) == 0 && plane_bytes % 16 == 0 &&
                tile_bytes % 16 == 0) ? 1 : 0;

    // H-tiles [o0, min(o0 + tile_oh, OH)), in launches of at most
    // kConvMaxHTiles; each tile's slice and pads come from htile_rows.
    const int64_t n_ht_total = (oh + tile_oh - 1) / tile_oh;
    for (int64_t first = 0; first < n_ht_total; first += kConvMaxHTiles) {
        const int count = static_cast<int>(std::min<int64_t>(kConvMaxHTiles, n_ht_total - first));
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
        }
        a.n_htiles = count;
        const int64_t tiles = static_cast<int64_t>(d->n) * count * a.m_blocks * a.n_blocks;
        if (tiles > INT32_MAX) return fail(TILES_ERR_TOO_LARGE, "too many tiles");
        a.tiles = static_cast<int32_t>(tiles);
        const int grid = static_cast<int>(std::min<int64_t>(tiles, sms));
        kernel<<<grid, kConvThreads, CL::SMEM_BYTES, static_cast<cudaStream_t>(stream)>>>(tw, a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return fail(TILES_ERR_CUDA, "conv launch: %s", cudaGetErrorString(e));
    }
    return TILES_OK;
}

int64_t conv_workspace_bytes(const tiles_conv_desc* d, int tile_oh) {
    if (!d || tile_oh < 1 || d->kh < 1 || d->kw < 1 || d->sh < 1 || d->sw < 1 || d->dh < 1 ||
        d->dw < 1 || d->n < 1 || d->c < 1 || d->h < 1 || d->w < 1 || d->c_out < 1)
        return 0;
    int64_t oh = 0, ow = 0;
    if (conv_out_hw(d, &oh, &ow) != TILES_OK) return 0;
    ConvTmaGeometry g;
    return conv_tma_geometry(d, oh, ow, tile_oh, static_cast<int>(std::min<int64_t>(ow, INT32_MAX)), &g)
               ? g.ws_bytes : 256;
}

int conv2d_htiled(const tiles_conv_desc* d, int tile_oh, const tiles_config* cfg, void* ws,
                  size_t ws_bytes, void* stream) {
    return conv2d_tiled(d, tile_oh, 0, 0, cfg, ws, ws_bytes, stream);
}

}  // namespace tiles
