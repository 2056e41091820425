// End-to-end calls: operands start in host memory and results end there.
//
// A call cuts its work into pieces and chains, for each piece, the upload of
// its inputs on the library's host-to-device stream, its kernels on the
// caller's stream and the download of its results on the library's
// device-to-host stream, linked by events.  The two copy directions run on
// separate copy engines and the kernels on the SMs, so piece p's upload,
// piece p-1's kernels and piece p-2's download overlap; the call costs about
// the upload of every input plus the last piece's kernels and download,
// instead of the sum of all three.  Each piece is an ordinary device call
// (tiles_gemm_batched, tiles_conv2d_htiled), so the results are those of the
// device calls on the same piece shapes.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "tiles.h"
#include "tiles_internal.h"

namespace tiles {
namespace {

constexpr int kMaxPieces = 16;
constexpr int kMaxPipeDevices = 64;

// The copy streams and events of one host thread on one device.  Per thread,
// so that two threads' calls never re-record each other's events; released
// when the thread exits.  Destroying a stream with work still queued on it
// is allowed: the work completes and the stream is released afterwards.
struct CopyPipe {
    bool ready = false;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t start = nullptr, done = nullptr, landed[kMaxPieces] = {}, computed[kMaxPieces] = {};

    CopyPipe() = default;
    CopyPipe(const CopyPipe&) = delete;
    CopyPipe& operator=(const CopyPipe&) = delete;
    ~CopyPipe() {
        // Errors are ignored: at process exit the runtime may already be
        // shutting down, and nothing can be reported from here.
        auto drop_event = [](cudaEvent_t e) { if (e) cudaEventDestroy(e); };
        drop_event(start);
        drop_event(done);
        for (int i = 0; i < kMaxPieces; ++i) {
            drop_event(landed[i]);
            drop_event(computed[i]);
        }
        if (up) cudaStreamDestroy(up);
        if (down) cudaStreamDestroy(down);
    }
};

thread_local CopyPipe t_pipes[kMaxPipeDevices];

int cuda_fail(cudaError_t e, const char* what) {
    return fail(TILES_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int pipe_for_current_device(CopyPipe** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxPipeDevices)
        return fail(TILES_ERR_INVALID_ARG, "device ordinal %d beyond %d", dev, kMaxPipeDevices);
    CopyPipe& p = t_pipes[dev];
    if (!p.ready) {
        // Each handle is recorded as soon as it exists, so a failure part
        // way leaves nothing that the destructor does not release.
        if (!p.up) e = cudaStreamCreateWithFlags(&p.up, cudaStreamNonBlocking);
        if (e == cudaSuccess && !p.down) e = cudaStreamCreateWithFlags(&p.down, cudaStreamNonBlocking);
        auto make = [&](cudaEvent_t* ev) {
            if (e == cudaSuccess && !*ev) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        };
        make(&p.start);
        make(&p.done);
        for (int i = 0; i < kMaxPieces; ++i) {
            make(&p.landed[i]);
            make(&p.computed[i]);
        }
        if (e != cudaSuccess) return cuda_fail(e, "creating the copy streams and events");
        p.ready = true;
    }
    *out = &p;
    return TILES_OK;
}

int copy_async(void* dst, const void* src, int64_t bytes, cudaMemcpyKind kind, cudaStream_t s) {
    if (bytes <= 0) return TILES_OK;
    const cudaError_t e = cudaMemcpyAsync(dst, src, static_cast<size_t>(bytes), kind, s);
    return e == cudaSuccess ? TILES_OK
                            : cuda_fail(e, kind == cudaMemcpyHostToDevice ? "upload" : "download");
}

// `later` runs after the work enqueued on `earlier` so far.
int order(cudaStream_t earlier, cudaStream_t later, cudaEvent_t ev) {
    cudaError_t e = cudaEventRecord(ev, earlier);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(later, ev, 0);
    return e == cudaSuccess ? TILES_OK : cuda_fail(e, "ordering the copy streams");
}

int bytes_of_dtype(int dt) {
    return dt == TILES_F32 ? 4 : (dt == TILES_F16 || dt == TILES_BF16) ? 2 : 0;
}

const char* at(const void* p, int64_t off) { return static_cast<const char*>(p) + off; }
char* at(void* p, int64_t off) { return static_cast<char*>(p) + off; }

}  // namespace
}  // namespace tiles

using namespace tiles;

extern "C" int tiles_gemm_host(const tiles_gemm_desc* d, const tiles_config* cfg,
                               const void* a_host, const void* b_host, void* c_host, int chunks,
                               void* ws, size_t ws_bytes, void* stream) {
    if (!d) return fail(TILES_ERR_INVALID_ARG, "null descriptor");
    if (!a_host || !b_host || !c_host) return fail(TILES_ERR_INVALID_ARG, "null host buffer");
    if (chunks < 1 || chunks > kMaxPieces)
        return fail(TILES_ERR_INVALID_ARG, "chunks must be in 1..%d (got %d)", kMaxPieces, chunks);
    // Every device-side argument is checked (and the tile chosen) before
    // anything is enqueued.
    tiles_schedule sch;
    int s = tiles_gemm_schedule(d, cfg, ws_bytes, &sch);
    if (s != TILES_OK) return s;
    const int64_t ei = bytes_of_dtype(d->a_dtype), ec = bytes_of_dtype(d->c_dtype);
    const bool batched = d->batch > 1;

    // Pieces: runs of batch items, or runs of whole-tile rows of one item.
    struct Piece { int64_t i0, i1, r0, r1; };
    Piece pc[kMaxPieces];
    int np = 0;
    if (batched) {
        np = static_cast<int>(std::min<int64_t>(chunks, d->batch));
        for (int p = 0; p < np; ++p)
            pc[p] = Piece{p * d->batch / np, (p + 1) * d->batch / np, 0, d->m};
    } else {
        const int64_t bm = std::max<int64_t>(sch.cfg.bm, 1);
        const int64_t rows = (((d->m + chunks - 1) / chunks) + bm - 1) / bm * bm;
        for (int64_t r0 = 0; r0 < d->m; r0 += rows) pc[np++] = Piece{0, 1, r0, std::min(d->m, r0 + rows)};
    }
    // Byte offsets of (item, row) and the extent of a run of rows/items.
    auto a_off = [&](int64_t i, int64_t r) { return (i * (batched ? d->stride_a : 0) + r * d->lda) * ei; };
    auto b_off = [&](int64_t i) { return i * (batched ? d->stride_b : 0) * ei; };
    auto c_off = [&](int64_t i, int64_t r) { return (i * (batched ? d->stride_c : 0) + r * d->ldc) * ec; };
    const int64_t b_item = ((d->k - 1) * d->ldb + d->n) * ei;

    CopyPipe* p = nullptr;
    s = pipe_for_current_device(&p);
    if (s != TILES_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((s = order(st, p->up, p->start)) != TILES_OK) return s;
    if (const cudaError_t e = cudaStreamWaitEvent(p->down, p->start, 0); e != cudaSuccess)
        return cuda_fail(e, "ordering the copy streams");
    if (!batched && (s = copy_async(const_cast<void*>(d->b), b_host, b_item, cudaMemcpyHostToDevice,
                                    p->up)) != TILES_OK)
        return s;
    for (int i = 0; i < np; ++i) {
        const Piece& q = pc[i];
        if (batched) {
            const int64_t off = b_off(q.i0), len = b_off(q.i1 - 1) + b_item - off;
            s = copy_async(const_cast<char*>(at(d->b, off)), at(b_host, off), len,
                           cudaMemcpyHostToDevice, p->up);
            if (s != TILES_OK) return s;
        }
        const int64_t a0 = a_off(q.i0, q.r0), a1 = a_off(q.i1 - 1, q.r1 - 1) + d->k * ei;
        s = copy_async(const_cast<char*>(at(d->a, a0)), at(a_host, a0), a1 - a0,
                       cudaMemcpyHostToDevice, p->up);
        if (s != TILES_OK) return s;
        if ((s = order(p->up, st, p->landed[i])) != TILES_OK) return s;
        tiles_gemm_desc g = *d;
        g.batch = q.i1 - q.i0;
        g.m = q.r1 - q.r0;
        g.a = at(d->a, a0);
        g.b = at(d->b, b_off(q.i0));
        g.c = at(d->c, c_off(q.i0, q.r0));
        if ((s = tiles_gemm_batched(&g, cfg, ws, ws_bytes, stream)) != TILES_OK) return s;
        if ((s = order(st, p->down, p->computed[i])) != TILES_OK) return s;
        const int64_t c0 = c_off(q.i0, q.r0), c1 = c_off(q.i1 - 1, q.r1 - 1) + d->n * ec;
        s = copy_async(at(c_host, c0), at(d->c, c0), c1 - c0, cudaMemcpyDeviceToHost, p->down);
        if (s != TILES_OK) return s;
    }
    return order(p->down, st, p->done);
}

extern "C" int tiles_conv2d_host(const tiles_conv_desc* d, int tile_oh, const tiles_config* cfg,
                                 const void* x_host, const void* w_host, void* y_host, int chunks,
                                 void* ws, size_t ws_bytes, void* stream) {
    if (!d) return fail(TILES_ERR_INVALID_ARG, "null descriptor");
    if (!x_host || !w_host || !y_host) return fail(TILES_ERR_INVALID_ARG, "null host buffer");
    if (!d->x || !d->wt || !d->y) return fail(TILES_ERR_INVALID_ARG, "null device buffer");
    if (chunks < 1 || chunks > kMaxPieces)
        return fail(TILES_ERR_INVALID_ARG, "chunks must be in 1..%d (got %d)", kMaxPieces, chunks);
    if (tiles_conv_workspace_bytes(d, tile_oh) == 0)
        return fail(TILES_ERR_INVALID_ARG, "invalid convolution shape");
    const int64_t ei = bytes_of_dtype(d->in_dtype), eo = bytes_of_dtype(d->out_dtype);
    if (!ei || !eo) return fail(TILES_ERR_UNSUPPORTED_DTYPE, "unsupported dtype");
    int64_t oh = 0, ow = 0;
    if (const int hw = conv_out_hw(d, &oh, &ow); hw != TILES_OK) return hw;
    // One image of x (either layout) and of y is contiguous.
    const int64_t x_img = static_cast<int64_t>(d->c) * d->h * d->w * ei;
    const int64_t y_img = static_cast<int64_t>(d->c_out) * oh * ow * eo;
    const int64_t w_bytes = static_cast<int64_t>(d->c_out) * d->c * d->kh * d->kw * ei;
    const int np = std::min(chunks, d->n);

    CopyPipe* p = nullptr;
    int s = pipe_for_current_device(&p);
    if (s != TILES_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((s = order(st, p->up, p->start)) != TILES_OK) return s;
    if (const cudaError_t e = cudaStreamWaitEvent(p->down, p->start, 0); e != cudaSuccess)
        return cuda_fail(e, "ordering the copy streams");
    s = copy_async(const_cast<void*>(d->wt), w_host, w_bytes, cudaMemcpyHostToDevice, p->up);
    if (s != TILES_OK) return s;
    for (int i = 0; i < np; ++i) {
        const int n0 = static_cast<int>(static_cast<int64_t>(i) * d->n / np);
        const int n1 = static_cast<int>(static_cast<int64_t>(i + 1) * d->n / np);
        s = copy_async(const_cast<char*>(at(d->x, n0 * x_img)), at(x_host, n0 * x_img),
                       (n1 - n0) * x_img, cudaMemcpyHostToDevice, p->up);
        if (s != TILES_OK) return s;
        if ((s = order(p->up, st, p->landed[i])) != TILES_OK) return s;
        tiles_conv_desc c = *d;
        c.n = n1 - n0;
        c.x = at(d->x, n0 * x_img);
        c.y = at(d->y, n0 * y_img);
        if ((s = tiles_conv2d_htiled(&c, tile_oh, cfg, ws, ws_bytes, stream)) != TILES_OK) return s;
        if ((s = order(st, p->down, p->computed[i])) != TILES_OK) return s;
        s = copy_async(at(y_host, n0 * y_img), at(d->y, n0 * y_img), (n1 - n0) * y_img,
                       cudaMemcpyDeviceToHost, p->down);
        if (s != TILES_OK) return s;
    }
    return order(p->down, st, p->done);
}
