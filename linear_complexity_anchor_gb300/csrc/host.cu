// Forward from host buffers.  The batch is cut into chunks of whole batch entries, or, when that
// gives too few chunks to overlap well (and there are fewer batch entries than chunks allowed),
// of head ranges of single batch entries.  U is copied once; a chunk is an ordinary forward
// problem on a range of U's rows, planned as the whole problem is (its slice count, the
// slice-streaming kernel's CTAs per slice), so that its result bits are the whole problem's.
// Chunk k's Q and V
// are copied in on one stream, its forward runs on the caller's stream and
// its H is copied out on a third stream, over two device buffer sets, so that the copies of
// one chunk overlap the forward of the next and the copies in and out run at the same time
// (Q and V on two streams of their own were no faster: the host link, not a copy engine, sets
// the rate, about 240 GB/s of copies in and out together).  Everything is enqueued: the call returns at once, and the caller's stream is
// ordered after the last copy out.  The streams and events are made once per device and
// reused; calls on one device take a lock while they enqueue.
#include "common.cuh"

#include <stdlib.h>

#include <mutex>

namespace anchor {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 16;
constexpr size_t kChunkBytes = size_t(64) << 20;  // Q, V and H bytes a chunk aims at
constexpr int kEvents = 2 + 3 * kMaxChunks;

struct Pipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;  // Q and V in, H out
    cudaEvent_t ev[kEvents];
};
Pipe g_pipes[kMaxDevices];
std::mutex g_pipe_lock[kMaxDevices];

cudaError_t get_pipe(int dev, Pipe *&pp) {
    Pipe &p = g_pipes[dev];
    if (!p.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
        for (int i = 0; i < kEvents && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&p.ev[i], cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
        p.ready = true;
    }
    pp = &p;
    return cudaSuccess;
}

}  // namespace

anchor_attn_status_t forward_host(const void *hQ, const void *hU, const void *hV, void *hH, int B, int heads, int n,
                                  int m, int d, float scale, bool f32, void *stream_v) {
    const Problem whole{hQ, hU, hV, hH, B, heads, n, m, d, scale, f32};
    const anchor_attn_status_t st = check_problem(whole);
    if (st != ANCHOR_ATTN_OK) return st;
    if (whole.slices() == 0 || n == 0) return ANCHOR_ATTN_OK;
    cudaStream_t user = (cudaStream_t)stream_v;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_pipe_lock[dev]);
    Pipe *pp = nullptr;
    if (get_pipe(dev, pp) != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_CUDA;
    }
    Pipe &P = *pp;
    const size_t elem = f32 ? 4 : 2;
    const size_t sbytes = (size_t)n * d * elem;  // one slice of Q, V or H
    const size_t ubytes = (size_t)heads * m * d * elem;
    const long long S = whole.slices();
    const long long want = (long long)((3 * sbytes * (size_t)S + kChunkBytes - 1) / kChunkBytes);
    const int cl_c = forward_stream_cluster(whole);
    // Chunks: whole batch entries while that gives enough of them (or there are kMaxChunks
    // entries or more); else each batch entry cut into head ranges (a chunk is always slices of
    // one head range of whole batch entries, so that it is an ordinary problem: its U is a range
    // of rows of U, its Q, V and H one run of memory)
    int chunks, hsplit, per_b = 1;
    if (want <= B || B >= kMaxChunks) {
        hsplit = 1;
        chunks = (int)std::max<long long>(1, std::min<long long>({(long long)B, (long long)kMaxChunks, want}));
        per_b = (B + chunks - 1) / chunks;
    } else {
        hsplit = (int)std::max<long long>(1, std::min<long long>({(long long)heads, (long long)(kMaxChunks / B),
                                                                    (want + B - 1) / B}));
        chunks = B * hsplit;
    }
    const int per_h = (heads + hsplit - 1) / hsplit;
    const size_t per = (size_t)(hsplit == 1 ? per_b * heads : per_h);  // slices of the largest chunk
    const int sets = chunks > 1 ? 2 : 1;
    // device workspace: U | sets x (Q | V | H) of the largest chunk
    const size_t setb = 3 * sbytes * per;
    const size_t ubytes_al = (ubytes + 255) / 256 * 256;
    uint8_t *ws = nullptr;
    if (getenv("ANCHOR_ATTN_TEST_FAIL_ALLOC") != nullptr) return ANCHOR_ATTN_ERR_ALLOC;
    if (cudaMallocAsync(reinterpret_cast<void **>(&ws), ubytes_al + sets * setb, user) != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_ALLOC;
    }
    cudaEvent_t ev_start = P.ev[0], ev_end_in = P.ev[1];
    cudaEvent_t *ev_in = P.ev + 2, *ev_comp = ev_in + kMaxChunks, *ev_out = ev_comp + kMaxChunks;
    anchor_attn_status_t status = ANCHOR_ATTN_OK;
    cudaError_t e = cudaEventRecord(ev_start, user);  // the workspace, and the caller's earlier work
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.in, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, ev_start, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(ws, hU, ubytes, cudaMemcpyHostToDevice, P.in);
    int issued_out = 0;
    for (int k = 0; k < chunks && e == cudaSuccess && status == ANCHOR_ATTN_OK; ++k) {
        // this chunk: batch entries [b0, b1) x heads [h0, h1), contiguous in memory
        int b0, b1, h0, h1;
        if (hsplit == 1) {
            b0 = (int)((long long)k * B / chunks);
            b1 = (int)((long long)(k + 1) * B / chunks);
            h0 = 0;
            h1 = heads;
        } else {
            b0 = k / hsplit;
            b1 = b0 + 1;
            const int j = k - b0 * hsplit;
            h0 = (int)((long long)j * heads / hsplit);
            h1 = (int)((long long)(j + 1) * heads / hsplit);
        }
        const size_t off = ((size_t)b0 * heads + h0) * sbytes;
        const size_t bytes = (size_t)(b1 - b0) * (h1 - h0) * sbytes;
        uint8_t *dQ = ws + ubytes_al + (k % sets) * setb, *dV = dQ + sbytes * per, *dH = dV + sbytes * per;
        // copy in (after the copy out of the chunk that last used this buffer set)
        if (k >= sets) e = cudaStreamWaitEvent(P.in, ev_out[k - sets], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dQ, static_cast<const uint8_t *>(hQ) + off, bytes, cudaMemcpyHostToDevice, P.in);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dV, static_cast<const uint8_t *>(hV) + off, bytes, cudaMemcpyHostToDevice, P.in);
        if (e == cudaSuccess) e = cudaEventRecord(ev_in[k], P.in);
        // the forward of the chunk on the caller's stream, planned as the whole problem would be
        // (the same result bits)
        if (e == cudaSuccess) e = cudaStreamWaitEvent(user, ev_in[k], 0);
        if (e != cudaSuccess) break;
        Problem cp{dQ, ws + (size_t)h0 * m * d * elem, dV, dH, b1 - b0, h1 - h0, n, m, d, scale, f32};
        cp.plan_slices = S;
        cp.plan_cl_c = cl_c;
        status = forward_problem(cp, user);
        if (status != ANCHOR_ATTN_OK) break;
        e = cudaEventRecord(ev_comp[k], user);
        // copy out
        if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, ev_comp[k], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(static_cast<uint8_t *>(hH) + off, dH, bytes, cudaMemcpyDeviceToHost, P.out);
        if (e == cudaSuccess) e = cudaEventRecord(ev_out[k], P.out);
        if (e == cudaSuccess) issued_out = k + 1;
    }
    // the caller's stream is ordered after every copy this call enqueued, then the workspace
    // goes back (also after a failure, so that nothing in flight still uses it)
    cudaError_t e2 = cudaEventRecord(ev_end_in, P.in);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(user, ev_end_in, 0);
    if (e2 == cudaSuccess && issued_out > 0) e2 = cudaStreamWaitEvent(user, ev_out[issued_out - 1], 0);
    const cudaError_t ef = cudaFreeAsync(ws, user);
    if (status != ANCHOR_ATTN_OK) return status;
    if (e != cudaSuccess || e2 != cudaSuccess || ef != cudaSuccess) {
        cudaGetLastError();
        return ANCHOR_ATTN_ERR_CUDA;
    }
    return ANCHOR_ATTN_OK;
}

}  // namespace anchor

extern "C" {

anchor_attn_status_t anchor_attn_forward_host(const void *Q, const void *U, const void *V, void *H, int B, int heads,
                                              int n, int m, int d, float scale, void *stream) {
    return anchor::forward_host(Q, U, V, H, B, heads, n, m, d, scale, false, stream);
}

anchor_attn_status_t anchor_attn_forward_host_f32(const float *Q, const float *U, const float *V, float *H, int B,
                                                  int heads, int n, int m, int d, float scale, void *stream) {
    return anchor::forward_host(Q, U, V, H, B, heads, n, m, d, scale, true, stream);
}

}  // extern "C"
