// lr_host.cu -- the engine behind the host-buffer entry points: a scan whose
// tensors live in host memory runs through the GPU in time chunks.
//
// Every scan here is a recurrence over time that carries a state, and each
// device entry point resumes from a given initial state, so a sequence can be
// cut into chunks of Lc steps and run chunk after chunk with the state handed
// over on the device.  Three streams of the library's own overlap the work:
//   in:   chunk k+1's inputs, host -> device (one 2-D copy per tensor: the
//         chunk is B rows of Lc x width elements, pitch L x width)
//   comp: chunk k's kernel, reading one staging buffer, writing another
//   out:  chunk k-1's outputs, device -> host
// with two staging buffers per direction and events between the streams:
//   in(k)   waits comp(k-2)   (its input buffer is free again)
//   comp(k) waits in(k) and out(k-2) (inputs landed, output buffer free)
//   out(k)  waits comp(k)
// Measured on GB300 the host link moves about 210 GB/s host -> device and
// 190 GB/s device -> host, and both directions together about 340 GB/s, so
// a streaming scan is copy-bound; the overlap hides the kernels and the
// outbound copies behind the inbound ones.  Pinned host memory is needed for
// the copies to run asynchronously (pageable memory gives the same results
// with the copies serialised).
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "lr_internal.h"

namespace lr {
namespace {

constexpr int kMaxHostDevices = 64;

// Streams and events of one device, created on first use and kept; calls on
// one device take the mutex, so they run one after another.
struct HostRes {
    std::once_flag once;
    bool ok = false;
    std::mutex mu;
    cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr, in_done[2] = {}, comp_done[2] = {}, out_done[2] = {};
};
HostRes g_host[kMaxHostDevices];

HostRes *host_res(int dev) {
    if (dev < 0 || dev >= kMaxHostDevices) return nullptr;
    HostRes &r = g_host[dev];
    std::call_once(r.once, [&r] {
        auto stream = [](cudaStream_t *s) {
            return cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) == cudaSuccess;
        };
        auto event = [](cudaEvent_t *e) {
            return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
        };
        bool ok = stream(&r.s_in) && stream(&r.s_comp) && stream(&r.s_out) && event(&r.start);
        for (int b = 0; b < 2 && ok; ++b)
            ok = event(&r.in_done[b]) && event(&r.comp_done[b]) && event(&r.out_done[b]);
        r.ok = ok;
    });
    return r.ok ? &r : nullptr;
}

size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

// B rows of `width` bytes: one 2-D copy, or one copy per row when a pitch
// exceeds what 2-D copies accept
bool copy_rows(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width, size_t rows,
               cudaMemcpyKind kind, cudaStream_t st, size_t max_pitch) {
    if (dpitch <= max_pitch && spitch <= max_pitch)
        return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, st) == cudaSuccess;
    for (size_t b = 0; b < rows; ++b)
        if (cudaMemcpyAsync(static_cast<char *>(dst) + b * dpitch, static_cast<const char *>(src) + b * spitch,
                            width, kind, st) != cudaSuccess)
            return false;
    return true;
}

// Workspace layout: the kernel workspace (so its call status sits at the
// start of the whole workspace), parameters, two states, then two input and
// two output staging buffers (every region 256-byte aligned).
struct Layout {
    size_t par[3] = {}, state[2] = {}, kws = 0, in_buf[2] = {}, out_buf[2] = {};
    size_t in_off[6] = {}, out_off[2] = {}, in_bytes = 0, out_bytes = 0, total = 0;
};

Layout layout(const HostJob &j) {
    Layout l;
    size_t at = 0;
    l.kws = at;
    at += al256(j.kernel_ws);
    for (int p = 0; p < j.n_par; ++p) {
        l.par[p] = at;
        at += al256(j.par[p].bytes);
    }
    for (int s = 0; s < 2; ++s) {
        l.state[s] = at;
        at += al256(j.state_bytes);
    }
    for (int i = 0; i < j.n_in; ++i) {
        l.in_off[i] = l.in_bytes;
        l.in_bytes += al256(size_t(j.B) * j.Lc * j.in[i].width * j.es);
    }
    for (int o = 0; o < j.n_out; ++o) {
        l.out_off[o] = l.out_bytes;
        l.out_bytes += al256(size_t(j.B) * j.Lc * j.out[o].width * j.es);
    }
    for (int b = 0; b < 2; ++b) {
        l.in_buf[b] = at;
        at += l.in_bytes;
    }
    for (int b = 0; b < 2; ++b) {
        l.out_buf[b] = at;
        at += l.out_bytes;
    }
    l.total = at;
    return l;
}

}  // namespace

int64_t g_host_chunk_override = 0;

int64_t host_chunk_steps(int64_t B, int64_t L, size_t in_bytes_per_step) {
    if (g_host_chunk_override > 0) return g_host_chunk_override;
    const size_t per_step = size_t(B > 0 ? B : 1) * (in_bytes_per_step > 0 ? in_bytes_per_step : 1);
    int64_t lc = int64_t((size_t(128) << 20) / per_step);
    lc = std::max<int64_t>(64, lc / 64 * 64);
    const int64_t l64 = std::max<int64_t>(64, (L + 63) / 64 * 64);
    return std::min(lc, l64);
}

size_t host_workspace_bytes(const HostJob &job) { return layout(job).total; }

int run_host_job(const HostJob &j, void *workspace, size_t ws_bytes, cudaStream_t caller, bool async_) {
    const Layout lay = layout(j);
    if (workspace == nullptr || ws_bytes < lay.total) return LR_ERR_WORKSPACE;
    int dev = 0, max_pitch = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_pitch, cudaDevAttrMaxPitch, dev) != cudaSuccess)
        return LR_ERR_CUDA;
    HostRes *r = host_res(dev);
    if (r == nullptr) return LR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(r->mu);
    char *ws = static_cast<char *>(workspace);
    float *state[2] = {reinterpret_cast<float *>(ws + lay.state[0]),
                       reinterpret_cast<float *>(ws + lay.state[1])};
    const void *par[3] = {};
    for (int p = 0; p < j.n_par; ++p) par[p] = j.par[p].host ? ws + lay.par[p] : nullptr;

    bool ok = cudaEventRecord(r->start, caller) == cudaSuccess &&
              cudaStreamWaitEvent(r->s_in, r->start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(r->s_comp, r->start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(r->s_out, r->start, 0) == cudaSuccess;
    for (int p = 0; p < j.n_par && ok; ++p)
        if (j.par[p].host)
            ok = cudaMemcpyAsync(ws + lay.par[p], j.par[p].host, j.par[p].bytes, cudaMemcpyHostToDevice,
                                 r->s_in) == cudaSuccess;
    if (ok && j.state0 != nullptr)
        ok = cudaMemcpyAsync(state[0], j.state0, j.state_bytes, cudaMemcpyHostToDevice, r->s_in) ==
             cudaSuccess;

    int rc = LR_OK;
    const SharedStamp one_call;   // every chunk launch records into the same call status
    const int64_t K = (j.L + j.Lc - 1) / j.Lc;
    for (int64_t k = 0; k < K && ok && rc == LR_OK; ++k) {
        const int b = int(k & 1);
        const int64_t t0 = k * j.Lc, lc = std::min(j.Lc, j.L - t0);
        char *ib = ws + lay.in_buf[b], *ob = ws + lay.out_buf[b];
        // inputs of chunk k (after chunk k-2 has consumed this buffer)
        if (k >= 2) ok = cudaStreamWaitEvent(r->s_in, r->comp_done[b], 0) == cudaSuccess;
        const void *din[6] = {};
        for (int i = 0; i < j.n_in && ok; ++i) {
            const size_t row = size_t(j.in[i].width) * j.es;
            din[i] = ib + lay.in_off[i];
            ok = copy_rows(ib + lay.in_off[i], lc * row, static_cast<const char *>(j.in[i].in) + t0 * row,
                           j.L * row, lc * row, j.B, cudaMemcpyHostToDevice, r->s_in, size_t(max_pitch));
        }
        ok = ok && cudaEventRecord(r->in_done[b], r->s_in) == cudaSuccess;
        // chunk k's kernel (after its inputs landed and chunk k-2's outputs left)
        ok = ok && cudaStreamWaitEvent(r->s_comp, r->in_done[b], 0) == cudaSuccess;
        if (ok && k >= 2) ok = cudaStreamWaitEvent(r->s_comp, r->out_done[b], 0) == cudaSuccess;
        void *dout[2] = {};
        for (int o = 0; o < j.n_out; ++o) dout[o] = ob + lay.out_off[o];
        if (ok) {
            const float *s_in = (k == 0 && j.state0 == nullptr) ? nullptr : state[k & 1];
            rc = j.launch(j.ctx, din, dout, par, lc, s_in, state[(k + 1) & 1], ws + lay.kws, j.kernel_ws,
                          r->s_comp);
        }
        ok = ok && rc == LR_OK && cudaEventRecord(r->comp_done[b], r->s_comp) == cudaSuccess;
        // outputs of chunk k
        ok = ok && cudaStreamWaitEvent(r->s_out, r->comp_done[b], 0) == cudaSuccess;
        for (int o = 0; o < j.n_out && ok; ++o) {
            const size_t row = size_t(j.out[o].width) * j.es;
            ok = copy_rows(static_cast<char *>(j.out[o].out) + t0 * row, j.L * row, ob + lay.out_off[o],
                           lc * row, lc * row, j.B, cudaMemcpyDeviceToHost, r->s_out, size_t(max_pitch));
        }
        ok = ok && cudaEventRecord(r->out_done[b], r->s_out) == cudaSuccess;
    }
    // the state after the last chunk (the out stream already follows it)
    if (ok && rc == LR_OK && j.state_final != nullptr)
        ok = cudaMemcpyAsync(j.state_final, state[K & 1], j.state_bytes, cudaMemcpyDeviceToHost,
                             r->s_out) == cudaSuccess;
    // the asynchronous form returns with the work queued: a later call's
    // copies follow this call's on the same streams and overlap its last
    // chunks; host_sync() waits for all of it, and the device-side status is
    // read from the workspace afterwards
    if (async_) {
        if (rc != LR_OK) return rc;
        return ok ? LR_OK : LR_ERR_CUDA;
    }
    // nothing may still use the workspace or the host buffers on return
    const bool synced = cudaStreamSynchronize(r->s_in) == cudaSuccess &&
                        cudaStreamSynchronize(r->s_comp) == cudaSuccess &&
                        cudaStreamSynchronize(r->s_out) == cudaSuccess;
    if (rc != LR_OK) return rc;
    if (!(ok && synced)) return LR_ERR_CUDA;
    // the chunks' device-side status (a bounded wait that ran out)
    int code = LR_OK;
    if (read_status(ws + lay.kws, r->s_comp, &code, false) != LR_OK) return LR_ERR_CUDA;
    return code;
}

int host_sync() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LR_ERR_CUDA;
    HostRes *r = host_res(dev);
    if (r == nullptr) return LR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(r->mu);
    const bool ok = cudaStreamSynchronize(r->s_in) == cudaSuccess && cudaStreamSynchronize(r->s_comp) == cudaSuccess &&
                    cudaStreamSynchronize(r->s_out) == cudaSuccess;
    return ok ? LR_OK : LR_ERR_CUDA;
}

}  // namespace lr
