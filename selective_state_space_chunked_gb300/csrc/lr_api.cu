// lr_api.cu -- the C ABI declared in include/lrscan.h: argument validation
// (pure host logic, run before any CUDA call), dispatch to the kernels'
// launchers, the per-call device status, and the tuning / test knobs.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "lr_internal.h"
#include "lrscan.h"

namespace lr {
int g_split_override = 0;
int g_withheld_split = -1;
int g_withheld_timeout_ms = 1000;
int64_t g_selective_warmup_steps = -1;   // automatic

namespace {
std::atomic<unsigned long long> g_stamp{0};
thread_local unsigned long long t_shared_stamp = 0;
thread_local int t_shared_depth = 0;

unsigned long long fresh_stamp() {
    unsigned long long s = 0;
    while (s == 0) s = (g_stamp.fetch_add(1, std::memory_order_relaxed) + 1) & ((1ull << 48) - 1);
    return s;
}
}  // namespace

StatusRef call_status(void *workspace) {
    return StatusRef{static_cast<unsigned long long *>(workspace),
                     t_shared_depth > 0 ? t_shared_stamp : fresh_stamp()};
}

SharedStamp::SharedStamp() {
    if (t_shared_depth++ == 0) t_shared_stamp = fresh_stamp();
}
SharedStamp::~SharedStamp() { --t_shared_depth; }

int read_status(void *workspace, cudaStream_t stream, int *code, bool clear) {
    unsigned long long word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return LR_ERR_CUDA;
    *code = static_cast<int>(static_cast<int16_t>(word & 0xffffu));
    if (clear && *code != LR_OK) {
        static const unsigned long long kZero = 0;
        // stamp 0 with code 0: no call's stamp, nothing recorded
        if (cudaMemcpyAsync(workspace, &kZero, sizeof(kZero), cudaMemcpyHostToDevice, stream) != cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess)
            return LR_ERR_CUDA;
    }
    return LR_OK;
}

int status_ok_no_launch(void *workspace, size_t ws_bytes, cudaStream_t stream) {
    if (workspace == nullptr || ws_bytes < kStatusBytes) return LR_OK;
    return cudaMemsetAsync(workspace, 0, sizeof(unsigned long long), stream) == cudaSuccess ? LR_OK
                                                                                              : LR_ERR_CUDA;
}
}  // namespace lr

namespace {

constexpr int kVersion = 10000;  // 1.0.0

bool misaligned(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

bool io_ok(lr_dtype io) { return io == LR_F32 || io == LR_BF16; }

// Channel counts must keep every TMA row stride a multiple of 16 bytes.
bool channels_ok(int64_t D, lr_dtype io) { return D % (io == LR_BF16 ? 8 : 4) == 0; }

bool fits_int(int64_t v) { return v <= INT_MAX; }

int check_workspace(const lr::DiagPlan &p, const void *ws, size_t ws_bytes) {
    if (p.ws_bytes == 0) return LR_OK;
    if (ws == nullptr || ws_bytes < p.ws_bytes) return LR_ERR_WORKSPACE;
    if (misaligned(ws)) return LR_ERR_MISALIGNED;
    return LR_OK;
}

// L == 0: the final state is the initial state (or zero).
int copy_state(const float *h0, float *h_final, size_t count, cudaStream_t stream) {
    if (h_final == nullptr || count == 0) return LR_OK;
    const cudaError_t e =
        h0 != nullptr
            ? cudaMemcpyAsync(h_final, h0, count * sizeof(float), cudaMemcpyDeviceToDevice, stream)
            : cudaMemsetAsync(h_final, 0, count * sizeof(float), stream);
    return e == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

int validate_selective(const void *x, const void *dt, const void *z, const void *Bm,
                       const void *Cm, const float *A_log, const float *Dskip, const float *h0,
                       const void *y, const float *h_final, int64_t B, int64_t L, int64_t D,
                       int64_t N, lr_dtype io) {
    if (B < 0 || L < 0 || D < 0 || N < 0 || !io_ok(io)) return LR_ERR_INVALID_ARG;
    // activation pointers may be NULL only when there are no activations
    const bool acts = B > 0 && L > 0 && D > 0;
    if ((acts && (!x || !dt || !Bm || !Cm || !y)) || (D > 0 && !A_log)) return LR_ERR_INVALID_ARG;
    if (N != 16 || !channels_ok(D, io)) return LR_ERR_UNSUPPORTED;
    if (!fits_int(B) || !fits_int(L) || !fits_int(D)) return LR_ERR_UNSUPPORTED;
    const void *ptrs[] = {x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final};
    for (const void *p : ptrs)
        if (misaligned(p)) return LR_ERR_MISALIGNED;
    return LR_OK;
}

int validate_rglru(const void *x, const void *r, const void *i, const float *a_log, float c,
                   const float *h0, const void *y, const float *h_final, int64_t B, int64_t L,
                   int64_t D, lr_dtype io) {
    if (B < 0 || L < 0 || D < 0 || !io_ok(io) || !std::isfinite(c)) return LR_ERR_INVALID_ARG;
    const bool acts = B > 0 && L > 0 && D > 0;
    if ((acts && (!x || !r || !i || !y)) || (D > 0 && !a_log)) return LR_ERR_INVALID_ARG;
    if (!channels_ok(D, io)) return LR_ERR_UNSUPPORTED;
    if (!fits_int(B) || !fits_int(L) || !fits_int(D)) return LR_ERR_UNSUPPORTED;
    const void *ptrs[] = {x, r, i, a_log, h0, y, h_final};
    for (const void *p : ptrs)
        if (misaligned(p)) return LR_ERR_MISALIGNED;
    return LR_OK;
}

int validate_hgrn2(const void *q, const void *k, const void *v, const void *g, const float *S0,
                   const void *o, const float *S_final, int64_t B, int64_t L, int64_t H,
                   int64_t dk, int64_t dv, int64_t chunk, lr_dtype io) {
    if (B < 0 || L < 0 || H <= 0 || dk <= 0 || dv <= 0 || chunk <= 0 || !io_ok(io))
        return LR_ERR_INVALID_ARG;
    if (B > 0 && L > 0 && (!q || !k || !v || !g || !o)) return LR_ERR_INVALID_ARG;
    if (dk > 512) return LR_ERR_UNSUPPORTED;
    if (!fits_int(B) || !fits_int(L) || !fits_int(H) || !fits_int(B * H)) return LR_ERR_UNSUPPORTED;
    const void *ptrs[] = {q, k, v, g, S0, o, S_final};
    for (const void *p : ptrs)
        if (misaligned(p)) return LR_ERR_MISALIGNED;
    return LR_OK;
}

// The tcgen05 chunked kernel serves dk = dv = 128, chunk 64, bf16 I/O; every
// other case runs on the general step-by-step kernel.
bool hgrn2_tensor_path(int64_t dk, int64_t dv, int64_t chunk, lr_dtype io) {
    return dk == 128 && dv == 128 && chunk == 64 && io == LR_BF16;
}
// fp32 I/O on the tensor cores (split bf16 operands): 128 x 128 heads, chunk 64
bool hgrn2_f32_tensor_path(int64_t dk, int64_t dv, int64_t chunk, lr_dtype io) {
    return dk == 128 && dv == 128 && chunk == 64 && io == LR_F32;
}

int validate_minmax(const void *r, const void *s, const float *x0, const void *y, const float *x_final,
                    int64_t B, int64_t L, int64_t D, lr_dtype io) {
    if (B < 0 || L < 0 || D < 0 || !io_ok(io)) return LR_ERR_INVALID_ARG;
    if (B > 0 && L > 0 && D > 0 && (!r || !s || !y)) return LR_ERR_INVALID_ARG;
    if (!channels_ok(D, io)) return LR_ERR_UNSUPPORTED;
    if (!fits_int(B) || !fits_int(L) || !fits_int(D)) return LR_ERR_UNSUPPORTED;
    const void *ptrs[] = {r, s, x0, y, x_final};
    for (const void *p : ptrs)
        if (misaligned(p)) return LR_ERR_MISALIGNED;
    return LR_OK;
}

// Decode steps: the state after the step is always written (h_out
// required); the state before it is optional (NULL = zero).
int validate_step_common(const void *const *required, int n_required, const void *const *all, int n_all) {
    for (int k = 0; k < n_required; ++k)
        if (required[k] == nullptr) return LR_ERR_INVALID_ARG;
    for (int k = 0; k < n_all; ++k)
        if (misaligned(all[k])) return LR_ERR_MISALIGNED;
    return LR_OK;
}

}  // namespace

extern "C" {

const char *lr_status_string(int code) {
    switch (code) {
        case LR_OK: return "LR_OK";
        case LR_ERR_INVALID_ARG: return "LR_ERR_INVALID_ARG: invalid argument";
        case LR_ERR_UNSUPPORTED: return "LR_ERR_UNSUPPORTED: unsupported shape or dtype";
        case LR_ERR_MISALIGNED: return "LR_ERR_MISALIGNED: tensor base not 16-byte aligned";
        case LR_ERR_WORKSPACE: return "LR_ERR_WORKSPACE: workspace missing or too small";
        case LR_ERR_CUDA: return "LR_ERR_CUDA: a CUDA call failed";
        case LR_ERR_TIMEOUT: return "LR_ERR_TIMEOUT: a bounded device-side wait ran out";
        case LR_ERR_RANGE: return "LR_ERR_RANGE: an HGRN2 gate is not a finite number";
        default: return "unknown lrscan status";
    }
}

int lr_version(void) { return kVersion; }

int lr_check_status(void *workspace, lr_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return LR_ERR_CUDA;
    void *ws = workspace;
    if (ws == nullptr && lr::rglru_builtin_scratch(&ws) != LR_OK) return LR_ERR_CUDA;
    if (misaligned(ws)) return LR_ERR_MISALIGNED;
    int code = LR_OK;
    if (lr::read_status(ws, st, &code, true) != LR_OK) return LR_ERR_CUDA;
    return code;
}

int lr_set_split_override(int splits) {
    const int prev = lr::g_split_override;
    lr::g_split_override = splits > 0 ? splits : 0;
    return prev;
}

int64_t lr_set_host_chunk_steps(int64_t steps) {
    const int64_t prev = lr::g_host_chunk_override;
    lr::g_host_chunk_override = steps > 0 ? steps : 0;
    return prev;
}

int64_t lr_set_selective_warmup(int64_t max_steps) {
    const int64_t prev = lr::g_selective_warmup_steps;
    lr::g_selective_warmup_steps =
        max_steps < 0 ? -1 : (max_steps < (int64_t(1) << 30) ? max_steps : (int64_t(1) << 30));
    return prev;
}

int lr_test_withhold_split(int split, int timeout_ms) {
    lr::g_withheld_split = split >= 1 ? split : -1;
    lr::g_withheld_timeout_ms = timeout_ms > 0 ? timeout_ms : 1000;
    return LR_OK;
}

// ---------------------------------------------------------------- selective
size_t lr_selective_scan_workspace_size(int64_t B, int64_t L, int64_t D, int64_t N, lr_dtype io) {
    if (B < 0 || L < 0 || D < 0 || N != 16 || !io_ok(io)) return 0;
    if (B == 0 || L == 0 || D == 0) return lr::kStatusBytes;
    lr::DiagPlan p;
    if (lr::selective_plan(B, L, D, io, &p) != LR_OK) return SIZE_MAX;
    return p.ws_bytes;
}

int lr_selective_scan_fwd(const void *x, const void *dt, const void *z, const void *Bm,
                          const void *Cm, const float *A_log, const float *Dskip, const float *h0,
                          void *y, float *h_final, int64_t B, int64_t L, int64_t D, int64_t N,
                          lr_dtype io, int dt_softplus, void *workspace, size_t ws_bytes,
                          lr_stream_t stream) {
    int rc = validate_selective(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final, B, L, D, N, io);
    if (rc != LR_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (B == 0 || D == 0) return lr::status_ok_no_launch(workspace, ws_bytes, st);
    if (L == 0) {
        if ((rc = copy_state(h0, h_final, size_t(B) * D * N, st)) != LR_OK) return rc;
        return lr::status_ok_no_launch(workspace, ws_bytes, st);
    }
    lr::DiagPlan p;
    if ((rc = lr::selective_plan(B, L, D, io, &p)) != LR_OK) return rc;
    if ((rc = check_workspace(p, workspace, ws_bytes)) != LR_OK) return rc;
    return lr::selective_launch(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final, B, L, D, io,
                                dt_softplus, p, workspace, st);
}

// ---------------------------------------------------------------- RG-LRU
size_t lr_rglru_scan_workspace_size(int64_t B, int64_t L, int64_t D, lr_dtype io) {
    if (B < 0 || L < 0 || D < 0 || !io_ok(io)) return 0;
    if (B == 0 || L == 0 || D == 0) return lr::kStatusBytes;
    lr::DiagPlan p;
    if (lr::rglru_plan(B, L, D, io, &p) != LR_OK) return SIZE_MAX;
    return p.ws_bytes;
}

int lr_rglru_scan_fwd(const void *x, const void *r, const void *i, const float *a_log, float c,
                      const float *h0, void *y, float *h_final, int64_t B, int64_t L, int64_t D,
                      lr_dtype io, void *workspace, size_t ws_bytes, lr_stream_t stream) {
    int rc = validate_rglru(x, r, i, a_log, c, h0, y, h_final, B, L, D, io);
    if (rc != LR_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (B == 0 || D == 0) return lr::status_ok_no_launch(workspace, ws_bytes, st);
    if (L == 0) {
        if ((rc = copy_state(h0, h_final, size_t(B) * D, st)) != LR_OK) return rc;
        return lr::status_ok_no_launch(workspace, ws_bytes, st);
    }
    lr::DiagPlan p;
    if ((rc = lr::rglru_plan(B, L, D, io, &p)) != LR_OK) return rc;
    if ((rc = check_workspace(p, workspace, ws_bytes)) != LR_OK) return rc;
    return lr::rglru_launch(x, r, i, a_log, c, h0, y, h_final, B, L, D, io, p, workspace, st);
}

// RG-LRU scan without a caller workspace: same arithmetic and launch as
// lr_rglru_scan_fwd, with the look-back scratch taken from the library's
// built-in array.  Allocates nothing.
int lr_rglru_scan_fwd_noalloc(const void *x, const void *r, const void *i, const float *a_log,
                              float c, const float *h0, void *y, float *h_final, int64_t B,
                              int64_t L, int64_t D, lr_dtype io, lr_stream_t stream) {
    int rc = validate_rglru(x, r, i, a_log, c, h0, y, h_final, B, L, D, io);
    if (rc != LR_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void *scratch = nullptr;
    if ((rc = lr::rglru_builtin_scratch(&scratch)) != LR_OK) return rc;
    if (B == 0 || D == 0) return lr::status_ok_no_launch(scratch, lr::kRglruScratchBytes, st);
    if (L == 0) {
        if ((rc = copy_state(h0, h_final, size_t(B) * D, st)) != LR_OK) return rc;
        return lr::status_ok_no_launch(scratch, lr::kRglruScratchBytes, st);
    }
    lr::DiagPlan p;
    if ((rc = lr::rglru_plan(B, L, D, io, &p)) != LR_OK) return rc;
    if (p.ws_bytes > lr::kRglruScratchBytes) return LR_ERR_WORKSPACE;
    return lr::rglru_launch(x, r, i, a_log, c, h0, y, h_final, B, L, D, io, p, scratch, st);
}

// ---------------------------------------------------------------- HGRN2
size_t lr_hgrn2_workspace_size(int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv,
                               lr_dtype io) {
    (void)dk;
    (void)dv;
    (void)io;
    size_t bytes = 0;
    if (B < 0 || L < 0 || H <= 0) return 0;
    if (B == 0 || L == 0) return lr::kStatusBytes;   // nothing launched: the status only
    if (lr::hgrn2_workspace(B, L, H, &bytes) != LR_OK) return SIZE_MAX;
    return bytes;
}

int lr_hgrn2_fwd(const void *q, const void *k, const void *v, const void *g, const float *S0,
                 void *o, float *S_final, int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv,
                 int64_t chunk, lr_dtype io, void *workspace, size_t ws_bytes,
                 lr_stream_t stream) {
    int rc = validate_hgrn2(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, chunk, io);
    if (rc != LR_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (B == 0) return lr::status_ok_no_launch(workspace, ws_bytes, st);
    if (L == 0) {
        if ((rc = copy_state(S0, S_final, size_t(B) * H * dk * dv, st)) != LR_OK) return rc;
        return lr::status_ok_no_launch(workspace, ws_bytes, st);
    }
    size_t need = 0;
    if ((rc = lr::hgrn2_workspace(B, L, H, &need)) != LR_OK) return rc;
    if (workspace == nullptr || ws_bytes < need) return LR_ERR_WORKSPACE;
    if (misaligned(workspace)) return LR_ERR_MISALIGNED;
    if (hgrn2_f32_tensor_path(dk, dv, chunk, io))
        return lr::hgrn2_f32_launch(q, k, v, g, S0, o, S_final, B, L, H, workspace, st, false, 0.0f);
    if (!hgrn2_tensor_path(dk, dv, chunk, io))
        return lr::hgrn2_general_launch(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, io == LR_BF16,
                                        false, 0.0f, workspace, st);
    return lr::hgrn2_launch(q, k, v, g, S0, o, S_final, B, L, H, workspace, st);
}

}  // extern "C"

extern "C" int lr_selective_scan_step(const void *x, const void *dt, const void *z, const void *Bm,
                                      const void *Cm, const float *A_log, const float *Dskip,
                                      const float *h_in, float *h_out, void *y, int64_t B, int64_t D,
                                      int64_t N, lr_dtype io, int dt_softplus, lr_stream_t stream) {
    if (B < 0 || D < 0 || N < 0 || !io_ok(io)) return LR_ERR_INVALID_ARG;
    if (N != 16) return LR_ERR_UNSUPPORTED;
    if (B * D > 0) {
        const void *req[] = {x, dt, Bm, Cm, A_log, h_out, y};
        const void *all[] = {x, dt, z, Bm, Cm, A_log, Dskip, h_in, h_out, y};
        const int rc = validate_step_common(req, 7, all, 10);
        if (rc != LR_OK) return rc;
    }
    return lr::selective_step_launch(x, dt, z, Bm, Cm, A_log, Dskip, h_in, h_out, y, B, D, io == LR_BF16,
                                     dt_softplus, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int lr_rglru_scan_step(const void *x, const void *r, const void *i, const float *a_log,
                                  float c, const float *h_in, float *h_out, void *y, int64_t B,
                                  int64_t D, lr_dtype io, lr_stream_t stream) {
    if (B < 0 || D < 0 || !io_ok(io) || !std::isfinite(c)) return LR_ERR_INVALID_ARG;
    if (B * D > 0) {
        const void *req[] = {x, r, i, a_log, h_out, y};
        const void *all[] = {x, r, i, a_log, h_in, h_out, y};
        const int rc = validate_step_common(req, 6, all, 7);
        if (rc != LR_OK) return rc;
    }
    return lr::rglru_step_launch(x, r, i, a_log, c, h_in, h_out, y, B, D, io == LR_BF16,
                                 reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int lr_hgrn2_step(const void *q, const void *k, const void *v, const void *g,
                             const float *S_in, float *S_out, void *o, int64_t B, int64_t H,
                             int64_t dk, int64_t dv, lr_dtype io, lr_stream_t stream) {
    if (B < 0 || H <= 0 || dk <= 0 || dv <= 0 || !io_ok(io)) return LR_ERR_INVALID_ARG;
    if (B > 0) {
        const void *req[] = {q, k, v, g, S_out, o};
        const void *all[] = {q, k, v, g, S_in, S_out, o};
        const int rc = validate_step_common(req, 6, all, 7);
        if (rc != LR_OK) return rc;
    }
    return lr::hgrn2_step_launch(q, k, v, g, S_in, S_out, o, B, H, dk, dv, io == LR_BF16,
                                 reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t lr_minmax_scan_workspace_size(int64_t B, int64_t L, int64_t D, lr_dtype io) {
    if (B < 0 || L < 0 || D < 0 || !io_ok(io)) return 0;
    if (B == 0 || L == 0 || D == 0) return lr::kStatusBytes;
    lr::DiagPlan p;
    if (lr::minmax_plan(B, L, D, io, &p) != LR_OK) return SIZE_MAX;
    return p.ws_bytes;
}

extern "C" int lr_minmax_scan_fwd(const void *r, const void *s, const float *x0, void *y, float *x_final,
                                  int64_t B, int64_t L, int64_t D, lr_dtype io, void *workspace,
                                  size_t ws_bytes, lr_stream_t stream) {
    int rc = validate_minmax(r, s, x0, y, x_final, B, L, D, io);
    if (rc != LR_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (B == 0 || D == 0) return lr::status_ok_no_launch(workspace, ws_bytes, st);
    if (L == 0) {
        if ((rc = copy_state(x0, x_final, size_t(B) * D, st)) != LR_OK) return rc;
        return lr::status_ok_no_launch(workspace, ws_bytes, st);
    }
    lr::DiagPlan p;
    if ((rc = lr::minmax_plan(B, L, D, io, &p)) != LR_OK) return rc;
    if ((rc = check_workspace(p, workspace, ws_bytes)) != LR_OK) return rc;
    return lr::minmax_launch(r, s, x0, y, x_final, B, L, D, io, p, workspace, st);
}

// RG-LRU with the gates given before their sigmoid ([RGLRU] forward applies
// sigmoid to the r and i projections before the scan); the sigmoid runs in
// the scan kernel.  Same workspace as lr_rglru_scan_fwd.
extern "C" int lr_rglru_scan_preact_fwd(const void *x, const void *r_pre, const void *i_pre,
                                        const float *a_log, float c, const float *h0, void *y,
                                        float *h_final, int64_t B, int64_t L, int64_t D, lr_dtype io,
                                        void *workspace, size_t ws_bytes, lr_stream_t stream) {
    int rc = validate_rglru(x, r_pre, i_pre, a_log, c, h0, y, h_final, B, L, D, io);
    if (rc != LR_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (B == 0 || D == 0) return lr::status_ok_no_launch(workspace, ws_bytes, st);
    if (L == 0) {
        if ((rc = copy_state(h0, h_final, size_t(B) * D, st)) != LR_OK) return rc;
        return lr::status_ok_no_launch(workspace, ws_bytes, st);
    }
    lr::DiagPlan p;
    if ((rc = lr::rglru_plan(B, L, D, io, &p)) != LR_OK) return rc;
    if ((rc = check_workspace(p, workspace, ws_bytes)) != LR_OK) return rc;
    return lr::rglru_launch(x, r_pre, i_pre, a_log, c, h0, y, h_final, B, L, D, io, p, workspace, st,
                            true);
}

// HGRN2 with the forget gate given as its pre-activation f: the kernel forms
// g = lb + (1 - lb) sigmoid(f) ([HGRN2] sigmoid-activated, lower-bounded
// gate) before the recurrence.  lb in [0, 1).
extern "C" int lr_hgrn2_preact_fwd(const void *q, const void *k, const void *v, const void *f, float lb,
                                   const float *S0, void *o, float *S_final, int64_t B, int64_t L,
                                   int64_t H, int64_t dk, int64_t dv, int64_t chunk, lr_dtype io,
                                   void *workspace, size_t ws_bytes, lr_stream_t stream) {
    if (!(lb >= 0.0f && lb < 1.0f)) return LR_ERR_INVALID_ARG;
    int rc = validate_hgrn2(q, k, v, f, S0, o, S_final, B, L, H, dk, dv, chunk, io);
    if (rc != LR_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (B == 0) return lr::status_ok_no_launch(workspace, ws_bytes, st);
    if (L == 0) {
        if ((rc = copy_state(S0, S_final, size_t(B) * H * dv * dk, st)) != LR_OK) return rc;
        return lr::status_ok_no_launch(workspace, ws_bytes, st);
    }
    size_t need = 0;
    if ((rc = lr::hgrn2_workspace(B, L, H, &need)) != LR_OK) return rc;
    if (workspace == nullptr || ws_bytes < need) return LR_ERR_WORKSPACE;
    if (misaligned(workspace)) return LR_ERR_MISALIGNED;
    if (hgrn2_f32_tensor_path(dk, dv, chunk, io))
        return lr::hgrn2_f32_launch(q, k, v, f, S0, o, S_final, B, L, H, workspace, st, true, lb);
    if (!hgrn2_tensor_path(dk, dv, chunk, io))
        return lr::hgrn2_general_launch(q, k, v, f, S0, o, S_final, B, L, H, dk, dv, io == LR_BF16,
                                        true, lb, workspace, st);
    return lr::hgrn2_launch(q, k, v, f, S0, o, S_final, B, L, H, workspace, st, true, lb);
}

extern "C" int lr_minmax_scan_step(const void *r, const void *s, const float *x_in, float *x_out,
                                   void *y, int64_t B, int64_t D, lr_dtype io, lr_stream_t stream) {
    if (B < 0 || D < 0 || !io_ok(io)) return LR_ERR_INVALID_ARG;
    if (B * D > 0) {
        const void *req[] = {r, s, x_out, y};
        const void *all[] = {r, s, x_in, x_out, y};
        const int rc = validate_step_common(req, 4, all, 5);
        if (rc != LR_OK) return rc;
    }
    return lr::minmax_step_launch(r, s, x_in, x_out, y, B, D, io == LR_BF16,
                                  reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- host buffers
// The same scans with every tensor in host memory: the engine in lr_host.cu
// runs the sequence through the GPU in time chunks, each chunk one call of
// the device entry point above (so every chunk is validated and launched
// exactly as a device call is), the state carried on the device.
namespace {

size_t io_bytes(lr_dtype io) { return io == LR_BF16 ? 2 : 4; }

// the final state of an empty sequence, in host memory
void host_state_copy(const float *s0, float *s_final, size_t count) {
    if (s_final == nullptr || count == 0) return;
    if (s0 != nullptr)
        std::memcpy(s_final, s0, count * sizeof(float));
    else
        std::memset(s_final, 0, count * sizeof(float));
}

int host_ws_check(const lr::HostJob &j, const void *ws, size_t ws_bytes) {
    if (j.kernel_ws == SIZE_MAX) return LR_ERR_CUDA;
    if (ws == nullptr || ws_bytes < lr::host_workspace_bytes(j)) return LR_ERR_WORKSPACE;
    return misaligned(ws) ? LR_ERR_MISALIGNED : LR_OK;
}

struct SelHost {
    int64_t B, D, N;
    lr_dtype io;
    int dt_softplus;
    bool has_z;
};

int sel_host_chunk(const void *c, const void *const *in, void *const *out, const void *const *par, int64_t lc,
                   const float *s_in, float *s_out, void *kws, size_t kws_bytes, cudaStream_t st) {
    const SelHost &a = *static_cast<const SelHost *>(c);
    const int b = a.has_z ? 3 : 2;   // inputs: x, dt, [z], Bm, Cm
    return lr_selective_scan_fwd(in[0], in[1], a.has_z ? in[2] : nullptr, in[b], in[b + 1],
                                 static_cast<const float *>(par[0]), static_cast<const float *>(par[1]), s_in,
                                 out[0], s_out, a.B, lc, a.D, a.N, a.io, a.dt_softplus, kws, kws_bytes,
                                 reinterpret_cast<lr_stream_t>(st));
}

// The chunk length always counts z's bytes, so the workspace query (which
// assumes z and Dskip) covers calls without them.
lr::HostJob sel_host_job(const SelHost &a, int64_t L, const void *x, const void *dt, const void *z,
                         const void *Bm, const void *Cm, const float *A_log, const float *Dskip,
                         const float *h0, void *y, float *h_final, bool with_dskip) {
    lr::HostJob j;
    j.B = a.B;
    j.L = L;
    j.es = io_bytes(a.io);
    int n = 0;
    j.in[n++] = {x, nullptr, a.D};
    j.in[n++] = {dt, nullptr, a.D};
    if (a.has_z) j.in[n++] = {z, nullptr, a.D};
    j.in[n++] = {Bm, nullptr, a.N};
    j.in[n++] = {Cm, nullptr, a.N};
    j.n_in = n;
    j.out[0] = {nullptr, y, a.D};
    j.n_out = 1;
    j.par[0] = {A_log, size_t(a.D) * a.N * sizeof(float)};
    j.par[1] = {Dskip, with_dskip ? size_t(a.D) * sizeof(float) : 0};
    j.n_par = 2;
    j.state0 = h0;
    j.state_final = h_final;
    j.state_bytes = size_t(a.B) * a.D * a.N * sizeof(float);
    j.Lc = lr::host_chunk_steps(a.B, L, j.es * size_t(3 * a.D + 2 * a.N));
    j.kernel_ws = lr_selective_scan_workspace_size(a.B, j.Lc, a.D, a.N, a.io);
    j.launch = sel_host_chunk;
    j.ctx = &a;
    return j;
}

struct RgHost {
    int64_t B, D;
    lr_dtype io;
    float c;
};

int rg_host_chunk(const void *c, const void *const *in, void *const *out, const void *const *par, int64_t lc,
                  const float *s_in, float *s_out, void *kws, size_t kws_bytes, cudaStream_t st) {
    const RgHost &a = *static_cast<const RgHost *>(c);
    return lr_rglru_scan_fwd(in[0], in[1], in[2], static_cast<const float *>(par[0]), a.c, s_in, out[0], s_out,
                             a.B, lc, a.D, a.io, kws, kws_bytes, reinterpret_cast<lr_stream_t>(st));
}

lr::HostJob rg_host_job(const RgHost &a, int64_t L, const void *x, const void *r, const void *i,
                        const float *a_log, const float *h0, void *y, float *h_final) {
    lr::HostJob j;
    j.B = a.B;
    j.L = L;
    j.es = io_bytes(a.io);
    j.in[0] = {x, nullptr, a.D};
    j.in[1] = {r, nullptr, a.D};
    j.in[2] = {i, nullptr, a.D};
    j.n_in = 3;
    j.out[0] = {nullptr, y, a.D};
    j.n_out = 1;
    j.par[0] = {a_log, size_t(a.D) * sizeof(float)};
    j.n_par = 1;
    j.state0 = h0;
    j.state_final = h_final;
    j.state_bytes = size_t(a.B) * a.D * sizeof(float);
    j.Lc = lr::host_chunk_steps(a.B, L, j.es * size_t(3 * a.D));
    j.kernel_ws = lr_rglru_scan_workspace_size(a.B, j.Lc, a.D, a.io);
    j.launch = rg_host_chunk;
    j.ctx = &a;
    return j;
}

struct HgHost {
    int64_t B, H, dk, dv, chunk;
    lr_dtype io;
};

int hg_host_chunk(const void *c, const void *const *in, void *const *out, const void *const *, int64_t lc,
                  const float *s_in, float *s_out, void *kws, size_t kws_bytes, cudaStream_t st) {
    const HgHost &a = *static_cast<const HgHost *>(c);
    return lr_hgrn2_fwd(in[0], in[1], in[2], in[3], s_in, out[0], s_out, a.B, lc, a.H, a.dk, a.dv, a.chunk, a.io,
                        kws, kws_bytes, reinterpret_cast<lr_stream_t>(st));
}

lr::HostJob hg_host_job(const HgHost &a, int64_t L, const void *q, const void *k, const void *v,
                        const void *g, const float *S0, void *o, float *S_final) {
    lr::HostJob j;
    j.B = a.B;
    j.L = L;
    j.es = io_bytes(a.io);
    j.in[0] = {q, nullptr, a.H * a.dk};
    j.in[1] = {k, nullptr, a.H * a.dk};
    j.in[2] = {v, nullptr, a.H * a.dv};
    j.in[3] = {g, nullptr, a.H * a.dv};
    j.n_in = 4;
    j.out[0] = {nullptr, o, a.H * a.dv};
    j.n_out = 1;
    j.n_par = 0;
    j.state0 = S0;
    j.state_final = S_final;
    j.state_bytes = size_t(a.B) * a.H * a.dv * a.dk * sizeof(float);
    j.Lc = lr::host_chunk_steps(a.B, L, j.es * size_t(2 * a.H * (a.dk + a.dv)));
    j.kernel_ws = lr_hgrn2_workspace_size(a.B, j.Lc, a.H, a.dk, a.dv, a.io);
    j.launch = hg_host_chunk;
    j.ctx = &a;
    return j;
}

struct MmHost {
    int64_t B, D;
    lr_dtype io;
};

int mm_host_chunk(const void *c, const void *const *in, void *const *out, const void *const *, int64_t lc,
                  const float *s_in, float *s_out, void *kws, size_t kws_bytes, cudaStream_t st) {
    const MmHost &a = *static_cast<const MmHost *>(c);
    return lr_minmax_scan_fwd(in[0], in[1], s_in, out[0], s_out, a.B, lc, a.D, a.io, kws, kws_bytes,
                              reinterpret_cast<lr_stream_t>(st));
}

lr::HostJob mm_host_job(const MmHost &a, int64_t L, const void *r, const void *s, const float *x0, void *y,
                        float *x_final) {
    lr::HostJob j;
    j.B = a.B;
    j.L = L;
    j.es = io_bytes(a.io);
    j.in[0] = {r, nullptr, a.D};
    j.in[1] = {s, nullptr, a.D};
    j.n_in = 2;
    j.out[0] = {nullptr, y, a.D};
    j.n_out = 1;
    j.n_par = 0;
    j.state0 = x0;
    j.state_final = x_final;
    j.state_bytes = size_t(a.B) * a.D * sizeof(float);
    j.Lc = lr::host_chunk_steps(a.B, L, j.es * size_t(2 * a.D));
    j.kernel_ws = lr_minmax_scan_workspace_size(a.B, j.Lc, a.D, a.io);
    j.launch = mm_host_chunk;
    j.ctx = &a;
    return j;
}

}  // namespace

extern "C" size_t lr_selective_scan_fwd_host_workspace_size(int64_t B, int64_t L, int64_t D, int64_t N,
                                                            lr_dtype io) {
    if (B <= 0 || L <= 0 || D <= 0 || N != 16 || !io_ok(io)) return 0;
    const SelHost a{B, D, N, io, 1, true};
    const lr::HostJob j = sel_host_job(a, L, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                       nullptr, nullptr, nullptr, true);
    return j.kernel_ws == SIZE_MAX ? SIZE_MAX : lr::host_workspace_bytes(j);
}

static int selective_host(const void *x, const void *dt, const void *z, const void *Bm, const void *Cm,
                          const float *A_log, const float *Dskip, const float *h0, void *y, float *h_final,
                          int64_t B, int64_t L, int64_t D, int64_t N, lr_dtype io, int dt_softplus,
                          void *workspace, size_t ws_bytes, lr_stream_t stream, bool async_) {
    int rc = validate_selective(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final, B, L, D, N, io);
    if (rc != LR_OK) return rc;
    if (B == 0 || D == 0) return LR_OK;
    if (L == 0) {
        host_state_copy(h0, h_final, size_t(B) * D * N);
        return LR_OK;
    }
    const SelHost a{B, D, N, io, dt_softplus, z != nullptr};
    const lr::HostJob j = sel_host_job(a, L, x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final, Dskip != nullptr);
    if ((rc = host_ws_check(j, workspace, ws_bytes)) != LR_OK) return rc;
    return lr::run_host_job(j, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream), async_);
}

extern "C" int lr_selective_scan_fwd_host(const void *x, const void *dt, const void *z, const void *Bm,
                                          const void *Cm, const float *A_log, const float *Dskip,
                                          const float *h0, void *y, float *h_final, int64_t B, int64_t L,
                                          int64_t D, int64_t N, lr_dtype io, int dt_softplus, void *workspace,
                                          size_t ws_bytes, lr_stream_t stream) {
    return selective_host(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final, B, L, D, N, io, dt_softplus,
                          workspace, ws_bytes, stream, false);
}

extern "C" int lr_selective_scan_fwd_host_async(const void *x, const void *dt, const void *z, const void *Bm,
                                                const void *Cm, const float *A_log, const float *Dskip,
                                                const float *h0, void *y, float *h_final, int64_t B,
                                                int64_t L, int64_t D, int64_t N, lr_dtype io, int dt_softplus,
                                                void *workspace, size_t ws_bytes, lr_stream_t stream) {
    return selective_host(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final, B, L, D, N, io, dt_softplus,
                          workspace, ws_bytes, stream, true);
}

extern "C" size_t lr_rglru_scan_fwd_host_workspace_size(int64_t B, int64_t L, int64_t D, lr_dtype io) {
    if (B <= 0 || L <= 0 || D <= 0 || !io_ok(io)) return 0;
    const RgHost a{B, D, io, 8.0f};
    const lr::HostJob j = rg_host_job(a, L, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
    return j.kernel_ws == SIZE_MAX ? SIZE_MAX : lr::host_workspace_bytes(j);
}

static int rglru_host(const void *x, const void *r, const void *i, const float *a_log, float c,
                      const float *h0, void *y, float *h_final, int64_t B, int64_t L, int64_t D, lr_dtype io,
                      void *workspace, size_t ws_bytes, lr_stream_t stream, bool async_) {
    int rc = validate_rglru(x, r, i, a_log, c, h0, y, h_final, B, L, D, io);
    if (rc != LR_OK) return rc;
    if (B == 0 || D == 0) return LR_OK;
    if (L == 0) {
        host_state_copy(h0, h_final, size_t(B) * D);
        return LR_OK;
    }
    const RgHost a{B, D, io, c};
    const lr::HostJob j = rg_host_job(a, L, x, r, i, a_log, h0, y, h_final);
    if ((rc = host_ws_check(j, workspace, ws_bytes)) != LR_OK) return rc;
    return lr::run_host_job(j, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream), async_);
}

extern "C" int lr_rglru_scan_fwd_host(const void *x, const void *r, const void *i, const float *a_log,
                                      float c, const float *h0, void *y, float *h_final, int64_t B, int64_t L,
                                      int64_t D, lr_dtype io, void *workspace, size_t ws_bytes,
                                      lr_stream_t stream) {
    return rglru_host(x, r, i, a_log, c, h0, y, h_final, B, L, D, io, workspace, ws_bytes, stream, false);
}

extern "C" int lr_rglru_scan_fwd_host_async(const void *x, const void *r, const void *i, const float *a_log,
                                            float c, const float *h0, void *y, float *h_final, int64_t B,
                                            int64_t L, int64_t D, lr_dtype io, void *workspace,
                                            size_t ws_bytes, lr_stream_t stream) {
    return rglru_host(x, r, i, a_log, c, h0, y, h_final, B, L, D, io, workspace, ws_bytes, stream, true);
}

extern "C" size_t lr_hgrn2_fwd_host_workspace_size(int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv,
                                                   lr_dtype io) {
    if (B <= 0 || L <= 0 || H <= 0 || dk <= 0 || dv <= 0 || !io_ok(io)) return 0;
    const HgHost a{B, H, dk, dv, 64, io};
    const lr::HostJob j = hg_host_job(a, L, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
    return j.kernel_ws == SIZE_MAX ? SIZE_MAX : lr::host_workspace_bytes(j);
}

static int hgrn2_host(const void *q, const void *k, const void *v, const void *g, const float *S0, void *o,
                      float *S_final, int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv, int64_t chunk,
                      lr_dtype io, void *workspace, size_t ws_bytes, lr_stream_t stream, bool async_) {
    int rc = validate_hgrn2(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, chunk, io);
    if (rc != LR_OK) return rc;
    if (B == 0) return LR_OK;
    if (L == 0) {
        host_state_copy(S0, S_final, size_t(B) * H * dk * dv);
        return LR_OK;
    }
    const HgHost a{B, H, dk, dv, chunk, io};
    const lr::HostJob j = hg_host_job(a, L, q, k, v, g, S0, o, S_final);
    if ((rc = host_ws_check(j, workspace, ws_bytes)) != LR_OK) return rc;
    return lr::run_host_job(j, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream), async_);
}

extern "C" int lr_hgrn2_fwd_host(const void *q, const void *k, const void *v, const void *g, const float *S0,
                                 void *o, float *S_final, int64_t B, int64_t L, int64_t H, int64_t dk,
                                 int64_t dv, int64_t chunk, lr_dtype io, void *workspace, size_t ws_bytes,
                                 lr_stream_t stream) {
    return hgrn2_host(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, chunk, io, workspace, ws_bytes, stream,
                      false);
}

extern "C" int lr_hgrn2_fwd_host_async(const void *q, const void *k, const void *v, const void *g,
                                       const float *S0, void *o, float *S_final, int64_t B, int64_t L,
                                       int64_t H, int64_t dk, int64_t dv, int64_t chunk, lr_dtype io,
                                       void *workspace, size_t ws_bytes, lr_stream_t stream) {
    return hgrn2_host(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, chunk, io, workspace, ws_bytes, stream,
                      true);
}

extern "C" size_t lr_minmax_scan_fwd_host_workspace_size(int64_t B, int64_t L, int64_t D, lr_dtype io) {
    if (B <= 0 || L <= 0 || D <= 0 || !io_ok(io)) return 0;
    const MmHost a{B, D, io};
    const lr::HostJob j = mm_host_job(a, L, nullptr, nullptr, nullptr, nullptr, nullptr);
    return j.kernel_ws == SIZE_MAX ? SIZE_MAX : lr::host_workspace_bytes(j);
}

static int minmax_host(const void *r, const void *s, const float *x0, void *y, float *x_final, int64_t B,
                       int64_t L, int64_t D, lr_dtype io, void *workspace, size_t ws_bytes,
                       lr_stream_t stream, bool async_) {
    int rc = validate_minmax(r, s, x0, y, x_final, B, L, D, io);
    if (rc != LR_OK) return rc;
    if (B == 0 || D == 0) return LR_OK;
    if (L == 0) {
        host_state_copy(x0, x_final, size_t(B) * D);
        return LR_OK;
    }
    const MmHost a{B, D, io};
    const lr::HostJob j = mm_host_job(a, L, r, s, x0, y, x_final);
    if ((rc = host_ws_check(j, workspace, ws_bytes)) != LR_OK) return rc;
    return lr::run_host_job(j, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream), async_);
}

extern "C" int lr_minmax_scan_fwd_host(const void *r, const void *s, const float *x0, void *y, float *x_final,
                                       int64_t B, int64_t L, int64_t D, lr_dtype io, void *workspace,
                                       size_t ws_bytes, lr_stream_t stream) {
    return minmax_host(r, s, x0, y, x_final, B, L, D, io, workspace, ws_bytes, stream, false);
}

extern "C" int lr_minmax_scan_fwd_host_async(const void *r, const void *s, const float *x0, void *y,
                                             float *x_final, int64_t B, int64_t L, int64_t D, lr_dtype io,
                                             void *workspace, size_t ws_bytes, lr_stream_t stream) {
    return minmax_host(r, s, x0, y, x_final, B, L, D, io, workspace, ws_bytes, stream, true);
}

extern "C" int lr_host_sync(void) { return lr::host_sync(); }
