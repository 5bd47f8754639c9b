// lr_internal.h -- host-side declarations shared by the library's .cu files.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda.h>
#include <cuda_runtime.h>

#include "lrscan.h"

namespace lr {

// Every workspace starts with this many bytes of call status (the 64-bit
// status word at offset 0, the rest reserved), then the kernel's scratch.
constexpr size_t kStatusBytes = 256;

// Where a launch records device-side errors, and the call's stamp (see
// status_begin / status_report in lr_device.cuh).
struct StatusRef {
    unsigned long long *word;   // NULL: the launch records nothing
    unsigned long long stamp;   // 48-bit, non-zero
};

// A fresh stamp for a call (or the stamp of the enclosing host-buffer call,
// whose chunk launches share one) with the status word at the start of
// `workspace` (NULL: nothing recorded).
StatusRef call_status(void *workspace);

// Runs the calls made by this thread under one stamp while it lives.
struct SharedStamp {
    SharedStamp();
    ~SharedStamp();
};

// Reads the status code recorded in a workspace's status word, in the order
// of `stream` (it synchronises `stream`); `clear` resets the code to LR_OK.
int read_status(void *workspace, cudaStream_t stream, int *code, bool clear = false);

// Records LR_OK for a call that launches nothing (an empty problem), so the
// workspace's status word describes that call.
int status_ok_no_launch(void *workspace, size_t ws_bytes, cudaStream_t stream);

// Work decomposition of a diagonal scan (selective or RG-LRU).
//   n_cb   channel blocks (batch x ceil(D / DC)); one thread block each when S == 1
//   S      time splits per channel block (S > 1: decoupled look-back between splits)
//   tps    tiles per split; n_tiles = ceil(L / T)
struct DiagPlan {
    int64_t n_cb = 0;
    int S = 1;
    int tps = 0;
    int n_tiles = 0;
    int dc = 0;           // channels per thread block
    int tile_t = 0;       // time steps per tile
    size_t ctrl_bytes = 0;  // flags + ticket (cleared at each call)
    size_t ws_bytes = 0;    // total workspace, status bytes included
    int warps = 0;          // selective scan: warps sharing the flat tile list
    int grid = 0;           // selective scan: thread blocks
};

// Process-wide knobs (see lr_set_split_override / lr_test_withhold_split).
extern int g_split_override;
extern int g_withheld_split;
extern int g_withheld_timeout_ms;
extern int64_t g_selective_warmup_steps;   // lr_set_selective_warmup

// Default wall-clock limit of every bounded device-side wait.
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // 1 s

int device_sm_count(int *sms);  // LR_OK / LR_ERR_CUDA

int rglru_plan(int64_t B, int64_t L, int64_t D, lr_dtype io, DiagPlan *p);
int rglru_launch(const void *x, const void *r, const void *i, const float *a_log, float c,
                 const float *h0, void *y, float *h_final, int64_t B, int64_t L, int64_t D,
                 lr_dtype io, const DiagPlan &p, void *workspace, cudaStream_t stream,
                 bool preact = false);

int selective_plan(int64_t B, int64_t L, int64_t D, lr_dtype io, DiagPlan *p);
int selective_launch(const void *x, const void *dt, const void *z, const void *Bm,
                     const void *Cm, const float *A_log, const float *Dskip, const float *h0,
                     void *y, float *h_final, int64_t B, int64_t L, int64_t D, lr_dtype io,
                     int dt_softplus, const DiagPlan &p, void *workspace, cudaStream_t stream);

int minmax_plan(int64_t B, int64_t L, int64_t D, lr_dtype io, DiagPlan *p);
int minmax_launch(const void *r, const void *s, const float *x0, void *y, float *x_final, int64_t B,
                  int64_t L, int64_t D, lr_dtype io, const DiagPlan &p, void *workspace,
                  cudaStream_t stream);

// Built-in scratch of lr_rglru_scan_fwd_noalloc (1 MiB per device; its first
// kStatusBytes hold the call status).
constexpr size_t kRglruScratchBytes = size_t(1) << 20;
int rglru_builtin_scratch(void **ptr);  // device address, set up once per device

// HGRN2 (chunked tcgen05 kernel)
int hgrn2_workspace(int64_t B, int64_t L, int64_t H, size_t *bytes);
int hgrn2_launch(const void *q, const void *k, const void *v, const void *g, const float *S0,
                 void *o, float *S_final, int64_t B, int64_t L, int64_t H, void *workspace,
                 cudaStream_t stream, bool preact = false, float lb = 0.0f);
// 3-D TMA map over a row-major (d2, d1, d0) tensor with a (b0, b1, b2) box,
// no swizzle, zero fill outside the tensor; false if the driver refuses it.
bool encode_map_3d(CUtensorMap *tm, const void *base, CUtensorMapDataType type, size_t esize,
                   uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, uint32_t b2);

// HGRN2 for fp32 I/O and head dims other than 128 x 128 (CUDA cores, step by step)
// redo != NULL: only the heads whose redo word holds `stamp` run (the heads
// a tensor-core pass of the same call marked), under that call's stamp.
int hgrn2_general_launch(const void *q, const void *k, const void *v, const void *g, const float *S0,
                         void *o, float *S_final, int64_t B, int64_t L, int64_t H, int64_t dk,
                         int64_t dv, int io_bf16, bool preact, float lb, void *workspace,
                         cudaStream_t stream, const unsigned long long *redo = nullptr,
                         unsigned long long stamp = 0);

// HGRN2 with fp32 I/O, 128 x 128 heads, on the tensor cores (split bf16
// operands); heads with steep chunks are re-run by the general kernel.
int hgrn2_f32_launch(const void *q, const void *k, const void *v, const void *g, const float *S0, void *o,
                     float *S_final, int64_t B, int64_t L, int64_t H, void *workspace, cudaStream_t stream,
                     bool preact, float lb);

// Single-token decode steps (plain one-pass kernels)
int selective_step_launch(const void *x, const void *dt, const void *z, const void *Bm, const void *Cm,
                          const float *A_log, const float *Dskip, const float *h_in, float *h_out,
                          void *y, int64_t B, int64_t D, int io_bf16, int dt_softplus,
                          cudaStream_t stream);
int rglru_step_launch(const void *x, const void *r, const void *i, const float *a_log, float c,
                      const float *h_in, float *h_out, void *y, int64_t B, int64_t D, int io_bf16,
                      cudaStream_t stream);
int minmax_step_launch(const void *r, const void *s, const float *x_in, float *x_out, void *y,
                       int64_t B, int64_t D, int io_bf16, cudaStream_t stream);
int hgrn2_step_launch(const void *q, const void *k, const void *v, const void *g, const float *S_in,
                      float *S_out, void *o, int64_t B, int64_t H, int64_t dk, int64_t dv, int io_bf16,
                      cudaStream_t stream);

// Host-buffer runs (lr_host.cu): a scan whose tensors live in host memory is
// moved through the GPU in chunks of Lc time steps on three streams of the
// library's own (copy in, compute, copy out), two chunks in flight in each
// direction, the carried state staying on the device between chunks.
struct HostSeq {          // a (B, L, width) host array of `es`-byte elements
    const void *in = nullptr;   // input sequence (copied in), or
    void *out = nullptr;        // output sequence (copied out)
    int64_t width = 0;
};
struct HostParam {        // a small host array copied to the device once
    const void *host = nullptr;
    size_t bytes = 0;
};
struct HostJob {
    int64_t B = 0, L = 0, Lc = 0;
    size_t es = 0;
    int n_in = 0, n_out = 0, n_par = 0;
    HostSeq in[6], out[2];
    HostParam par[3];
    const float *state0 = nullptr;   // host initial state (NULL: zero)
    float *state_final = nullptr;    // host final state (NULL: not written)
    size_t state_bytes = 0;
    size_t kernel_ws = 0;            // device workspace of one chunk's launch
    // one chunk: device inputs / outputs / parameters, its length, the state
    // it starts from (NULL: zero) and ends in, the kernel workspace
    int (*launch)(const void *ctx, const void *const *in, void *const *out, const void *const *par,
                  int64_t lc, const float *s_in, float *s_out, void *kws, size_t kws_bytes,
                  cudaStream_t stream) = nullptr;
    const void *ctx = nullptr;
};
// chunk length: a multiple of 64 steps (every kernel's tile) holding about
// 64 MB of inputs; `in_bytes_per_step` counts one batch row
int64_t host_chunk_steps(int64_t B, int64_t L, size_t in_bytes_per_step);
extern int64_t g_host_chunk_override;   // lr_set_host_chunk_steps
size_t host_workspace_bytes(const HostJob &job);
// async_: return once the work is queued (no synchronisation, the device-side
// status is left in the workspace); host_sync() waits for every queued call
// of the current device.
int run_host_job(const HostJob &job, void *workspace, size_t ws_bytes, cudaStream_t caller,
                 bool async_ = false);
int host_sync();

}  // namespace lr
