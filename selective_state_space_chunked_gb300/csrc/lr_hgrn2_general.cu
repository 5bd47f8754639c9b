// lr_hgrn2_general.cu -- HGRN2 recurrence (frankenstein-transformer docs,
// HGRN2 Attention page: S_t = diag(g_t) S_{t-1} + v_t k_t^T, o_t = S_t q_t)
// for the shapes and I/O types the tcgen05 chunked kernel does not take:
// fp32 I/O (whose 1e-4 parity bar bf16 tensor-core operands cannot meet) and
// head dims other than dk = dv = 128.
//
// One warp owns one row i of one (batch, head) state and walks the sequence
// step by step, exactly as the page's recurrence reads: lane l holds
// S[i][j] for j = l, l + 32, ... (dk <= 32 * M) in registers,
//   S[i][:] = g_t[i] S[i][:] + v_t[i] k_t,   o_t[i] = S[i][:] . q_t,
// with the dot product finished by a warp reduction.  All arithmetic is
// fp32; bf16 outputs are rounded at the store.  The eight warps of a block
// take consecutive rows of one head, so k_t and q_t are read from L1 after
// the first warp; the next step's operands are loaded before the current
// step's arithmetic.  The cost is O(L dv dk) on the CUDA cores, with no
// chunking and hence no range limit on the gates.
#include <cuda_runtime.h>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

constexpr int kGenWarps = 8;

// PRE: g arrives as the pre-activation f; g = lb + (1 - lb) sigmoid(f).
template <typename IO, int M, bool PRE>
__global__ void __launch_bounds__(32 * kGenWarps)
    hgrn2_general_kernel(const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
                         const IO *__restrict__ g, const float *__restrict__ S0,
                         IO *__restrict__ o, float *__restrict__ S_final, int64_t B, int64_t L,
                         int64_t H, int64_t dk, int64_t dv, float lb) {
    const int64_t row = (int64_t(blockIdx.x) * kGenWarps) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= B * H * dv) return;   // warp-uniform
    const int64_t bh = row / dv, i = row - bh * dv;
    const int64_t b = bh / H, h = bh - b * H;
    const int64_t HK = H * dk, HV = H * dv;
    float S[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const int64_t j = lane + 32 * m;
        S[m] = (S0 != nullptr && j < dk) ? S0[row * dk + j] : 0.0f;
    }
    const IO *kb = k + b * L * HK + h * dk;
    const IO *qb = q + b * L * HK + h * dk;
    const IO *vb = v + b * L * HV + h * dv + i;
    const IO *gb = g + b * L * HV + h * dv + i;
    IO *ob = o + b * L * HV + h * dv + i;

    // operands of step t, loaded one step ahead
    float kn[M], qn[M], vn = 0.0f, gn = 1.0f;
    auto load = [&](int64_t t) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int64_t j = lane + 32 * m;
            kn[m] = j < dk ? Io<IO>::to_f(kb[t * HK + j]) : 0.0f;
            qn[m] = j < dk ? Io<IO>::to_f(qb[t * HK + j]) : 0.0f;
        }
        vn = Io<IO>::to_f(vb[t * HV]);
        gn = Io<IO>::to_f(gb[t * HV]);
        if (PRE) gn = fmaf(1.0f - lb, 1.0f / (1.0f + expf(-gn)), lb);
    };
    if (L > 0) load(0);
    for (int64_t t = 0; t < L; ++t) {
        float kc[M], qc[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
            kc[m] = kn[m];
            qc[m] = qn[m];
        }
        const float vc = vn, gc = gn;
        if (t + 1 < L) load(t + 1);
        float acc = 0.0f;
#pragma unroll
        for (int m = 0; m < M; ++m) {
            S[m] = fmaf(gc, S[m], vc * kc[m]);
            acc = fmaf(S[m], qc[m], acc);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) ob[t * HV] = Io<IO>::from_f(acc);
    }
    if (S_final != nullptr) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int64_t j = lane + 32 * m;
            if (j < dk) S_final[row * dk + j] = S[m];
        }
    }
}

template <typename IO, int M>
int launch_m(const void *q, const void *k, const void *v, const void *g, const float *S0, void *o,
             float *S_final, int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv, bool pre,
             float lb, cudaStream_t stream) {
    const int64_t rows = B * H * dv;
    const unsigned grid = unsigned((rows + kGenWarps - 1) / kGenWarps);
    auto kern = pre ? hgrn2_general_kernel<IO, M, true> : hgrn2_general_kernel<IO, M, false>;
    kern<<<grid, 32 * kGenWarps, 0, stream>>>(
        static_cast<const IO *>(q), static_cast<const IO *>(k), static_cast<const IO *>(v),
        static_cast<const IO *>(g), S0, static_cast<IO *>(o), S_final, B, L, H, dk, dv, lb);
    return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

template <typename IO>
int launch_io(const void *q, const void *k, const void *v, const void *g, const float *S0, void *o,
              float *S_final, int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv,
              bool pre, float lb, cudaStream_t stream) {
    if (dk <= 32) return launch_m<IO, 1>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, stream);
    if (dk <= 64) return launch_m<IO, 2>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, stream);
    if (dk <= 128) return launch_m<IO, 4>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, stream);
    if (dk <= 256) return launch_m<IO, 8>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, stream);
    return launch_m<IO, 16>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, stream);
}

}  // namespace

int hgrn2_general_launch(const void *q, const void *k, const void *v, const void *g, const float *S0,
                         void *o, float *S_final, int64_t B, int64_t L, int64_t H, int64_t dk,
                         int64_t dv, int io_bf16, bool preact, float lb, cudaStream_t stream) {
    if (B * H * dv == 0) return LR_OK;
    return io_bf16 ? launch_io<__nv_bfloat16>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, preact, lb,
                                              stream)
                   : launch_io<float>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, preact, lb, stream);
}

}  // namespace lr
