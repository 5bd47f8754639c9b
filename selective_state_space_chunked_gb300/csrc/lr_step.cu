// lr_step.cu -- single-token decode steps of the three recurrences: one
// update of the carried state and its readout, the L = 1 case the pages run
// token by token ([SSM] MultiScaleSSM.forward with past_state and one token,
// [RGLRU] RGLRU.step, [HGRN2] the per-token state update).
//
// A step reads and writes the whole state once and touches every input
// element once, so it is bound by HBM traffic and launch latency; the
// kernels are plain one-pass kernels (no tiling, no tensor cores), with the
// state streamed by 16-byte vector accesses.  They use the accurate math
// library functions: a decode loop runs many steps back to back and the cost
// of an accurate exp is invisible here.  Input and output state may be the
// same buffer (each thread reads its part of the state before writing it).
#include <cuda_runtime.h>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

constexpr int kStepThreads = 128;

__device__ __forceinline__ float softplus_acc(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

// Selective SSM, four lanes per (b, d), four of its 16 states each (so the
// state moves in coalesced 16-byte pieces and each lane runs a quarter of
// the exp chain):
//   delta = softplus(dt); h[n] = exp(delta A[n]) h[n] + delta B[n] x;
//   y = (sum_n C[n] h[n] + D x) silu(z)
// Every lane computes delta and u itself (cheap, shared loads); the partial
// C . h sums meet by two xor shuffles and the group's first lane stores y.
// A lane reads its 16 bytes of h_in before writing the same 16 bytes of
// h_out, so the update may run in place.
template <typename IO, bool HAS_Z, bool SOFTPLUS>
__global__ void __launch_bounds__(kStepThreads)
    selective_step_kernel(const IO *__restrict__ x, const IO *__restrict__ dt, const IO *__restrict__ z,
                          const IO *__restrict__ Bm, const IO *__restrict__ Cm,
                          const float *__restrict__ A_log, const float *__restrict__ Dskip,
                          const float *h_in, float *h_out, IO *__restrict__ y, int64_t B, int64_t D) {
    const int64_t g = int64_t(blockIdx.x) * kStepThreads + threadIdx.x;
    const int64_t idx = g >> 2;            // (b, d)
    const int q = int(g & 3);              // states 4q .. 4q+3
    const bool valid = idx < B * D;        // whole groups of four share validity
    float acc = 0.0f, xv = 0.0f;
    int64_t d = 0;
    if (valid) {
        const int64_t b = idx / D;
        d = idx - b * D;
        xv = Io<IO>::to_f(x[idx]);
        const float dtv = Io<IO>::to_f(dt[idx]);
        const float dl = SOFTPLUS ? softplus_acc(dtv) : dtv;
        const float u = dl * xv;
        const IO *Bb = Bm + b * 16 + 4 * q, *Cb = Cm + b * 16 + 4 * q;
        const float4 a4 = reinterpret_cast<const float4 *>(A_log + d * 16)[q];
        float4 h = h_in != nullptr ? reinterpret_cast<const float4 *>(h_in + idx * 16)[q]
                                   : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        float *hv = reinterpret_cast<float *>(&h);
        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float decay = expf(dl * -expf(av[e]));
            hv[e] = fmaf(decay, hv[e], u * Io<IO>::to_f(Bb[e]));
            acc = fmaf(Io<IO>::to_f(Cb[e]), hv[e], acc);
        }
        reinterpret_cast<float4 *>(h_out + idx * 16)[q] = h;
    }
    // the four lanes of a group are consecutive lanes of one warp
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    if (valid && q == 0) {
        float o = fmaf(Dskip != nullptr ? Dskip[d] : 0.0f, xv, acc);
        if (HAS_Z) {
            const float zv = Io<IO>::to_f(z[idx]);
            o *= zv / (1.0f + expf(-zv));
        }
        y[idx] = Io<IO>::from_f(o);
    }
}

// RG-LRU, one thread per (b, d):
//   a = exp(c r a_log); h = a h + sqrt(1 - a^2) i x; y = h
template <typename IO>
__global__ void __launch_bounds__(kStepThreads)
    rglru_step_kernel(const IO *__restrict__ x, const IO *__restrict__ r, const IO *__restrict__ ig,
                      const float *__restrict__ a_log, float c, const float *h_in, float *h_out,
                      IO *__restrict__ y, int64_t B, int64_t D) {
    const int64_t idx = int64_t(blockIdx.x) * kStepThreads + threadIdx.x;
    if (idx >= B * D) return;
    const int64_t d = idx - (idx / D) * D;
    const float eps = c * Io<IO>::to_f(r[idx]) * a_log[d];
    const float a = expf(eps);
    const float mult = sqrtf(-expm1f(2.0f * eps));   // sqrt(1 - a^2) without cancellation
    const float h0 = h_in != nullptr ? h_in[idx] : 0.0f;
    const float h = fmaf(a, h0, mult * Io<IO>::to_f(ig[idx]) * Io<IO>::to_f(x[idx]));
    h_out[idx] = h;
    y[idx] = Io<IO>::from_f(h);
}

// MinMax, one thread per (b, d): x = max(min(r, x), s); y = x.  min.NaN /
// max.NaN propagate NaN like torch.minimum / torch.maximum.
template <typename IO>
__global__ void __launch_bounds__(kStepThreads)
    minmax_step_kernel(const IO *__restrict__ r, const IO *__restrict__ s, const float *x_in,
                       float *x_out, IO *__restrict__ y, int64_t B, int64_t D) {
    const int64_t idx = int64_t(blockIdx.x) * kStepThreads + threadIdx.x;
    if (idx >= B * D) return;
    float x = x_in != nullptr ? x_in[idx] : 0.0f;
    float lo;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(lo) : "f"(Io<IO>::to_f(r[idx])), "f"(x));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(x) : "f"(lo), "f"(Io<IO>::to_f(s[idx])));
    x_out[idx] = x;
    y[idx] = Io<IO>::from_f(x);
}

// Four consecutive elements as fp32 (16-byte fp32 or 8-byte bf16 load).
__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// HGRN2, one warp per state row (b, head, value channel i):
//   S[i][:] = g_i S[i][:] + v_i k;  o_i = S[i][:] . q
// VEC: dk is a multiple of 128, each lane takes 4 consecutive keys per 128.
template <typename IO, bool VEC>
__global__ void __launch_bounds__(256)
    hgrn2_step_kernel(const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
                      const IO *__restrict__ g, const float *S_in, float *S_out, IO *__restrict__ o,
                      int64_t B, int64_t H, int64_t dk, int64_t dv) {
    const int64_t row = (int64_t(blockIdx.x) * 256 + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= B * H * dv) return;   // warp-uniform
    const int64_t bh = row / dv, i = row - bh * dv;
    const int64_t b = bh / H, h = bh - b * H;
    const int64_t vi_idx = b * H * dv + h * dv + i;
    const float gi = Io<IO>::to_f(g[vi_idx]), vi = Io<IO>::to_f(v[vi_idx]);
    const IO *kb = k + b * H * dk + h * dk, *qb = q + b * H * dk + h * dk;
    const float *si = S_in != nullptr ? S_in + row * dk : nullptr;
    float *so = S_out + row * dk;
    float acc = 0.0f;
    if (VEC) {
        for (int64_t j = 4 * lane; j < dk; j += 128) {
            const float4 s0 = si != nullptr ? ld4(si + j) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            const float4 k4 = ld4(kb + j), q4 = ld4(qb + j);
            const float4 s4 = make_float4(fmaf(gi, s0.x, vi * k4.x), fmaf(gi, s0.y, vi * k4.y),
                                          fmaf(gi, s0.z, vi * k4.z), fmaf(gi, s0.w, vi * k4.w));
            *reinterpret_cast<float4 *>(so + j) = s4;
            acc = fmaf(s4.x, q4.x, fmaf(s4.y, q4.y, fmaf(s4.z, q4.z, fmaf(s4.w, q4.w, acc))));
        }
    } else {
        for (int64_t j = lane; j < dk; j += 32) {
            const float s = fmaf(gi, si != nullptr ? si[j] : 0.0f, vi * Io<IO>::to_f(kb[j]));
            so[j] = s;
            acc = fmaf(s, Io<IO>::to_f(qb[j]), acc);
        }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (lane == 0) o[vi_idx] = Io<IO>::from_f(acc);
}

unsigned blocks_for(int64_t n, int64_t per_block) { return unsigned((n + per_block - 1) / per_block); }

template <typename IO>
int selective_step_io(const void *x, const void *dt, const void *z, const void *Bm, const void *Cm,
                      const float *A_log, const float *Dskip, const float *h_in, float *h_out, void *y,
                      int64_t B, int64_t D, int dt_softplus, cudaStream_t s) {
    const unsigned grid = blocks_for(4 * B * D, kStepThreads);   // four lanes per (b, d)
    const IO *xi = static_cast<const IO *>(x), *di = static_cast<const IO *>(dt),
             *zi = static_cast<const IO *>(z), *bi = static_cast<const IO *>(Bm),
             *ci = static_cast<const IO *>(Cm);
    IO *yo = static_cast<IO *>(y);
    if (z != nullptr && dt_softplus)
        selective_step_kernel<IO, true, true><<<grid, kStepThreads, 0, s>>>(xi, di, zi, bi, ci, A_log, Dskip,
                                                                           h_in, h_out, yo, B, D);
    else if (z != nullptr)
        selective_step_kernel<IO, true, false><<<grid, kStepThreads, 0, s>>>(xi, di, zi, bi, ci, A_log, Dskip,
                                                                            h_in, h_out, yo, B, D);
    else if (dt_softplus)
        selective_step_kernel<IO, false, true><<<grid, kStepThreads, 0, s>>>(xi, di, zi, bi, ci, A_log, Dskip,
                                                                            h_in, h_out, yo, B, D);
    else
        selective_step_kernel<IO, false, false><<<grid, kStepThreads, 0, s>>>(xi, di, zi, bi, ci, A_log,
                                                                             Dskip, h_in, h_out, yo, B, D);
    return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

}  // namespace

int selective_step_launch(const void *x, const void *dt, const void *z, const void *Bm, const void *Cm,
                          const float *A_log, const float *Dskip, const float *h_in, float *h_out,
                          void *y, int64_t B, int64_t D, int io_bf16, int dt_softplus,
                          cudaStream_t stream) {
    if (B * D == 0) return LR_OK;
    return io_bf16 ? selective_step_io<__nv_bfloat16>(x, dt, z, Bm, Cm, A_log, Dskip, h_in, h_out, y, B, D,
                                                      dt_softplus, stream)
                   : selective_step_io<float>(x, dt, z, Bm, Cm, A_log, Dskip, h_in, h_out, y, B, D,
                                              dt_softplus, stream);
}

int rglru_step_launch(const void *x, const void *r, const void *i, const float *a_log, float c,
                      const float *h_in, float *h_out, void *y, int64_t B, int64_t D, int io_bf16,
                      cudaStream_t stream) {
    if (B * D == 0) return LR_OK;
    const unsigned grid = blocks_for(B * D, kStepThreads);
    if (io_bf16)
        rglru_step_kernel<__nv_bfloat16><<<grid, kStepThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(r),
            static_cast<const __nv_bfloat16 *>(i), a_log, c, h_in, h_out, static_cast<__nv_bfloat16 *>(y),
            B, D);
    else
        rglru_step_kernel<float><<<grid, kStepThreads, 0, stream>>>(
            static_cast<const float *>(x), static_cast<const float *>(r), static_cast<const float *>(i),
            a_log, c, h_in, h_out, static_cast<float *>(y), B, D);
    return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

int hgrn2_step_launch(const void *q, const void *k, const void *v, const void *g, const float *S_in,
                      float *S_out, void *o, int64_t B, int64_t H, int64_t dk, int64_t dv, int io_bf16,
                      cudaStream_t stream) {
    const int64_t rows = B * H * dv;
    if (rows == 0) return LR_OK;
    const unsigned grid = blocks_for(rows * 32, 256);
    // 16-byte state rows and 8/16-byte key/query groups need dk % 128 == 0
    const bool vec = dk % 128 == 0;
    using bf = __nv_bfloat16;
    if (io_bf16) {
        auto kern = vec ? hgrn2_step_kernel<bf, true> : hgrn2_step_kernel<bf, false>;
        kern<<<grid, 256, 0, stream>>>(static_cast<const bf *>(q), static_cast<const bf *>(k),
                                       static_cast<const bf *>(v), static_cast<const bf *>(g), S_in,
                                       S_out, static_cast<bf *>(o), B, H, dk, dv);
    } else {
        auto kern = vec ? hgrn2_step_kernel<float, true> : hgrn2_step_kernel<float, false>;
        kern<<<grid, 256, 0, stream>>>(static_cast<const float *>(q), static_cast<const float *>(k),
                                       static_cast<const float *>(v), static_cast<const float *>(g),
                                       S_in, S_out, static_cast<float *>(o), B, H, dk, dv);
    }
    return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

int minmax_step_launch(const void *r, const void *s, const float *x_in, float *x_out, void *y,
                       int64_t B, int64_t D, int io_bf16, cudaStream_t stream) {
    if (B * D == 0) return LR_OK;
    const unsigned grid = blocks_for(B * D, kStepThreads);
    if (io_bf16)
        minmax_step_kernel<__nv_bfloat16><<<grid, kStepThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(r), static_cast<const __nv_bfloat16 *>(s), x_in, x_out,
            static_cast<__nv_bfloat16 *>(y), B, D);
    else
        minmax_step_kernel<float><<<grid, kStepThreads, 0, stream>>>(
            static_cast<const float *>(r), static_cast<const float *>(s), x_in, x_out,
            static_cast<float *>(y), B, D);
    return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

}  // namespace lr
