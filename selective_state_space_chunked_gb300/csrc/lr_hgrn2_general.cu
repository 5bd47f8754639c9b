// lr_hgrn2_general.cu -- HGRN2 recurrence (frankenstein-transformer docs,
// HGRN2 Attention page: S_t = diag(g_t) S_{t-1} + v_t k_t^T, o_t = S_t q_t)
// for the shapes and I/O types the tcgen05 chunked kernel does not take:
// fp32 I/O (whose 1e-4 parity bar bf16 tensor-core operands cannot meet) and
// head dims other than dk = dv = 128.
//
// Step by step, exactly as the page's recurrence reads, on the CUDA cores in
// fp32.  A block of 64 threads owns RB value rows of one (batch, head); a
// thread owns RT of those rows and CPT key columns of each, in registers, so
// P = dk_pad / CPT consecutive lanes share a row.  The columns come in groups
// of four dealt round-robin (thread p takes groups p, p + P, ...), so the P
// lanes of a row read consecutive 16 bytes of k_t, q_t at a time (no bank
// conflicts):
//     S[i][j] = g_t[i] S[i][j] + v_t[i] k_t[j]    (packed fp32x2 mul + fma)
//     o_t[i]  = sum_j S[i][j] q_t[j]              (packed fma, then a
//                                                  butterfly over the P lanes)
// Each k/q value read from shared memory serves all of the thread's rows.
// The recurrence is serial in time, so the parallelism is B H dv dk / (RT CPT)
// threads: the host takes RT = 2, CPT = 32 (most work per staged value) when
// that still gives 1.5 blocks per SM, else RT = 1, then CPT = 16.
//
// k_t and q_t (shared by every row of the head) and the block's v_t, g_t
// arrive in chunks of TC steps.  When every row start is 16-byte aligned one
// thread stages a chunk with four TMA tensor copies (3-D maps over
// (columns, heads, batch x time); key columns past dk and value rows past dv
// arrive as zeros) into one of three buffers, two chunks ahead of the
// compute, counted on the buffer's mbarrier; otherwise the block copies
// element by element, synchronously.  Per-thread 16-byte copies or one bulk
// copy per row cost more to issue than the updates they feed.  Outputs are
// staged per chunk and written back row-contiguous.  The cost is O(L dv dk)
// with no chunking of the recurrence, hence no range limit on the gates.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {
namespace {

constexpr int kNT = 64;   // threads per block
constexpr int kNB = 3;    // staging buffers: copies run two chunks ahead

// P lanes of CPT key columns share RT value rows
template <int P, int CPT, int RT>
struct GenCfg {
    static constexpr int DKP = P * CPT;                 // padded key dim
    static constexpr int KB = DKP < 256 ? DKP : 256;    // key columns per TMA box (<= 256)
    static constexpr int NH = DKP / KB;                 // key boxes per row
    static constexpr int RB = RT * kNT / P;             // value rows per block
    static constexpr int TC = DKP <= 128 ? 16 : 2048 / DKP;   // steps per staged chunk
    static constexpr int KT = TC * DKP, VT = TC * RB;   // elements per buffer
    // buffer pitch in elements: every TMA destination starts 128-byte aligned
    template <typename IO>
    __host__ __device__ static constexpr int pitch(int n) {
        return int((n * sizeof(IO) + 127) / 128 * 128 / sizeof(IO));
    }
    template <typename IO>
    static constexpr size_t smem_bytes() {
        return sizeof(IO) * size_t(kNB) * (2 * pitch<IO>(KT) + 2 * pitch<IO>(VT)) +
               sizeof(float) * VT + kNB * sizeof(uint64_t);
    }
};

// four consecutive staged values as fp32 (16-byte / 8-byte aligned loads)
template <typename IO>
__device__ __forceinline__ float4 ld4f(const IO *p);
template <>
__device__ __forceinline__ float4 ld4f<float>(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
template <>
__device__ __forceinline__ float4 ld4f<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

// PRE: g arrives as the pre-activation f; g = lb + (1 - lb) sigmoid(f).
// TMA: staged by tensor copies (the host checked alignment and ranges).
// A staged key row lives in NH boxes of KB columns: column j of step t of a
// buffer sits at (j / KB) * TC * KB + t * KB + j % KB.
template <typename IO, int P, int CPT, int RT, bool PRE, bool TMA>
__global__ void __launch_bounds__(kNT, 1)
    hgrn2_general_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                         const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
                         const IO *__restrict__ g, const float *__restrict__ S0,
                         IO *__restrict__ o, float *__restrict__ S_final, int L, int H, int dk,
                         int dv, int nrb, float lb, uint64_t timeout_ns, StatusRef sref,
                         const unsigned long long *__restrict__ redo) {
    using C = GenCfg<P, CPT, RT>;
    constexpr int kCPT = CPT, kRT = RT;
    constexpr int KB = C::KB, RB = C::RB, TC = C::TC, VT = C::VT;
    constexpr int KT = C::template pitch<IO>(C::KT), VTP = C::template pitch<IO>(VT);
    extern __shared__ __align__(128) unsigned char smem[];
    IO *ks = reinterpret_cast<IO *>(smem);   // [NB][NH][TC][KB] (pitch KT)
    IO *qs = ks + kNB * KT;                  // [NB][NH][TC][KB]
    IO *vs = qs + kNB * KT;                  // [NB][TC][RB] (pitch VTP)
    IO *gs = vs + kNB * VTP;                 // [NB][TC][RB]
    float *os = reinterpret_cast<float *>(gs + kNB * VTP);     // [TC][RB]
    uint64_t *full = reinterpret_cast<uint64_t *>(os + VT);    // [NB]: chunk staged

    const int tid = threadIdx.x;
    const int bh = blockIdx.x / nrb, rb = blockIdx.x - bh * nrb;
    // re-running the heads a tensor-core pass marked (with that call's stamp)
    if (redo != nullptr && redo[bh] != sref.stamp) return;
    if (tid == 0 && blockIdx.x == 0) status_begin(sref);
    const int p = tid % P, rg = tid / P;
    const int b = bh / H, h = bh - b * H;
    const int row0 = rb * RB;
    const int rbv = min(RB, dv - row0);      // rows of this block inside dv
    const size_t HK = size_t(H) * dk, HV = size_t(H) * dv;
    const IO *kb = k + size_t(b) * L * HK + size_t(h) * dk;
    const IO *qb = q + size_t(b) * L * HK + size_t(h) * dk;
    const IO *vb = v + size_t(b) * L * HV + size_t(h) * dv + row0;
    const IO *gb = g + size_t(b) * L * HV + size_t(h) * dv + row0;
    IO *ob = o + size_t(b) * L * HV + size_t(h) * dv + row0;

    if (TMA) {
        if (tid == 0) {
            for (int i = 0; i < kNB; ++i) mbar_init(&full[i], 1);
            fence_mbar_init();
        }
    } else {
        // zero what the element copies never write: key columns past dk,
        // value rows past dv
        for (int e = tid; e < kNB * KT; e += kNT) {
            const int ei = e % KT;
            if (ei >= C::KT || (ei / (TC * KB)) * KB + ei % KB >= dk) {
                ks[e] = Io<IO>::from_f(0.0f);
                qs[e] = Io<IO>::from_f(0.0f);
            }
        }
        for (int e = tid; e < kNB * VTP; e += kNT) {
            if (e % VTP >= VT || (e % VTP) % RB >= rbv) {
                vs[e] = Io<IO>::from_f(0.0f);
                gs[e] = Io<IO>::from_f(0.0f);
            }
        }
    }

    // the thread's state: rows row0 + rg*RT + rr; S[rr][2m + e] holds columns
    // 4 (m P + p) + 2e + {0, 1}
    float2 S[kRT][kCPT / 2];
#pragma unroll
    for (int rr = 0; rr < kRT; ++rr) {
        const int i = row0 + rg * kRT + rr;
#pragma unroll
        for (int m2 = 0; m2 < kCPT / 2; ++m2) {
            const int j = 4 * ((m2 >> 1) * P + p) + 2 * (m2 & 1);
            float2 s = make_float2(0.0f, 0.0f);
            if (S0 != nullptr && i < dv) {
                const float *src = S0 + (size_t(bh) * dv + i) * dk;
                if (j < dk) s.x = src[j];
                if (j + 1 < dk) s.y = src[j + 1];
            }
            S[rr][m2] = s;
        }
    }

    const int nchunks = (L + TC - 1) / TC;
    auto stage = [&](int c, int buf) {
        const int t0 = c * TC;
        IO *kd = ks + buf * KT, *qd = qs + buf * KT;
        IO *vd = vs + buf * VTP, *gd = gs + buf * VTP;
        if (TMA) {
            // whole boxes, rows past L included (zero-filled past the tensor)
            if (tid == 0) {
                mbar_arrive_expect_tx(&full[buf], uint32_t(sizeof(IO)) * (2 * C::KT + 2 * VT));
                const int row = b * L + t0;
#pragma unroll
                for (int hh = 0; hh < C::NH; ++hh) {
                    tma_load_3d(kd + hh * TC * KB, &tm_k, &full[buf], hh * KB, h, row);
                    tma_load_3d(qd + hh * TC * KB, &tm_q, &full[buf], hh * KB, h, row);
                }
                tma_load_3d(vd, &tm_v, &full[buf], row0, h, row);
                tma_load_3d(gd, &tm_g, &full[buf], row0, h, row);
            }
        } else {
            const int nt = min(TC, L - t0);
            for (int t = 0; t < nt; ++t) {
                const size_t sk = size_t(t0 + t) * HK, sv = size_t(t0 + t) * HV;
                for (int j = tid; j < dk; j += kNT) {
                    const int at = (j / KB) * TC * KB + t * KB + j % KB;
                    kd[at] = kb[sk + j];
                    qd[at] = qb[sk + j];
                }
                for (int r = tid; r < rbv; r += kNT) {
                    vd[t * RB + r] = vb[sv + r];
                    gd[t * RB + r] = gb[sv + r];
                }
            }
        }
    };

    if (TMA) __syncthreads();   // barriers initialised before anyone waits on them
    for (int c = 0; c < kNB - 1 && c < nchunks; ++c) stage(c, c);
    for (int c = 0; c < nchunks; ++c) {
        const int buf = c % kNB;
        // the buffer chunk c - 1 used is free again: refill it kNB - 1 chunks ahead
        if (c + kNB - 1 < nchunks) stage(c + kNB - 1, (c + kNB - 1) % kNB);
        const bool ok = !TMA || mbar_wait_bounded(&full[buf], (c / kNB) & 1, timeout_ns);
        if (__syncthreads_or(!ok)) {   // chunk c never arrived: report and stop
            if (tid == 0) {
                status_report(sref, LR_ERR_TIMEOUT);
                // let the copies already issued land (bounded) before the block exits
                for (int c2 = c + 1; c2 < c + kNB && c2 < nchunks; ++c2)
                    mbar_wait_bounded(&full[c2 % kNB], (c2 / kNB) & 1, timeout_ns);
            }
            break;
        }
        const int t0 = c * TC, nt = min(TC, L - t0);
#pragma unroll 2
        for (int t = 0; t < nt; ++t) {
            const IO *kr = ks + buf * KT + t * KB + 4 * p;
            const IO *qr = qs + buf * KT + t * KB + 4 * p;
            float2 g2[kRT], v2[kRT], acc[kRT][2];
#pragma unroll
            for (int rr = 0; rr < kRT; ++rr) {
                const int il = rg * kRT + rr;
                float gv = Io<IO>::to_f(gs[buf * VTP + t * RB + il]);
                if (PRE) gv = fmaf(1.0f - lb, 1.0f / (1.0f + expf(-gv)), lb);
                const float vv = Io<IO>::to_f(vs[buf * VTP + t * RB + il]);
                g2[rr] = make_float2(gv, gv);
                v2[rr] = make_float2(vv, vv);
                acc[rr][0] = acc[rr][1] = make_float2(0.0f, 0.0f);
            }
#pragma unroll
            for (int m = 0; m < kCPT / 4; ++m) {
                // column group m P + p: box (4 P m) / KB, offset (4 P m) % KB + 4 p
                const int off = ((4 * P * m) / KB) * TC * KB + (4 * P * m) % KB;
                const float4 k4 = ld4f<IO>(kr + off);
                const float4 q4 = ld4f<IO>(qr + off);
                const float2 k01 = make_float2(k4.x, k4.y), k23 = make_float2(k4.z, k4.w);
                const float2 q01 = make_float2(q4.x, q4.y), q23 = make_float2(q4.z, q4.w);
#pragma unroll
                for (int rr = 0; rr < kRT; ++rr) {
                    S[rr][2 * m] = __ffma2_rn(g2[rr], S[rr][2 * m], __fmul2_rn(v2[rr], k01));
                    S[rr][2 * m + 1] = __ffma2_rn(g2[rr], S[rr][2 * m + 1], __fmul2_rn(v2[rr], k23));
                    acc[rr][0] = __ffma2_rn(S[rr][2 * m], q01, acc[rr][0]);
                    acc[rr][1] = __ffma2_rn(S[rr][2 * m + 1], q23, acc[rr][1]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < kRT; ++rr) {
                float ov = (acc[rr][0].x + acc[rr][0].y) + (acc[rr][1].x + acc[rr][1].y);
#pragma unroll
                for (int off = P / 2; off >= 1; off >>= 1) ov += __shfl_xor_sync(0xffffffffu, ov, off);
                if (p == rr % P) os[t * RB + rg * kRT + rr] = ov;
            }
        }
        __syncthreads();   // chunk c's buffer and every os entry are done
        for (int e = tid; e < TC * RB; e += kNT) {   // RB is a power of two
            const int t = e / RB, r = e % RB;
            if (t < nt && r < rbv) ob[size_t(t0 + t) * HV + r] = Io<IO>::from_f(os[e]);
        }
    }

    if (S_final != nullptr) {
#pragma unroll
        for (int rr = 0; rr < kRT; ++rr) {
            const int i = row0 + rg * kRT + rr;
            if (i >= dv) continue;
            float *dst = S_final + (size_t(bh) * dv + i) * dk;
#pragma unroll
            for (int m2 = 0; m2 < kCPT / 2; ++m2) {
                const int j = 4 * ((m2 >> 1) * P + p) + 2 * (m2 & 1);
                if (j < dk) dst[j] = S[rr][m2].x;
                if (j + 1 < dk) dst[j + 1] = S[rr][m2].y;
            }
        }
    }
}

inline bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

template <typename IO, int P, int CPT, int RT>
int launch_p(const void *q, const void *k, const void *v, const void *g, const float *S0, void *o,
             float *S_final, int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv, bool pre,
             float lb, StatusRef st, cudaStream_t stream, const unsigned long long *redo) {
    using C = GenCfg<P, CPT, RT>;
    const int nrb = static_cast<int>((dv + C::RB - 1) / C::RB);
    const int64_t grid = B * H * nrb;
    if (dv > INT32_MAX || grid > INT32_MAX) return LR_ERR_UNSUPPORTED;
    const size_t es = sizeof(IO);
    // tensor copies need 16-byte row starts and strides and 32-bit row coordinates
    bool tma = (dk * int64_t(es)) % 16 == 0 && (dv * int64_t(es)) % 16 == 0 && (C::RB * es) % 16 == 0 &&
               aligned16(q) && aligned16(k) && aligned16(v) && aligned16(g) && B * L <= INT32_MAX;
    CUtensorMap mq{}, mk{}, mv{}, mg{};
    if (tma) {
        const auto tt = Io<IO>::kTmType;
        const uint64_t rows = uint64_t(B) * L;
        tma = encode_map_3d(&mq, q, tt, es, dk, H, rows, C::KB, 1, C::TC) &&
              encode_map_3d(&mk, k, tt, es, dk, H, rows, C::KB, 1, C::TC) &&
              encode_map_3d(&mv, v, tt, es, dv, H, rows, C::RB, 1, C::TC) &&
              encode_map_3d(&mg, g, tt, es, dv, H, rows, C::RB, 1, C::TC);
    }
    const size_t smem = C::template smem_bytes<IO>();
    auto kern = pre ? (tma ? hgrn2_general_kernel<IO, P, CPT, RT, true, true>
                           : hgrn2_general_kernel<IO, P, CPT, RT, true, false>)
                    : (tma ? hgrn2_general_kernel<IO, P, CPT, RT, false, true>
                           : hgrn2_general_kernel<IO, P, CPT, RT, false, false>);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return LR_ERR_CUDA;
    kern<<<static_cast<unsigned>(grid), kNT, smem, stream>>>(
        mq, mk, mv, mg, static_cast<const IO *>(q), static_cast<const IO *>(k),
        static_cast<const IO *>(v), static_cast<const IO *>(g), S0, static_cast<IO *>(o), S_final,
        static_cast<int>(L), static_cast<int>(H), static_cast<int>(dk), static_cast<int>(dv), nrb, lb,
        kDefaultTimeoutNs, st, redo);
    return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

// DKP = padded key dim: (32 columns, 2 rows) per thread while that gives
// 1.5 blocks per SM, else (32, 1), else (16, 1); DKP = 512 always (32, 2)
template <typename IO, int DKP>
int launch_dk(const void *q, const void *k, const void *v, const void *g, const float *S0, void *o,
              float *S_final, int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv, bool pre,
              float lb, StatusRef st, cudaStream_t stream, const unsigned long long *redo) {
    int sms = 0;
    if (device_sm_count(&sms) != LR_OK) return LR_ERR_CUDA;
    auto blocks = [&](int rb) { return B * H * ((dv + rb - 1) / rb); };
    const int64_t want = 3 * int64_t(sms) / 2;
    if (DKP > 256 || blocks(2 * kNT / (DKP / 32)) >= want)
        return launch_p<IO, DKP / 32, 32, 2>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, st, stream, redo);
    if constexpr (DKP <= 256) {
        if (blocks(kNT / (DKP / 32)) >= want)
            return launch_p<IO, DKP / 32, 32, 1>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb,
                                                 st, stream, redo);
        return launch_p<IO, DKP / 16, 16, 1>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, st, stream, redo);
    }
    return LR_ERR_UNSUPPORTED;
}

template <typename IO>
int launch_io(const void *q, const void *k, const void *v, const void *g, const float *S0, void *o,
              float *S_final, int64_t B, int64_t L, int64_t H, int64_t dk, int64_t dv,
              bool pre, float lb, StatusRef st, cudaStream_t stream, const unsigned long long *redo) {
    if (dk <= 32) return launch_dk<IO, 32>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, st, stream, redo);
    if (dk <= 64) return launch_dk<IO, 64>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, st, stream, redo);
    if (dk <= 128) return launch_dk<IO, 128>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, st, stream, redo);
    if (dk <= 256) return launch_dk<IO, 256>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, st, stream, redo);
    return launch_dk<IO, 512>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, pre, lb, st, stream, redo);
}

}  // namespace

int hgrn2_general_launch(const void *q, const void *k, const void *v, const void *g, const float *S0,
                         void *o, float *S_final, int64_t B, int64_t L, int64_t H, int64_t dk,
                         int64_t dv, int io_bf16, bool preact, float lb, void *workspace,
                         cudaStream_t stream, const unsigned long long *redo, unsigned long long stamp) {
    if (B * H * dv == 0) return LR_OK;
    StatusRef st = call_status(workspace);
    if (redo != nullptr) st.stamp = stamp;   // part of the call that marked the heads
    return io_bf16 ? launch_io<__nv_bfloat16>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, preact, lb,
                                              st, stream, redo)
                   : launch_io<float>(q, k, v, g, S0, o, S_final, B, L, H, dk, dv, preact, lb, st, stream, redo);
}

}  // namespace lr
