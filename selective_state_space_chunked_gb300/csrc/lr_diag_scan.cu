// lr_diag_scan.cu -- the two diagonal-state scans on sm_103a:
//
//   * RG-LRU   (lrnnx rglru module source, RGLRU.step fallback update):
//       a_t = exp(c r_t a_log),  h = a_t h + sqrt(1 - a_t^2) (i_t x_t),  y_t = h
//   * selective SSM (cortexnet 3.2.1, cortexnet/ssm.py, MultiScaleSSM):
//       delta = softplus(dt), h[n] = exp(delta A[n]) h[n] + delta B_t[n] x,
//       y_t = (C_t . h + D x) silu(z)
//
// Design (both kernels):
//   * A thread block owns a block of DC consecutive channels of one batch row
//     and streams a range of time tiles (T steps x DC channels) through a
//     multi-stage shared-memory ring filled by TMA (cp.async.bulk.tensor,
//     3-D maps over (D, L, B); out-of-range rows and channels arrive as
//     zeros).  Warps are specialised: a producer warp keeps the ring full
//     (and widens shared per-step operands once per tile), compute warps
//     run the recurrence of their channels (one thread per channel, or a
//     lane pair per channel for the 16-state selective scan) with the state
//     in registers, in batches of 8 steps whose loads and coefficients are
//     independent, and store outputs straight from registers.  Stages pass
//     between the roles through full / empty mbarriers, not block barriers.
//   * When batch x channel blocks fill the GPU (S == 1) a block streams the
//     whole sequence once, carrying the state across tiles in registers.
//   * Otherwise the sequence is cut into S time splits that run in parallel.
//     Each split first scans its range from a zero state to get its
//     aggregate (product of decays, state), publishes it, and
//     takes its carry-in from a decoupled look-back over the preceding
//     splits' descriptors (Merrill & Garland, "Single-pass Parallel Prefix
//     Scan with Decoupled Look-back", 2016).  Split order comes from an
//     atomic ticket, so every split a block waits for is already running.
//     It then re-streams its range (an L2 hit for the small problems this
//     mode serves) and writes the outputs.  Every wait is bounded in time.
//   * A split descriptor is (product of decays, h) per channel for RG-LRU and
//     (sum of delta, h[16]) for the selective scan, whose 16 decay products
//     over a range are exp(A[n] sum delta) and need not be stored.
#include <cudaTypedefs.h>

#include <mutex>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {

__device__ int g_diag_status = 0;

__device__ __forceinline__ void report_status(int code) { atomicCAS(&g_diag_status, 0, code); }

// Flag values of a split descriptor.
constexpr uint32_t kFlagNone = 0, kFlagAggregate = 1, kFlagInclusive = 2;

struct LookbackWs {
    uint32_t *flags;   // [n_cb * S]
    uint32_t *ticket;  // [1]
    float *agg;        // [n_cb * S][kAgg][DC]
    float *incl;       // [n_cb * S][kIncl][DC]
};

// Polls a split flag (thread 0 only) until it is non-zero or the limit runs
// out; returns the flag value (kFlagNone on timeout).
__device__ __forceinline__ uint32_t poll_flag(const uint32_t *flag, uint64_t limit_ns) {
    uint32_t v = ld_acquire_gpu(flag);
    if (v != kFlagNone) return v;
    const uint64_t t0 = globaltimer_ns();
    while ((v = ld_acquire_gpu(flag)) == kFlagNone) {
        if (globaltimer_ns() - t0 > limit_ns) return kFlagNone;
        __nanosleep(100);
    }
    return v;
}

// ----------------------------------------------------------------------------
// Accurate helpers (fp32 I/O path)
// ----------------------------------------------------------------------------

// exp(x) - 1 without cancellation: Taylor series (coefficients 1/k!) for
// |x| < 0.3, where nine terms leave a truncation error below 2e-12 relative;
// expf(x) - 1 elsewhere, where |exp(x) - 1| > 0.25 keeps the subtraction
// exact to a few ulp.
__device__ __forceinline__ float expm1_accurate(float x) {
    if (fabsf(x) < 0.3f) {
        float p = 1.0f / 362880.0f;
        p = fmaf(p, x, 1.0f / 40320.0f);
        p = fmaf(p, x, 1.0f / 5040.0f);
        p = fmaf(p, x, 1.0f / 720.0f);
        p = fmaf(p, x, 1.0f / 120.0f);
        p = fmaf(p, x, 1.0f / 24.0f);
        p = fmaf(p, x, 1.0f / 6.0f);
        p = fmaf(p, x, 0.5f);
        p = fmaf(p, x, 1.0f);
        return p * x;
    }
    return expf(x) - 1.0f;
}

// torch softplus (beta 1, threshold 20).
template <bool ACC>
__device__ __forceinline__ float softplus_t(float x) {
    if (ACC) return x > 20.0f ? x : log1pf(expf(x));
    const float e = ex2_approx(x * kLog2e);
    // log(1 + e): below 2^-10 it is e within e/2 relative (< 5e-4, under the
    // bf16 output rounding), where 1 + e would round e's digits away.
    const float l = e < 9.765625e-4f ? e : lg2_approx(1.0f + e) * kLn2;
    return x > 20.0f ? x : l;
}

// Two fast-form softplus values at once (packed fp32x2 arithmetic).
__device__ __forceinline__ float2 softplus2_fast(float2 x) {
    const float2 t = __fmul2_rn(x, make_float2(kLog2e, kLog2e));
    const float2 e = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    const float2 e1 = __fadd2_rn(e, make_float2(1.0f, 1.0f));
    const float2 l = __fmul2_rn(make_float2(lg2_approx(e1.x), lg2_approx(e1.y)), make_float2(kLn2, kLn2));
    return make_float2(x.x > 20.0f ? x.x : (e.x < 9.765625e-4f ? e.x : l.x),
                       x.y > 20.0f ? x.y : (e.y < 9.765625e-4f ? e.y : l.y));
}

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// silu(z) = z sigmoid(z).  ACC (fp32 I/O): from exp2 and a reciprocal,
// ~1e-6 relative.  Otherwise (bf16 I/O) as z/2 (1 + tanh(z/2)) with the
// single-instruction tanh (about 5e-4 relative, far below the bf16 output
// rounding), which saves one SFU op per (step, channel).
template <bool ACC>
__device__ __forceinline__ float silu_t(float z) {
    if (ACC) return z * rcp_approx(1.0f + ex2_approx(-z * kLog2e));
    const float hz = 0.5f * z;
    return fmaf(hz, tanh_approx(hz), hz);
}

template <bool ACC>
__device__ __forceinline__ float pow2_t(float e) {
    return ACC ? exp2f(e) : ex2_approx(e);
}

// ============================================================================
// Shared tile helpers
// ============================================================================

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Two consecutive bf16 / fp32 values as a float2.
__device__ __forceinline__ float2 ld2(const float *p) { return *reinterpret_cast<const float2 *>(p); }
__device__ __forceinline__ float2 ld2(const __nv_bfloat16 *p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}

// Per-block abort word: once any wait of the block has run out, later waits
// are skipped so that every warp still walks the same barrier sequence and
// the block finishes.
__device__ __noinline__ bool block_wait_slow(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                             volatile int *flag) {
    if (*flag != 0) return false;
    if (mbar_wait_bounded(bar, parity, limit_ns)) return true;
    *flag = 1;
    report_status(LR_ERR_TIMEOUT);
    return false;
}

struct BlockAbort {
    volatile int *flag;
    // Fast path: one try_wait when the phase has already completed.
    __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) const {
        if (mbar_try_wait(bar, parity)) return true;
        return block_wait_slow(bar, parity, limit_ns, flag);
    }
};

// ============================================================================
// RG-LRU
// ============================================================================
// Warp roles in a block of DC channels:
//   compute warps (one channel per thread): wait for a TMA-staged tile, then
//     run the recurrence through it in batches of 8 steps (loads, a_t, b_t of
//     the batch are independent; only the h chain is sequential) and store
//     y straight from registers; then release the stage (one arrive per warp).
//   producer warp: lane 0 keeps STAGES tiles of x, r, i in flight by TMA,
//     re-arming a stage as soon as every compute warp released it.
template <typename IO>
struct RgCfg {
    static constexpr int DC = 64;                        // channels per block
    // time steps per tile; bf16 tiles are 64 steps deep in 3 stages (the same
    // 72 KB as 6 x 32 steps, so 3 blocks stay resident per SM, with half the
    // handshakes per step)
    static constexpr int T = sizeof(IO) == 2 ? 64 : 32;
    static constexpr int CWARPS = DC / 32;
    static constexpr int THREADS = 32 * (CWARPS + 1);    // + producer warp
    static constexpr int STAGES = sizeof(IO) == 2 ? 3 : 4;
    static constexpr int BATCH = 8;
    static constexpr int TILE = T * DC;
    static constexpr uint32_t STAGE_BYTES = 3u * TILE * sizeof(IO);
    static constexpr size_t OFF_BAR = size_t(STAGES) * STAGE_BYTES;   // full[], empty[]
    static constexpr size_t SMEM = OFF_BAR + 2 * STAGES * 8 + 16;
    static constexpr int kAgg = 2, kIncl = 1;  // descriptor floats per channel
};

// a_t and b_t = sqrt(1 - a_t^2) u of one (t, channel); cl = c a_log,
// cl2 = cl log2(e).
template <bool ACC>
__device__ __forceinline__ void rglru_ab(float r, float u, float cl, float cl2, float &a,
                                         float &bb) {
    if (ACC) {
        const float em1 = expm1_accurate(cl * r);   // a_t - 1
        a = 1.0f + em1;
        bb = sqrtf(-em1 * (2.0f + em1)) * u;        // 1 - a^2 = -em1 (2 + em1)
    } else {
        a = ex2_approx(cl2 * r);
        bb = sqrt_approx(fmaf(-a, a, 1.0f)) * u;
    }
}

// Tile modes: the aggregate pass, an output tile whose rows and channels are
// all in range (no per-step predicate, so a batch is one basic block the
// scheduler can interleave), and a ragged output tile.
enum TileMode { kAggregate = 0, kFull = 1, kRagged = 2 };

// Logistic sigmoids of both pre-activation gates.  The fast form shares one
// reciprocal: with e = exp(-v) clamped to 2^60 (so the product stays finite;
// sigma moves by less than 1e-18), sigma(r) = (1 + e_i) / ((1 + e_r)(1 + e_i))
// and likewise for i -- five special-function operations per step, not six.
template <bool ACC>
__device__ __forceinline__ void sigmoid_pair(float &r, float &i) {
    if (ACC) {
        r = 1.0f / (1.0f + expf(-r));
        i = 1.0f / (1.0f + expf(-i));
    } else {
        const float er1 = 1.0f + fminf(ex2_approx(-r * kLog2e), 0x1p60f);
        const float ei1 = 1.0f + fminf(ex2_approx(-i * kLog2e), 0x1p60f);
        const float inv = rcp_approx(er1 * ei1);
        r = ei1 * inv;
        i = er1 * inv;
    }
}

// One T-step tile of one channel's recurrence.  PRE: r and i arrive before
// their sigmoid, which is applied here.  `rows` = steps of the tile inside
// the sequence (0 for a channel past D).
template <typename IO, bool ACC, bool PRE, int MODE>
__device__ __forceinline__ void rglru_tile(const IO *xs, const IO *rs, const IO *is, float cl,
                                           float cl2, float &h, float &P, IO *yp, int D, int rows) {
    using C = RgCfg<IO>;
    // the whole tile unrolled keeps every batch's loads ahead of the chain;
    // with the two sigmoids per step that would take 191 registers, so the
    // pre-activation form unrolls four batches (96 registers)
    constexpr int kUnroll = PRE ? 4 : C::T / C::BATCH;
#pragma unroll kUnroll
    for (int j0 = 0; j0 < C::T; j0 += C::BATCH) {
        float a[C::BATCH], bb[C::BATCH];
        if (PRE && !ACC) {
            // two steps at a time in packed fp32x2: both gates' sigmoids (one
            // shared reciprocal per step, as sigmoid_pair), the decays and the
            // input terms (as rglru_ab); each lane of a packed operation rounds
            // as the scalar one, so the results are the scalar form's bit for bit
#pragma unroll
            for (int u = 0; u < C::BATCH; u += 2) {
                const int o0 = (j0 + u) * C::DC, o1 = o0 + C::DC;
                const float2 r2 = make_float2(Io<IO>::to_f(rs[o0]), Io<IO>::to_f(rs[o1]));
                const float2 i2 = make_float2(Io<IO>::to_f(is[o0]), Io<IO>::to_f(is[o1]));
                const float2 x2 = make_float2(Io<IO>::to_f(xs[o0]), Io<IO>::to_f(xs[o1]));
                const float2 tr = __fmul2_rn(r2, make_float2(-kLog2e, -kLog2e));
                const float2 ti = __fmul2_rn(i2, make_float2(-kLog2e, -kLog2e));
                const float2 er1 = __fadd2_rn(make_float2(fminf(ex2_approx(tr.x), 0x1p60f),
                                                          fminf(ex2_approx(tr.y), 0x1p60f)),
                                              make_float2(1.0f, 1.0f));
                const float2 ei1 = __fadd2_rn(make_float2(fminf(ex2_approx(ti.x), 0x1p60f),
                                                          fminf(ex2_approx(ti.y), 0x1p60f)),
                                              make_float2(1.0f, 1.0f));
                const float2 den = __fmul2_rn(er1, ei1);
                const float2 inv = make_float2(rcp_approx(den.x), rcp_approx(den.y));
                const float2 sr = __fmul2_rn(ei1, inv), si = __fmul2_rn(er1, inv);
                const float2 la = __fmul2_rn(sr, make_float2(cl2, cl2));
                const float2 a2 = make_float2(ex2_approx(la.x), ex2_approx(la.y));
                const float2 om = __ffma2_rn(make_float2(-a2.x, -a2.y), a2, make_float2(1.0f, 1.0f));
                const float2 u2 = __fmul2_rn(si, x2);
                const float2 b2 = __fmul2_rn(make_float2(sqrt_approx(om.x), sqrt_approx(om.y)), u2);
                a[u] = a2.x;
                a[u + 1] = a2.y;
                bb[u] = b2.x;
                bb[u + 1] = b2.y;
                if (MODE != kFull) {   // rows past L: identity steps
                    if (j0 + u >= rows) { a[u] = 1.0f; bb[u] = 0.0f; }
                    if (j0 + u + 1 >= rows) { a[u + 1] = 1.0f; bb[u + 1] = 0.0f; }
                }
            }
        } else
#pragma unroll
        for (int u = 0; u < C::BATCH; ++u) {
            const int o = (j0 + u) * C::DC;
            float rv = Io<IO>::to_f(rs[o]), iv = Io<IO>::to_f(is[o]);
            if (PRE) sigmoid_pair<ACC>(rv, iv);
            rglru_ab<ACC>(rv, iv * Io<IO>::to_f(xs[o]), cl, cl2, a[u], bb[u]);
            // rows past L arrive zero-filled; with raw gates r = 0 is the
            // identity step (a = 1, b = 0), after a sigmoid it is not
            if (PRE && MODE != kFull && j0 + u >= rows) {
                a[u] = 1.0f;
                bb[u] = 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < C::BATCH; ++u) {
            h = fmaf(a[u], h, bb[u]);
            if (MODE == kAggregate) P *= a[u];
            if (MODE == kFull) __stcs(yp + size_t(j0 + u) * D, Io<IO>::from_f(h));
            if (MODE == kRagged && j0 + u < rows) __stcs(yp + size_t(j0 + u) * D, Io<IO>::from_f(h));
        }
    }
}

template <typename IO, bool ACC, bool PRE>
__global__ void __launch_bounds__(RgCfg<IO>::THREADS, 1)  // registers for a whole batch in flight
    rglru_scan_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_r,
                      const __grid_constant__ CUtensorMap tm_i, const float *__restrict__ a_log,
                      float c, const float *__restrict__ h0, IO *__restrict__ y,
                      float *__restrict__ h_final, int L, int D, int n_db, int S, int tps,
                      int n_tiles, LookbackWs ws, int withheld, uint64_t timeout_ns) {
    using C = RgCfg<IO>;
    extern __shared__ __align__(128) unsigned char smem[];
    IO *tiles = reinterpret_cast<IO *>(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::STAGES;
    int *bcast = reinterpret_cast<int *>(empty + C::STAGES);
    int *abort_word = bcast + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const BlockAbort ab{abort_word};

    if (tid == 0) {
        for (int st = 0; st < C::STAGES; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], C::CWARPS);
        }
        *abort_word = 0;
        fence_mbar_init();
        if (S > 1) *bcast = static_cast<int>(atomicAdd(ws.ticket, 1u));
    }
    __syncthreads();
    const int tk = S > 1 ? *bcast : static_cast<int>(blockIdx.x);
    const int cb = tk / S, s = tk - (tk / S) * S;
    const int b = cb / n_db;
    const int d0 = (cb - b * n_db) * C::DC;
    const int k0 = s * tps;
    const int ntl = min(k0 + tps, n_tiles) - k0;
    const int V = S > 1 ? 2 * ntl : ntl;  // virtual tiles: aggregate pass, then output pass

    if (warp == C::CWARPS) {  // ---------------------------------- producer warp
        if (lane == 0) {
            prefetch_tensormap(&tm_x);
            prefetch_tensormap(&tm_r);
            prefetch_tensormap(&tm_i);
            for (int v = 0; v < V; ++v) {
                const int st = v % C::STAGES;
                if (v >= C::STAGES && !ab.wait(&empty[st], ((v / C::STAGES) - 1) & 1, timeout_ns))
                    break;
                const int t0 = (k0 + v % ntl) * C::T;
                IO *base = tiles + size_t(st) * 3 * C::TILE;
                mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
                tma_load_3d(base, &tm_x, &full[st], d0, t0, b);
                tma_load_3d(base + C::TILE, &tm_r, &full[st], d0, t0, b);
                tma_load_3d(base + 2 * C::TILE, &tm_i, &full[st], d0, t0, b);
            }
        }
        return;
    }

    // ------------------------------------------------------------ compute warps
    const int ch = tid;  // channel within the block
    const int d = d0 + ch;
    const bool vd = d < D;
    const float cl = vd ? c * a_log[d] : 0.0f;
    const float cl2 = cl * kLog2e;
    const float h0v = (vd && h0 != nullptr) ? h0[size_t(b) * D + d] : 0.0f;
    float h = S > 1 ? 0.0f : h0v;  // the aggregate pass starts from zero
    float P = 1.0f;                // product of decays over the aggregate pass

    for (int v = 0; v < V; ++v) {
        const int st = v % C::STAGES;
        const bool agg_pass = S > 1 && v < ntl;
        const int t0 = (k0 + v % ntl) * C::T;
        ab.wait(&full[st], (v / C::STAGES) & 1, timeout_ns);
        const IO *xs = tiles + size_t(st) * 3 * C::TILE + ch;
        const IO *rs = xs + C::TILE;
        const IO *is = rs + C::TILE;
        IO *yp = y + (size_t(b) * L + t0) * D + d;
        // warp-uniform choice: the whole warp's channels and rows in range?
        const bool full_tile = t0 + C::T <= L && d0 + 32 * (warp + 1) <= D;
        if (agg_pass)
            rglru_tile<IO, ACC, PRE, kAggregate>(xs, rs, is, cl, cl2, h, P, yp, D, min(C::T, L - t0));
        else if (full_tile)
            rglru_tile<IO, ACC, PRE, kFull>(xs, rs, is, cl, cl2, h, P, yp, D, C::T);
        else
            rglru_tile<IO, ACC, PRE, kRagged>(xs, rs, is, cl, cl2, h, P, yp, D,
                                              vd ? min(C::T, L - t0) : 0);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);

        if (agg_pass && v == ntl - 1) {
            // ---- publish this split's aggregate, look back, publish inclusive
            constexpr int NC = 32 * C::CWARPS;
            const size_t slot = size_t(cb) * S + s;
            float carry = h0v;
            if (s > 0) {
                ws.agg[(slot * C::kAgg + 0) * C::DC + ch] = P;
                ws.agg[(slot * C::kAgg + 1) * C::DC + ch] = h;
                __threadfence();
                named_bar_sync(1, NC);
                if (tid == 0 && s != withheld) st_release_gpu(&ws.flags[slot], kFlagAggregate);
                float acc_p = 1.0f, acc_h = 0.0f;  // composition of splits sp+1 .. s-1
                carry = 0.0f;
                for (int sp = s - 1; sp >= 0; --sp) {
                    const size_t sl = size_t(cb) * S + sp;
                    if (tid == 0) *bcast = static_cast<int>(poll_flag(&ws.flags[sl], timeout_ns));
                    named_bar_sync(1, NC);
                    const int fv = *bcast;
                    named_bar_sync(1, NC);
                    if (fv == static_cast<int>(kFlagInclusive)) {
                        carry = fmaf(acc_p, __ldcg(&ws.incl[sl * C::DC + ch]), acc_h);
                        break;
                    }
                    if (fv == static_cast<int>(kFlagAggregate)) {
                        const float px = __ldcg(&ws.agg[(sl * C::kAgg + 0) * C::DC + ch]);
                        const float hx = __ldcg(&ws.agg[(sl * C::kAgg + 1) * C::DC + ch]);
                        acc_h = fmaf(acc_p, hx, acc_h);
                        acc_p *= px;
                        continue;
                    }
                    if (tid == 0) report_status(LR_ERR_TIMEOUT);
                    carry = acc_h;
                    break;
                }
            }
            ws.incl[slot * C::DC + ch] = fmaf(P, carry, h);
            __threadfence();
            named_bar_sync(1, NC);
            if (tid == 0 && s != withheld) st_release_gpu(&ws.flags[slot], kFlagInclusive);
            h = carry;  // the output pass restarts the range from its carry-in
        }
    }
    if (h_final != nullptr && vd && s == S - 1) h_final[size_t(b) * D + d] = h;
}

// ============================================================================
// MinMax recurrence
// ============================================================================
// x_t = max(min(r_t, x_{t-1}), s_t)  (minmaxrnc MinMaxNeuron; the operator
// f(x) = max(min(a, x), b) of minmax_operator.apply with a = r_t, b = s_t).
// Same skeleton as the RG-LRU scan: one channel per thread, TMA-staged tiles
// of r and s, and for time splits a decoupled look-back whose aggregate is
// the split's composed operator (A, Bc) with f(x) = max(min(A, x), Bc):
// composing f_t after F gives (min(r_t, A), max(min(r_t, Bc), s_t))
// (minmax_operator.compose).  min / max select one argument exactly, so the
// scan is exact in any order; NaN arguments give NaN, as torch.minimum and
// torch.maximum do.
__device__ __forceinline__ float min_nan(float a, float b) {
    float d;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ float max_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

template <typename IO>
struct MmCfg {
    static constexpr int DC = 64;                        // channels per block
    static constexpr int T = 32;                         // time steps per tile
    static constexpr int CWARPS = DC / 32;
    static constexpr int THREADS = 32 * (CWARPS + 1);    // + producer warp
    static constexpr int STAGES = sizeof(IO) == 2 ? 8 : 5;
    static constexpr int TILE = T * DC;
    static constexpr uint32_t STAGE_BYTES = 2u * TILE * sizeof(IO);
    static constexpr size_t OFF_BAR = size_t(STAGES) * STAGE_BYTES;   // full[], empty[]
    static constexpr size_t SMEM = OFF_BAR + 2 * STAGES * 8 + 16;
    static constexpr int kAgg = 2, kIncl = 1;  // (A, Bc) and the inclusive state
};

template <typename IO, int MODE>
__device__ __forceinline__ void minmax_tile(const IO *rs, const IO *ss, float &x, float &A, float &Bc,
                                            IO *yp, int D, int rows) {
    using C = MmCfg<IO>;
#pragma unroll
    for (int j = 0; j < C::T; ++j) {
        const float r = Io<IO>::to_f(rs[j * C::DC]);
        const float sv = Io<IO>::to_f(ss[j * C::DC]);
        if (MODE == kAggregate) {
            Bc = max_nan(min_nan(r, Bc), sv);
            A = min_nan(r, A);
        } else {
            x = max_nan(min_nan(r, x), sv);
            if (MODE == kFull) __stcs(yp + size_t(j) * D, Io<IO>::from_f(x));
            if (MODE == kRagged && j < rows) __stcs(yp + size_t(j) * D, Io<IO>::from_f(x));
        }
    }
}

template <typename IO>
__global__ void __launch_bounds__(MmCfg<IO>::THREADS, 1)
    minmax_scan_kernel(const __grid_constant__ CUtensorMap tm_r, const __grid_constant__ CUtensorMap tm_s,
                       const float *__restrict__ x0, IO *__restrict__ y, float *__restrict__ x_final,
                       int L, int D, int n_db, int S, int tps, int n_tiles, LookbackWs ws,
                       int withheld, uint64_t timeout_ns) {
    using C = MmCfg<IO>;
    extern __shared__ __align__(128) unsigned char smem[];
    IO *tiles = reinterpret_cast<IO *>(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::STAGES;
    int *bcast = reinterpret_cast<int *>(empty + C::STAGES);
    int *abort_word = bcast + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const BlockAbort ab{abort_word};

    if (tid == 0) {
        for (int st = 0; st < C::STAGES; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], C::CWARPS);
        }
        *abort_word = 0;
        fence_mbar_init();
        if (S > 1) *bcast = static_cast<int>(atomicAdd(ws.ticket, 1u));
    }
    __syncthreads();
    const int tk = S > 1 ? *bcast : static_cast<int>(blockIdx.x);
    const int cb = tk / S, s = tk - (tk / S) * S;
    const int b = cb / n_db;
    const int d0 = (cb - b * n_db) * C::DC;
    const int k0 = s * tps;
    const int ntl = min(k0 + tps, n_tiles) - k0;
    const int V = S > 1 ? 2 * ntl : ntl;  // virtual tiles: aggregate pass, then output pass

    if (warp == C::CWARPS) {  // ---------------------------------- producer warp
        if (lane == 0) {
            prefetch_tensormap(&tm_r);
            prefetch_tensormap(&tm_s);
            for (int v = 0; v < V; ++v) {
                const int st = v % C::STAGES;
                if (v >= C::STAGES && !ab.wait(&empty[st], ((v / C::STAGES) - 1) & 1, timeout_ns))
                    break;
                const int t0 = (k0 + v % ntl) * C::T;
                IO *base = tiles + size_t(st) * 2 * C::TILE;
                mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
                tma_load_3d(base, &tm_r, &full[st], d0, t0, b);
                tma_load_3d(base + C::TILE, &tm_s, &full[st], d0, t0, b);
            }
        }
        return;
    }

    // ------------------------------------------------------------ compute warps
    const int ch = tid;
    const int d = d0 + ch;
    const bool vd = d < D;
    const float x0v = (vd && x0 != nullptr) ? x0[size_t(b) * D + d] : 0.0f;
    float x = x0v;
    float A = __int_as_float(0x7f800000), Bc = __int_as_float(0xff800000);  // identity: +inf, -inf

    for (int v = 0; v < V; ++v) {
        const int st = v % C::STAGES;
        const bool agg_pass = S > 1 && v < ntl;
        const int t0 = (k0 + v % ntl) * C::T;
        ab.wait(&full[st], (v / C::STAGES) & 1, timeout_ns);
        const IO *rs = tiles + size_t(st) * 2 * C::TILE + ch;
        const IO *ss = rs + C::TILE;
        IO *yp = y + (size_t(b) * L + t0) * D + d;
        const bool full_tile = t0 + C::T <= L && d0 + 32 * (warp + 1) <= D;
        // rows past L (zero-filled by TMA) must not act: clamp them out of the
        // aggregate by treating them as identity steps
        const int rows = vd ? min(C::T, L - t0) : 0;
        if (agg_pass) {
            if (t0 + C::T <= L) {
                minmax_tile<IO, kAggregate>(rs, ss, x, A, Bc, yp, D, 0);
            } else {
                for (int j = 0; j < L - t0; ++j) {
                    const float r = Io<IO>::to_f(rs[j * C::DC]), sv = Io<IO>::to_f(ss[j * C::DC]);
                    Bc = max_nan(min_nan(r, Bc), sv);
                    A = min_nan(r, A);
                }
            }
        } else if (full_tile) {
            minmax_tile<IO, kFull>(rs, ss, x, A, Bc, yp, D, C::T);
        } else {
            // the state must not run through the zero-filled rows past L either
            const float keep = x;
            float xr = x;
            for (int j = 0; j < min(C::T, L - t0); ++j) {
                xr = max_nan(min_nan(Io<IO>::to_f(rs[j * C::DC]), xr), Io<IO>::to_f(ss[j * C::DC]));
                if (j < rows) __stcs(yp + size_t(j) * D, Io<IO>::from_f(xr));
            }
            x = L - t0 > 0 ? xr : keep;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);

        if (agg_pass && v == ntl - 1) {
            // ---- publish this split's operator, look back, publish inclusive
            constexpr int NC = 32 * C::CWARPS;
            const size_t slot = size_t(cb) * S + s;
            float carry = x0v;
            if (s > 0) {
                ws.agg[(slot * C::kAgg + 0) * C::DC + ch] = A;
                ws.agg[(slot * C::kAgg + 1) * C::DC + ch] = Bc;
                __threadfence();
                named_bar_sync(1, NC);
                if (tid == 0 && s != withheld) st_release_gpu(&ws.flags[slot], kFlagAggregate);
                // composition G of splits sp+1 .. s-1 (starts as the identity)
                float gA = __int_as_float(0x7f800000), gB = __int_as_float(0xff800000);
                carry = 0.0f;
                for (int sp = s - 1; sp >= 0; --sp) {
                    const size_t sl = size_t(cb) * S + sp;
                    if (tid == 0) *bcast = static_cast<int>(poll_flag(&ws.flags[sl], timeout_ns));
                    named_bar_sync(1, NC);
                    const int fv = *bcast;
                    named_bar_sync(1, NC);
                    if (fv == static_cast<int>(kFlagInclusive)) {
                        carry = max_nan(min_nan(gA, __ldcg(&ws.incl[sl * C::DC + ch])), gB);
                        break;
                    }
                    if (fv == static_cast<int>(kFlagAggregate)) {
                        const float fA = __ldcg(&ws.agg[(sl * C::kAgg + 0) * C::DC + ch]);
                        const float fB = __ldcg(&ws.agg[(sl * C::kAgg + 1) * C::DC + ch]);
                        gB = max_nan(min_nan(gA, fB), gB);   // G o F
                        gA = min_nan(gA, fA);
                        continue;
                    }
                    if (tid == 0) report_status(LR_ERR_TIMEOUT);
                    carry = max_nan(min_nan(gA, 0.0f), gB);
                    break;
                }
            }
            ws.incl[slot * C::DC + ch] = max_nan(min_nan(A, carry), Bc);
            __threadfence();
            named_bar_sync(1, NC);
            if (tid == 0 && s != withheld) st_release_gpu(&ws.flags[slot], kFlagInclusive);
            x = carry;  // the output pass restarts the range from its carry-in
        }
    }
    if (x_final != nullptr && vd && s == S - 1) x_final[size_t(b) * D + d] = x;
}

// ============================================================================
// Selective SSM
// ============================================================================
// Warp roles in a block of DC channels:
//   compute warps: LPC lanes per channel, N / LPC states per lane.  In
//     batches of 8 steps each lane computes delta = softplus(dt) and
//     u = delta x for 8 / LPC of the steps and the channel's lanes share them
//     by shuffles; every lane advances its states through the 8 steps
//     (h[n] = exp(delta A[n]) h[n] + u B_t[n], partial C_t . h); a butterfly
//     over the channel's lanes sums the partials so that each lane ends up
//     with the full C_t . h of its own steps, finishes
//     y = (C.h + D x) silu(z) for them and stores it.  LPC = 2 (8 states per
//     lane) is the measured optimum on GB300: 4 lanes double the resident
//     warps but cost more shuffles and fewer independent chains per lane and
//     ran 1.5x slower; 1 lane per channel leaves too few warps per SM.
//   producer warp: keeps STAGES tiles of x, dt, z, B_t, C_t in flight by TMA
//     and widens each tile's B_t, C_t rows (shared by all channels) to fp32
//     once, so the compute lanes read them with broadcast 16-byte loads.
// Decays.  In general each state's decay is one exp2 of delta A[n] log2(e).
// The SSM's initialisation puts A on a lattice, A[n] = (n + 1) A[0] per
// channel (cortexnet MultiScaleSSM.__init__: A_log[d, n] = log((n+1) 2^s)).
// There the 16 decays of a step are the powers E, E^2, .., E^16 of
// E = exp(delta A[0]); a lane holding states k0 .. k0+7 takes
// (E^(k0+1), E^(k0+2)) and E^2 from three exps and the rest of its pairs as
// P * (E^2, E^2), five exps fewer per lane and step.  The kernel checks the
// lattice itself, per warp, from the A_log it is given: every state of every
// channel of the warp must satisfy |A[n] - (n+1) A[0]| <= 2^-20 |A[n]| in
// fp32, else the warp keeps the general form.  Trained A_log leaves the
// lattice and takes the general form; nothing is assumed.
template <typename IO, int DC_, int LPC_>
struct SelCfg {
    static constexpr int DC = DC_;                       // channels per block
    static constexpr int LPC = LPC_;                     // lanes per channel
    static constexpr int CWARPS = DC * LPC / 32;
    static constexpr int THREADS = 32 * (CWARPS + 1);    // + producer warp
    static constexpr int N = 16, NS = N / LPC, NP = NS / 2;
    static constexpr int T = 64;                         // steps per tile
    static constexpr int STAGES = 2;                     // 2 x 64 steps in flight (48 KB with the fp32 B/C copies)
    static constexpr int BATCH = 8;
    static constexpr int OWN = BATCH / LPC;              // steps a lane prepares per batch
    static constexpr int TILE = T * DC;                  // x / dt / z tile elements
    static constexpr int TILE_N = T * N;                 // B / C tile elements
    static constexpr int STAGE_ELEMS = 3 * TILE + 2 * TILE_N;
    static constexpr size_t STAGE_IO_BYTES = size_t(STAGE_ELEMS) * sizeof(IO);
    static constexpr size_t OFF_BC = size_t(STAGES) * STAGE_IO_BYTES;     // float [STAGES][T][2N]
    static constexpr size_t OFF_BAR = OFF_BC + size_t(STAGES) * T * 2 * N * 4;
    static constexpr size_t SMEM = OFF_BAR + 3 * STAGES * 8 + 16;
    static constexpr int kAgg = 1 + N, kIncl = N;
    // two lanes per channel (the exchange and the packed finish assume it;
    // four measured slower, one leaves too few warps)
    static_assert(T % BATCH == 0 && (DC * LPC) % 32 == 0 && LPC == 2, "tile shape");
};

// One T-step tile of one lane's states.  `rows` = steps of the tile inside
// the sequence (and 0 for a channel past D in the ragged mode).  MODE is
// warp-uniform, so the shuffles always run converged.  Lane r of a channel's
// group (r = lane % LPC) prepares steps j0 + r + LPC m of each batch and
// finishes the outputs of the same steps.  Inside a batch the lane walks its
// states in groups of four (one 16-byte B_t and C_t load per step and group)
// and, per group, all 8 steps: the group's decays for the 8 steps are
// independent of each other and of the state, so they issue ahead of the
// serial h chain.
template <typename IO, int DC, int LPC, bool ACC, bool HAS_Z, bool SOFTPLUS, int MODE, bool LAT = false>
__device__ __forceinline__ void sel_tile(const IO *xs, const IO *dts, const IO *zs, const float *bc,
                                         const float2 (&A2)[SelCfg<IO, DC, LPC>::NP],
                                         float2 (&h)[SelCfg<IO, DC, LPC>::NP], float &dsum,
                                         float dsk, IO *yp, int D, int rows, int r, int lane,
                                         float3 latc = make_float3(0.0f, 0.0f, 0.0f)) {
    using C = SelCfg<IO, DC, LPC>;
    constexpr int OWN = C::OWN;
    const unsigned FULL = 0xffffffffu;
#pragma unroll 2   // two batches in flight: the next batch's softplus overlaps this one's updates
    for (int j0 = 0; j0 < C::T; j0 += C::BATCH) {
        float xv[OWN], dl[OWN], u[OWN];
        if (!ACC) {
            // the lane's own steps two at a time, in packed fp32x2 arithmetic
#pragma unroll
            for (int m = 0; m < OWN; m += 2) {
                const int ja = j0 + r + LPC * m, jb = ja + LPC;
                const float2 x2 = make_float2(Io<IO>::to_f(xs[ja * DC]), Io<IO>::to_f(xs[jb * DC]));
                float2 d2 = make_float2(Io<IO>::to_f(dts[ja * DC]), Io<IO>::to_f(dts[jb * DC]));
                if (SOFTPLUS) d2 = softplus2_fast(d2);
                if (MODE != kFull) {   // rows past L: identity steps
                    d2.x = ja < rows ? d2.x : 0.0f;
                    d2.y = jb < rows ? d2.y : 0.0f;
                }
                const float2 u2 = __fmul2_rn(d2, x2);
                xv[m] = x2.x;
                xv[m + 1] = x2.y;
                dl[m] = d2.x;
                dl[m + 1] = d2.y;
                u[m] = u2.x;
                u[m + 1] = u2.y;
            }
        } else {
#pragma unroll
            for (int m = 0; m < OWN; ++m) {
                const int j = j0 + r + LPC * m;
                xv[m] = Io<IO>::to_f(xs[j * DC]);
                const float dtv = Io<IO>::to_f(dts[j * DC]);
                dl[m] = SOFTPLUS ? softplus_t<ACC>(dtv) : dtv;
                if (MODE != kFull) dl[m] = j < rows ? dl[m] : 0.0f;  // rows past L: identity steps
                u[m] = dl[m] * xv[m];
            }
        }
        // the partner lane prepared the other parity of steps: one xor
        // exchange per value, then pick own / other per step
        float dqs[C::BATCH], uqs[C::BATCH];
#pragma unroll
        for (int m = 0; m < OWN; ++m) {
            const float od = __shfl_xor_sync(FULL, dl[m], 1);
            const float ou = __shfl_xor_sync(FULL, u[m], 1);
            dqs[2 * m] = r == 0 ? dl[m] : od;
            dqs[2 * m + 1] = r == 0 ? od : dl[m];
            uqs[2 * m] = r == 0 ? u[m] : ou;
            uqs[2 * m + 1] = r == 0 ? ou : u[m];
        }
        if (MODE == kAggregate) {
#pragma unroll
            for (int q = 0; q < C::BATCH; ++q) dsum += dqs[q];
        }
        float2 ya[C::BATCH];
#pragma unroll
        for (int q = 0; q < C::BATCH; ++q) ya[q] = make_float2(0.0f, 0.0f);
        if (LAT) {
            // lattice decays: the lane's states k0 .. k0+7 decay by E^(k0+1) ..
            // E^(k0+8), E = 2^(delta A2[0]); (E^(k0+1), E^(k0+2)) and
            // M = E^2 from three exps, the other pairs as P * (M, M)
#pragma unroll
            for (int q = 0; q < C::BATCH; q += 2) {
                const float2 dq2 = make_float2(dqs[q], dqs[q + 1]);
                const float2 a1 = __fmul2_rn(dq2, make_float2(latc.x, latc.x));
                const float2 a2 = __fmul2_rn(dq2, make_float2(latc.y, latc.y));
                const float2 am = __fmul2_rn(dq2, make_float2(latc.z, latc.z));
                const float e1[2] = {ex2_approx(a1.x), ex2_approx(a1.y)};
                const float e2[2] = {ex2_approx(a2.x), ex2_approx(a2.y)};
                const float em[2] = {ex2_approx(am.x), ex2_approx(am.y)};
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const int qi = q + qq;
                    const float2 mm = make_float2(em[qq], em[qq]);
                    float2 P[C::NP];
                    P[0] = make_float2(e1[qq], e2[qq]);
#pragma unroll
                    for (int k = 1; k < C::NP; ++k) P[k] = __fmul2_rn(P[k - 1], mm);
                    const float *row = bc + (j0 + qi) * 2 * C::N;
                    const float2 uu = make_float2(uqs[qi], uqs[qi]);
#pragma unroll
                    for (int g = 0; g < C::NP / 2; ++g) {
                        const float4 b4 = *reinterpret_cast<const float4 *>(row + 4 * g);
                        h[2 * g] = __ffma2_rn(P[2 * g], h[2 * g], __fmul2_rn(uu, make_float2(b4.x, b4.y)));
                        h[2 * g + 1] = __ffma2_rn(P[2 * g + 1], h[2 * g + 1],
                                                  __fmul2_rn(uu, make_float2(b4.z, b4.w)));
                        const float4 c4 = *reinterpret_cast<const float4 *>(row + C::N + 4 * g);
                        ya[qi] = __ffma2_rn(make_float2(c4.x, c4.y), h[2 * g], ya[qi]);
                        ya[qi] = __ffma2_rn(make_float2(c4.z, c4.w), h[2 * g + 1], ya[qi]);
                    }
                }
            }
        } else
#pragma unroll
        for (int g = 0; g < C::NP / 2; ++g) {
#pragma unroll
            for (int q = 0; q < C::BATCH; q += 2) {
                // the group's four decays at steps q and q + 1: (delta_q, delta_q+1) x (A_n, A_n)
                const float2 dq2 = make_float2(dqs[q], dqs[q + 1]);
                float ea[4], eb[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float an = (k & 1) ? A2[2 * g + (k >> 1)].y : A2[2 * g + (k >> 1)].x;
                    const float2 a = __fmul2_rn(dq2, make_float2(an, an));
                    ea[k] = ex2_approx(a.x);
                    eb[k] = ex2_approx(a.y);
                }
#pragma unroll
                for (int qq = 0; qq < 2; ++qq) {
                    const int qi = q + qq;
                    const float *e = qq ? eb : ea;
                    const float *row = bc + (j0 + qi) * 2 * C::N + 4 * g;
                    const float2 uu = make_float2(uqs[qi], uqs[qi]);
                    const float4 b4 = *reinterpret_cast<const float4 *>(row);
                    h[2 * g] = __ffma2_rn(make_float2(e[0], e[1]), h[2 * g],
                                          __fmul2_rn(uu, make_float2(b4.x, b4.y)));
                    h[2 * g + 1] = __ffma2_rn(make_float2(e[2], e[3]), h[2 * g + 1],
                                              __fmul2_rn(uu, make_float2(b4.z, b4.w)));
                    if (MODE != kAggregate) {
                        const float4 c4 = *reinterpret_cast<const float4 *>(row + C::N);
                        ya[qi] = __ffma2_rn(make_float2(c4.x, c4.y), h[2 * g], ya[qi]);
                        ya[qi] = __ffma2_rn(make_float2(c4.z, c4.w), h[2 * g + 1], ya[qi]);
                    }
                }
            }
        }
        float yq[C::BATCH];
#pragma unroll
        for (int q = 0; q < C::BATCH; ++q) yq[q] = ya[q].x + ya[q].y;
        if (MODE != kAggregate) {
            // butterfly over the group: at the level of bit b a lane keeps the
            // steps whose bit b matches its own and adds its partner's share
#pragma unroll
            for (int bb = LPC / 2; bb >= 1; bb >>= 1) {
                const bool hi = (r & bb) != 0;
#pragma unroll
                for (int q = 0; q < C::BATCH; ++q) {
                    if ((q & (LPC - 1) & ~(2 * bb - 1)) != 0 || (q & bb) != 0) continue;
                    const float send = hi ? yq[q] : yq[q | bb];
                    const float keep = hi ? yq[q | bb] : yq[q];
                    yq[q] = keep + __shfl_xor_sync(FULL, send, bb);
                }
            }
            if (!ACC) {
#pragma unroll
                for (int m = 0; m < OWN; m += 2) {
                    const int ja = j0 + r + LPC * m, jb = ja + LPC;
                    float2 o2 = __ffma2_rn(make_float2(dsk, dsk), make_float2(xv[m], xv[m + 1]),
                                           make_float2(yq[LPC * m], yq[LPC * (m + 1)]));
                    if (HAS_Z) {   // silu(z) = z/2 (1 + tanh(z/2))
                        const float2 hz = __fmul2_rn(
                            make_float2(Io<IO>::to_f(zs[ja * DC]), Io<IO>::to_f(zs[jb * DC])),
                            make_float2(0.5f, 0.5f));
                        o2 = __fmul2_rn(o2, __ffma2_rn(hz, make_float2(tanh_approx(hz.x), tanh_approx(hz.y)), hz));
                    }
                    if (MODE == kFull || ja < rows) __stcs(yp + size_t(ja) * D, Io<IO>::from_f(o2.x));
                    if (MODE == kFull || jb < rows) __stcs(yp + size_t(jb) * D, Io<IO>::from_f(o2.y));
                }
            } else {
#pragma unroll
                for (int m = 0; m < OWN; ++m) {
                    const int j = j0 + r + LPC * m;
                    float o = fmaf(dsk, xv[m], yq[LPC * m]);
                    if (HAS_Z) o *= silu_t<ACC>(Io<IO>::to_f(zs[j * DC]));
                    if (MODE == kFull || j < rows) __stcs(yp + size_t(j) * D, Io<IO>::from_f(o));
                }
            }
        }
    }
}

// The minimum of one resident block lets ptxas keep the batch's decays and
// partial sums in registers (~130) instead of serialising the update to fit a
// smaller budget; shared memory, not registers, bounds the blocks per SM.
template <typename IO, int DC, int LPC, bool ACC, bool HAS_Z, bool SOFTPLUS>
__global__ void __launch_bounds__(SelCfg<IO, DC, LPC>::THREADS, 1)
    selective_scan_kernel(const __grid_constant__ CUtensorMap tm_x,
                          const __grid_constant__ CUtensorMap tm_dt,
                          const __grid_constant__ CUtensorMap tm_z,
                          const __grid_constant__ CUtensorMap tm_B,
                          const __grid_constant__ CUtensorMap tm_C, const float *__restrict__ A_log,
                          const float *__restrict__ Dskip, const float *__restrict__ h0,
                          IO *__restrict__ y, float *__restrict__ h_final, int L, int D, int n_db,
                          int S, int tps, int n_tiles, LookbackWs ws, int withheld,
                          uint64_t timeout_ns) {
    using C = SelCfg<IO, DC, LPC>;
    constexpr bool has_z = HAS_Z;
    extern __shared__ __align__(128) unsigned char smem[];
    IO *tiles = reinterpret_cast<IO *>(smem);
    float *BCf = reinterpret_cast<float *>(smem + C::OFF_BC);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *ready = full + C::STAGES;   // B/C widened: producer -> compute
    uint64_t *empty = ready + C::STAGES;  // stage released: compute -> producer
    int *bcast = reinterpret_cast<int *>(empty + C::STAGES);
    int *abort_word = bcast + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const BlockAbort abt{abort_word};
    const unsigned FULL = 0xffffffffu;

    if (tid == 0) {
        for (int st = 0; st < C::STAGES; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&ready[st], 1);
            mbar_init(&empty[st], C::CWARPS);
        }
        *abort_word = 0;
        fence_mbar_init();
        if (S > 1) *bcast = static_cast<int>(atomicAdd(ws.ticket, 1u));
    }
    __syncthreads();
    const int tk = S > 1 ? *bcast : static_cast<int>(blockIdx.x);
    const int cb = tk / S, s = tk - (tk / S) * S;
    const int b = cb / n_db;
    const int d0 = (cb - b * n_db) * DC;
    const int k0 = s * tps;
    const int ntl = min(k0 + tps, n_tiles) - k0;
    const int V = S > 1 ? 2 * ntl : ntl;
    const uint32_t stage_bytes =
        uint32_t((has_z ? 3 : 2) * C::TILE + 2 * C::TILE_N) * uint32_t(sizeof(IO));

    if (warp == C::CWARPS) {  // ---------------------------------- producer warp
        auto issue = [&](int v) {  // lane 0 only
            const int st = v % C::STAGES;
            const int t0 = (k0 + v % ntl) * C::T;
            IO *base = tiles + size_t(st) * C::STAGE_ELEMS;
            mbar_arrive_expect_tx(&full[st], stage_bytes);
            tma_load_3d(base, &tm_x, &full[st], d0, t0, b);
            tma_load_3d(base + C::TILE, &tm_dt, &full[st], d0, t0, b);
            if (has_z) tma_load_3d(base + 2 * C::TILE, &tm_z, &full[st], d0, t0, b);
            tma_load_3d(base + 3 * C::TILE, &tm_B, &full[st], 0, t0, b);
            tma_load_3d(base + 3 * C::TILE + C::TILE_N, &tm_C, &full[st], 0, t0, b);
        };
        if (lane == 0) {
            prefetch_tensormap(&tm_x);
            prefetch_tensormap(&tm_dt);
            if (has_z) prefetch_tensormap(&tm_z);
            prefetch_tensormap(&tm_B);
            prefetch_tensormap(&tm_C);
            for (int v = 0; v < min(C::STAGES, V); ++v) issue(v);
        }
        for (int v = 0; v < V; ++v) {
            const int st = v % C::STAGES;
            // widen tile v's B_t, C_t rows into BCf[st] = [T][B(16) | C(16)]
            bool ok = true;
            if (lane == 0) ok = abt.wait(&full[st], (v / C::STAGES) & 1, timeout_ns);
            ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
            if (ok) {
                const IO *Bs = tiles + size_t(st) * C::STAGE_ELEMS + 3 * C::TILE;
                float *dst = BCf + size_t(st) * C::T * 2 * C::N;
#pragma unroll
                for (int k = 0; k < C::TILE_N / 32; ++k) {   // pairs over B then C
                    const int p = lane + 32 * k;
                    const int which = p / (C::TILE_N / 2);
                    const int e = 2 * (p - which * (C::TILE_N / 2));
                    const float2 v2 = ld2(Bs + which * C::TILE_N + e);
                    *reinterpret_cast<float2 *>(dst + (e / C::N) * 2 * C::N + which * C::N +
                                                e % C::N) = v2;
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ready[st]);
                // re-arm the stage of tile v - 1 once the compute warps released it
                const int nv = v - 1 + C::STAGES;
                if (v >= 1 && nv < V) {
                    const int ps = (v - 1) % C::STAGES;
                    if (abt.wait(&empty[ps], ((v - 1) / C::STAGES) & 1, timeout_ns)) issue(nv);
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------ compute warps
    const int ch = tid / LPC;   // channel within the block
    const int r = tid % LPC;    // states [NS r, NS r + NS)
    const int d = d0 + ch;
    const bool vd = d < D;
    float2 A2[C::NP], h[C::NP]; // A2 = A log2(e) = -exp(A_log) log2(e)
#pragma unroll
    for (int q = 0; q < C::NP; ++q) {
        const int n = r * C::NS + 2 * q;
        A2[q] = vd ? make_float2(-expf(A_log[size_t(d) * C::N + n]) * kLog2e,
                                 -expf(A_log[size_t(d) * C::N + n + 1]) * kLog2e)
                   : make_float2(0.0f, 0.0f);
        h[q] = (vd && h0 != nullptr && S == 1)
                   ? make_float2(h0[(size_t(b) * D + d) * C::N + n],
                                 h0[(size_t(b) * D + d) * C::N + n + 1])
                   : make_float2(0.0f, 0.0f);
    }
    const float dsk = (vd && Dskip != nullptr) ? Dskip[d] : 0.0f;
    float dsum = 0.0f;  // sum of delta over the aggregate pass
    // lattice check (see above): A2[n] = (n + 1) A2[0] to 2^-20 relative for
    // every state of every channel of the warp; channels past D pass
    const float a20 = vd ? -expf(A_log[size_t(d) * C::N]) * kLog2e : 0.0f;
    bool on = true;
#pragma unroll
    for (int q = 0; q < C::NP; ++q) {
        const int n = r * C::NS + 2 * q;
        on = on && fabsf(A2[q].x - float(n + 1) * a20) <= 0x1p-20f * fabsf(A2[q].x);
        on = on && fabsf(A2[q].y - float(n + 2) * a20) <= 0x1p-20f * fabsf(A2[q].y);
    }
    const bool lat = __all_sync(FULL, on);
    const float3 latc = make_float3(float(r * C::NS + 1) * a20, float(r * C::NS + 2) * a20, 2.0f * a20);

    for (int v = 0; v < V; ++v) {
        const int st = v % C::STAGES;
        const bool agg_pass = S > 1 && v < ntl;
        const int t0 = (k0 + v % ntl) * C::T;
        abt.wait(&ready[st], (v / C::STAGES) & 1, timeout_ns);
        const IO *base = tiles + size_t(st) * C::STAGE_ELEMS;
        const IO *xs = base + ch;
        const IO *dts = base + C::TILE + ch;
        const IO *zs = base + 2 * C::TILE + ch;
        const float *bc = BCf + size_t(st) * C::T * 2 * C::N + r * C::NS;
        IO *yp = y + (size_t(b) * L + t0) * D + d;
        (void)FULL;
        const bool full_tile = t0 + C::T <= L && d0 + (32 / LPC) * (warp + 1) <= D;
        if (agg_pass)
            sel_tile<IO, DC, LPC, ACC, HAS_Z, SOFTPLUS, kAggregate>(xs, dts, zs, bc, A2, h, dsum, dsk,
                                                                     yp, D, L - t0, r, lane);
        else if (full_tile && lat)
            sel_tile<IO, DC, LPC, ACC, HAS_Z, SOFTPLUS, kFull, true>(xs, dts, zs, bc, A2, h, dsum, dsk,
                                                                      yp, D, C::T, r, lane, latc);
        else if (full_tile)
            sel_tile<IO, DC, LPC, ACC, HAS_Z, SOFTPLUS, kFull>(xs, dts, zs, bc, A2, h, dsum, dsk, yp,
                                                                D, C::T, r, lane);
        else
            sel_tile<IO, DC, LPC, ACC, HAS_Z, SOFTPLUS, kRagged>(xs, dts, zs, bc, A2, h, dsum, dsk,
                                                                  yp, D, vd ? L - t0 : 0, r, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);

        if (agg_pass && v == ntl - 1) {
            constexpr int NC = 32 * C::CWARPS;
            const size_t slot = size_t(cb) * S + s;
            float2 carry[C::NP];
#pragma unroll
            for (int q = 0; q < C::NP; ++q) {
                const int n = r * C::NS + 2 * q;
                carry[q] = (vd && h0 != nullptr)
                               ? make_float2(h0[(size_t(b) * D + d) * C::N + n],
                                             h0[(size_t(b) * D + d) * C::N + n + 1])
                               : make_float2(0.0f, 0.0f);
            }
            if (s > 0) {
                float *ag = ws.agg + slot * C::kAgg * DC;
                if (r == 0) ag[ch] = dsum;
#pragma unroll
                for (int q = 0; q < C::NP; ++q) {
                    const int n = r * C::NS + 2 * q;
                    ag[(1 + n) * DC + ch] = h[q].x;
                    ag[(2 + n) * DC + ch] = h[q].y;
                }
                __threadfence();
                named_bar_sync(1, NC);
                if (tid == 0 && s != withheld) st_release_gpu(&ws.flags[slot], kFlagAggregate);
                float acc_d = 0.0f;  // composition of splits sp+1 .. s-1
                float2 acc_h[C::NP];
#pragma unroll
                for (int q = 0; q < C::NP; ++q) acc_h[q] = make_float2(0.0f, 0.0f);
                bool done = false;
                for (int sp = s - 1; sp >= 0 && !done; --sp) {
                    const size_t sl = size_t(cb) * S + sp;
                    if (tid == 0) *bcast = static_cast<int>(poll_flag(&ws.flags[sl], timeout_ns));
                    named_bar_sync(1, NC);
                    const int fv = *bcast;
                    named_bar_sync(1, NC);
                    if (fv == static_cast<int>(kFlagInclusive)) {
                        const float *in = ws.incl + sl * C::kIncl * DC;
#pragma unroll
                        for (int q = 0; q < C::NP; ++q) {
                            const int n = r * C::NS + 2 * q;
                            const float px = pow2_t<ACC>(A2[q].x * acc_d);
                            const float py = pow2_t<ACC>(A2[q].y * acc_d);
                            carry[q].x = fmaf(px, __ldcg(&in[n * DC + ch]), acc_h[q].x);
                            carry[q].y = fmaf(py, __ldcg(&in[(n + 1) * DC + ch]), acc_h[q].y);
                        }
                        done = true;
                    } else if (fv == static_cast<int>(kFlagAggregate)) {
                        const float *ax = ws.agg + sl * C::kAgg * DC;
#pragma unroll
                        for (int q = 0; q < C::NP; ++q) {
                            const int n = r * C::NS + 2 * q;
                            const float px = pow2_t<ACC>(A2[q].x * acc_d);
                            const float py = pow2_t<ACC>(A2[q].y * acc_d);
                            acc_h[q].x = fmaf(px, __ldcg(&ax[(1 + n) * DC + ch]), acc_h[q].x);
                            acc_h[q].y = fmaf(py, __ldcg(&ax[(2 + n) * DC + ch]), acc_h[q].y);
                        }
                        acc_d += __ldcg(&ax[ch]);
                    } else {
                        if (tid == 0) report_status(LR_ERR_TIMEOUT);
#pragma unroll
                        for (int q = 0; q < C::NP; ++q) carry[q] = acc_h[q];
                        done = true;
                    }
                }
            }
            float *in = ws.incl + slot * C::kIncl * DC;
#pragma unroll
            for (int q = 0; q < C::NP; ++q) {
                const int n = r * C::NS + 2 * q;
                in[n * DC + ch] = fmaf(pow2_t<ACC>(A2[q].x * dsum), carry[q].x, h[q].x);
                in[(n + 1) * DC + ch] = fmaf(pow2_t<ACC>(A2[q].y * dsum), carry[q].y, h[q].y);
                h[q] = carry[q];
            }
            __threadfence();
            named_bar_sync(1, NC);
            if (tid == 0 && s != withheld) st_release_gpu(&ws.flags[slot], kFlagInclusive);
        }
    }
    if (h_final != nullptr && vd && s == S - 1) {
#pragma unroll
        for (int q = 0; q < C::NP; ++q) {
            const int n = r * C::NS + 2 * q;
            h_final[(size_t(b) * D + d) * C::N + n] = h[q].x;
            h_final[(size_t(b) * D + d) * C::N + n + 1] = h[q].y;
        }
    }
}

// ============================================================================
// Host side
// ============================================================================
namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

bool encode_map_3d(CUtensorMap *tm, const void *base, CUtensorMapDataType type, size_t esize,
                   uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, uint32_t b2) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * esize, d0 * d1 * esize};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(tm, type, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// 3-D map over a row-major (d2, d1, d0) tensor, box (b0, b1, 1).
bool make_map_3d(CUtensorMap *tm, const void *base, CUtensorMapDataType type, size_t esize,
                 uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1) {
    return encode_map_3d(tm, base, type, esize, d0, d1, d2, b0, b1, 1);
}

// Per-device facts and per-kernel attributes, looked up once.
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    std::once_flag once;
    int sms = 0;
};
DeviceInfo g_dev[kMaxDevices];

// Sets a kernel's dynamic shared-memory limit once per device and returns
// how many of its blocks fit on one SM (0 on error).
template <auto Kernel>
int kernel_blocks_per_sm(int threads, size_t smem, int dev) {
    static std::once_flag once[kMaxDevices];
    static int blocks[kMaxDevices];
    std::call_once(once[dev], [&] {
        blocks[dev] = 0;
        if (cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, Kernel, threads, smem) == cudaSuccess)
            blocks[dev] = n;
    });
    return blocks[dev];
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Splits are used only when the channel blocks alone leave most SMs idle; the
// split count then targets every resident block slot.  Two splits would
// only double the work per split, so fewer than three means one.
void choose_splits(DiagPlan *p, int sms, int resident_per_sm, int agg_floats, int incl_floats) {
    int S = 1;
    if (g_split_override > 0) {
        S = g_split_override;
    } else if (p->n_cb * 2 < sms) {
        const int64_t slots = int64_t(sms) * (resident_per_sm > 0 ? resident_per_sm : 1);
        const int64_t want = (slots + p->n_cb - 1) / p->n_cb;
        S = want >= 3 ? static_cast<int>(want < (1 << 20) ? want : (1 << 20)) : 1;
    }
    S = S < 1 ? 1 : (S > p->n_tiles ? p->n_tiles : S);
    p->tps = (p->n_tiles + S - 1) / S;
    p->S = (p->n_tiles + p->tps - 1) / p->tps;
    if (p->S <= 1) {
        p->S = 1;
        p->tps = p->n_tiles;
        p->ctrl_bytes = 0;
        p->ws_bytes = 0;
        return;
    }
    const size_t slots = size_t(p->n_cb) * p->S;
    p->ctrl_bytes = align_up((slots + 1) * sizeof(uint32_t), 256);
    const size_t agg = align_up(slots * agg_floats * p->dc * sizeof(float), 256);
    const size_t incl = align_up(slots * incl_floats * p->dc * sizeof(float), 256);
    p->ws_bytes = p->ctrl_bytes + agg + incl;
}

LookbackWs carve(const DiagPlan &p, void *workspace, int agg_floats) {
    LookbackWs w{};
    if (p.S <= 1) return w;
    char *base = static_cast<char *>(workspace);
    const size_t slots = size_t(p.n_cb) * p.S;
    w.flags = reinterpret_cast<uint32_t *>(base);
    w.ticket = w.flags + slots;
    w.agg = reinterpret_cast<float *>(base + p.ctrl_bytes);
    w.incl = reinterpret_cast<float *>(
        base + p.ctrl_bytes + align_up(slots * agg_floats * p.dc * sizeof(float), 256));
    return w;
}

uint64_t timeout_ns() {
    return g_withheld_split >= 1 ? uint64_t(g_withheld_timeout_ms) * 1000000ull : kDefaultTimeoutNs;
}

constexpr int kSelDC = 32;
constexpr int kSelLPC = 2;   // lanes per channel

int current_device(int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return LR_ERR_CUDA;
    return LR_OK;
}

}  // namespace

int device_sm_count(int *sms) {
    int dev = 0;
    if (current_device(&dev) != LR_OK) return LR_ERR_CUDA;
    DeviceInfo &di = g_dev[dev];
    std::call_once(di.once, [&] {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) di.sms = n;
    });
    if (di.sms <= 0) return LR_ERR_CUDA;
    *sms = di.sms;
    return LR_OK;
}

// ---------------------------------------------------------------- RG-LRU host
template <typename IO, bool ACC>
static int rglru_resident(int dev) {
    // both gate variants share block size and shared memory; each needs its
    // own dynamic shared-memory attribute
    const int a = kernel_blocks_per_sm<rglru_scan_kernel<IO, ACC, false>>(RgCfg<IO>::THREADS,
                                                                          RgCfg<IO>::SMEM, dev);
    const int b = kernel_blocks_per_sm<rglru_scan_kernel<IO, ACC, true>>(RgCfg<IO>::THREADS,
                                                                         RgCfg<IO>::SMEM, dev);
    return a < b ? a : b;
}

int rglru_plan(int64_t B, int64_t L, int64_t D, lr_dtype io, DiagPlan *p) {
    int sms = 0, dev = 0;
    if (device_sm_count(&sms) != LR_OK || current_device(&dev) != LR_OK) return LR_ERR_CUDA;
    *p = DiagPlan{};
    p->dc = RgCfg<float>::DC;
    p->tile_t = io == LR_BF16 ? RgCfg<__nv_bfloat16>::T : RgCfg<float>::T;
    p->n_cb = B * ((D + p->dc - 1) / p->dc);
    p->n_tiles = static_cast<int>((L + p->tile_t - 1) / p->tile_t);
    const int per_sm = io == LR_BF16 ? rglru_resident<__nv_bfloat16, false>(dev)
                                     : rglru_resident<float, true>(dev);
    if (per_sm <= 0) return LR_ERR_CUDA;
    choose_splits(p, sms, per_sm, RgCfg<float>::kAgg, RgCfg<float>::kIncl);
    return LR_OK;
}

template <typename IO, bool ACC>
static int rglru_launch_t(const void *x, const void *r, const void *i, const float *a_log, float c,
                          const float *h0, void *y, float *h_final, int64_t B, int64_t L,
                          int64_t D, const DiagPlan &p, void *workspace, bool preact,
                          cudaStream_t stream) {
    using C = RgCfg<IO>;
    CUtensorMap mx, mr, mi;
    const auto tt = Io<IO>::kTmType;
    if (!make_map_3d(&mx, x, tt, sizeof(IO), D, L, B, C::DC, C::T) ||
        !make_map_3d(&mr, r, tt, sizeof(IO), D, L, B, C::DC, C::T) ||
        !make_map_3d(&mi, i, tt, sizeof(IO), D, L, B, C::DC, C::T))
        return LR_ERR_CUDA;
    if (p.S > 1 && cudaMemsetAsync(workspace, 0, p.ctrl_bytes, stream) != cudaSuccess)
        return LR_ERR_CUDA;
    const LookbackWs ws = carve(p, workspace, C::kAgg);
    const int n_db = static_cast<int>((D + C::DC - 1) / C::DC);
    const int64_t grid = p.n_cb * p.S;
    auto kern = preact ? rglru_scan_kernel<IO, ACC, true> : rglru_scan_kernel<IO, ACC, false>;
    kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, stream>>>(
        mx, mr, mi, a_log, c, h0, static_cast<IO *>(y), h_final, static_cast<int>(L),
        static_cast<int>(D), n_db, p.S, p.tps, p.n_tiles, ws, g_withheld_split, timeout_ns());
    return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

int rglru_launch(const void *x, const void *r, const void *i, const float *a_log, float c,
                 const float *h0, void *y, float *h_final, int64_t B, int64_t L, int64_t D,
                 lr_dtype io, const DiagPlan &p, void *workspace, cudaStream_t stream, bool preact) {
    if (io == LR_BF16)
        return rglru_launch_t<__nv_bfloat16, false>(x, r, i, a_log, c, h0, y, h_final, B, L, D, p,
                                                    workspace, preact, stream);
    return rglru_launch_t<float, true>(x, r, i, a_log, c, h0, y, h_final, B, L, D, p, workspace,
                                       preact, stream);
}

// ---------------------------------------------------------------- minmax host
template <typename IO>
static int minmax_resident(int dev) {
    using C = MmCfg<IO>;
    return kernel_blocks_per_sm<minmax_scan_kernel<IO>>(C::THREADS, C::SMEM, dev);
}

int minmax_plan(int64_t B, int64_t L, int64_t D, lr_dtype io, DiagPlan *p) {
    int sms = 0, dev = 0;
    if (device_sm_count(&sms) != LR_OK || current_device(&dev) != LR_OK) return LR_ERR_CUDA;
    *p = DiagPlan{};
    p->dc = MmCfg<float>::DC;
    p->tile_t = MmCfg<float>::T;
    p->n_cb = B * ((D + p->dc - 1) / p->dc);
    p->n_tiles = static_cast<int>((L + p->tile_t - 1) / p->tile_t);
    const int per_sm = io == LR_BF16 ? minmax_resident<__nv_bfloat16>(dev) : minmax_resident<float>(dev);
    if (per_sm <= 0) return LR_ERR_CUDA;
    choose_splits(p, sms, per_sm, MmCfg<float>::kAgg, MmCfg<float>::kIncl);
    return LR_OK;
}

template <typename IO>
static int minmax_launch_t(const void *r, const void *s, const float *x0, void *y, float *x_final,
                           int64_t B, int64_t L, int64_t D, const DiagPlan &p, void *workspace,
                           cudaStream_t stream) {
    using C = MmCfg<IO>;
    CUtensorMap mr, ms;
    const auto tt = Io<IO>::kTmType;
    if (!make_map_3d(&mr, r, tt, sizeof(IO), D, L, B, C::DC, C::T) ||
        !make_map_3d(&ms, s, tt, sizeof(IO), D, L, B, C::DC, C::T))
        return LR_ERR_CUDA;
    if (p.S > 1 && cudaMemsetAsync(workspace, 0, p.ctrl_bytes, stream) != cudaSuccess)
        return LR_ERR_CUDA;
    const LookbackWs ws = carve(p, workspace, C::kAgg);
    const int n_db = static_cast<int>((D + C::DC - 1) / C::DC);
    const int64_t grid = p.n_cb * p.S;
    minmax_scan_kernel<IO><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, stream>>>(
        mr, ms, x0, static_cast<IO *>(y), x_final, static_cast<int>(L), static_cast<int>(D), n_db, p.S,
        p.tps, p.n_tiles, ws, g_withheld_split, timeout_ns());
    return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

int minmax_launch(const void *r, const void *s, const float *x0, void *y, float *x_final, int64_t B,
                  int64_t L, int64_t D, lr_dtype io, const DiagPlan &p, void *workspace,
                  cudaStream_t stream) {
    if (io == LR_BF16)
        return minmax_launch_t<__nv_bfloat16>(r, s, x0, y, x_final, B, L, D, p, workspace, stream);
    return minmax_launch_t<float>(r, s, x0, y, x_final, B, L, D, p, workspace, stream);
}

// ------------------------------------------------------------- selective host
template <typename IO, bool ACC, bool HZ, bool SP>
static int selective_resident(int dev) {
    using C = SelCfg<IO, kSelDC, kSelLPC>;
    return kernel_blocks_per_sm<selective_scan_kernel<IO, kSelDC, kSelLPC, ACC, HZ, SP>>(C::THREADS, C::SMEM,
                                                                               dev);
}

template <typename IO, bool ACC>
static int selective_resident_any(int dev, bool hz, bool sp) {
    // all four variants share block size and shared memory; each needs its
    // own dynamic shared-memory attribute, so every one is set up here
    const int a = selective_resident<IO, ACC, true, true>(dev);
    const int b = selective_resident<IO, ACC, true, false>(dev);
    const int c = selective_resident<IO, ACC, false, true>(dev);
    const int d = selective_resident<IO, ACC, false, false>(dev);
    return hz ? (sp ? a : b) : (sp ? c : d);
}

int selective_plan(int64_t B, int64_t L, int64_t D, lr_dtype io, DiagPlan *p) {
    int sms = 0, dev = 0;
    if (device_sm_count(&sms) != LR_OK || current_device(&dev) != LR_OK) return LR_ERR_CUDA;
    *p = DiagPlan{};
    p->dc = kSelDC;
    p->tile_t = SelCfg<float, kSelDC, kSelLPC>::T;
    p->n_cb = B * ((D + p->dc - 1) / p->dc);
    p->n_tiles = static_cast<int>((L + p->tile_t - 1) / p->tile_t);
    const int per_sm = io == LR_BF16 ? selective_resident_any<__nv_bfloat16, false>(dev, true, true)
                                     : selective_resident_any<float, true>(dev, true, true);
    if (per_sm <= 0) return LR_ERR_CUDA;
    choose_splits(p, sms, per_sm, SelCfg<float, kSelDC, kSelLPC>::kAgg, SelCfg<float, kSelDC, kSelLPC>::kIncl);
    return LR_OK;
}

template <typename IO, bool ACC, bool HZ, bool SP>
static int selective_launch_v(const CUtensorMap &mx, const CUtensorMap &mdt, const CUtensorMap &mz,
                              const CUtensorMap &mB, const CUtensorMap &mC, const float *A_log,
                              const float *Dskip, const float *h0, void *y, float *h_final,
                              int64_t L, int64_t D, const DiagPlan &p, const LookbackWs &ws,
                              cudaStream_t stream) {
    using C = SelCfg<IO, kSelDC, kSelLPC>;
    const int n_db = static_cast<int>((D + C::DC - 1) / C::DC);
    const int64_t grid = p.n_cb * p.S;
    selective_scan_kernel<IO, kSelDC, kSelLPC, ACC, HZ, SP>
        <<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, stream>>>(
            mx, mdt, mz, mB, mC, A_log, Dskip, h0, static_cast<IO *>(y), h_final,
            static_cast<int>(L), static_cast<int>(D), n_db, p.S, p.tps, p.n_tiles, ws,
            g_withheld_split, timeout_ns());
    return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

template <typename IO, bool ACC>
static int selective_launch_t(const void *x, const void *dt, const void *z, const void *Bm,
                              const void *Cm, const float *A_log, const float *Dskip,
                              const float *h0, void *y, float *h_final, int64_t B, int64_t L,
                              int64_t D, int dt_softplus, const DiagPlan &p, void *workspace,
                              cudaStream_t stream) {
    using C = SelCfg<IO, kSelDC, kSelLPC>;
    CUtensorMap mx, mdt, mz, mB, mC;
    const auto tt = Io<IO>::kTmType;
    if (!make_map_3d(&mx, x, tt, sizeof(IO), D, L, B, C::DC, C::T) ||
        !make_map_3d(&mdt, dt, tt, sizeof(IO), D, L, B, C::DC, C::T) ||
        !make_map_3d(&mz, z != nullptr ? z : x, tt, sizeof(IO), D, L, B, C::DC, C::T) ||
        !make_map_3d(&mB, Bm, tt, sizeof(IO), C::N, L, B, C::N, C::T) ||
        !make_map_3d(&mC, Cm, tt, sizeof(IO), C::N, L, B, C::N, C::T))
        return LR_ERR_CUDA;
    if (p.S > 1 && cudaMemsetAsync(workspace, 0, p.ctrl_bytes, stream) != cudaSuccess)
        return LR_ERR_CUDA;
    const LookbackWs ws = carve(p, workspace, C::kAgg);
    const bool hz = z != nullptr, sp = dt_softplus != 0;
    if (hz && sp)
        return selective_launch_v<IO, ACC, true, true>(mx, mdt, mz, mB, mC, A_log, Dskip, h0, y,
                                                       h_final, L, D, p, ws, stream);
    if (hz)
        return selective_launch_v<IO, ACC, true, false>(mx, mdt, mz, mB, mC, A_log, Dskip, h0, y,
                                                        h_final, L, D, p, ws, stream);
    if (sp)
        return selective_launch_v<IO, ACC, false, true>(mx, mdt, mz, mB, mC, A_log, Dskip, h0, y,
                                                        h_final, L, D, p, ws, stream);
    return selective_launch_v<IO, ACC, false, false>(mx, mdt, mz, mB, mC, A_log, Dskip, h0, y,
                                                     h_final, L, D, p, ws, stream);
}

int selective_launch(const void *x, const void *dt, const void *z, const void *Bm, const void *Cm,
                     const float *A_log, const float *Dskip, const float *h0, void *y,
                     float *h_final, int64_t B, int64_t L, int64_t D, lr_dtype io, int dt_softplus,
                     const DiagPlan &p, void *workspace, cudaStream_t stream) {
    if (io == LR_BF16)
        return selective_launch_t<__nv_bfloat16, false>(x, dt, z, Bm, Cm, A_log, Dskip, h0, y,
                                                        h_final, B, L, D, dt_softplus, p,
                                                        workspace, stream);
    return selective_launch_t<float, true>(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final, B, L, D,
                                           dt_softplus, p, workspace, stream);
}

// ---------------------------------------------------- built-in scratch (RG-LRU)
// Scratch for lr_rglru_scan_fwd_noalloc: the look-back flags, ticket and split
// descriptors of the RG-LRU scan live in this fixed array instead of a
// caller-provided workspace.  Every GPU that loads the library holds it until
// the process exits; all calls on a device share it.
static __device__ __align__(256) unsigned char g_rglru_scratch[kRglruScratchBytes];

int rglru_builtin_scratch(void **ptr) {
    int dev = 0;
    if (current_device(&dev) != LR_OK) return LR_ERR_CUDA;
    static std::once_flag once[kMaxDevices];
    static void *addr[kMaxDevices];
    static cudaError_t err[kMaxDevices];
    // Host code sees the array only through a stand-in symbol: its device
    // address is looked up once per device, with that device current.
    std::call_once(once[dev], [&] {
        addr[dev] = nullptr;
        err[dev] = cudaGetSymbolAddress(&addr[dev], g_rglru_scratch);
    });
    if (err[dev] != cudaSuccess || addr[dev] == nullptr) return LR_ERR_CUDA;
    *ptr = addr[dev];
    return LR_OK;
}

int diag_status_read_and_clear(int *status) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_diag_status, sizeof(int)) != cudaSuccess) return LR_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_diag_status, &zero, sizeof(int)) != cudaSuccess)
            return LR_ERR_CUDA;
    }
    *status = v;
    return LR_OK;
}

}  // namespace lr
