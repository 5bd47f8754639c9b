// lr_diag_scan.cu -- the scalar-state scans on sm_103a:
//
//   * RG-LRU   (lrnnx rglru module source, RGLRU.step fallback update):
//       a_t = exp(c r_t a_log),  h = a_t h + sqrt(1 - a_t^2) (i_t x_t),  y_t = h
//   * MinMax   (minmaxrnc MinMaxNeuron): x_t = max(min(r_t, x_{t-1}), s_t)
//
// Design (both kernels):
//   * A thread block owns a block of DC consecutive channels of one batch row
//     and streams a range of time tiles (T steps x DC channels) through a
//     multi-stage shared-memory ring filled by TMA (cp.async.bulk.tensor,
//     3-D maps over (D, L, B); out-of-range rows and channels arrive as
//     zeros).  Warps are specialised: a producer warp keeps the ring full,
//     compute warps run the recurrence of their channels (one thread per
//     channel) with the state in registers, in batches of 8 steps whose loads
//     and coefficients are independent, and store outputs straight from
//     registers.  Stages pass between the roles through full / empty
//     mbarriers, not block barriers.
//   * When batch x channel blocks fill the GPU (S == 1) a block streams the
//     whole sequence once, carrying the state across tiles in registers.
//   * Otherwise the sequence is cut into S time splits that run in parallel.
//     Each split first scans its range from a zero state to get its
//     aggregate, publishes it, and takes its carry-in from a decoupled
//     look-back over the preceding splits' descriptors (Merrill & Garland,
//     "Single-pass Parallel Prefix Scan with Decoupled Look-back", 2016).
//     Split order comes from an atomic ticket, so every split a block waits
//     for is already running.  It then re-streams its range (an L2 hit for
//     the small problems this mode serves) and writes the outputs.  Every
//     wait is bounded in time.
//   * A split descriptor is (product of decays, h) per channel for RG-LRU and
//     the composed (min, max) operator for MinMax.
#include <cudaTypedefs.h>

#include <mutex>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {

// Flag values of a split descriptor.
constexpr uint32_t kFlagNone = 0, kFlagAggregate = 1, kFlagInclusive = 2;

struct LookbackWs {
    uint32_t *flags;   // [n_cb * S]
    uint32_t *ticket;  // [1]
    float *agg;        // [n_cb * S][kAgg][DC]
    float *incl;       // [n_cb * S][kIncl][DC]
};

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
                                             volatile int *flag, StatusRef st) {
    if (*flag != 0) return false;
    if (mbar_wait_bounded(bar, parity, limit_ns)) return true;
    *flag = 1;
    status_report(st, LR_ERR_TIMEOUT);
    return false;
}

struct BlockAbort {
    volatile int *flag;
    StatusRef st;
    // Fast path: one try_wait when the phase has already completed.
    __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) const {
        if (mbar_try_wait(bar, parity)) return true;
        return block_wait_slow(bar, parity, limit_ns, flag, st);
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
                      int n_tiles, LookbackWs ws, int withheld, uint64_t timeout_ns, StatusRef sref) {
    using C = RgCfg<IO>;
    extern __shared__ __align__(128) unsigned char smem[];
    IO *tiles = reinterpret_cast<IO *>(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::STAGES;
    int *bcast = reinterpret_cast<int *>(empty + C::STAGES);
    int *abort_word = bcast + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const BlockAbort ab{abort_word, sref};

    if (tid == 0) {
        for (int st = 0; st < C::STAGES; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], C::CWARPS);
        }
        *abort_word = 0;
        fence_mbar_init();
        if (S > 1) *bcast = static_cast<int>(atomicAdd(ws.ticket, 1u));
        if (blockIdx.x == 0) status_begin(sref);
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
                    if (tid == 0) status_report(sref, LR_ERR_TIMEOUT);
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
                       int withheld, uint64_t timeout_ns, StatusRef sref) {
    using C = MmCfg<IO>;
    extern __shared__ __align__(128) unsigned char smem[];
    IO *tiles = reinterpret_cast<IO *>(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::STAGES;
    int *bcast = reinterpret_cast<int *>(empty + C::STAGES);
    int *abort_word = bcast + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const BlockAbort ab{abort_word, sref};

    if (tid == 0) {
        for (int st = 0; st < C::STAGES; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], C::CWARPS);
        }
        *abort_word = 0;
        fence_mbar_init();
        if (S > 1) *bcast = static_cast<int>(atomicAdd(ws.ticket, 1u));
        if (blockIdx.x == 0) status_begin(sref);
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
                    if (tid == 0) status_report(sref, LR_ERR_TIMEOUT);
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
        p->ws_bytes = kStatusBytes;
        return;
    }
    const size_t slots = size_t(p->n_cb) * p->S;
    p->ctrl_bytes = align_up((slots + 1) * sizeof(uint32_t), 256);
    const size_t agg = align_up(slots * agg_floats * p->dc * sizeof(float), 256);
    const size_t incl = align_up(slots * incl_floats * p->dc * sizeof(float), 256);
    p->ws_bytes = kStatusBytes + p->ctrl_bytes + agg + incl;
}

LookbackWs carve(const DiagPlan &p, void *workspace, int agg_floats) {
    LookbackWs w{};
    if (p.S <= 1) return w;
    char *base = static_cast<char *>(workspace) + kStatusBytes;
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
    if (p.S > 1 && cudaMemsetAsync(static_cast<char *>(workspace) + kStatusBytes, 0, p.ctrl_bytes, stream) !=
                       cudaSuccess)
        return LR_ERR_CUDA;
    const LookbackWs ws = carve(p, workspace, C::kAgg);
    const int n_db = static_cast<int>((D + C::DC - 1) / C::DC);
    const int64_t grid = p.n_cb * p.S;
    auto kern = preact ? rglru_scan_kernel<IO, ACC, true> : rglru_scan_kernel<IO, ACC, false>;
    kern<<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, stream>>>(
        mx, mr, mi, a_log, c, h0, static_cast<IO *>(y), h_final, static_cast<int>(L),
        static_cast<int>(D), n_db, p.S, p.tps, p.n_tiles, ws, g_withheld_split, timeout_ns(),
        call_status(workspace));
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
    if (p.S > 1 && cudaMemsetAsync(static_cast<char *>(workspace) + kStatusBytes, 0, p.ctrl_bytes, stream) !=
                       cudaSuccess)
        return LR_ERR_CUDA;
    const LookbackWs ws = carve(p, workspace, C::kAgg);
    const int n_db = static_cast<int>((D + C::DC - 1) / C::DC);
    const int64_t grid = p.n_cb * p.S;
    minmax_scan_kernel<IO><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM, stream>>>(
        mr, ms, x0, static_cast<IO *>(y), x_final, static_cast<int>(L), static_cast<int>(D), n_db, p.S,
        p.tps, p.n_tiles, ws, g_withheld_split, timeout_ns(), call_status(workspace));
    return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

int minmax_launch(const void *r, const void *s, const float *x0, void *y, float *x_final, int64_t B,
                  int64_t L, int64_t D, lr_dtype io, const DiagPlan &p, void *workspace,
                  cudaStream_t stream) {
    if (io == LR_BF16)
        return minmax_launch_t<__nv_bfloat16>(r, s, x0, y, x_final, B, L, D, p, workspace, stream);
    return minmax_launch_t<float>(r, s, x0, y, x_final, B, L, D, p, workspace, stream);
}

// ---------------------------------------------------- built-in scratch (RG-LRU)
// Scratch for lr_rglru_scan_fwd_noalloc: the status word, look-back flags,
// ticket and split descriptors of the RG-LRU scan live in this fixed array
// instead of a caller-provided workspace.  Every GPU that loads the library
// holds it until the process exits; all calls on a device share it.
static __device__ __align__(256) unsigned char g_rglru_scratch[kRglruScratchBytes];

int rglru_builtin_scratch(void **ptr) {
    int dev = 0;
    if (current_device(&dev) != LR_OK) return LR_ERR_CUDA;
    static std::mutex mu;
    static void *addr[kMaxDevices];
    // Host code sees the array only through a stand-in symbol: its device
    // address is looked up with that device current, and only a successful
    // lookup is kept (a failed one, e.g. during stream capture, is retried by
    // the next call).
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_rglru_scratch) != cudaSuccess || a == nullptr) return LR_ERR_CUDA;
        addr[dev] = a;
    }
    *ptr = addr[dev];
    return LR_OK;
}

}  // namespace lr
