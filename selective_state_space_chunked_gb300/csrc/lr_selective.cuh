// lr_selective.cuh -- the selective SSM scan on sm_103a: device code and the
// kernel variants (instantiated in lr_sel_*.cu; host plan in lr_selective.cu).
//
// [SSM] cortexnet 3.2.1, cortexnet/ssm.py: MultiScaleSSM._selective_scan (the
// recurrence) with the D skip and silu(z) gate of MultiScaleSSM.forward:
//
//   delta_t = softplus(dt_t),  h[n] = exp(delta_t A[n]) h[n] + delta_t B_t[n] x_t,
//   y_t = (C_t . h + D x_t) silu(z_t)
//
// Work decomposition.  A warp owns a "chain": 32 * CPL consecutive channels
// of one batch row, CPL per lane (two or four), the 16 fp32 states of each
// in registers.  The chains' 8-step time tiles form one flat list
// (chain-major), and each warp of the launch starts with an equal contiguous
// share of it.  The grid is one resident wave.  Chains are numbered batch row
// first (chain c is channel group c / B of batch row c % B), so that the
// blocks an SM holds, which lie far apart in the list, cover different
// channel groups: how long a warm-up or a carry correction runs depends on
// its channels' decay rates, and mixing channel groups spreads that work
// evenly over the SMs.
//
// Equal shares do not finish together: the warps sharing a scheduler do not
// get equal issue shares, so some finish in half the time of others, and an
// SM whose warps have finished runs its last ones at a fraction of its
// throughput (measured: 4.8 tiles/us with 16 warps, 2.4 with 4, 0.4 with one).
// With warm-ups on, a share therefore runs as a claimable range with work
// stealing (see "Ranges and work stealing"): a warp that has run out of work
// splits off the back half of the largest remainder still unclaimed, warms up
// to its start and runs it, so the SMs stay busy until the list is done.
//
// A piece that starts inside a chain needs the state its chain reaches just
// before it.  Because every state decays, that state depends, to any given
// relative accuracy, only on a window of preceding steps: the piece first
// walks back over them (the "warm-up"), summing their contributions
//   h_{s-1}[n] = sum_t exp(A[n] (Lambda_{s-1} - Lambda_t)) delta_t B_t[n] x_t
// from the latest step back -- each term independent of the others, so no
// serial chain -- until, for every channel of the warp, the slowest decay
// over the walked steps has fallen below 2^-c, or until the chain start (the
// initial state, decayed over the whole prefix, is then added and the state
// is exact).  The omitted history contributes less than 2^-c of the size the
// state had at the window start: c = 32 for fp32 outputs, 10 for bf16
// outputs (half the bf16 output's half-ulp 2^-9, far inside the bf16
// tolerance; measured on the pages' workload at B1 L4096 with 16 pieces per
// chain, the fp32 final state moves by 4e-6 of its maximum and y not at all
// beyond its bf16 rounding).  The warm-up reads each window's x, dt, B_t
// once more (about one tenth of the data for the pages' sequences) but
// never waits for another warp.
//
// When the window would exceed a limit (lr_set_selective_warmup; slow decays
// or tiny steps; by default always for fp32 outputs, whose window is as long
// as the pages' sequences), the piece instead runs from a zero state and its carry-in,
// the state at the end of the preceding piece, arrives afterwards through a
// decoupled look-back over the preceding warps' piece descriptors (Merrill &
// Garland, "Single-pass Parallel Prefix Scan with Decoupled Look-back",
// 2016), compressed to (sum of delta, h[16]) per channel because the decay of
// state n over a range is exp(A[n] * sum of delta).  The piece's outputs are
// then corrected in place, y_t += silu(z_t) sum_n C_t[n] exp(A[n] Lambda_t)
// carry[n] with Lambda_t the sum of delta from the piece start to t, until
// every remaining term is below 2^-c of its value at the piece start.  In
// the stealing kernel a share whose warm-up would exceed the limit is left
// to a second launch (the static kernel, run for the marked shares only),
// which takes that path.
//
// Data movement.  Each warp streams its tiles through a private ring of
// shared-memory stages filled by TMA (one lane issues the copies of x, dt, z,
// B_t, C_t; out-of-range rows and channels arrive as zeros), so warps never
// wait for each other; bf16 B_t, C_t rows (shared by all channels) are widened
// to fp32 once per tile by the whole warp and read back as broadcast 16-byte
// loads, each feeding all the channels of a lane.
//
// Decays.  In general each state's decay is one exp2 of delta A[n] log2(e).
// The cortexnet 3.2.1 ssm.py page (class MultiScaleSSM, its initialiser)
// sets A_log[d, n] = log((n+1) 2^s), so that
// A[n] = (n + 1) A[0]; on that lattice the 16 decays of a step are the powers
// E, E^2, .., E^16 of E = exp(delta A[0]), taken as (E, E^2) from two exp2 and
// the other pairs as P * (E^2, E^2).  Each warp checks the lattice itself from
// the A_log it is given (|A[n] - (n+1) A[0]| <= 2^-20 |A[n]| in fp32 for every
// state of its channels); trained A_log leaves the lattice and takes the
// general form.
#pragma once

#include <cudaTypedefs.h>

#include <mutex>

#include "lr_device.cuh"
#include "lr_internal.h"

// Channels per lane of the bf16 and fp32 kernels (2 or 4), steps per tile,
// and the resident blocks per SM that the two-channel bf16 kernel's register
// budget targets (4: 128 registers per thread, 3: 168).
#ifndef LR_SEL_CPL_BF16
#define LR_SEL_CPL_BF16 2
#endif
#ifndef LR_SEL_T
#define LR_SEL_T 8
#endif
#ifndef LR_SEL_MINB2_BF16
#define LR_SEL_MINB2_BF16 4
#endif

#ifndef LR_SEL_CPL_F32
#define LR_SEL_CPL_F32 2
#endif
// log2 of the share of the state's size below which the history a warm-up
// or a correction leaves out must fall (bf16 outputs; fp32: -32)
#ifndef LR_SEL_CUT_BF16
#define LR_SEL_CUT_BF16 -10.0f
#endif

namespace lr {
namespace sel {

// Arguments of one launch of the selective kernel.
struct SelArgs {
    const float *A_log;     // (D, 16)
    const float *Dskip;     // (D) or NULL
    const float *h0;        // (B, D, 16) or NULL
    void *y;                // (B, L, D)
    float *h_final;         // (B, D, 16) or NULL
    int B, L, D, ntt;       // batch, sequence, channels, tiles per chain
    long long F;            // chains x ntt
    int W;                  // warps sharing the flat tile list
    uint32_t *ticket;       // block order (a block waits only on blocks that started before it)
    uint32_t *ticket2;      // block order of the second (deferred) launch
    unsigned long long *ctl;   // [W] range of each warp: claim cursor (low 32 bits), end (high 32 bits)
    uint32_t *defer;        // [W] 1: the share is left to the second launch
    int steal;              // ranges are claimed in steps and split by idle warps (warm-up mode)
    int deferred;           // second launch: only the deferred shares run
    uint32_t *flags;        // [W] descriptor flag of each warp's last piece
    float *agg;             // [W][1 + 16][chain width]: sum of delta, state of a piece run from zero
    float *incl;            // [W][16][chain width]: state at the end of a warp's last piece
    StatusRef st;
    int withheld;           // test hook: pieces with this ordinal in their chain never publish
    int warmup_tiles;       // longest warm-up (tiles); 0: carries always by look-back
    uint64_t timeout_ns;
};

}  // namespace sel

namespace {

constexpr int kN = 16;                // states per channel
constexpr int kT = LR_SEL_T;          // steps per tile
constexpr int kWpb = 4;               // warps per thread block
constexpr int kMinTiles = 8;          // fewest tiles a warp is given
#ifndef LR_SEL_CLAIM
#define LR_SEL_CLAIM 8
#endif
#ifndef LR_SEL_MIN_STEAL
#define LR_SEL_MIN_STEAL 64
#endif
constexpr int kClaim = LR_SEL_CLAIM;          // tiles a warp claims at a time from its own range
constexpr int kMinSteal = LR_SEL_MIN_STEAL;   // a range is split only with this many tiles unclaimed
constexpr uint32_t kFlagAggregate = 1, kFlagInclusive = 2;
constexpr unsigned kFull = 0xffffffffu;

template <typename IO>
constexpr int cpl_of() { return sizeof(IO) == 2 ? LR_SEL_CPL_BF16 : LR_SEL_CPL_F32; }

template <typename IO, int CPL>
struct SelCfg {
    static constexpr int WCH = 32 * CPL;                         // channels per warp
    static constexpr int NP = CPL / 2;                           // channel pairs per lane
    static constexpr int TILE = kT * WCH;                        // x | y, dt, z elements
    static constexpr int TILE_N = kT * kN;                       // B, C elements
    static constexpr size_t SLOT = size_t(TILE) * sizeof(IO);
    static constexpr size_t SLOT_N = size_t(TILE_N) * sizeof(IO);
    static constexpr size_t OFF_DT = SLOT, OFF_Z = 2 * SLOT, OFF_B = 3 * SLOT, OFF_C = 3 * SLOT + SLOT_N;
    static constexpr size_t STAGE = 3 * SLOT + 2 * SLOT_N;
    // three stages while a warp's ring stays within 24 KB, else two
    static constexpr int STAGES = 3 * STAGE <= 24576 ? 3 : 2;
    static constexpr size_t OFF_BCF = STAGES * STAGE;            // fp32 [kT][B(16) | C(16)], bf16 I/O only
    static constexpr size_t BCF = sizeof(IO) == 2 ? size_t(kT) * 2 * kN * sizeof(float) : 0;
    static constexpr size_t OFF_BAR = OFF_BCF + BCF;
    static constexpr size_t WARP_SMEM = (OFF_BAR + STAGES * 8 + 127) / 128 * 128;
    static constexpr size_t SMEM = kWpb * WARP_SMEM;
    // register budget: resident blocks per SM (4 x 128 registers per thread
    // with two channels per lane, 2 x 255 with four)
    static constexpr int MINB = CPL == 2 ? (sizeof(IO) == 2 ? LR_SEL_MINB2_BF16 : 3) : 2;
    // log2 of the relative size where the carry correction stops
    static constexpr float CUT = sizeof(IO) == 2 ? LR_SEL_CUT_BF16 : -32.0f;
    static_assert(CPL == 2 || CPL == 4, "two or four channels per lane");
    static_assert(kT % 8 == 0, "tiles of whole 8-step passes");
    static_assert(STAGE % 128 == 0 && SLOT_N % 128 == 0, "TMA destinations stay 128-byte aligned");
};

// CPL adjacent channels of one step as a raw word (bf16x2 words or floats)
// and as NP fp32 pairs.
template <typename IO, int CPL> struct Vec;
template <> struct Vec<__nv_bfloat16, 2> {
    using raw = uint32_t;
    __device__ __forceinline__ static void get(raw v, float2 (&f)[1]) {
        f[0] = make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
    }
    __device__ __forceinline__ static raw put(const float2 (&f)[1]) {
        const __nv_bfloat162 b = __float22bfloat162_rn(f[0]);
        return *reinterpret_cast<const uint32_t *>(&b);
    }
};
template <> struct Vec<__nv_bfloat16, 4> {
    using raw = uint2;
    __device__ __forceinline__ static void get(raw v, float2 (&f)[2]) {
        f[0] = make_float2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
        f[1] = make_float2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    }
    __device__ __forceinline__ static raw put(const float2 (&f)[2]) {
        const __nv_bfloat162 a = __float22bfloat162_rn(f[0]), b = __float22bfloat162_rn(f[1]);
        return make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
    }
};
template <> struct Vec<float, 2> {
    using raw = float2;
    __device__ __forceinline__ static void get(raw v, float2 (&f)[1]) { f[0] = v; }
    __device__ __forceinline__ static raw put(const float2 (&f)[1]) { return f[0]; }
};
template <> struct Vec<float, 4> {
    using raw = float4;
    __device__ __forceinline__ static void get(raw v, float2 (&f)[2]) {
        f[0] = make_float2(v.x, v.y);
        f[1] = make_float2(v.z, v.w);
    }
    __device__ __forceinline__ static raw put(const float2 (&f)[2]) {
        return make_float4(f[0].x, f[0].y, f[1].x, f[1].y);
    }
};

// torch softplus (beta 1, threshold 20) of two values.  ACC (fp32 I/O):
// libm log1p / exp.  Otherwise max(x, log(1 + e^x)) from exp2 / log2 with
// the exponent clamped at 2^126: above 20 that is x (log(1 + e^x) rounds to
// x there, as torch's threshold returns), and where 1 + e^x rounds to 1
// (x < -17) it gives 0 for a step of under 4e-8, which moves no bf16 output.
template <bool ACC>
__device__ __forceinline__ float2 softplus2(float2 x) {
    if (ACC)
        return make_float2(x.x > 20.0f ? x.x : log1pf(expf(x.x)), x.y > 20.0f ? x.y : log1pf(expf(x.y)));
    const float2 t = __fmul2_rn(x, make_float2(kLog2e, kLog2e));
    const float2 e = make_float2(ex2_approx(fminf(t.x, 126.0f)), ex2_approx(fminf(t.y, 126.0f)));
    const float2 e1 = __fadd2_rn(e, make_float2(1.0f, 1.0f));
    const float2 l = __fmul2_rn(make_float2(lg2_approx(e1.x), lg2_approx(e1.y)), make_float2(kLn2, kLn2));
    return make_float2(fmaxf(x.x, l.x), fmaxf(x.y, l.y));
}

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// silu(z) = z sigmoid(z) of two values.  ACC (fp32 I/O): from exp2 and a
// reciprocal, ~1e-6 relative.  Otherwise z/2 (1 + tanh(z/2)) with the
// single-instruction tanh (~5e-4 relative, under the bf16 output rounding).
template <bool ACC>
__device__ __forceinline__ float2 silu2(float2 z) {
    if (ACC)
        return make_float2(z.x * rcp_approx(1.0f + ex2_approx(-z.x * kLog2e)),
                           z.y * rcp_approx(1.0f + ex2_approx(-z.y * kLog2e)));
    const float2 hz = __fmul2_rn(z, make_float2(0.5f, 0.5f));
    return __ffma2_rn(hz, make_float2(tanh_approx(hz.x), tanh_approx(hz.y)), hz);
}

template <bool ACC>
__device__ __forceinline__ float pow2_t(float e) {
    return ACC ? exp2f(e) : ex2_approx(e);
}

__device__ __forceinline__ void st_cs(uint32_t *p, uint32_t v) { __stcs(reinterpret_cast<unsigned int *>(p), v); }
__device__ __forceinline__ void st_cs(uint2 *p, uint2 v) { __stcs(p, v); }
__device__ __forceinline__ void st_cs(float2 *p, float2 v) { __stcs(p, v); }
__device__ __forceinline__ void st_cs(float4 *p, float4 v) { __stcs(p, v); }

using sel::SelArgs;

// Per-lane constants of a chain: channel pair j of the lane holds channels
// d + 2j, d + 2j + 1.
template <int CPL>
struct Lane {
    int b, d0, d;           // batch row, first channel of the chain, the lane's first channel
    bool valid;             // d < D (D is a multiple of 4, so all CPL channels are in or out)
    float2 a20[CPL / 2];    // A[0] log2(e) per channel pair
    float2 a2min[CPL / 2];  // max over n of A[n] log2(e): the slowest decay
    float2 dsk[CPL / 2];    // D skip
};

// A[n] log2(e) of the lane's channels as (n, n+1) pairs.
template <int CPL>
__device__ __forceinline__ void load_A2(const float *A_log, const Lane<CPL> &ln, float2 (&A2)[CPL][8]) {
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const float *a = A_log + size_t(ln.d + k) * kN;
#pragma unroll
        for (int g = 0; g < 8; ++g)
            A2[k][g] = ln.valid ? make_float2(-expf(a[2 * g]) * kLog2e, -expf(a[2 * g + 1]) * kLog2e)
                                : make_float2(0.0f, 0.0f);
    }
}

// Lane constants of chain c and the warp's decision for the lattice form.
template <int CPL>
__device__ __forceinline__ bool chain_lane(const SelArgs &a, int c, Lane<CPL> &ln) {
    const int lane = threadIdx.x & 31;
    ln.b = c % a.B;
    ln.d0 = (c / a.B) * 32 * CPL;
    ln.d = ln.d0 + CPL * lane;
    ln.valid = ln.d < a.D;
    bool on = true;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const float *al = a.A_log + size_t(ln.d + k) * kN;
        float a0 = 0.0f, mn = 0.0f;
        if (ln.valid) {
            a0 = -expf(al[0]) * kLog2e;
            mn = a0;
#pragma unroll
            for (int n = 0; n < kN; ++n) {
                const float v = -expf(al[n]) * kLog2e;
                mn = fmaxf(mn, v);
                on = on && fabsf(v - float(n + 1) * a0) <= 0x1p-20f * fabsf(v);
            }
        }
        if (k & 1) {
            ln.a20[k / 2].y = a0;
            ln.a2min[k / 2].y = mn;
        } else {
            ln.a20[k / 2].x = a0;
            ln.a2min[k / 2].x = mn;
        }
    }
#pragma unroll
    for (int j = 0; j < CPL / 2; ++j)
        ln.dsk[j] = (ln.valid && a.Dskip != nullptr) ? make_float2(a.Dskip[ln.d + 2 * j], a.Dskip[ln.d + 2 * j + 1])
                                                     : make_float2(0.0f, 0.0f);
    return __all_sync(kFull, on);
}

// ----------------------------------------------------------------------------
// Tiles
// ----------------------------------------------------------------------------
// B_t / C_t rows of a tile in fp32: bf16 I/O widens them into the warp's
// buffer (row q = B(16) | C(16)); fp32 I/O reads the TMA slots directly.
template <typename IO>
struct BCRows {
    static constexpr int STRIDE = sizeof(IO) == 2 ? 2 * kN : kN;
    const float *b, *c;
};

template <typename IO, int CPL>
__device__ __forceinline__ BCRows<IO> widen_bc(const unsigned char *st, float *bcf) {
    using Cf = SelCfg<IO, CPL>;
    if constexpr (sizeof(IO) == 2) {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int r = 0; r < kT / 8; ++r) {
            // 8 rows x (B lo, B hi, C lo, C hi) per pass
            const int q = 8 * r + (lane >> 2), part = lane & 3;
            const uint4 raw = *reinterpret_cast<const uint4 *>(
                st + (part < 2 ? Cf::OFF_B : Cf::OFF_C) + size_t(q * kN + 8 * (part & 1)) * 2);
            float4 *dst = reinterpret_cast<float4 *>(bcf + q * 2 * kN + 8 * part);
            dst[0] = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                                 __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u));
            dst[1] = make_float4(__uint_as_float(raw.z << 16), __uint_as_float(raw.z & 0xffff0000u),
                                 __uint_as_float(raw.w << 16), __uint_as_float(raw.w & 0xffff0000u));
        }
        __syncwarp();
        return BCRows<IO>{bcf, bcf + kN};
    } else {
        return BCRows<IO>{reinterpret_cast<const float *>(st + Cf::OFF_B),
                          reinterpret_cast<const float *>(st + Cf::OFF_C)};
    }
}

// One tile of the scan: steps t0 .. t0 + rows - 1 of the lane's channels
// (rows = 0 for a lane past D).  FULL: every row and channel is in range, so
// no step carries a predicate.
template <typename IO, int CPL, bool ACC, bool HAS_Z, bool SP, bool LAT, bool FULL>
__device__ __forceinline__ void tile_scan(const unsigned char *st, const BCRows<IO> &bc, float2 (&h)[CPL][8],
                                          const float2 (&A2)[CPL][8], const Lane<CPL> &ln,
                                          float2 (&dsum)[CPL / 2], IO *yp, int D, int rows) {
    using Cf = SelCfg<IO, CPL>;
    using V = Vec<IO, CPL>;
    using R = typename V::raw;
    constexpr int NP = CPL / 2;
    const int lane = threadIdx.x & 31;
    const R *xs = reinterpret_cast<const R *>(st) + lane;
    const R *ds = reinterpret_cast<const R *>(st + Cf::OFF_DT) + lane;
    const R *zs = reinterpret_cast<const R *>(st + Cf::OFF_Z) + lane;
#pragma unroll
    for (int q = 0; q < kT; ++q) {
        float2 xv[NP], dl[NP], u[NP];
        V::get(xs[q * 32], xv);
        V::get(ds[q * 32], dl);
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            if (SP) dl[j] = softplus2<ACC>(dl[j]);
            if (!FULL && q >= rows) dl[j] = make_float2(0.0f, 0.0f);   // rows past L: identity steps
            dsum[j] = __fadd2_rn(dsum[j], dl[j]);
            u[j] = __fmul2_rn(dl[j], xv[j]);
        }
        float2 Pk[CPL], Mk[CPL], uu[CPL], ya[CPL];
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            uu[2 * j] = make_float2(u[j].x, u[j].x);
            uu[2 * j + 1] = make_float2(u[j].y, u[j].y);
            if (LAT) {
                // (E, E^2) per channel; later pairs by (E^2, E^2)
                const float2 ar = __fmul2_rn(dl[j], ln.a20[j]);
                const float2 ar2 = __fadd2_rn(ar, ar);
                Pk[2 * j] = make_float2(ex2_approx(ar.x), ex2_approx(ar2.x));
                Pk[2 * j + 1] = make_float2(ex2_approx(ar.y), ex2_approx(ar2.y));
                Mk[2 * j] = make_float2(Pk[2 * j].y, Pk[2 * j].y);
                Mk[2 * j + 1] = make_float2(Pk[2 * j + 1].y, Pk[2 * j + 1].y);
            }
        }
#pragma unroll
        for (int k = 0; k < CPL; ++k) ya[k] = make_float2(0.0f, 0.0f);
        const float *brow = bc.b + q * BCRows<IO>::STRIDE;
        const float *crow = bc.c + q * BCRows<IO>::STRIDE;
#pragma unroll
        for (int g4 = 0; g4 < kN / 4; ++g4) {
            const float4 b4 = *reinterpret_cast<const float4 *>(brow + 4 * g4);
            const float4 c4 = *reinterpret_cast<const float4 *>(crow + 4 * g4);
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
                const int g = 2 * g4 + gg;
                const float2 bp = gg ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
                const float2 cp = gg ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
#pragma unroll
                for (int k = 0; k < CPL; ++k) {
                    float2 dec;
                    if (LAT) {
                        if (g > 0) Pk[k] = __fmul2_rn(Pk[k], Mk[k]);
                        dec = Pk[k];
                    } else {
                        const float dk = (k & 1) ? dl[k / 2].y : dl[k / 2].x;
                        const float2 ar = __fmul2_rn(make_float2(dk, dk), A2[k][g]);
                        dec = make_float2(ex2_approx(ar.x), ex2_approx(ar.y));
                    }
                    h[k][g] = __ffma2_rn(dec, h[k][g], __fmul2_rn(uu[k], bp));
                    ya[k] = __ffma2_rn(cp, h[k][g], ya[k]);
                }
            }
        }
        float2 o[NP], zv[NP];
        if (HAS_Z) V::get(zs[q * 32], zv);
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            o[j] = __ffma2_rn(ln.dsk[j], xv[j],
                              make_float2(ya[2 * j].x + ya[2 * j].y, ya[2 * j + 1].x + ya[2 * j + 1].y));
            if (HAS_Z) o[j] = __fmul2_rn(o[j], silu2<ACC>(zv[j]));
        }
        if (FULL || q < rows) st_cs(reinterpret_cast<R *>(yp + size_t(q) * D), V::put(o));
    }
}

// One tile of the backward warm-up of a piece that starts at step s: adds
// the tile's steps' contributions to the state just before s,
//   acc[n] += G_t^(n+1) u_t B_t[n]     (lattice; exp2(A2[n] S_t) in general)
// with G_t = exp(A[0] S_t) and S_t the sum of delta over steps t+1 .. s-1,
// which `lamb` carries in (the steps after this tile) and out (this tile
// added).  Each step's term is independent of the others, so there is no
// serial chain.  Every step of a tile before s lies inside the sequence.
// Bit g of `act` (warp-uniform) set: state pair g (n = 2g, 2g+1) still takes
// terms; a pair whose decay over S already fell below the cut-off for every
// channel of the warp is left out (on the lattice the active pairs are a
// prefix, as pair g decays 2g+1 times faster than state 0).
template <typename IO, int CPL, bool ACC, bool SP, bool LAT>
__device__ __forceinline__ void tile_back(const unsigned char *st, const BCRows<IO> &bc, float2 (&acc)[CPL][8],
                                          const float2 (&A2)[CPL][8], const Lane<CPL> &ln,
                                          float2 (&lamb)[CPL / 2], unsigned act) {
    using Cf = SelCfg<IO, CPL>;
    using V = Vec<IO, CPL>;
    using R = typename V::raw;
    constexpr int NP = CPL / 2;
    const int lane = threadIdx.x & 31;
    const R *xs = reinterpret_cast<const R *>(st) + lane;
    const R *ds = reinterpret_cast<const R *>(st + Cf::OFF_DT) + lane;
#pragma unroll
    for (int q = kT - 1; q >= 0; --q) {
        float2 xv[NP], dl[NP], u[NP], sa[NP];
        V::get(xs[q * 32], xv);
        V::get(ds[q * 32], dl);
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            if (SP) dl[j] = softplus2<ACC>(dl[j]);
            u[j] = __fmul2_rn(dl[j], xv[j]);
            sa[j] = lamb[j];                       // S_t: the steps after t
            lamb[j] = __fadd2_rn(lamb[j], dl[j]);
        }
        const float *brow = bc.b + q * BCRows<IO>::STRIDE;
        float2 Pk[CPL], Mk[CPL], uu[CPL];
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            uu[2 * j] = make_float2(u[j].x, u[j].x);
            uu[2 * j + 1] = make_float2(u[j].y, u[j].y);
            if (LAT) {
                const float2 ar = __fmul2_rn(sa[j], ln.a20[j]);
                const float2 ar2 = __fadd2_rn(ar, ar);
                Pk[2 * j] = make_float2(ex2_approx(ar.x), ex2_approx(ar2.x));
                Pk[2 * j + 1] = make_float2(ex2_approx(ar.y), ex2_approx(ar2.y));
                Mk[2 * j] = make_float2(Pk[2 * j].y, Pk[2 * j].y);
                Mk[2 * j + 1] = make_float2(Pk[2 * j + 1].y, Pk[2 * j + 1].y);
            }
        }
#pragma unroll
        for (int g4 = 0; g4 < kN / 4; ++g4) {
            if (!(act & (3u << (2 * g4)))) continue;
            const float4 b4 = *reinterpret_cast<const float4 *>(brow + 4 * g4);
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
                const int g = 2 * g4 + gg;
                if (!(act & (1u << g))) continue;
                const float2 bp = gg ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
#pragma unroll
                for (int k = 0; k < CPL; ++k) {
                    float2 dec;
                    if (LAT) {
                        if (g > 0) Pk[k] = __fmul2_rn(Pk[k], Mk[k]);
                        dec = Pk[k];
                    } else {
                        const float sk = (k & 1) ? sa[k / 2].y : sa[k / 2].x;
                        const float2 ar = __fmul2_rn(make_float2(sk, sk), A2[k][g]);
                        dec = make_float2(ex2_approx(ar.x), ex2_approx(ar.y));
                    }
                    acc[k][g] = __ffma2_rn(__fmul2_rn(uu[k], dec), bp, acc[k][g]);
                }
            }
        }
    }
}

// One tile of the carry correction of a piece: the TMA slot of x holds the
// piece's outputs y.  lam accumulates delta from the piece start; cy = the
// carry-in state.  y_t += silu(z_t) sum_n C_t[n] exp2(A2[n] lam_t) cy[n].
template <typename IO, int CPL, bool ACC, bool HAS_Z, bool SP, bool LAT, bool FULL>
__device__ __forceinline__ void tile_correct(const unsigned char *st, const BCRows<IO> &bc,
                                             const float2 (&cy)[CPL][8], const float2 (&A2)[CPL][8],
                                             const Lane<CPL> &ln, float2 (&lam)[CPL / 2], IO *yp, int D,
                                             int rows) {
    using Cf = SelCfg<IO, CPL>;
    using V = Vec<IO, CPL>;
    using R = typename V::raw;
    constexpr int NP = CPL / 2;
    const int lane = threadIdx.x & 31;
    const R *ys = reinterpret_cast<const R *>(st) + lane;
    const R *ds = reinterpret_cast<const R *>(st + Cf::OFF_DT) + lane;
    const R *zs = reinterpret_cast<const R *>(st + Cf::OFF_Z) + lane;
#pragma unroll
    for (int q = 0; q < kT; ++q) {
        float2 dl[NP];
        V::get(ds[q * 32], dl);
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            if (SP) dl[j] = softplus2<ACC>(dl[j]);
            if (!FULL && q >= rows) dl[j] = make_float2(0.0f, 0.0f);
            lam[j] = __fadd2_rn(lam[j], dl[j]);
        }
        const float *crow = bc.c + q * BCRows<IO>::STRIDE;
        float cr[CPL];
        if (LAT) {
            // sum_n c_n E^(n+1), c_n = C[n] cy[n], E = 2^(A2[0] lam): Horner in
            // E^2 on (even, odd) coefficient pairs
            float E[CPL];
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                const float2 ar = __fmul2_rn(lam[j], ln.a20[j]);
                E[2 * j] = ex2_approx(ar.x);
                E[2 * j + 1] = ex2_approx(ar.y);
            }
            float2 acc[CPL];
#pragma unroll
            for (int k = 0; k < CPL; ++k) acc[k] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int g = 7; g >= 0; --g) {
                const float2 cp = *reinterpret_cast<const float2 *>(crow + 2 * g);
#pragma unroll
                for (int k = 0; k < CPL; ++k) {
                    const float e2 = E[k] * E[k];
                    acc[k] = __ffma2_rn(acc[k], make_float2(e2, e2), __fmul2_rn(cp, cy[k][g]));
                }
            }
#pragma unroll
            for (int k = 0; k < CPL; ++k) cr[k] = E[k] * fmaf(E[k], acc[k].y, acc[k].x);
        } else {
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
                const float lk = (k & 1) ? lam[k / 2].y : lam[k / 2].x;
                float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const float2 ar = __fmul2_rn(make_float2(lk, lk), A2[k][g]);
                    const float2 dec = make_float2(ex2_approx(ar.x), ex2_approx(ar.y));
                    const float2 cp = *reinterpret_cast<const float2 *>(crow + 2 * g);
                    acc = __ffma2_rn(__fmul2_rn(cp, cy[k][g]), dec, acc);
                }
                cr[k] = acc.x + acc.y;
            }
        }
        float2 yv[NP], zv[NP], o[NP];
        V::get(ys[q * 32], yv);
        if (HAS_Z) V::get(zs[q * 32], zv);
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            const float2 corr = make_float2(cr[2 * j], cr[2 * j + 1]);
            o[j] = HAS_Z ? __ffma2_rn(silu2<ACC>(zv[j]), corr, yv[j]) : __fadd2_rn(yv[j], corr);
        }
        if (FULL || q < rows) st_cs(reinterpret_cast<R *>(yp + size_t(q) * D), V::put(o));
    }
}

// ----------------------------------------------------------------------------
// The warp's TMA ring
// ----------------------------------------------------------------------------
struct Maps {
    const CUtensorMap *x, *dt, *z, *B, *C, *y;
};

struct Ring {
    unsigned char *base;
    uint64_t *full;
    uint32_t it;   // tiles taken through the ring so far: stage it % STAGES, parity (it / STAGES) & 1
    bool ok;       // false once a wait ran out
};

// Lane 0: copies tile t0 of chain (b, d0) into ring slot `slot`; slot 0 of
// the stage gets x (scan) or y (correction).
// KIND 0: x (or y), dt, z, B, C; KIND 1: x, dt, B (the backward warm-up).
template <typename IO, int CPL, bool HAS_Z, int KIND = 0>
__device__ __forceinline__ void issue_tile(const Ring &rg, uint32_t slot, const CUtensorMap *m0, const Maps &m,
                                           int b, int d0, int t0) {
    using Cf = SelCfg<IO, CPL>;
    const uint32_t s = slot % Cf::STAGES;
    unsigned char *st = rg.base + s * Cf::STAGE;
    uint64_t *bar = &rg.full[s];
    constexpr uint32_t bytes =
        KIND == 1 ? uint32_t(2 * Cf::SLOT + Cf::SLOT_N) : uint32_t((HAS_Z ? 3 : 2) * Cf::SLOT + 2 * Cf::SLOT_N);
    // the lanes' generic reads of this stage's previous tile come first
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, bytes);
    if (KIND == 1) {
        tma_load_3d(st, m.x, bar, d0, t0, b);
        tma_load_3d(st + Cf::OFF_DT, m.dt, bar, d0, t0, b);
        tma_load_3d(st + Cf::OFF_B, m.B, bar, 0, t0, b);
        return;
    }
    tma_load_3d(st, m0, bar, d0, t0, b);
    tma_load_3d(st + Cf::OFF_DT, m.dt, bar, d0, t0, b);
    if (HAS_Z) tma_load_3d(st + Cf::OFF_Z, m.z, bar, d0, t0, b);
    tma_load_3d(st + Cf::OFF_B, m.B, bar, 0, t0, b);
    tma_load_3d(st + Cf::OFF_C, m.C, bar, 0, t0, b);
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(kFull, ok)) return true;
    if (!ok) ok = mbar_wait_bounded(bar, parity, limit_ns);
    return __all_sync(kFull, ok);
}

// Streams n tiles of chain (b, d0) through the ring -- v0, v0 + 1, ... (DIR
// = 1) or v0, v0 - 1, ... (DIR = -1) -- and calls body(stage, bc, t0) for
// each; body returns false to stop early.  Tiles already in flight when it
// stops are waited for, so no copy is pending when the ring is reused or the
// warp exits.  KIND 1 copies x, dt and B only.
template <typename IO, int CPL, bool HAS_Z, int KIND = 0, int DIR = 1, typename Body>
__device__ __forceinline__ void stream_tiles(Ring &rg, const CUtensorMap *m0, const Maps &m, int b, int d0,
                                             int v0, int n, uint64_t timeout_ns, const StatusRef &st,
                                             Body &&body) {
    using Cf = SelCfg<IO, CPL>;
    const int lane = threadIdx.x & 31;
    float *bcf = reinterpret_cast<float *>(rg.base + Cf::OFF_BCF);
    if (n <= 0 || !rg.ok) return;
    const uint32_t it0 = rg.it;
    int issued = n < Cf::STAGES - 1 ? n : Cf::STAGES - 1;
    if (lane == 0)
        for (int k = 0; k < issued; ++k)
            issue_tile<IO, CPL, HAS_Z, KIND>(rg, it0 + k, m0, m, b, d0, (v0 + DIR * k) * kT);
    int k = 0;
    while (k < n) {
        if (issued < n) {   // into the stage the previous tile released
            if (lane == 0) issue_tile<IO, CPL, HAS_Z, KIND>(rg, it0 + issued, m0, m, b, d0, (v0 + DIR * issued) * kT);
            ++issued;
        }
        const uint32_t slot = it0 + k;
        const uint32_t s = slot % Cf::STAGES;
        ++k;
        if (!warp_wait(&rg.full[s], (slot / Cf::STAGES) & 1, timeout_ns)) {
            if (lane == 0) status_report(st, LR_ERR_TIMEOUT);
            rg.ok = false;
            break;
        }
        const unsigned char *stg = rg.base + s * Cf::STAGE;
        const BCRows<IO> bc = widen_bc<IO, CPL>(stg, bcf);
        const bool go = body(stg, bc, (v0 + DIR * (k - 1)) * kT);
        __syncwarp();
        if (!go) break;
    }
    for (; k < issued; ++k) {   // drain
        const uint32_t slot = it0 + k;
        if (rg.ok && !warp_wait(&rg.full[slot % Cf::STAGES], (slot / Cf::STAGES) & 1, timeout_ns)) {
            if (lane == 0) status_report(st, LR_ERR_TIMEOUT);
            rg.ok = false;
        }
    }
    rg.it = it0 + issued;
}

template <int CPL>
__device__ __forceinline__ void write_h_final(const SelArgs &a, const Lane<CPL> &ln, const float2 (&h)[CPL][8]) {
    if (a.h_final == nullptr || !ln.valid) return;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        float4 *dst = reinterpret_cast<float4 *>(a.h_final + (size_t(ln.b) * a.D + ln.d + k) * kN);
#pragma unroll
        for (int g = 0; g < 4; ++g)
            dst[g] = make_float4(h[k][2 * g].x, h[k][2 * g].y, h[k][2 * g + 1].x, h[k][2 * g + 1].y);
    }
}

template <int CPL>
__device__ __forceinline__ void load_h0(const SelArgs &a, const Lane<CPL> &ln, float2 (&h)[CPL][8]) {
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const float4 *src = reinterpret_cast<const float4 *>(a.h0 + (size_t(ln.b) * a.D + ln.d + k) * kN);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float4 v = (a.h0 != nullptr && ln.valid) ? src[g] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            h[k][2 * g] = make_float2(v.x, v.y);
            h[k][2 * g + 1] = make_float2(v.z, v.w);
        }
    }
}

// ----------------------------------------------------------------------------
// Pieces
// ----------------------------------------------------------------------------
// The scan of tiles [lo, hi) of chain (ln.b, ln.d0) from state h; dsum gets
// the sum of delta over them.
template <typename IO, int CPL, bool ACC, bool HAS_Z, bool SP, bool LAT>
__device__ __forceinline__ void scan_piece(Ring &rg, const Maps &m, const SelArgs &a, const Lane<CPL> &ln,
                                           int lo, int hi, float2 (&h)[CPL][8], float2 (&dsum)[CPL / 2]) {
    float2 A2[CPL][8];
    if (!LAT) load_A2<CPL>(a.A_log, ln, A2);
    IO *y = static_cast<IO *>(a.y);
    const bool full_ch = ln.d0 + 32 * CPL <= a.D;
    stream_tiles<IO, CPL, HAS_Z>(rg, m.x, m, ln.b, ln.d0, lo, hi - lo, a.timeout_ns, a.st,
                                 [&](const unsigned char *stg, const BCRows<IO> &bc, int t0) {
                                     IO *yp = y + (size_t(ln.b) * a.L + t0) * a.D + ln.d;
                                     if (full_ch && t0 + kT <= a.L) {
                                         tile_scan<IO, CPL, ACC, HAS_Z, SP, LAT, true>(stg, bc, h, A2, ln, dsum,
                                                                                       yp, a.D, kT);
                                     } else {
                                         const int rows = ln.valid ? min(kT, a.L - t0) : 0;
                                         tile_scan<IO, CPL, ACC, HAS_Z, SP, LAT, false>(stg, bc, h, A2, ln,
                                                                                        dsum, yp, a.D, rows);
                                     }
                                     return true;
                                 });
}

// The backward warm-up of a piece starting at tile lo: the state just before
// it, summed over the preceding steps from the latest back (tile_back) until,
// for every channel of the warp, the slowest decay since then has fallen
// below 2^CUT -- the rest of the history then contributes less than that
// share of its size -- or the chain start is reached (the initial state,
// decayed over the whole range, is then added and the result is exact).
// Returns false (h untouched) when `cap` tiles did not reach either.
template <typename IO, int CPL, bool ACC, bool HAS_Z, bool SP, bool LAT>
__device__ __forceinline__ bool warm_up(Ring &rg, const Maps &m, const SelArgs &a, const Lane<CPL> &ln, int lo,
                                        int cap, float2 (&h)[CPL][8]) {
    using Cf = SelCfg<IO, CPL>;
    float2 A2[CPL][8], acc[CPL][8], lamb[CPL / 2];
    if (!LAT) load_A2<CPL>(a.A_log, ln, A2);
#pragma unroll
    for (int k = 0; k < CPL; ++k)
#pragma unroll
        for (int g = 0; g < 8; ++g) acc[k][g] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < CPL / 2; ++j) lamb[j] = make_float2(0.0f, 0.0f);
    const int n = lo < cap ? lo : cap;
    int walked = 0;
    bool reached = false;
    stream_tiles<IO, CPL, HAS_Z, 1, -1>(rg, m.x, m, ln.b, ln.d0, lo - 1, n, a.timeout_ns, a.st,
                                        [&](const unsigned char *stg, const BCRows<IO> &bc, int) {
                                            // pairs whose slowest decay over the steps
                                            // already summed is still above the cut-off
                                            unsigned bits = 0;
#pragma unroll
                                            for (int g = 0; g < 8; ++g) {
                                                bool on = false;
#pragma unroll
                                                for (int k = 0; k < CPL; ++k) {
                                                    const float lk = (k & 1) ? lamb[k / 2].y : lamb[k / 2].x;
                                                    const float ak = LAT ? float(2 * g + 1) *
                                                                               ((k & 1) ? ln.a20[k / 2].y
                                                                                        : ln.a20[k / 2].x)
                                                                         : fmaxf(A2[k][g].x, A2[k][g].y);
                                                    on = on || ak * lk > Cf::CUT;
                                                }
                                                bits |= on ? 1u << g : 0u;
                                            }
                                            const unsigned act = __reduce_or_sync(kFull, ln.valid ? bits : 0u);
                                            tile_back<IO, CPL, ACC, SP, LAT>(stg, bc, acc, A2, ln, lamb, act);
                                            ++walked;
                                            bool done = true;
#pragma unroll
                                            for (int j = 0; j < CPL / 2; ++j)
                                                done = done && ln.a2min[j].x * lamb[j].x <= Cf::CUT &&
                                                       ln.a2min[j].y * lamb[j].y <= Cf::CUT;
                                            reached = __all_sync(kFull, done || !ln.valid);
                                            return !reached;
                                        });
    if (!rg.ok || !(reached || walked == lo)) return false;
    if (walked == lo) {
        // the whole prefix: add the initial state decayed over it
        float2 h0v[CPL][8];
        if (LAT) load_A2<CPL>(a.A_log, ln, A2);
        load_h0<CPL>(a, ln, h0v);
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            const float lk = (k & 1) ? lamb[k / 2].y : lamb[k / 2].x;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const float2 dec = make_float2(pow2_t<ACC>(A2[k][g].x * lk), pow2_t<ACC>(A2[k][g].y * lk));
                acc[k][g] = __ffma2_rn(dec, h0v[k][g], acc[k][g]);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < CPL; ++k)
#pragma unroll
        for (int g = 0; g < 8; ++g) h[k][g] = acc[k][g];
    return true;
}

// The carry correction of tiles [lo, hi) of a chain, stopping once every
// remaining term is below 2^CUT of its value at the piece start.
template <typename IO, int CPL, bool ACC, bool HAS_Z, bool SP, bool LAT>
__device__ __forceinline__ void correct_piece(Ring &rg, const Maps &m, const SelArgs &a, const Lane<CPL> &ln,
                                              int lo, int hi, const float2 (&cy)[CPL][8]) {
    using Cf = SelCfg<IO, CPL>;
    float2 A2[CPL][8];
    if (!LAT) load_A2<CPL>(a.A_log, ln, A2);
    IO *y = static_cast<IO *>(a.y);
    const bool full_ch = ln.d0 + 32 * CPL <= a.D;
    float2 lam[CPL / 2];
#pragma unroll
    for (int j = 0; j < CPL / 2; ++j) lam[j] = make_float2(0.0f, 0.0f);
    stream_tiles<IO, CPL, HAS_Z>(rg, m.y, m, ln.b, ln.d0, lo, hi - lo, a.timeout_ns, a.st,
                                 [&](const unsigned char *stg, const BCRows<IO> &bc, int t0) {
                                     IO *yp = y + (size_t(ln.b) * a.L + t0) * a.D + ln.d;
                                     if (full_ch && t0 + kT <= a.L) {
                                         tile_correct<IO, CPL, ACC, HAS_Z, SP, LAT, true>(stg, bc, cy, A2, ln,
                                                                                          lam, yp, a.D, kT);
                                     } else {
                                         const int rows = ln.valid ? min(kT, a.L - t0) : 0;
                                         tile_correct<IO, CPL, ACC, HAS_Z, SP, LAT, false>(stg, bc, cy, A2, ln,
                                                                                           lam, yp, a.D, rows);
                                     }
                                     bool done = true;
#pragma unroll
                                     for (int j = 0; j < CPL / 2; ++j)
                                         done = done && ln.a2min[j].x * lam[j].x <= Cf::CUT &&
                                                ln.a2min[j].y * lam[j].y <= Cf::CUT;
                                     return !__all_sync(kFull, done || !ln.valid);
                                 });
}

// Descriptor rows of warp `wi`: row r holds one value per channel of the
// chain; the lane's CPL channels are adjacent.
template <int CPL>
__device__ __forceinline__ float *agg_row(const SelArgs &a, int wi, int r) {
    return a.agg + (size_t(wi) * (kN + 1) + r) * (32 * CPL) + CPL * (threadIdx.x & 31);
}
template <int CPL>
__device__ __forceinline__ float *incl_row(const SelArgs &a, int wi, int r) {
    return a.incl + (size_t(wi) * kN + r) * (32 * CPL) + CPL * (threadIdx.x & 31);
}

__device__ __forceinline__ void publish(const SelArgs &a, int wi, uint32_t flag) {
    __threadfence();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) st_release_gpu(&a.flags[wi], flag);
}

// State n of channel k lives at row r0 + n, column k.
template <int CPL>
__device__ __forceinline__ void write_rows(float *(*row)(const SelArgs &, int, int), const SelArgs &a, int wi,
                                           int r0, const float2 (&h)[CPL][8]) {
#pragma unroll
    for (int n = 0; n < kN; ++n) {
        float *p = row(a, wi, r0 + n);
#pragma unroll
        for (int k = 0; k < CPL; ++k) p[k] = (n & 1) ? h[k][n / 2].y : h[k][n / 2].x;
    }
}

template <int CPL>
__device__ __forceinline__ void read_rows(float *(*row)(const SelArgs &, int, int), const SelArgs &a, int wi,
                                          int r0, float2 (&h)[CPL][8]) {
#pragma unroll
    for (int n = 0; n < kN; ++n) {
        const float *p = row(a, wi, r0 + n);
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            const float v = __ldcg(p + k);
            if (n & 1) h[k][n / 2].y = v;
            else h[k][n / 2].x = v;
        }
    }
}

// The carry-in of warp wi's first piece: the state at the end of warp
// wi - 1's last piece, composed back over aggregates until an inclusive
// state is found.  A2: the channels' exponents (general form).
template <int CPL, bool ACC>
__device__ __forceinline__ void look_back(const SelArgs &a, int wi, const float2 (&A2)[CPL][8],
                                          float2 (&carry)[CPL][8]) {
    const int lane = threadIdx.x & 31;
    float acc_d[CPL];
    float2 acc_h[CPL][8];
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        acc_d[k] = 0.0f;
#pragma unroll
        for (int g = 0; g < 8; ++g) acc_h[k][g] = make_float2(0.0f, 0.0f);
    }
    for (int v = wi - 1; v >= 0; --v) {
        uint32_t fv = 0;
        if (lane == 0) fv = poll_flag(&a.flags[v], a.timeout_ns);
        fv = __shfl_sync(kFull, fv, 0);
        __syncwarp();
        float2 s[CPL][8];
        if (fv == kFlagInclusive) {
            read_rows<CPL>(incl_row<CPL>, a, v, 0, s);
#pragma unroll
            for (int k = 0; k < CPL; ++k)
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const float2 dec = make_float2(pow2_t<ACC>(A2[k][g].x * acc_d[k]),
                                                   pow2_t<ACC>(A2[k][g].y * acc_d[k]));
                    carry[k][g] = __ffma2_rn(dec, s[k][g], acc_h[k][g]);
                }
            return;
        }
        if (fv == kFlagAggregate) {
            read_rows<CPL>(agg_row<CPL>, a, v, 1, s);
            const float *d = agg_row<CPL>(a, v, 0);
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const float2 dec = make_float2(pow2_t<ACC>(A2[k][g].x * acc_d[k]),
                                                   pow2_t<ACC>(A2[k][g].y * acc_d[k]));
                    acc_h[k][g] = __ffma2_rn(dec, s[k][g], acc_h[k][g]);
                }
                acc_d[k] += __ldcg(d + k);
            }
            continue;
        }
        if (lane == 0) status_report(a.st, LR_ERR_TIMEOUT);   // predecessor never published
        break;
    }
#pragma unroll
    for (int k = 0; k < CPL; ++k)
#pragma unroll
        for (int g = 0; g < 8; ++g) carry[k][g] = acc_h[k][g];
}

// Warp owning flat tile f.
__device__ __forceinline__ long long owner_of(long long f, long long F, int W) {
    return ((f + 1) * W + F - 1) / F - 1;
}


// ----------------------------------------------------------------------------
// Ranges and work stealing (warm-up mode)
// ----------------------------------------------------------------------------
// A warp whose state is exact at the start of its share runs the share as a
// range: a 64-bit word per warp holds the range's claim cursor and end, the
// warp claims kClaim tiles at a time (atomicAdd on the cursor, issued a
// chunk ahead), and a warp that has run out of work takes the back half of
// the largest unclaimed remainder it finds (atomicCAS on the end, which
// fails if the owner claimed in between), warms its state up to the start
// of that half and runs it as its own range.  So no tile is run twice or
// left out, and the warps of an SM stay busy until the whole list is done
// instead of finishing one by one.  Every range lies inside one warp's
// original share; whoever runs the last tile of a share publishes its
// inclusive state for the look-back of a successor that could not warm up.
__device__ __forceinline__ unsigned long long range_word(long long p, long long e) {
    return (static_cast<unsigned long long>(e) << 32) | static_cast<unsigned long long>(p);
}
__device__ __forceinline__ void range_split(unsigned long long w, long long &p, long long &e) {
    p = static_cast<long long>(w & 0xffffffffull);
    e = static_cast<long long>(w >> 32);
}

// The tiles of chain c from local tile lo that the warp's range holds, claimed
// on the way; returns how many it ran.  ce: the claimed end (flat), more:
// whether the range may still hold unclaimed tiles.
template <typename IO, int CPL, bool ACC, bool HAS_Z, bool SP, bool LAT>
__device__ __forceinline__ int scan_claimed(Ring &rg, const Maps &m, const SelArgs &a, int wi, const Lane<CPL> &ln,
                                            long long cbase, int lo, long long &ce, bool &more,
                                            float2 (&h)[CPL][8]) {
    using Cf = SelCfg<IO, CPL>;
    const int lane = threadIdx.x & 31;
    float2 A2[CPL][8], dsum[CPL / 2];
    if (!LAT) load_A2<CPL>(a.A_log, ln, A2);
#pragma unroll
    for (int j = 0; j < CPL / 2; ++j) dsum[j] = make_float2(0.0f, 0.0f);
    IO *y = static_cast<IO *>(a.y);
    const bool full_ch = ln.d0 + 32 * CPL <= a.D;
    float *bcf = reinterpret_cast<float *>(rg.base + Cf::OFF_BCF);
    // chain-local tile indices: lim = the claimed end inside this chain, cl =
    // the claimed end (may lie past the chain); both change only when a
    // claim returns
    const long long cend = cbase + a.ntt;
    int lim = static_cast<int>((ce < cend ? ce : cend) - cbase);
    int cl = static_cast<int>((ce < cend + 2 * kClaim ? ce : cend + 2 * kClaim) - cbase);
    const uint32_t it0 = rg.it;
    int t = lo;   // next tile to run
    int ti = lo + (lim - lo < Cf::STAGES - 1 ? lim - lo : Cf::STAGES - 1);   // next tile to copy
    if (lane == 0)
        for (int j = lo; j < ti; ++j) issue_tile<IO, CPL, HAS_Z>(rg, it0 + (j - lo), m.x, m, ln.b, ln.d0, j * kT);
    unsigned long long pend = 0;
    bool pending = false;
    for (;;) {
        if (pending) {   // the claim issued during the previous tile
            long long p, e;
            range_split(__shfl_sync(kFull, pend, 0), p, e);
            if (p < e)
                ce = p + kClaim < e ? p + kClaim : e;
            else
                more = false;
            lim = static_cast<int>((ce < cend ? ce : cend) - cbase);
            cl = static_cast<int>((ce < cend + 2 * kClaim ? ce : cend + 2 * kClaim) - cbase);
            pending = false;
        }
        if (t >= lim) break;
        if (ti < lim) {
            if (lane == 0) issue_tile<IO, CPL, HAS_Z>(rg, it0 + (ti - lo), m.x, m, ln.b, ln.d0, ti * kT);
            ++ti;
        }
        if (more && cl - t < 2 * kClaim) {   // claim ahead; read after this tile
            if (lane == 0) pend = atomicAdd(a.ctl + wi, static_cast<unsigned long long>(kClaim));
            pending = true;
        }
        const uint32_t slot = it0 + (t - lo);
        const uint32_t s = slot % Cf::STAGES;
        if (!warp_wait(&rg.full[s], (slot / Cf::STAGES) & 1, a.timeout_ns)) {
            if (lane == 0) status_report(a.st, LR_ERR_TIMEOUT);
            rg.ok = false;
            break;
        }
        const unsigned char *stg = rg.base + s * Cf::STAGE;
        const BCRows<IO> bc = widen_bc<IO, CPL>(stg, bcf);
        const int t0 = t * kT;
        IO *yp = y + (size_t(ln.b) * a.L + t0) * a.D + ln.d;
        if (full_ch && t0 + kT <= a.L) {
            tile_scan<IO, CPL, ACC, HAS_Z, SP, LAT, true>(stg, bc, h, A2, ln, dsum, yp, a.D, kT);
        } else {
            const int rows = ln.valid ? min(kT, a.L - t0) : 0;
            tile_scan<IO, CPL, ACC, HAS_Z, SP, LAT, false>(stg, bc, h, A2, ln, dsum, yp, a.D, rows);
        }
        __syncwarp();
        ++t;
    }
    if (pending) more = false;   // only after a failed wait
    for (int j = t + (rg.ok ? 0 : 1); j < ti; ++j) {   // drain (after a failed wait)
        const uint32_t slot = it0 + (j - lo);
        if (rg.ok && !warp_wait(&rg.full[slot % Cf::STAGES], (slot / Cf::STAGES) & 1, a.timeout_ns)) {
            if (lane == 0) status_report(a.st, LR_ERR_TIMEOUT);
            rg.ok = false;
        }
    }
    const int issued = ti - lo, k = t - lo;
    rg.it = it0 + issued;
    return rg.ok ? k : 0;
}

// Runs the warp's range from flat tile cur; h is the exact state before cur
// (or anything when cur starts a chain).
template <typename IO, int CPL, bool ACC, bool HAS_Z, bool SP>
__device__ __forceinline__ void run_range(Ring &rg, const Maps &m, const SelArgs &a, int wi, long long cur,
                                          float2 (&h)[CPL][8]) {
    const int lane = threadIdx.x & 31;
    long long ce = cur;
    bool more = true;
    long long last = -1;
    while (rg.ok) {
        if (cur >= ce) {   // nothing claimed ahead: claim now
            if (!more) break;
            unsigned long long r = 0;
            if (lane == 0) r = atomicAdd(a.ctl + wi, static_cast<unsigned long long>(kClaim));
            long long p, e;
            range_split(__shfl_sync(kFull, r, 0), p, e);
            if (p >= e) break;
            ce = p + kClaim < e ? p + kClaim : e;
        }
        const int c = static_cast<int>(cur / a.ntt);
        const long long cbase = static_cast<long long>(c) * a.ntt;
        const int lo = static_cast<int>(cur - cbase);
        Lane<CPL> ln;
        const bool lat = chain_lane<CPL>(a, c, ln);
        if (lo == 0) load_h0<CPL>(a, ln, h);
        const int n = lat ? scan_claimed<IO, CPL, ACC, HAS_Z, SP, true>(rg, m, a, wi, ln, cbase, lo, ce, more, h)
                          : scan_claimed<IO, CPL, ACC, HAS_Z, SP, false>(rg, m, a, wi, ln, cbase, lo, ce, more, h);
        if (n <= 0) break;
        cur += n;
        last = cur - 1;
        if (cur == cbase + a.ntt) write_h_final<CPL>(a, ln, h);
    }
    if (last < 0 || !rg.ok) return;
    // the last tile of a share that ends inside its chain: publish the state
    const int u = static_cast<int>(owner_of(last, a.F, a.W));
    const long long f1u = a.F * (u + 1) / a.W;
    if (last + 1 == f1u && f1u % a.ntt != 0) {
        write_rows<CPL>(incl_row<CPL>, a, u, 0, h);
        publish(a, u, kFlagInclusive);
    }
}

// Takes the back half of the largest unclaimed remainder among 128 warps
// sampled across the grid; true with [m, e) now this warp's range.  (The
// half split measured best: a thief pays a warm-up of its own before it
// starts, and splits that try to balance that cost, or give the thief more
// than half, ran slower.)
__device__ __forceinline__ bool steal_range(const SelArgs &a, int wi, int attempt, long long &m_out, long long &e_out) {
    const int lane = threadIdx.x & 31;
    long long best = 0;
    int bv = -1;
    unsigned long long bw = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int v = static_cast<int>((wi + 1 + attempt + (static_cast<long long>(lane + 32 * j) * a.W) / 128) % a.W);
        const unsigned long long w = __ldcg(a.ctl + v);
        long long p, e;
        range_split(w, p, e);
        if (v != wi && e - p > best) {
            best = e - p;
            bv = v;
            bw = w;
        }
    }
    const unsigned top = __reduce_max_sync(kFull, static_cast<unsigned>(best));
    if (top < static_cast<unsigned>(kMinSteal)) return false;
    const int who = __ffs(__ballot_sync(kFull, static_cast<unsigned>(best) == top)) - 1;
    long long p, e;
    range_split(bw, p, e);
    const long long mid = p + (e - p) / 2;
    int ok = 0;
    if (lane == who) ok = atomicCAS(a.ctl + bv, bw, range_word(p, mid)) == bw;
    ok = __shfl_sync(kFull, ok, who);
    if (!ok) return false;
    m_out = __shfl_sync(kFull, mid, who);
    e_out = __shfl_sync(kFull, e, who);
    if (lane == 0) atomicExch(a.ctl + wi, range_word(m_out, e_out));
    return true;
}

template <typename IO, int CPL, bool ACC, bool HAS_Z, bool SP>
__device__ __forceinline__ void scan_piece_any(bool lat, Ring &rg, const Maps &m, const SelArgs &a,
                                               const Lane<CPL> &ln, int lo, int hi, float2 (&h)[CPL][8],
                                               float2 (&dsum)[CPL / 2]) {
    if (lat)
        scan_piece<IO, CPL, ACC, HAS_Z, SP, true>(rg, m, a, ln, lo, hi, h, dsum);
    else
        scan_piece<IO, CPL, ACC, HAS_Z, SP, false>(rg, m, a, ln, lo, hi, h, dsum);
}

// A warp's share as static pieces: the end of one chain (warmed up, or run
// from zero with its carry by look-back and correction), whole chains, the
// start of the next.  try_warm false: the first piece takes the look-back
// path without trying the warm-up.
template <typename IO, int CPL, bool ACC, bool HAS_Z, bool SP>
__device__ __forceinline__ void static_share(Ring &rg, const Maps &m, const SelArgs &a, int wi, bool try_warm) {
    constexpr int NP = CPL / 2;
    const long long f0 = a.F * wi / a.W, f1 = a.F * (wi + 1) / a.W;

    // the first piece: the end of chain c1 from tile lo1
    const int c1 = static_cast<int>(f0 / a.ntt);
    const int lo1 = static_cast<int>(f0 - static_cast<long long>(c1) * a.ntt);
    const int hi1 = static_cast<int>(min(static_cast<long long>(a.ntt), lo1 + (f1 - f0)));
    const bool single = f0 + (hi1 - lo1) >= f1;
    Lane<CPL> ln;
    const bool lat = chain_lane<CPL>(a, c1, ln);
    float2 h[CPL][8], dsum[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) dsum[j] = make_float2(0.0f, 0.0f);
    if (lo1 == 0) {
        load_h0<CPL>(a, ln, h);
    } else {
#pragma unroll
        for (int k = 0; k < CPL; ++k)
#pragma unroll
            for (int g = 0; g < 8; ++g) h[k][g] = make_float2(0.0f, 0.0f);
    }
    // a piece that starts inside its chain first warms up its state over the
    // preceding steps where the carry still counts, when that horizon is
    // short enough; otherwise it runs from zero and takes its carry by
    // look-back and correction below
    bool warmed = lo1 == 0;   // h carries the true state
    if (try_warm && !warmed && a.warmup_tiles > 0)
        warmed = lat ? warm_up<IO, CPL, ACC, HAS_Z, SP, true>(rg, m, a, ln, lo1, a.warmup_tiles, h)
                     : warm_up<IO, CPL, ACC, HAS_Z, SP, false>(rg, m, a, ln, lo1, a.warmup_tiles, h);
    scan_piece_any<IO, CPL, ACC, HAS_Z, SP>(lat, rg, m, a, ln, lo1, hi1, h, dsum);
    const long long ord1 = wi - owner_of(static_cast<long long>(c1) * a.ntt, a.F, a.W);
    const bool withhold = single && ord1 == a.withheld;
    if (warmed) {
        if (hi1 == a.ntt) {
            write_h_final<CPL>(a, ln, h);
        } else if (single && !withhold) {
            write_rows<CPL>(incl_row<CPL>, a, wi, 0, h);
            publish(a, wi, kFlagInclusive);
        }
    } else {
        // keep the piece's aggregate in this warp's descriptor; announce it
        // when it is the warp's last piece and a successor continues the chain
        float *d = agg_row<CPL>(a, wi, 0);
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            d[2 * j] = dsum[j].x;
            d[2 * j + 1] = dsum[j].y;
        }
        write_rows<CPL>(agg_row<CPL>, a, wi, 1, h);
        if (single && hi1 < a.ntt && !withhold) publish(a, wi, kFlagAggregate);
    }

    // whole chains, then the start of the next
    for (long long f = f0 + (hi1 - lo1); f < f1;) {
        const int c = static_cast<int>(f / a.ntt);
        const int hi = static_cast<int>(min(static_cast<long long>(a.ntt), f1 - f));
        Lane<CPL> lc;
        const bool lt = chain_lane<CPL>(a, c, lc);
        load_h0<CPL>(a, lc, h);
        scan_piece_any<IO, CPL, ACC, HAS_Z, SP>(lt, rg, m, a, lc, 0, hi, h, dsum);
        if (hi == a.ntt) {
            write_h_final<CPL>(a, lc, h);
        } else {
            write_rows<CPL>(incl_row<CPL>, a, wi, 0, h);
            publish(a, wi, kFlagInclusive);
        }
        f += hi;
    }

    if (!warmed) {
        // carry-in of the first piece, its true final state, the correction
        float2 A2[CPL][8], carry[CPL][8];
        load_A2<CPL>(a.A_log, ln, A2);
        __syncwarp();
        float dsk[CPL];
        const float *d = agg_row<CPL>(a, wi, 0);
#pragma unroll
        for (int k = 0; k < CPL; ++k) dsk[k] = __ldcg(d + k);
        read_rows<CPL>(agg_row<CPL>, a, wi, 1, h);
        look_back<CPL, ACC>(a, wi, A2, carry);
#pragma unroll
        for (int k = 0; k < CPL; ++k)
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const float2 dec = make_float2(pow2_t<ACC>(A2[k][g].x * dsk[k]), pow2_t<ACC>(A2[k][g].y * dsk[k]));
                h[k][g] = __ffma2_rn(dec, carry[k][g], h[k][g]);
            }
        if (hi1 == a.ntt) {
            write_h_final<CPL>(a, ln, h);
        } else if (single && !withhold) {
            write_rows<CPL>(incl_row<CPL>, a, wi, 0, h);
            publish(a, wi, kFlagInclusive);
        }
        // the piece's outputs were written by this warp's lanes: make them
        // visible to the TMA reads of the correction
        fence_proxy_async_global();
        __syncwarp();
        if (lat)
            correct_piece<IO, CPL, ACC, HAS_Z, SP, true>(rg, m, a, ln, lo1, hi1, carry);
        else
            correct_piece<IO, CPL, ACC, HAS_Z, SP, false>(rg, m, a, ln, lo1, hi1, carry);
    }
}

// A warp's share in the stealing kernel: the own share as a range after its
// warm-up (left to the second launch, which takes its carry by look-back,
// when the warm-up does not reach its horizon), then ranges taken from other
// warps, each warmed up however far back it needs, until no range is left
// worth splitting.
template <typename IO, int CPL, bool ACC, bool HAS_Z, bool SP>
__device__ __forceinline__ void steal_share(Ring &rg, const Maps &m, const SelArgs &a, int wi) {
    const int lane = threadIdx.x & 31;
    const long long f0 = a.F * wi / a.W, f1 = a.F * (wi + 1) / a.W;
    float2 h[CPL][8];
    long long r0 = f0, e0 = f1;   // the range to run next: the own share first
    bool own = true;
    for (int attempt = 0; rg.ok;) {
        const int c = static_cast<int>(r0 / a.ntt);
        const int lo = static_cast<int>(r0 - static_cast<long long>(c) * a.ntt);
        bool ok = true;
        if (lo > 0) {   // the state before the range (a stolen one: however far back it takes)
            Lane<CPL> ln;
            const bool lat = chain_lane<CPL>(a, c, ln);
            const int cap = own ? a.warmup_tiles : lo;
            ok = lat ? warm_up<IO, CPL, ACC, HAS_Z, SP, true>(rg, m, a, ln, lo, cap, h)
                     : warm_up<IO, CPL, ACC, HAS_Z, SP, false>(rg, m, a, ln, lo, cap, h);
        }
        if (!rg.ok) return;
        if (ok) {
            // the own share becomes a range that idle warps may split
            if (own && lane == 0) atomicExch(a.ctl + wi, range_word(f0, f1));
            run_range<IO, CPL, ACC, HAS_Z, SP>(rg, m, a, wi, r0, h);
        } else if (lane == 0) {
            a.defer[wi] = 1;   // the own share's horizon is too long: the second launch runs it
        }
        own = false;
        int misses = 0;
        while (rg.ok && misses < 4 && !steal_range(a, wi, attempt++, r0, e0)) ++misses;
        if (misses >= 4) return;
    }
}

// STEAL: ranges with work stealing (warm-up mode); else static shares.
template <typename IO, bool ACC, bool HAS_Z, bool SP, bool STEAL, int CPL = cpl_of<IO>()>
__global__ void __launch_bounds__(kWpb * 32, SelCfg<IO, CPL>::MINB)
    selective_scan_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dt,
                          const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
                          const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_y,
                          const SelArgs a) {
    using Cf = SelCfg<IO, CPL>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_ticket;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (STEAL)
        launch_dependents();   // the launch for deferred shares may start; it waits for this grid
    else if (a.deferred)
        grid_dependency_wait();   // the stealing launch has completed and its writes are visible
    Ring rg{smem + warp * Cf::WARP_SMEM, nullptr, 0, true};
    rg.full = reinterpret_cast<uint64_t *>(rg.base + Cf::OFF_BAR);
    if (threadIdx.x == 0) {
        s_ticket = static_cast<int>(atomicAdd(a.deferred ? a.ticket2 : a.ticket, 1u));
        if (blockIdx.x == 0 && !a.deferred) status_begin(a.st);
    }
    if (lane == 0) {
        for (int s = 0; s < Cf::STAGES; ++s) mbar_init(&rg.full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int wi = s_ticket * kWpb + warp;
    if (wi >= a.W) return;
    const Maps m{&tm_x, &tm_dt, &tm_z, &tm_B, &tm_C, &tm_y};
    if constexpr (STEAL) {
        steal_share<IO, CPL, ACC, HAS_Z, SP>(rg, m, a, wi);
    } else {
        if (a.deferred && __ldcg(a.defer + wi) == 0) return;   // run by the first launch
        static_share<IO, CPL, ACC, HAS_Z, SP>(rg, m, a, wi, !a.deferred);
    }
}

// ----------------------------------------------------------------------------
// Compiled variants
// ----------------------------------------------------------------------------
constexpr int kMaxDevices = 64;

template <typename IO>
using HostCfg = SelCfg<IO, cpl_of<IO>()>;

template <auto Kernel>
int blocks_per_sm(size_t smem, int dev) {
    static std::once_flag once[kMaxDevices];
    static int blocks[kMaxDevices];
    std::call_once(once[dev], [&] {
        blocks[dev] = 0;
        if (cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, Kernel, kWpb * 32, smem) == cudaSuccess)
            blocks[dev] = n;
    });
    return blocks[dev];
}

// Launches variant (IO, HZ, SP) of the kernel: the stealing form when the
// arguments ask for it.
template <typename IO, bool ACC, bool HZ, bool SP>
int launch_variant(const CUtensorMap *mp, const SelArgs &a, int grid, cudaStream_t stream) {
    constexpr size_t smem = SelCfg<IO, cpl_of<IO>()>::SMEM;
    if (!a.steal) {
        selective_scan_kernel<IO, ACC, HZ, SP, false>
            <<<static_cast<unsigned>(grid), kWpb * 32, smem, stream>>>(mp[0], mp[1], mp[2], mp[3], mp[4], mp[5], a);
        return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
    }
    // stealing launch, then the shares it deferred (most warps return at once)
    selective_scan_kernel<IO, ACC, HZ, SP, true>
        <<<static_cast<unsigned>(grid), kWpb * 32, smem, stream>>>(mp[0], mp[1], mp[2], mp[3], mp[4], mp[5], a);
    if (cudaGetLastError() != cudaSuccess) return LR_ERR_CUDA;
    SelArgs b = a;
    b.deferred = 1;
    // a programmatic dependent launch: it starts launching while the stealing
    // grid runs, and its blocks wait for that grid before reading the marks
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kWpb * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, selective_scan_kernel<IO, ACC, HZ, SP, false>, mp[0], mp[1], mp[2],
                                             mp[3], mp[4], mp[5], b);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

// Resident blocks per SM of variant (IO, HZ, SP) (both forms; sets their
// dynamic shared-memory attribute once per device).
template <typename IO, bool ACC, bool HZ, bool SP>
int variant_blocks(int dev) {
    constexpr size_t smem = SelCfg<IO, cpl_of<IO>()>::SMEM;
    const int a = blocks_per_sm<selective_scan_kernel<IO, ACC, HZ, SP, true>>(smem, dev);
    const int b = blocks_per_sm<selective_scan_kernel<IO, ACC, HZ, SP, false>>(smem, dev);
    return a < b ? a : b;
}

}  // namespace

namespace sel {
// Each (I/O type, z gate, softplus on dt) variant of the kernel is compiled
// in its own translation unit (lr_sel_<io>_<z>_<sp>.cu), so that they build
// in parallel.
#define LR_SEL_VARIANTS(X)                                                   \
    X(bf16_z_sp, __nv_bfloat16, false, true, true)                           \
    X(bf16_z_nosp, __nv_bfloat16, false, true, false)                        \
    X(bf16_noz_sp, __nv_bfloat16, false, false, true)                        \
    X(bf16_noz_nosp, __nv_bfloat16, false, false, false)                     \
    X(f32_z_sp, float, true, true, true)                                     \
    X(f32_z_nosp, float, true, true, false)                                  \
    X(f32_noz_sp, float, true, false, true)                                  \
    X(f32_noz_nosp, float, true, false, false)
#define LR_SEL_DECLARE(NAME, IO, ACC, HZ, SP)                                 \
    int launch_##NAME(const CUtensorMap *mp, const SelArgs &a, int grid, cudaStream_t stream); \
    int blocks_##NAME(int dev);
LR_SEL_VARIANTS(LR_SEL_DECLARE)
#undef LR_SEL_DECLARE
// Defines the entry points of one variant (in its translation unit).
#define LR_SEL_DEFINE(NAME, IO, ACC, HZ, SP)                                                       \
    int launch_##NAME(const CUtensorMap *mp, const SelArgs &a, int grid, cudaStream_t stream) {    \
        return launch_variant<IO, ACC, HZ, SP>(mp, a, grid, stream);                               \
    }                                                                                              \
    int blocks_##NAME(int dev) { return variant_blocks<IO, ACC, HZ, SP>(dev); }
}  // namespace sel
}  // namespace lr
