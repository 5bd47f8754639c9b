// lr_hgrn2.cu -- HGRN2 matrix-state recurrence (frankenstein-transformer docs,
// HGRN2 Attention page: S_t = diag(g_t) S_{t-1} + v_t k_t^T, readout
// o_t = S_t q_t) in chunked form on the sm_103a tensor cores.
//
// Per chunk of C = 64 steps, with Lambda_t[i] = sum_{u <= t} log2 g_u[i]
// (cumulative inside the chunk, fp32) and S the state at the chunk start:
//
//   o_t[i] = sum_{s <= t} (q_t . k_s) 2^(Lambda_t[i] - Lambda_s[i]) v_s[i]
//          + 2^Lambda_t[i] (S q_t)[i]
//   S'[i][j] = 2^Lambda_C[i] S[i][j] + sum_s 2^(Lambda_C[i] - Lambda_s[i]) v_s[i] k_s[j]
//
// The gate decays rows i of S (value channels), so the per-(t, s, i) factor
// splits through a per-channel reference m[i] (the chunk's mid-range of
// Lambda): 2^(Lambda_t - Lambda_s) = 2^(Lambda_t - m) 2^(m - Lambda_s).  With
// V~ = 2^(m - Lambda) (.) V and V~' = 2^(Lambda_C - Lambda) (.) V,
//
//   O    = 2^(Lambda - m) (.) ( tril(Q K^T) V~  +  2^m (.) Q S^T )
//   dS^T = K^T V~'                                  (state update: S' = 2^Lambda_C (.) S + dS)
//
// Both factors stay within 2^(+-spread/2), where the spread is the sum of
// |log2 g| over the range.  A chunk whose spread exceeds 160 for some
// channel (small gates: the page's lower bound may be 0) is run as 2, 4, ..
// "virtual chunks" of 32, 16, .. steps -- the smallest split whose pieces all
// stay within 160 -- each one a pass through the same pipeline with the
// steps outside it masked out; the terms between virtual chunks then flow
// through the state, whose factors never exceed 1.  Log-gates are clamped at
// -120 per step (a gate below 2^-120, e.g. 0, resets the state to within
// fp32 resolution), so a single step always fits.  Non-finite gates set
// LR_ERR_RANGE.
//
// A thread block owns 64 value rows of one (batch, head) (rows of S evolve
// independently because diag(g) scales rows): grid = B * H * 2, one block per
// SM (224,512 bytes of shared memory, all 512 TMEM columns).  Four tcgen05 MMAs per
// chunk (bf16 operands in shared memory, fp32 accumulators in TMEM):
//   P    = Q K^T       M=64  N=64 K=128  A = Q (K-major), B = K (K-major), TMA 128B-swizzled
//   dS^T = K^T V~'     M=128 N=64 K=64   A = the same K tile read MN-major, B = V~' (K-major)
//   OI   = tril(P) V~  M=64  N=64 K=64   A = masked P (bf16), B = V~ (K-major)
//   OX   = Q S^T       M=64  N=64 K=128  B = bf16 state, MN-major [key j][value row i]
// Roles (warp specialised, connected by mbarriers, so consecutive chunks
// overlap instead of running one serial chain per block):
//   TMA warp   keeps 3 chunks of Q, K and the block's V, g columns in flight;
//   MMA warp   one thread issues P, dS and OI and commits them to mbarriers;
//   OX warp    one thread issues OX = Q S^T as soon as the back published the
//              state it needs (a second issuer keeps this state-dependent MMA
//              from queueing behind the front's work on the next chunk);
//   front (8)  gates -> Lambda, m; V~, V~' and 2^(Lambda - m) for chunk c; the
//              causal mask of P_c (runs up to a chunk ahead of the back).  In
//              a whole chunk the per-step factors are running products of the
//              gates, so a thread takes two exp2 and one log2 per chunk
//              instead of one per step.  One block barrier per chunk (the
//              exchange of quarter totals); each warp hands its operands over
//              with its own mbarrier arrival.  Two warps per scheduler;
//   back (4)   state update S = 2^Lambda_C S + dS (fp32, in registers: thread j
//              holds key column j of the 64 rows), its bf16 copy for the next
//              OX, then the outputs of chunk c.
// TMEM holds two buffers of every accumulator (P, OI, OX, dS: 8 x 64 columns)
// so the MMAs of chunk c+1 run while the back reads chunk c.
#include <cudaTypedefs.h>

#include <mutex>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {

namespace hg {
constexpr int C = 64;          // chunk length
constexpr int DK = 128;        // key channels per head
constexpr int DV = 128;        // value channels per head
constexpr int RB = 64;         // value rows of S per thread block
constexpr int NRB = DV / RB;   // blocks per head
constexpr int KW = 4;          // back warps 0..3
constexpr int FW = 8;          // front warps 4..11
constexpr int FQ = FW * 32 / 64;   // front threads per value row = quarters of the chunk's steps
constexpr int FSTEPS = 64 / FQ;    // steps per front thread
constexpr int TMA_WARP = KW + FW, MMA_WARP = KW + FW + 1, OX_WARP = KW + FW + 2;
constexpr int THREADS = 32 * (KW + FW + 3);
constexpr int NST = 3;         // TMA stages
// largest spread of Lambda (log2 units) over a virtual chunk that the
// reference split keeps inside fp32 range with headroom: 2^(+-80) factors
constexpr float kMaxSpread = 160.0f;
// per-step floor of log2 g: one step always fits a virtual chunk
constexpr float kMinLog2 = -120.0f;

// stage: Q [64 t][128 j] and K [64 s][128 j] as two 128B-swizzled 64-column
// halves each; V and g [64 t][64 i] as plain bf16 rows
constexpr uint32_t QK_BYTES = C * DK * 2;
constexpr uint32_t VG_BYTES = C * RB * 2;
constexpr uint32_t OFF_K = QK_BYTES, OFF_V = 2 * QK_BYTES, OFF_G = OFF_V + VG_BYTES;
constexpr uint32_t STAGE_BYTES = 2 * QK_BYTES + 2 * VG_BYTES;
constexpr uint32_t OFF_PS = NST * STAGE_BYTES;     // masked P [64 t][64 s], swizzled
constexpr uint32_t OFF_VT = OFF_PS + 8192;         // V~  [64 i][64 s], swizzled
constexpr uint32_t OFF_VTP = OFF_VT + 8192;        // V~' [64 i][64 s], swizzled
constexpr uint32_t OFF_SBT = OFF_VTP + 8192;       // bf16 state [128 j][64 i], swizzled
constexpr uint32_t OFF_E1 = OFF_SBT + 16384;       // 2 x 2^(Lambda - m), fp32 [64 t][64 i]
constexpr uint32_t OFF_EM = OFF_E1 + 2 * 16384;    // 2 x 2^m [64]
constexpr uint32_t OFF_GC = OFF_EM + 2 * 256;      // 2 x 2^Lambda_C [64]
constexpr uint32_t OFF_TOT = OFF_GC + 2 * 256;     // front: per-quarter totals [2][FQ][64] (by chunk parity)
constexpr uint32_t OFF_VI = OFF_TOT + 2 * FQ * 256;    // 2 x virtual chunk (chunk, lo, hi, last)
constexpr uint32_t OFF_SPL = OFF_VI + 32;          // front: split flags of the chunk; [4..7]
                                                   // virtual chunks of chunk c % 4
constexpr uint32_t OFF_BAR = OFF_SPL + 32;
// full[3] empty[3] bar_p[2] bar_o[2] bar_x[2] fdone[2] kdone[2] sbready mma_done splitr[2] bar_ds[2]
constexpr int NBAR = 3 + 3 + 2 + 2 + 2 + 2 + 2 + 1 + 1 + 2 + 2;
// the local test that rules out a split: every quarter (16 steps) of every
// row within a quarter of the limit
constexpr float kQuarterSafe = kMaxSpread / 4;
constexpr uint32_t OFF_TMEM = OFF_BAR + NBAR * 8;
constexpr uint32_t OFF_FLAG = OFF_TMEM + 8;
constexpr uint32_t SMEM = OFF_FLAG + 8;
static_assert(STAGE_BYTES % 1024 == 0 && OFF_PS % 1024 == 0 && OFF_VT % 1024 == 0 &&
                  OFF_VTP % 1024 == 0 && OFF_SBT % 1024 == 0 && OFF_E1 % 16 == 0,
              "swizzled operand tiles must be 1024-byte aligned");
static_assert(SMEM <= 227 * 1024, "one block per SM");

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_P = 0, T_OI = 128, T_OX = 256, T_DS = 384;   // + 64 * buffer

constexpr uint32_t IDESC_P = umma_idesc_bf16(64, 64, 0, 0);
constexpr uint32_t IDESC_OI = umma_idesc_bf16(64, 64, 0, 0);
constexpr uint32_t IDESC_OX = umma_idesc_bf16(64, 64, 0, 1);
constexpr uint32_t IDESC_DS = umma_idesc_bf16(128, 64, 1, 0);

// 2^(Lambda - m)[t][i] with 16-byte groups XOR-swizzled by the row, so the
// 16 lanes of an epilogue warp (16 consecutive rows, same columns) hit 16
// different bank groups.
__device__ __forceinline__ int e1_index(int t, int i) {
    return t * RB + ((((i >> 2) ^ (t & 15))) << 2) + (i & 3);
}

__device__ __forceinline__ void named_bar(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also ORs a predicate over its threads.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1 : 0), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&p);
}

// Bounded mbarrier wait of the block's roles: the first wait to run out sets
// the block's abort flag, so that every role leaves its loop instead of
// waiting out its own limit.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              uint64_t timeout_ns, StatusRef sref) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag != 0) return false;
        if (globaltimer_ns() - t0 > timeout_ns) {
            *abort_flag = 1;
            status_report(sref, LR_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// What a front thread works with.
struct FrontEnv {
    unsigned char *sm;
    uint32_t tmem;
    uint64_t *empty, *bar_p, *bar_o, *fdone, *kdone, *splitr;
    volatile int *abort_flag;
    volatile int *VI;          // [2][chunk, lo, hi, last]
    volatile unsigned *NVC;    // [4] virtual chunks of chunk c % 4
    int L;
    float lb;
    uint64_t timeout_ns;
    StatusRef sref;
};

// One virtual chunk [lo, hi) of chunk c by the front: V~, V~', the masked P,
// 2^(Lambda - m), 2^(m - B0) and the decay 2^(B1 - B0), then the hand-over to
// the MMA issuer and the back.  B0, B1: Lambda before the virtual chunk and at
// its last step.  Returns false, for the whole warp, when one of its waits
// failed; the warp then skips its hand-over.
//   WHOLE = false (a piece of a split chunk): a = this thread's cumulative
//   log2 gates from the chunk start; the factors are exp2 of their
//   differences, zero outside [lo, hi).
//   WHOLE = true (lo = 0, hi = 64, nothing masked): a = the running products
//   of this thread's gates (a[u] = g_tb ... g_tb+u), r = the products of the
//   gates after each step (r[u] = g_tb+u+1 ... g_tb+15), off = Lambda before
//   the thread's first step and qsum = log2 of its 16 gates' product.  Then
//   2^(Lambda_t - m) = 2^(off - m) a[u] and 2^(m - Lambda_t) = 2^(m - off -
//   qsum) r[u]: two exp2 per thread instead of one per step (no quarter of
//   a whole chunk decays by more than 2^-40, so the products stay normal).
template <bool SPLIT, bool WHOLE>
__device__ __forceinline__ bool front_vc(const FrontEnv &x, int c, int j, int nvc, int lo, int hi,
                                         const float (&a)[FSTEPS], const float (&r)[FSTEPS], float off,
                                         float qsum, float B0, float B1, int &v) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int f = tid - 32 * KW, fw = warp - KW;
    const int i = f & (RB - 1), qt = f / RB;
    const int tb = FSTEPS * qt;
    const int st = c % NST, bi = v & 1;
    const unsigned char *stg = x.sm + st * STAGE_BYTES;
    const __nv_bfloat16 *sV = reinterpret_cast<const __nv_bfloat16 *>(stg + OFF_V);
    float *E1 = reinterpret_cast<float *>(x.sm + OFF_E1);
    float *EM = reinterpret_cast<float *>(x.sm + OFF_EM);
    float *GC = reinterpret_cast<float *>(x.sm + OFF_GC);
    unsigned char *Ps = x.sm + OFF_PS, *VT = x.sm + OFF_VT, *VTP = x.sm + OFF_VTP;
    // 2^(Lambda - m) buffer free (back done with virtual chunk v-2)
    bool ok = v < 2 || wait_or_abort(&x.kdone[bi], ((v - 2) >> 1) & 1, x.abort_flag, x.timeout_ns, x.sref);
    // m = the mean of B0 and B1 keeps every factor within 2^(+-spread/2)
    const float m = 0.5f * (B0 + B1);
    float *e1 = E1 + bi * (C * RB);
    const float ea = WHOLE ? ex2_approx(off - m) : 0.0f, eb = WHOLE ? ex2_approx(m - off - qsum) : 0.0f;
#pragma unroll
    for (int u = 0; u < FSTEPS; ++u) {
        const int t = tb + u;
        if (WHOLE)
            e1[e1_index(t, i)] = ea * a[u];
        else
            e1[e1_index(t, i)] = (t >= lo && t < hi) ? ex2_approx(a[u] - m) : 0.0f;
    }
    if (WHOLE ? qt == 0 : qt == lo / FSTEPS) {
        EM[bi * RB + i] = ex2_approx(m - B0);
        GC[bi * RB + i] = ex2_approx(B1 - B0);
    }
    // V~ = 2^(m - Lambda) v and V~' = 2^(B1 - m) V~ for row i, this thread's
    // steps inside the virtual chunk
    const float cm = ex2_approx(B1 - m);
    uint32_t vt[FSTEPS / 2], vtp[FSTEPS / 2];
#pragma unroll
    for (int u = 0; u < FSTEPS; u += 2) {
        const int t = tb + u;
        float w0, w1;
        if (WHOLE) {
            w0 = eb * r[u] * __bfloat162float(sV[t * RB + i]);
            w1 = eb * r[u + 1] * __bfloat162float(sV[(t + 1) * RB + i]);
        } else {
            w0 = (t >= lo && t < hi) ? ex2_approx(m - a[u]) * __bfloat162float(sV[t * RB + i]) : 0.0f;
            w1 = (t + 1 >= lo && t + 1 < hi) ? ex2_approx(m - a[u + 1]) * __bfloat162float(sV[(t + 1) * RB + i])
                                             : 0.0f;
        }
        vt[u / 2] = pack_bf16(w0, w1);
        vtp[u / 2] = pack_bf16(w0 * cm, w1 * cm);
    }
    // the V~, V~' and masked-P buffers are free once dS and OI of virtual
    // chunk v-1 completed (the work above overlapped with them); P_c is ready
    if (ok && v >= 1)
        ok = wait_or_abort(&x.bar_o[(v - 1) & 1], ((v - 1) >> 1) & 1, x.abort_flag, x.timeout_ns, x.sref);
    if (ok) ok = wait_or_abort(&x.bar_p[c & 1], (c >> 1) & 1, x.abort_flag, x.timeout_ns, x.sref);
    ok = __all_sync(0xffffffffu, ok);   // the TMEM load below is warp-collective
    if (ok) {
#pragma unroll
        for (int k = 0; k < FSTEPS / 8; ++k) {
            const uint32_t o8 = sw128_offset(i, tb + 8 * k);
            *reinterpret_cast<uint4 *>(VT + o8) = make_uint4(vt[4 * k], vt[4 * k + 1], vt[4 * k + 2], vt[4 * k + 3]);
            *reinterpret_cast<uint4 *>(VTP + o8) =
                make_uint4(vtp[4 * k], vtp[4 * k + 1], vtp[4 * k + 2], vtp[4 * k + 3]);
        }
        // causal mask of P_c inside the virtual chunk: the M = 64 rows t sit in
        // lanes 0..15 of each warp quarter; the two warps of a quarter take 32
        // columns s each, their half-warps 16 columns each (two-half TMEM load)
        tc_fence_after();
        const int quarter = fw & 3;
        const int s_base = 32 * (fw >> 2) + 16 * (lane >> 4);
        float pv[16];
        tmem_ld16x2_nowait<16>(x.tmem + T_P + (c & 1) * 64 + 32 * (fw >> 2) + (uint32_t(quarter * 32) << 16), pv);
        tmem_ld_wait_tied(pv);
        const int t = 16 * quarter + (lane & 15);
        const bool row_in = WHOLE || (t >= lo && t < hi);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int s0 = s_base + ch * 8 + 2 * e;
                w4[e] = pack_bf16(row_in && s0 <= t && (WHOLE || s0 >= lo) ? pv[ch * 8 + 2 * e] : 0.0f,
                                  row_in && s0 + 1 <= t && (WHOLE || s0 + 1 >= lo) ? pv[ch * 8 + 2 * e + 1] : 0.0f);
            }
            const int chunk = (s_base >> 3) + ch;
            *reinterpret_cast<uint4 *>(Ps + t * 128 + ((chunk ^ (t & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
    }
    // each front warp hands over on its own: the MMA issuer and the back wait
    // for all eight arrivals (no block barrier, so a warp that is done goes on
    // to the next chunk's gates); ok is uniform over the warp
    fence_proxy_async_smem();
    tc_fence_before();
    if (!ok) return false;
    const bool last = j == nvc - 1;
    if (SPLIT && f == 0) {
        x.VI[4 * bi] = c;
        x.VI[4 * bi + 1] = lo;
        x.VI[4 * bi + 2] = hi;
        x.VI[4 * bi + 3] = last ? 1 : 0;
    }
    __syncwarp();
    if (lane == 0) {
        arrive(&x.fdone[bi]);
        if (last) arrive(&x.empty[st]);   // V, g of stage st no longer read
    }
    ++v;
    return true;
}

// A chunk some quarter of which decays beyond kQuarterSafe: its log-gates
// again with the per-step floor kMinLog2 (a gate of 0 gives -inf), the
// finest split into virtual chunks of 64 >> lvl steps whose every piece
// stays within kMaxSpread for every row, and the virtual chunks.
template <bool PRE>
__device__ __forceinline__ bool front_split_chunk(const FrontEnv &x, int c, int &v) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int f = tid - 32 * KW;
    const int i = f & (RB - 1), qt = f / RB;
    const int tb = FSTEPS * qt;
    const int t0 = c * C;
    const __nv_bfloat16 *sG = reinterpret_cast<const __nv_bfloat16 *>(x.sm + (c % NST) * STAGE_BYTES + OFF_G);
    float *TOTF = reinterpret_cast<float *>(x.sm + OFF_TOT);
    unsigned *SPL = reinterpret_cast<unsigned *>(x.sm + OFF_SPL);
    float loc[FSTEPS];
    float acc = 0.0f;
#pragma unroll
    for (int u = 0; u < FSTEPS; ++u) {
        const int t = tb + u;
        float gv = __bfloat162float(sG[t * RB + i]);
        if (PRE) gv = fmaf(1.0f - x.lb, rcp_approx(1.0f + ex2_approx(-gv * kLog2e)), x.lb);
        acc += t0 + t < x.L ? fmaxf(lg2_approx(gv), kMinLog2) : 0.0f;
        loc[u] = acc;
    }
    // bit k of `need` set = some aligned run of 64 >> k steps of some row
    // sums to more than kMaxSpread in |log2 g|
    unsigned need = 0;
    if (-acc > kMaxSpread) {   // runs inside this quarter (16 .. 1 steps)
        need |= 4u;
#pragma unroll 1
        for (int k = 3; k <= 6; ++k) {
            const int len = 64 >> k;
#pragma unroll 1
            for (int a0 = 0; a0 < FSTEPS; a0 += len) {
                float before = 0.0f, end = 0.0f;
#pragma unroll
                for (int u = 0; u < FSTEPS; ++u) {
                    if (u == a0 - 1) before = loc[u];
                    if (u == a0 + len - 1) end = loc[u];
                }
                if (before - end > kMaxSpread) need |= 1u << k;
            }
        }
    }
    named_bar(3, 32 * FW);   // every thread is past its reads of the previous totals
    TOTF[qt * RB + i] = acc;
    if (f == 0) SPL[0] = 0;
    named_bar(3, 32 * FW);
    float off = 0.0f, cq[FQ + 1];
    cq[0] = 0.0f;
#pragma unroll
    for (int q = 0; q < FQ; ++q) {
        const float tq = TOTF[q * RB + i];
        off += q < qt ? tq : 0.0f;
        cq[q + 1] = cq[q] + tq;   // cumulative Lambda at the end of quarter q
    }
    if (qt == 0) {
        if (-cq[FQ] > kMaxSpread) need |= 1u;
        if (-cq[2] > kMaxSpread || cq[2] - cq[FQ] > kMaxSpread) need |= 2u;
    }
    need = __reduce_or_sync(0xffffffffu, need);
    if (lane == 0 && need != 0) atomicOr(SPL, need);
    named_bar(3, 32 * FW);
    need = SPL[0];
    int lvl = 0;
    while (lvl < 6 && ((need >> lvl) & 1u)) ++lvl;
#pragma unroll
    for (int u = 0; u < FSTEPS; ++u) loc[u] += off;
    const int len = C >> lvl, nvc = 1 << lvl;
    if (f == 0) {   // tell the OX issuer
        x.NVC[c & 3] = nvc;
        arrive(&x.splitr[c & 1]);
    }
    for (int j = 0; j < nvc; ++j) {
        const int lo = j * len, hi = lo + len;
        float B0 = 0.0f, B1 = 0.0f;
        if (len >= FSTEPS) {
            B0 = cq[lo / FSTEPS];
            B1 = cq[hi / FSTEPS];
        } else if (qt == lo / FSTEPS) {   // inside this row's quarter
            B0 = lo == tb ? off : 0.0f;
#pragma unroll
            for (int u = 0; u < FSTEPS; ++u) {
                if (tb + u == lo - 1) B0 = loc[u];
                if (tb + u == hi - 1) B1 = loc[u];
            }
        }
        if (!front_vc<true, false>(x, c, j, nvc, lo, hi, loc, loc, 0.0f, 0.0f, B0, B1, v)) return false;
    }
    return true;
}
}  // namespace hg

// PRE: the gate arrives as the pre-activation f and the front forms
// g = lb + (1 - lb) sigmoid(f) ([HGRN2] lower-bounded, sigmoid-activated gate).
//
// A call runs in two passes over the same grid.  SPLIT = false: every chunk
// whole; a block that meets a chunk some quarter of which decays beyond
// kQuarterSafe (a split may be needed) writes the call's stamp into its
// redo word and carries on (its results are then discarded).  SPLIT = true:
// only the blocks whose redo word holds the stamp run, from the start,
// splitting chunks into virtual chunks where needed; the others return at
// once.  So the common case runs code without the split path's registers
// and branches.
template <bool PRE, bool SPLIT>
__global__ void __launch_bounds__(hg::THREADS, 1)
    hgrn2_chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                       const float *__restrict__ S0, float *__restrict__ S_final,
                       __nv_bfloat16 *__restrict__ o, int L, int H, int n_chunks, float lb,
                       uint64_t timeout_ns, StatusRef sref, unsigned long long *__restrict__ redo) {
    using namespace hg;
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (SPLIT) {
        grid_dependency_wait();   // launched as the first pass's dependent
        if (redo[blockIdx.x] != sref.stamp) return;   // the first pass was right
    } else {
        launch_dependents();   // the redo pass may launch; its blocks wait for this grid
        if (tid == 0 && blockIdx.x == 0) status_begin(sref);
    }
    if ((smem_u32(sm) & 1023u) != 0) {  // swizzled tiles need a 1024-byte aligned base
        if (tid == 0) status_report(sref, LR_ERR_CUDA);
        return;
    }
    const int blk = blockIdx.x;
    const int rb = blk % NRB, bh = blk / NRB;
    const int b = bh / H, h = bh - (bh / H) * H;
    const int qcol = h * DK, vcol = h * DV + rb * RB;
    const int HV = H * DV;

    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *full = bars, *empty = bars + 3, *bar_p = bars + 6, *bar_o = bars + 8,
             *bar_x = bars + 10, *fdone = bars + 12, *kdone = bars + 14, *sbready = bars + 16,
             *mma_done = bars + 17, *splitr = bars + 18, *bar_ds = bars + 20;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TMEM);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_FLAG);
    float *E1 = reinterpret_cast<float *>(sm + OFF_E1);
    float *EM = reinterpret_cast<float *>(sm + OFF_EM);
    float *GC = reinterpret_cast<float *>(sm + OFF_GC);
    unsigned char *Ps = sm + OFF_PS, *VT = sm + OFF_VT, *VTP = sm + OFF_VTP, *SBT = sm + OFF_SBT;
    volatile int *VI = reinterpret_cast<volatile int *>(sm + OFF_VI);   // [2][chunk, lo, hi, last]
    volatile unsigned *NVC = reinterpret_cast<volatile unsigned *>(sm + OFF_SPL) + 4;   // [4]

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2 + FW);   // the two MMA issuers' commits and each front warp
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&bar_p[k], 1);
            mbar_init(&bar_o[k], 1);
            mbar_init(&bar_x[k], 1);
            mbar_init(&fdone[k], FW);   // each front warp
            mbar_init(&kdone[k], KW);
        }
        mbar_init(sbready, KW);   // each back warp publishes its own 32 rows
        mbar_init(mma_done, 2);
        mbar_init(&splitr[0], 1);
        mbar_init(&splitr[1], 1);
        mbar_init(&bar_ds[0], 1);
        mbar_init(&bar_ds[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto hw = [&](uint64_t *bar, uint32_t parity) -> bool {
        return hg::wait_or_abort(bar, parity, abort_flag, timeout_ns, sref);
    };

    if (warp == TMA_WARP) {  // ------------------------------------------- TMA
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            prefetch_tensormap(&tm_g);
            int c = 0;
            for (; c < n_chunks; ++c) {
                const int st = c % NST;
                if (c >= NST && !hw(&empty[st], ((c - NST) / NST) & 1)) break;
                unsigned char *stg = sm + st * STAGE_BYTES;
                mbar_arrive_expect_tx(&full[st], STAGE_BYTES);
                tma_load_3d(stg, &tm_q, &full[st], qcol, c * C, b);
                tma_load_3d(stg + 8192, &tm_q, &full[st], qcol + 64, c * C, b);
                tma_load_3d(stg + OFF_K, &tm_k, &full[st], qcol, c * C, b);
                tma_load_3d(stg + OFF_K + 8192, &tm_k, &full[st], qcol + 64, c * C, b);
                tma_load_3d(stg + OFF_V, &tm_v, &full[st], vcol, c * C, b);
                tma_load_3d(stg + OFF_G, &tm_g, &full[st], vcol, c * C, b);
            }
            // copies still in flight land before the block exits
            for (int k = c > NST ? c - NST : 0; k < c; ++k)
                mbar_wait_bounded(&full[k % NST], (k / NST) & 1, timeout_ns);
        }
    } else if (warp == MMA_WARP) {  // ------------------------------------- MMA
        if (lane == 0) {
            auto issue_p = [&](int c) {  // P_c = Q_c K_c^T into buffer c & 1
                const uint32_t sQ = smem_u32(sm + (c % NST) * STAGE_BYTES), sK = sQ + OFF_K;
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                    umma_bf16(tmem + T_P + (c & 1) * 64, umma_smem_desc(sQ + off, 16, 1024),
                              umma_smem_desc(sK + off, 16, 1024), IDESC_P, kk > 0);
                }
                umma_commit(&bar_p[c & 1]);
            };
            bool ok = n_chunks > 0 && hw(&full[0], 0);
            if (ok) {
                tc_fence_after();
                issue_p(0);
            }
            bool first = true;   // virtual chunk v starts chunk c
            for (int c = 0, v = 0; ok && c < n_chunks; ++v) {
                const int st = c % NST, bi = v & 1;
                const uint32_t sK = smem_u32(sm + st * STAGE_BYTES) + OFF_K;
                // P of the next chunk: its buffer held P_{c-1}, which the front
                // masked for the last time in virtual chunk v-1
                if (first && c + 1 < n_chunks) {
                    if (!hw(&full[(c + 1) % NST], ((c + 1) / NST) & 1)) break;
                    tc_fence_after();
                    issue_p(c + 1);
                }
                // dS_v and OI_v once the front wrote V~', V~ and the masked P of
                // virtual chunk v and the back released the accumulators of v-2
                if (!hw(&fdone[bi], (v >> 1) & 1)) break;
                const bool last = !SPLIT || VI[4 * bi + 3] != 0;
                if (v >= 2 && !hw(&kdone[bi], ((v - 2) >> 1) & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < C / 16; ++kk)
                    umma_bf16(tmem + T_DS + bi * 64, umma_smem_desc(sK + kk * 2048, 8192, 1024),
                              umma_smem_desc(smem_u32(VTP) + kk * 32, 16, 1024), IDESC_DS, kk > 0);
                umma_commit(&bar_ds[bi]);   // the back's state update need not wait for OI
#pragma unroll
                for (int kk = 0; kk < C / 16; ++kk)
                    umma_bf16(tmem + T_OI + bi * 64, umma_smem_desc(smem_u32(Ps) + kk * 32, 16, 1024),
                              umma_smem_desc(smem_u32(VT) + kk * 32, 16, 1024), IDESC_OI, kk > 0);
                umma_commit(&bar_o[bi]);
                if (last) {
                    umma_commit(&empty[st]);   // K_c no longer read once these complete
                    ++c;
                }
                first = last;
            }
            // nothing of this block's may still run on the tensor cores when
            // its TMEM is released
            umma_commit(mma_done);
            mbar_wait_bounded(mma_done, 0, timeout_ns);
        }
    } else if (warp == OX_WARP) {  // -------------------------------------- OX
        if (lane == 0) {
            unsigned nvc = 0, j = 0;   // virtual chunks of chunk c, this one's index
            for (int c = 0, v = 0; c < n_chunks; ++v) {
                const int st = c % NST, bi = v & 1;
                // the bf16 state after virtual chunk v-1, how many virtual
                // chunks chunk c has (the front publishes it as soon as it has
                // decided), Q_c, and the OX buffer of v-2 released by the back
                if (!hw(sbready, v & 1)) break;
                if (!SPLIT) {
                    nvc = 1;
                } else if (j == 0) {
                    if (!hw(&splitr[c & 1], (c >> 1) & 1)) break;
                    nvc = NVC[c & 3];
                }
                const bool last = ++j == nvc;
                if (!hw(&full[st], (c / NST) & 1)) break;
                if (v >= 2 && !hw(&kdone[bi], ((v - 2) >> 1) & 1)) break;
                tc_fence_after();
                const uint32_t sQ = smem_u32(sm + st * STAGE_BYTES);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t qoff = (kk >> 2) * 8192 + (kk & 3) * 32;
                    umma_bf16(tmem + T_OX + bi * 64, umma_smem_desc(sQ + qoff, 16, 1024),
                              umma_smem_desc(smem_u32(SBT) + kk * 2048, 8192, 1024), IDESC_OX, kk > 0);
                }
                umma_commit(&bar_x[bi]);
                if (last) {
                    umma_commit(&empty[st]);   // Q_c no longer read once these complete
                    j = 0;
                    ++c;
                }
            }
            umma_commit(mma_done);
            mbar_wait_bounded(mma_done, 0, timeout_ns);
        }
    } else if (warp >= KW) {  // ----------------------------------------- front
        const int f = tid - 32 * KW;
        const int i = f & (RB - 1), qt = f / RB;   // value row, quarter of the chunk's steps
        const int tb = FSTEPS * qt;
        float *TOTF = reinterpret_cast<float *>(sm + OFF_TOT);
        const hg::FrontEnv fx{sm, tmem, empty, bar_p, bar_o, fdone, kdone, splitr, abort_flag, VI, NVC,
                              L, lb, timeout_ns, sref};
        int v = 0;   // virtual chunks so far
        // a wait of this warp ran out (or saw the abort flag) in an earlier
        // chunk's hand-over: the warp carries that to the next quarter-total
        // exchange, where all front warps leave the loop together (a warp that
        // left alone would leave the others at that barrier)
        bool failed = false;
        for (int c = 0; c < n_chunks; ++c) {
            const int st = c % NST;
            const __nv_bfloat16 *sG = reinterpret_cast<const __nv_bfloat16 *>(sm + st * STAGE_BYTES + OFF_G);
            const bool ok = !failed && hw(&full[st], (c / NST) & 1);   // inputs landed

            // running products of this thread's gates, forward and backward
            // (steps past L: g = 1), and the log2 of their product
            const int t0 = c * C;
            float pf[FSTEPS], pr[FSTEPS], gq[FSTEPS];
            float prod = 1.0f;
#pragma unroll
            for (int u = 0; u < FSTEPS; ++u) {
                const int t = tb + u;
                float gv = __bfloat162float(sG[t * RB + i]);
                if (PRE) gv = fmaf(1.0f - lb, rcp_approx(1.0f + ex2_approx(-gv * kLog2e)), lb);
                gq[u] = t0 + t < L ? gv : 1.0f;
                prod *= gq[u];
                pf[u] = prod;
            }
            pr[FSTEPS - 1] = 1.0f;
#pragma unroll
            for (int u = FSTEPS - 2; u >= 0; --u) pr[u] = pr[u + 1] * gq[u + 1];
            const float acc = lg2_approx(prod);
            // a gate that is not a number (or infinite) leaves NaN or +inf here
            if (!(acc == acc) || acc == __int_as_float(0x7f800000)) status_report(sref, LR_ERR_RANGE);
            float *tot = TOTF + (c & 1) * (FQ * RB);   // by chunk parity: a warp ahead may
                                                        // write the next chunk's totals
            tot[qt * RB + i] = acc;
            // the quarter totals are exchanged here.  The barrier also ORs the
            // local test that rules out a split (this quarter's |sum of log2 g|
            // within kQuarterSafe) with a failed wait; only when it fires do
            // the front threads tell the two apart and, rarely, split the chunk
            if (named_bar_or(2, 32 * FW, !ok || -acc > kQuarterSafe)) {
                if (named_bar_or(3, 32 * FW, !ok)) break;
                if constexpr (SPLIT) {
                    if (!hg::front_split_chunk<PRE>(fx, c, v)) failed = true;
                    continue;
                } else {
                    if (f == 0) redo[blockIdx.x] = sref.stamp;   // the second pass redoes this block
                }
            }
            float off = 0.0f, lc = 0.0f;
#pragma unroll
            for (int q = 0; q < FQ; ++q) {
                const float tq = tot[q * RB + i];
                off += q < qt ? tq : 0.0f;
                lc += tq;
            }
            if (SPLIT && f == 0) {   // one virtual chunk: tell the OX issuer
                NVC[c & 3] = 1;
                arrive(&splitr[c & 1]);
            }
            if (!hg::front_vc<SPLIT, true>(fx, c, 0, 1, 0, C, pf, pr, off, acc, 0.0f, lc, v)) failed = true;
        }
    } else {  // ------------------------------------------------------------ back
        // key column j = tid of value rows rb*64 .. rb*64+63 of S[b, h].  The
        // four back warps share no data: each publishes the bf16 rows of its
        // own 32 keys and releases its own TMEM lanes, so they run without a
        // block barrier and the abort decision is taken per warp.
        const unsigned FULLM = 0xffffffffu;
        const size_t srow0 = size_t(bh) * DV + size_t(rb) * RB;
        float S[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) S[r] = S0 != nullptr ? S0[(srow0 + r) * DK + tid] : 0.0f;
        // bf16 copy, MN-major: row j holds the 64 value rows in 8 swizzled 16-byte groups
        auto write_state = [&]() {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                *reinterpret_cast<uint4 *>(SBT + sw128_offset(tid, 8 * k)) =
                    make_uint4(pack_bf16(S[8 * k], S[8 * k + 1]), pack_bf16(S[8 * k + 2], S[8 * k + 3]),
                               pack_bf16(S[8 * k + 4], S[8 * k + 5]), pack_bf16(S[8 * k + 6], S[8 * k + 7]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) arrive(sbready);
        };
        write_state();
        const uint32_t lanes = uint32_t(warp * 32) << 16;
        // o_t = 2^(Lambda_t - m) (OI_t + 2^m OX_t); the M = 64 rows sit in lanes
        // 0..15 of the quarter, so the two half-warps take row t = 16 warp +
        // lane % 16 at columns [16 hh, +16) and [32 + 16 hh, +16)
        const int t = 16 * warp + (lane & 15);
        const int cb = 32 * (lane >> 4);
        for (int c = 0, v = 0; c < n_chunks; ++v) {
            const int bi = v & 1;
            bool ok = hw(&fdone[bi], (v >> 1) & 1);
            if (ok) ok = hw(&bar_ds[bi], (v >> 1) & 1);
            if (!__all_sync(FULLM, ok)) break;
            const int lo = SPLIT ? VI[4 * bi + 1] : 0, hi = SPLIT ? VI[4 * bi + 2] : C;
            const bool last = !SPLIT || VI[4 * bi + 3] != 0;
            tc_fence_after();
            {   // S = diag(2^Lambda_C) S + dS   (dS^T lane j, column i)
                const float *gc = GC + bi * RB;
#pragma unroll
                for (int hh = 0; hh < 4; hh += 2) {
                    float d0[16], d1[16];
                    tmem_ld16_nowait(tmem + T_DS + bi * 64 + 16 * hh + lanes, d0);
                    tmem_ld16_nowait(tmem + T_DS + bi * 64 + 16 * hh + 16 + lanes, d1);
                    tmem_ld_wait_tied(d0, d1);
#pragma unroll
                    for (int q = 0; q < 16; q += 4) {
                        const float4 g0 = *reinterpret_cast<const float4 *>(gc + 16 * hh + q);
                        const float4 g1 = *reinterpret_cast<const float4 *>(gc + 16 * hh + 16 + q);
                        float *s0 = S + 16 * hh + q, *s1 = S + 16 * hh + 16 + q;
                        s0[0] = fmaf(g0.x, s0[0], d0[q]);
                        s0[1] = fmaf(g0.y, s0[1], d0[q + 1]);
                        s0[2] = fmaf(g0.z, s0[2], d0[q + 2]);
                        s0[3] = fmaf(g0.w, s0[3], d0[q + 3]);
                        s1[0] = fmaf(g1.x, s1[0], d1[q]);
                        s1[1] = fmaf(g1.y, s1[1], d1[q + 1]);
                        s1[2] = fmaf(g1.z, s1[2], d1[q + 2]);
                        s1[3] = fmaf(g1.w, s1[3], d1[q + 3]);
                    }
                }
            }
            // OI_v, and OX_v, which reads the previous bf16 state until bar_x
            ok = hw(&bar_o[bi], (v >> 1) & 1);
            if (ok) ok = hw(&bar_x[bi], (v >> 1) & 1);
            if (!__all_sync(FULLM, ok)) break;
            tc_fence_after();
            // the first output columns' accumulator loads overlap the state write
            float oi[16], ox[16];
            tmem_ld16x2_nowait<32>(tmem + T_OI + bi * 64 + lanes, oi);
            tmem_ld16x2_nowait<32>(tmem + T_OX + bi * 64 + lanes, ox);
            write_state();
            const float *e1 = E1 + bi * (C * RB);
            const float *em = EM + bi * RB;
            const bool store = c * C + t < L && t >= lo && t < hi;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                if (hh > 0) {
                    tmem_ld16x2_nowait<32>(tmem + T_OI + bi * 64 + 16 * hh + lanes, oi);
                    tmem_ld16x2_nowait<32>(tmem + T_OX + bi * 64 + 16 * hh + lanes, ox);
                }
                tmem_ld_wait_tied(oi, ox);
                if (store) {
                    const int ib = cb + 16 * hh;
                    uint32_t w[8];
#pragma unroll
                    for (int q = 0; q < 16; q += 4) {
                        const int i0 = ib + q;
                        const float4 e = *reinterpret_cast<const float4 *>(e1 + e1_index(t, i0));
                        const float4 mm = *reinterpret_cast<const float4 *>(em + i0);
                        w[q / 2] = pack_bf16(fmaf(mm.x, ox[q], oi[q]) * e.x,
                                             fmaf(mm.y, ox[q + 1], oi[q + 1]) * e.y);
                        w[q / 2 + 1] = pack_bf16(fmaf(mm.z, ox[q + 2], oi[q + 2]) * e.z,
                                                 fmaf(mm.w, ox[q + 3], oi[q + 3]) * e.w);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(o + (size_t(b) * L + c * C + t) * HV +
                                                           vcol + ib);
                    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive(&kdone[bi]);
            if (last) ++c;
        }
        if (S_final != nullptr) {
#pragma unroll
            for (int r = 0; r < RB; ++r) S_final[(srow0 + r) * DK + tid] = S[r];
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// ============================================================================
// Host side
// ============================================================================
namespace {

PFN_cuTensorMapEncodeTiled_v12000 hg_encoder() {
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

// 3-D bf16 map over (cols, L, B), box (box_cols, 64, 1).
bool hg_map(CUtensorMap *tm, const void *base, uint64_t cols, uint64_t L, uint64_t B,
            uint32_t box_cols, bool swizzle128) {
    auto enc = hg_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {cols, L, B};
    const cuuint64_t strides[2] = {cols * 2, cols * L * 2};
    const cuuint32_t box[3] = {box_cols, uint32_t(hg::C), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename K>
bool hg_smem_attr(K kern) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(hg::SMEM)) ==
           cudaSuccess;
}

bool hg_setup_once() {
    static std::once_flag once;
    static bool ok = false;
    std::call_once(once, [] {
        ok = hg_smem_attr(hgrn2_chunk_kernel<false, false>) && hg_smem_attr(hgrn2_chunk_kernel<false, true>) &&
             hg_smem_attr(hgrn2_chunk_kernel<true, false>) && hg_smem_attr(hgrn2_chunk_kernel<true, true>);
    });
    return ok;
}

// A lower-bounded gate g >= lb keeps every quarter of a chunk within
// kQuarterSafe when 16 * -log2(lb) <= kQuarterSafe, i.e. lb >= 2^-2.5 =
// 0.177; above 0.18 the second pass cannot have work and is not launched.
constexpr float kLbNoSplit = 0.18f;

}  // namespace

int hgrn2_workspace(int64_t B, int64_t, int64_t H, size_t *bytes) {
    // the call status, then one redo word per thread block
    *bytes = kStatusBytes + size_t(B) * size_t(H) * hg::NRB * sizeof(unsigned long long);
    return LR_OK;
}

int hgrn2_launch(const void *q, const void *k, const void *v, const void *g, const float *S0,
                 void *o, float *S_final, int64_t B, int64_t L, int64_t H, void *workspace,
                 cudaStream_t stream, bool preact, float lb) {
    const uint64_t HK = uint64_t(H) * hg::DK, HV = uint64_t(H) * hg::DV;
    CUtensorMap mq, mk, mv, mg;
    if (!hg_map(&mq, q, HK, L, B, 64, true) || !hg_map(&mk, k, HK, L, B, 64, true) ||
        !hg_map(&mv, v, HV, L, B, hg::RB, false) || !hg_map(&mg, g, HV, L, B, hg::RB, false))
        return LR_ERR_CUDA;
    if (!hg_setup_once()) return LR_ERR_CUDA;
    const int n_chunks = static_cast<int>((L + hg::C - 1) / hg::C);
    const int64_t grid = B * H * hg::NRB;
    const uint64_t timeout = g_withheld_split >= 1 ? uint64_t(g_withheld_timeout_ms) * 1000000ull
                                                   : kDefaultTimeoutNs;
    const StatusRef sref = call_status(workspace);   // one stamp for both passes
    auto *redo = reinterpret_cast<unsigned long long *>(static_cast<unsigned char *>(workspace) + kStatusBytes);
    auto first = preact ? hgrn2_chunk_kernel<true, false> : hgrn2_chunk_kernel<false, false>;
    first<<<static_cast<unsigned>(grid), hg::THREADS, hg::SMEM, stream>>>(
        mq, mk, mv, mg, S0, S_final, static_cast<__nv_bfloat16 *>(o), static_cast<int>(L),
        static_cast<int>(H), n_chunks, lb, timeout, sref, redo);
    if (cudaGetLastError() != cudaSuccess) return LR_ERR_CUDA;
    if (preact && lb >= kLbNoSplit) return LR_OK;
    // the redo pass as a programmatic dependent launch: its launch overlaps the
    // first pass, and its blocks wait for the first pass's completion before
    // they read the redo words
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(hg::THREADS);
    cfg.dynamicSmemBytes = hg::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto second = preact ? hgrn2_chunk_kernel<true, true> : hgrn2_chunk_kernel<false, true>;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, second, mq, mk, mv, mg, S0, S_final,
                                             static_cast<__nv_bfloat16 *>(o), static_cast<int>(L),
                                             static_cast<int>(H), n_chunks, lb, timeout, sref, redo);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

}  // namespace lr
