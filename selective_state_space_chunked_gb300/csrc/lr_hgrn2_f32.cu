// lr_hgrn2_f32.cu -- HGRN2 matrix-state recurrence with fp32 I/O on the
// sm_103a tensor cores (frankenstein-transformer docs, HGRN2 Attention page:
// S_t = diag(g_t) S_{t-1} + v_t k_t^T, readout o_t = S_t q_t), for 128 x 128
// heads.
//
// The chunked form is the one of the bf16 kernel (lr_hgrn2.cu): per chunk of
// C = 64 steps, with Lambda the cumulative log2 gates of each value row and
// m its mid-range,
//
//   O    = 2^(Lambda - m) (.) ( tril(Q K^T) V~  +  2^m (.) Q S^T )
//   S^T <- 2^Lambda_C (.) S^T + K^T V~',   V~ = 2^(m - Lambda) (.) V,
//                                         V~' = 2^(Lambda_C - m) V~
//
// To meet fp32 accuracy every tensor-core operand is split into two bf16
// parts, x = x_hi + x_lo with x_hi = bf16(x) and x_lo = bf16(x - x_hi) (16
// mantissa bits between them), and each product X Y is taken as
// X_hi Y_hi + X_hi Y_lo + X_lo Y_hi, accumulated in fp32 TMEM; the dropped
// X_lo Y_lo term is below 2^-16 of the product.  Q and K arrive as fp32 by
// TMA and are split in shared memory; the block itself writes the split
// V~, V~', masked P and state copies.  The factors 2^(Lambda - m), 2^m and
// 2^Lambda_C stay fp32.
//
// A thread block owns 64 value rows of one (batch, head) (grid B * H * 2)
// and runs each chunk in phases separated by block barriers: split Q, K;
// P = Q K^T; gates, factors and the split V~, V~'; the causal mask of P;
// dS^T, OI and OX; the state update and the outputs.  The copies of the
// next chunk's Q, K run during the current chunk.  A chunk whose gates decay
// so steeply that some 16-step quarter of a row falls by more than 2^-40
// (where the factorisation could leave fp32 range) marks its head for the
// step-by-step CUDA-core kernel, which re-runs it in the same call; a gate
// that is not a finite number sets LR_ERR_RANGE.
#include <cudaTypedefs.h>

#include <mutex>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {

namespace hf {
constexpr int C = 64;          // chunk length
constexpr int DK = 128;        // key channels per head
constexpr int DV = 128;        // value channels per head
constexpr int RB = 64;         // value rows per block
constexpr int NRB = DV / RB;
constexpr int NT = 256;        // threads: 8 warps
constexpr int FQ = 4;          // front: quarters of the chunk's steps per value row
constexpr int FS = C / FQ;     // steps per front thread
constexpr float kQuarterSafe = 40.0f;

// shared memory (bytes)
constexpr uint32_t QS = 0;                 // Q fp32 [64 t][128 j], TMA destination
constexpr uint32_t KS = QS + 32768;        // K fp32
constexpr uint32_t QH = KS + 32768;        // Q hi / lo: two 128B-swizzled 64-column halves
constexpr uint32_t QL = QH + 16384;
constexpr uint32_t KH = QL + 16384;        // K hi / lo
constexpr uint32_t KL = KH + 16384;
constexpr uint32_t PH = KL + 16384;        // masked P hi / lo [64 t][64 s], swizzled
constexpr uint32_t PL = PH + 8192;
constexpr uint32_t VH = PL + 8192;         // V~ hi / lo [64 i][64 s], swizzled
constexpr uint32_t VL = VH + 8192;
constexpr uint32_t WH = VL + 8192;         // V~' hi / lo
constexpr uint32_t WL = WH + 8192;
constexpr uint32_t SH = WL + 8192;         // state hi / lo [128 j][64 i], swizzled (MN-major B of OX)
constexpr uint32_t SL = SH + 16384;
constexpr uint32_t E1 = SL + 16384;        // 2^(Lambda - m), fp32 [64 t][64 i] (row-swizzled groups)
constexpr uint32_t EM = E1 + 16384;        // 2^m [64]
constexpr uint32_t GC = EM + 256;          // 2^Lambda_C [64]
constexpr uint32_t TOT = GC + 256;         // quarter totals [4][64]
constexpr uint32_t BAR = TOT + 1024;       // full, mma, done, mma2
constexpr uint32_t TSLOT = BAR + 32;
constexpr uint32_t FLAGS = TSLOT + 16;     // [0] abort, [1] steep chunk seen
constexpr uint32_t SMEM = FLAGS + 16;
static_assert(QH % 1024 == 0 && PH % 1024 == 0 && VH % 1024 == 0 && WH % 1024 == 0 && SH % 1024 == 0,
              "swizzled operand tiles must be 1024-byte aligned");
static_assert(SMEM <= 227 * 1024, "one block per SM");

constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t T_P = 0, T_OI = 64, T_OX = 128, T_DS = 192;

constexpr uint32_t IDESC_P = umma_idesc_bf16(64, 64, 0, 0);
constexpr uint32_t IDESC_OI = umma_idesc_bf16(64, 64, 0, 0);
constexpr uint32_t IDESC_OX = umma_idesc_bf16(64, 64, 0, 1);
constexpr uint32_t IDESC_DS = umma_idesc_bf16(128, 64, 1, 0);

// fp32 [t][i] with 16-byte groups XOR-swizzled by the row, so the 16 rows an
// epilogue half-warp reads at the same columns hit different bank groups
__device__ __forceinline__ int e1_index(int t, int i) {
    return t * RB + ((((i >> 2) ^ (t & 15))) << 2) + (i & 3);
}

// x = hi + lo, both bf16; returns the packed pairs of (a, b)
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}
// eight consecutive values into one 16-byte group of the hi and lo tiles
__device__ __forceinline__ void split8(const float (&x)[8], unsigned char *hi, unsigned char *lo, uint32_t off) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) split2(x[2 * k], x[2 * k + 1], h[k], l[k]);
    *reinterpret_cast<uint4 *>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// the three bf16 products of a split X Y accumulated into d
__device__ __forceinline__ void umma3(uint32_t d, uint64_t ah, uint64_t al, uint64_t bh, uint64_t bl, uint32_t idesc,
                                      bool first) {
    umma_bf16(d, ah, bh, idesc, first ? 0u : 1u);
    umma_bf16(d, ah, bl, idesc, 1u);
    umma_bf16(d, al, bh, idesc, 1u);
}
}  // namespace hf

// PRE: the gate arrives as the pre-activation f, g = lb + (1 - lb) sigmoid(f).
template <bool PRE>
__global__ void __launch_bounds__(hf::NT, 1)
    hgrn2_f32_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const float *__restrict__ v, const float *__restrict__ g, const float *__restrict__ S0,
                     float *__restrict__ S_final, float *__restrict__ o, int L, int H, int n_chunks, float lb,
                     uint64_t timeout_ns, StatusRef sref, unsigned long long *__restrict__ redo) {
    using namespace hf;
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0 && blockIdx.x == 0) status_begin(sref);
    if ((smem_u32(sm) & 1023u) != 0) {   // swizzled tiles need a 1024-byte aligned base
        if (tid == 0) status_report(sref, LR_ERR_CUDA);
        return;
    }
    const int rb = blockIdx.x % NRB, bh = blockIdx.x / NRB;
    const int b = bh / H, h = bh - b * H;
    const int qcol = h * DK, vcol = h * DV + rb * RB;
    const int HV = H * DV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + BAR);
    uint64_t *full = bars, *mma = bars + 1, *done = bars + 2, *mma2 = bars + 3;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + TSLOT);
    volatile int *flags = reinterpret_cast<volatile int *>(sm + FLAGS);
    float *e1 = reinterpret_cast<float *>(sm + E1);
    float *em = reinterpret_cast<float *>(sm + EM);
    float *gc = reinterpret_cast<float *>(sm + GC);
    float *tot = reinterpret_cast<float *>(sm + TOT);

    if (tid == 0) {
        mbar_init(full, 1);
        mbar_init(mma, 1);
        mbar_init(done, 2);   // both MMA issuers (threads 0 and 32)
        mbar_init(mma2, 2);   // dS, OI from thread 0; OX from thread 32
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t s_base = smem_u32(sm);
    if (tid == 0 && n_chunks > 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        mbar_arrive_expect_tx(full, 2 * 32768);
        tma_load_3d(sm + QS, &tm_q, full, qcol, 0, b);
        tma_load_3d(sm + KS, &tm_k, full, qcol, 0, b);
    }

    // state: key column j = 32 (warp % 4) + lane, value rows [32 rh, 32 rh + 32)
    const int j = 32 * (warp & 3) + lane, rh = warp >> 2;
    const size_t srow = size_t(bh) * DV + size_t(rb) * RB + 32 * rh;
    float S[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) S[r] = S0 != nullptr ? S0[(srow + r) * DK + j] : 0.0f;
    auto write_state = [&]() {   // row j of the [128 j][64 i] tiles, columns 32 rh ..
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = S[8 * k + e];
            split8(x, sm + SH, sm + SL, sw128_offset(j, 32 * rh + 8 * k));
        }
    };
    write_state();

    // front: value row i, steps [fs0, fs0 + 16) of the chunk
    const int fi = tid & (RB - 1), fq = tid >> 6, fs0 = FS * fq;
    // epilogue / mask: rows t of the warp's quarter, column halves
    const int quarter = warp & 3;
    const int et = 16 * quarter + (lane & 15);
    uint32_t mma_phase = 0, mma2_phase = 0;
    bool ok = true;
    int pending = n_chunks > 0 ? 0 : -1;   // chunk whose Q, K copy is in flight

    for (int c = 0; c < n_chunks && ok; ++c) {
        const int t0 = c * C;
        // this thread's gates and values (global, coalesced over the rows)
        float gv[FS], vv[FS];
#pragma unroll
        for (int u = 0; u < FS; ++u) {
            const int t = t0 + fs0 + u;
            const size_t a = (size_t(b) * L + t) * HV + vcol + fi;
            gv[u] = t < L ? g[a] : (PRE ? 0.0f : 1.0f);
            vv[u] = t < L ? v[a] : 0.0f;
        }
        // Q, K of chunk c landed: split them
        if (!mbar_wait_bounded(full, c & 1, timeout_ns)) flags[0] = 1;
        if (__syncthreads_or(flags[0] != 0)) {
            ok = false;
            break;
        }
        pending = -1;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int gi = tid + NT * k;           // 2048 groups of 8 columns: Q then K
            const int tens = gi >> 10, gr = gi & 1023;
            const int t = gr >> 4, c8 = gr & 15;
            const float *src = reinterpret_cast<const float *>(sm + (tens ? KS : QS)) + t * DK + 8 * c8;
            const float4 a0 = *reinterpret_cast<const float4 *>(src);
            const float4 a1 = *reinterpret_cast<const float4 *>(src + 4);
            const float x[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint32_t off = (c8 >> 3) * 8192u + sw128_offset(t, (c8 & 7) * 8);
            split8(x, sm + (tens ? KH : QH), sm + (tens ? KL : QL), off);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            if (c + 1 < n_chunks) {   // the staging is free: copy the next chunk
                pending = c + 1;
                mbar_arrive_expect_tx(full, 2 * 32768);
                tma_load_3d(sm + QS, &tm_q, full, qcol, (c + 1) * C, b);
                tma_load_3d(sm + KS, &tm_k, full, qcol, (c + 1) * C, b);
            }
        }

        // gates: running products over this thread's 16 steps, forward
        // (pf[u] = g_0 .. g_u) and backward (pr[u] = g_u+1 .. g_15), and the
        // log2 of their product.  A head whose quarter product falls below
        // 2^-kQuarterSafe is re-run step by step, so on the heads kept the
        // products stay normal and the per-step factors need no exp2 of their
        // own: 2^(Lambda_t - m) = 2^(off - m) pf[u], 2^(m - Lambda_t) =
        // 2^(m - off - acc) pr[u]
        float pf[FS], pr[FS];
        float prod = 1.0f;
#pragma unroll
        for (int u = 0; u < FS; ++u) {
            float gg = gv[u];
            if (PRE) gg = t0 + fs0 + u < L ? fmaf(1.0f - lb, rcp_approx(1.0f + ex2_approx(-gg * kLog2e)), lb) : 1.0f;
            gv[u] = gg;
            prod *= gg;
            pf[u] = prod;
        }
        pr[FS - 1] = 1.0f;
#pragma unroll
        for (int u = FS - 2; u >= 0; --u) pr[u] = pr[u + 1] * gv[u + 1];
        const float acc = lg2_approx(prod);
        if (!(acc == acc) || acc == __int_as_float(0x7f800000)) status_report(sref, LR_ERR_RANGE);
        if (-acc > kQuarterSafe) flags[1] = 1;   // steep: the head is re-run step by step
        tot[fq * RB + fi] = acc;
        __syncthreads();
        if (tid == 0) {   // P = Q K^T, after this thread's share of the gate work
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
                umma3(tmem + T_P, umma_smem_desc(s_base + QH + off, 16, 1024),
                      umma_smem_desc(s_base + QL + off, 16, 1024), umma_smem_desc(s_base + KH + off, 16, 1024),
                      umma_smem_desc(s_base + KL + off, 16, 1024), IDESC_P, kk == 0);
            }
            umma_commit(mma);
        }
        float off = 0.0f, lc = 0.0f;
#pragma unroll
        for (int q = 0; q < FQ; ++q) {
            const float tq = tot[q * RB + fi];
            off += q < fq ? tq : 0.0f;
            lc += tq;
        }
        const float m = 0.5f * lc;
        if (fq == 0) {
            em[fi] = ex2_approx(m);
            gc[fi] = ex2_approx(lc);
        }
        const float cm = ex2_approx(lc - m);
        const float ea = ex2_approx(off - m), eb = ex2_approx(m - off - acc);
        float vt[FS], vtp[FS];
#pragma unroll
        for (int u = 0; u < FS; ++u) {
            e1[e1_index(fs0 + u, fi)] = ea * pf[u];
            vt[u] = eb * pr[u] * vv[u];
            vtp[u] = vt[u] * cm;
        }
#pragma unroll
        for (int k = 0; k < FS / 8; ++k) {
            float x[8], y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                x[e] = vt[8 * k + e];
                y[e] = vtp[8 * k + e];
            }
            split8(x, sm + VH, sm + VL, sw128_offset(fi, fs0 + 8 * k));
            split8(y, sm + WH, sm + WL, sw128_offset(fi, fs0 + 8 * k));
        }

        // P ready: causal mask into the split tiles
        if (!mbar_wait_bounded(mma, mma_phase & 1, timeout_ns)) flags[0] = 1;
        ++mma_phase;
        tc_fence_after();
        if (__syncthreads_or(flags[0] != 0)) {
            ok = false;
            break;
        }
        {
            const int s0 = 32 * (warp >> 2) + 16 * (lane >> 4);
            float pv[16];
            tmem_ld16x2_nowait<16>(tmem + T_P + 32 * (warp >> 2) + (uint32_t(quarter * 32) << 16), pv);
            tmem_ld_wait_tied(pv);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = s0 + 8 * k + e <= et ? pv[8 * k + e] : 0.0f;
                split8(x, sm + PH, sm + PL, sw128_offset(et, s0 + 8 * k));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // dS^T = K^T V~' and OI = tril(P) V~ from thread 0, OX = Q S^T from
        // thread 32 (a lane of another warp): two issuers halve the time the
        // MMAs take to issue; each accumulator has one issuer, so its order
        // of accumulation is unchanged
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                umma3(tmem + T_DS, umma_smem_desc(s_base + KH + kk * 2048, 8192, 1024),
                      umma_smem_desc(s_base + KL + kk * 2048, 8192, 1024),
                      umma_smem_desc(s_base + WH + kk * 32, 16, 1024), umma_smem_desc(s_base + WL + kk * 32, 16, 1024),
                      IDESC_DS, kk == 0);
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                umma3(tmem + T_OI, umma_smem_desc(s_base + PH + kk * 32, 16, 1024),
                      umma_smem_desc(s_base + PL + kk * 32, 16, 1024), umma_smem_desc(s_base + VH + kk * 32, 16, 1024),
                      umma_smem_desc(s_base + VL + kk * 32, 16, 1024), IDESC_OI, kk == 0);
            umma_commit(mma2);
        } else if (tid == 32) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                const uint32_t qoff = (kk >> 2) * 8192 + (kk & 3) * 32;
                umma3(tmem + T_OX, umma_smem_desc(s_base + QH + qoff, 16, 1024),
                      umma_smem_desc(s_base + QL + qoff, 16, 1024),
                      umma_smem_desc(s_base + SH + kk * 2048, 8192, 1024),
                      umma_smem_desc(s_base + SL + kk * 2048, 8192, 1024), IDESC_OX, kk == 0);
            }
            umma_commit(mma2);
        }
        if (!mbar_wait_bounded(mma2, mma2_phase & 1, timeout_ns)) flags[0] = 1;
        ++mma2_phase;
        tc_fence_after();
        if (__syncthreads_or(flags[0] != 0)) {
            ok = false;
            break;
        }

        // state: S = diag(2^Lambda_C) S + dS  (dS^T: lane j, columns = value rows)
        {
            float d[32];
            tmem_ld32_nowait(tmem + T_DS + 32 * rh + (uint32_t(32 * (warp & 3)) << 16), d);
            tmem_ld_wait_tied(d);
#pragma unroll
            for (int r = 0; r < 32; ++r) S[r] = fmaf(gc[32 * rh + r], S[r], d[r]);
        }
        // outputs o_t = 2^(Lambda_t - m) (OI_t + 2^m OX_t), rows t of the
        // quarter, columns [c0, c0 + 16) and [c0 + 32, c0 + 48)
        {
            const int c0 = 16 * rh;
            float oi[16], ox[16];
            tmem_ld16x2_nowait<32>(tmem + T_OI + c0 + (uint32_t(quarter * 32) << 16), oi);
            tmem_ld16x2_nowait<32>(tmem + T_OX + c0 + (uint32_t(quarter * 32) << 16), ox);
            tmem_ld_wait_tied(oi, ox);
            const int i0 = c0 + 32 * (lane >> 4);
            if (t0 + et < L) {
                float4 *dst = reinterpret_cast<float4 *>(o + (size_t(b) * L + t0 + et) * HV + vcol + i0);
#pragma unroll
                for (int q = 0; q < 16; q += 4) {
                    const float4 e = *reinterpret_cast<const float4 *>(e1 + e1_index(et, i0 + q));
                    const float4 mm = *reinterpret_cast<const float4 *>(em + i0 + q);
                    dst[q / 4] = make_float4(fmaf(mm.x, ox[q], oi[q]) * e.x, fmaf(mm.y, ox[q + 1], oi[q + 1]) * e.y,
                                             fmaf(mm.z, ox[q + 2], oi[q + 2]) * e.z,
                                             fmaf(mm.w, ox[q + 3], oi[q + 3]) * e.w);
                }
            }
        }
        tc_fence_before();
        __syncthreads();   // every thread is past its reads of OX's operand and of E1, 2^m
        write_state();
        fence_proxy_async_smem();
        __syncthreads();
    }

    if (ok && S_final != nullptr) {
#pragma unroll
        for (int r = 0; r < 32; ++r) S_final[(srow + r) * DK + j] = S[r];
    }
    if (tid == 0 && flags[1] != 0) redo[bh] = sref.stamp;   // both blocks of the head may write it
    // nothing of this block's may still run on the tensor cores or land in its
    // shared memory when it exits
    if (tid == 0 || tid == 32) umma_commit(done);   // each issuer's MMAs
    if (tid == 0) {
        mbar_wait_bounded(done, 0, timeout_ns);
        if (pending >= 0) mbar_wait_bounded(full, pending & 1, timeout_ns);   // after a failed wait only
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

template <typename K>
bool hf_smem_attr(K kern) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(hf::SMEM)) ==
           cudaSuccess;
}

bool hf_setup_once() {
    static std::once_flag once;
    static bool ok = false;
    std::call_once(once, [] { ok = hf_smem_attr(hgrn2_f32_kernel<false>) && hf_smem_attr(hgrn2_f32_kernel<true>); });
    return ok;
}

}  // namespace

int hgrn2_f32_launch(const void *q, const void *k, const void *v, const void *g, const float *S0, void *o,
                     float *S_final, int64_t B, int64_t L, int64_t H, void *workspace, cudaStream_t stream,
                     bool preact, float lb) {
    const uint64_t HK = uint64_t(H) * hf::DK;
    CUtensorMap mq, mk;
    if (!encode_map_3d(&mq, q, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, HK, uint64_t(L), uint64_t(B), hf::DK, hf::C, 1) ||
        !encode_map_3d(&mk, k, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, HK, uint64_t(L), uint64_t(B), hf::DK, hf::C, 1))
        return LR_ERR_CUDA;
    if (!hf_setup_once()) return LR_ERR_CUDA;
    const int n_chunks = static_cast<int>((L + hf::C - 1) / hf::C);
    const int64_t grid = B * H * hf::NRB;
    const uint64_t timeout = g_withheld_split >= 1 ? uint64_t(g_withheld_timeout_ms) * 1000000ull : kDefaultTimeoutNs;
    const StatusRef sref = call_status(workspace);
    auto *redo = reinterpret_cast<unsigned long long *>(static_cast<unsigned char *>(workspace) + kStatusBytes);
    auto kern = preact ? hgrn2_f32_kernel<true> : hgrn2_f32_kernel<false>;
    kern<<<static_cast<unsigned>(grid), hf::NT, hf::SMEM, stream>>>(
        mq, mk, static_cast<const float *>(v), static_cast<const float *>(g), S0, S_final, static_cast<float *>(o),
        static_cast<int>(L), static_cast<int>(H), n_chunks, lb, timeout, sref, redo);
    if (cudaGetLastError() != cudaSuccess) return LR_ERR_CUDA;
    // heads with a steep chunk: the step-by-step kernel re-runs them (its
    // blocks of other heads return at once); not needed when lb rules them out
    if (preact && lb >= 0.18f) return LR_OK;
    return hgrn2_general_launch(q, k, v, g, S0, o, S_final, B, L, H, hf::DK, hf::DV, 0, preact, lb, workspace,
                                stream, redo, sref.stamp);
}

}  // namespace lr
