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
// V~ = 2^(m - Lambda) (.) V and S~ = diag(2^m) S,
//
//   O   = 2^(Lambda - m) (.) ( tril(Q K^T) V~  +  2^m (.) Q S^T )
//   dS^T = K^T (2^(Lambda_C - Lambda) (.) V)                       (state update, in TMEM)
//
// Four tcgen05 MMAs per chunk (bf16 operands in shared memory, fp32
// accumulators in tensor memory):
//   P   = Q K^T            M=64  N=64 K=128   A = Q (K-major),  B = K (K-major)
//   OX  = Q S^T            M=64  N=32 K=128   B = bf16 state rows (K-major, written by the block)
//   dSt = K^T V~'          M=128 N=32 K=64    A = the same K tile read MN-major
//   OI  = tril(P) V~       M=64  N=32 K=64    A = masked P (bf16, written by the block)
// P and OX of chunk c+1 depend only on its Q, K and the state after chunk c,
// so they are issued as soon as chunk c's state update is written and run
// while the block computes chunk c+1's gates.  Q, K (128B-swizzled) and the
// block's V, g columns arrive by TMA, two chunks in flight.  Rows of S evolve independently (diag(g) scales rows), so a
// thread block owns 32 value rows of one (batch, head): 4 blocks per head.
// The fp32 state lives in registers (thread j holds column j of its 32 rows)
// and is updated elementwise from dS^T; it never leaves the chip between
// chunks.
#include <cudaTypedefs.h>

#include <mutex>

#include "lr_device.cuh"
#include "lr_internal.h"

namespace lr {

__device__ int g_hgrn2_status = 0;

__device__ __forceinline__ void hg_report(int code) { atomicCAS(&g_hgrn2_status, 0, code); }

namespace hg {
constexpr int C = 64;          // chunk length
constexpr int DK = 128;        // key channels per head
constexpr int DV = 128;        // value channels per head
constexpr int RB = 32;         // value rows of S per thread block
constexpr int NRB = DV / RB;   // blocks per head
constexpr int THREADS = 128;
constexpr int STAGES = 2;
// largest per-chunk spread of Lambda (log2 units) the reference split keeps
// inside fp32 range with headroom: 2^(+-80) factors
constexpr float kMaxSpread = 160.0f;

constexpr uint32_t Q_BYTES = C * DK * 2;   // two 64-column 128B-swizzled halves
constexpr uint32_t VG_BYTES = C * RB * 2;  // plain rows of 32 bf16
constexpr uint32_t STAGE_BYTES = 2 * Q_BYTES + 2 * VG_BYTES;
constexpr uint32_t OFF_P = STAGES * STAGE_BYTES;   // masked P, [64 t][64 s] swizzled
constexpr uint32_t OFF_VT = OFF_P + 8192;          // V~ as [32 i][64 s] swizzled
constexpr uint32_t OFF_VTP = OFF_VT + 4096;        // V~' as [32 i][64 s] swizzled
constexpr uint32_t OFF_SB = OFF_VTP + 4096;        // bf16 state rows [32 i][128 j], two swizzled halves
constexpr uint32_t OFF_LAM = OFF_SB + 8192;        // 2^(Lambda - m), float [64][32], 16-byte groups XOR-swizzled
constexpr uint32_t OFF_TOT = OFF_LAM + 8192;       // per-warp partial sums, float [4][32]
constexpr uint32_t OFF_L0 = OFF_TOT + 512;         // Lambda_0, float [32]
constexpr uint32_t OFF_M = OFF_L0 + 128;           // m, float [32]
constexpr uint32_t OFF_LC = OFF_M + 128;           // 2^Lambda_C, float [32]
constexpr uint32_t OFF_BAR = OFF_LC + 128;         // full[2], bar_p, bar_o
constexpr uint32_t OFF_TMEM = OFF_BAR + 32;
constexpr uint32_t SMEM = OFF_TMEM + 16;
static_assert(OFF_P % 1024 == 0 && OFF_VT % 1024 == 0 && OFF_VTP % 1024 == 0 &&
                  OFF_SB % 1024 == 0 && STAGE_BYTES % 1024 == 0,
              "swizzled operand tiles must be 1024-byte aligned");

constexpr uint32_t TMEM_COLS = 256;  // two blocks per SM fill the 512 columns exactly
constexpr uint32_t T_P = 0, T_OI = 64, T_OX = 96, T_S = 128;   // accumulator columns

constexpr uint32_t IDESC_P = umma_idesc_bf16(64, 64, 0, 0);
constexpr uint32_t IDESC_O = umma_idesc_bf16(64, RB, 0, 0);
constexpr uint32_t IDESC_S = umma_idesc_bf16(128, RB, 1, 0);
// Lambda[t][i] lives at a row-wise XOR swizzle of 4-float groups, so 16 lanes
// reading 16 rows at the same channel group hit 8 different bank groups.
__device__ __forceinline__ int lam_index(int t, int i) {
    return t * RB + ((((i >> 2) ^ (t & 7))) << 2) + (i & 3);
}
}  // namespace hg

__global__ void __launch_bounds__(hg::THREADS)
    hgrn2_chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                       const float *__restrict__ S0, float *__restrict__ S_final,
                       __nv_bfloat16 *__restrict__ o, int L, int H, int n_chunks,
                       uint64_t timeout_ns) {
    using namespace hg;
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((smem_u32(sm) & 1023u) != 0) {  // swizzled tiles need a 1024-byte aligned base
        if (tid == 0) hg_report(LR_ERR_CUDA);
        return;
    }
    const int blk = blockIdx.x;
    const int rb = blk % NRB, bh = blk / NRB;
    const int b = bh / H, h = bh - (bh / H) * H;
    const int qcol = h * DK, vcol = h * DV + rb * RB;
    const int HV = H * DV;

    uint64_t *full = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    uint64_t *bar_p = full + 2;
    uint64_t *bar_o = full + 3;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_TMEM);
    float *LAM = reinterpret_cast<float *>(sm + OFF_LAM);  // 2^(Lambda - m) per [t][i]
    float *TOT = reinterpret_cast<float *>(sm + OFF_TOT);
    float *L0S = reinterpret_cast<float *>(sm + OFF_L0);
    float *MS = reinterpret_cast<float *>(sm + OFF_M);
    float *LCS = reinterpret_cast<float *>(sm + OFF_LC);
    unsigned char *Ps = sm + OFF_P, *VT = sm + OFF_VT, *VTP = sm + OFF_VTP, *SB = sm + OFF_SB;

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(bar_p, 1);
        mbar_init(bar_o, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_g);
    }
    if (warp == 0) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // state rows rb*32 .. rb*32+31 of S[b, h]; this thread holds column j = tid
    const size_t srow0 = (size_t(b) * H + h) * DV + size_t(rb) * RB;
    float S[RB];
#pragma unroll
    for (int i = 0; i < RB; ++i) S[i] = S0 != nullptr ? S0[(srow0 + i) * DK + tid] : 0.0f;

    auto issue = [&](int c, int st) {  // thread 0: TMA for chunk c into stage st
        unsigned char *stg = sm + st * STAGE_BYTES;
        mbar_arrive_expect_tx(&full[st], STAGE_BYTES);
        tma_load_3d(stg, &tm_q, &full[st], qcol, c * C, b);
        tma_load_3d(stg + 8192, &tm_q, &full[st], qcol + 64, c * C, b);
        tma_load_3d(stg + Q_BYTES, &tm_k, &full[st], qcol, c * C, b);
        tma_load_3d(stg + Q_BYTES + 8192, &tm_k, &full[st], qcol + 64, c * C, b);
        tma_load_3d(stg + 2 * Q_BYTES, &tm_v, &full[st], vcol, c * C, b);
        tma_load_3d(stg + 2 * Q_BYTES + VG_BYTES, &tm_g, &full[st], vcol, c * C, b);
    };
    // thread 0: P = Q K^T and OX = Q S^T for the chunk whose inputs sit in stage st
    auto issue_p_ox = [&](int st) {
        const uint32_t sQ = smem_u32(sm + st * STAGE_BYTES), sK = sQ + Q_BYTES;
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
            umma_bf16(tmem + T_P, umma_smem_desc(sQ + off, 16, 1024),
                      umma_smem_desc(sK + off, 16, 1024), IDESC_P, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 8192 + (kk & 3) * 32;
            umma_bf16(tmem + T_OX, umma_smem_desc(sQ + off, 16, 1024),
                      umma_smem_desc(smem_u32(SB) + (kk >> 2) * 4096 + (kk & 3) * 32, 16, 1024),
                      IDESC_O, kk > 0);
        }
        umma_commit(bar_p);
    };
    // bf16 copy of the state rows [i][j] (K-major B operand of Q S^T)
    auto write_state_bf16 = [&]() {
        const int j = tid, hj = j >> 6, jc = j & 63;
#pragma unroll
        for (int i = 0; i < RB; ++i)
            *reinterpret_cast<__nv_bfloat16 *>(SB + hj * 4096 + sw128_offset(i, jc)) =
                __float2bfloat16_rn(S[i]);
    };

    write_state_bf16();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        issue(0, 0);
        if (n_chunks > 1) issue(1, 1);
        if (mbar_wait_bounded(&full[0], 0, timeout_ns)) {
            tc_fence_after();
            issue_p_ox(0);
        }
    }

    for (int c = 0; c < n_chunks; ++c) {
        const int st = c & 1;
        unsigned char *stg = sm + st * STAGE_BYTES;
        const uint32_t sK = smem_u32(stg) + Q_BYTES;
        const __nv_bfloat16 *sV = reinterpret_cast<const __nv_bfloat16 *>(stg + 2 * Q_BYTES);
        const __nv_bfloat16 *sG = sV + C * RB;
        const int t0 = c * C;

        const bool ok_in = mbar_wait_bounded(&full[st], (c >> 1) & 1, timeout_ns);
        if (__syncthreads_or(!ok_in)) {
            if (tid == 0) hg_report(LR_ERR_TIMEOUT);
            break;
        }

        // ---- cumulative log2 gates: warp w takes rows 16w..16w+15, lane = value channel
        float loc[16];
        {
            float acc = 0.0f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int t = 16 * warp + u;
                const float gv = __bfloat162float(sG[t * RB + lane]);
                acc += t0 + t < L ? lg2_approx(gv) : 0.0f;  // rows past L: g = 1
                loc[u] = acc;
            }
            TOT[warp * 32 + lane] = acc;
            if (warp == 0) L0S[lane] = loc[0];
        }
        __syncthreads();

        // ---- causal mask of P = Q K^T (issued at the end of the previous chunk)
        bool ok = mbar_wait_bounded(bar_p, c & 1, timeout_ns);
        tc_fence_after();
        {
            const uint32_t ta = tmem + T_P + (uint32_t(warp * 32) << 16);
            const int t = 16 * warp + lane;  // valid for lane < 16 (M = 64 layout)
            float pa[32], pb[32];
            tmem_ld32_nowait(ta, pa);
            tmem_ld32_nowait(ta + 32, pb);
            tmem_ld_wait();
            if (lane < 16) {
#pragma unroll
                for (int chunk = 0; chunk < 8; ++chunk) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s0 = chunk * 8 + 2 * e;
                        const float v0 = s0 < 32 ? pa[s0] : pb[s0 - 32];
                        const float v1 = s0 + 1 < 32 ? pa[s0 + 1] : pb[s0 + 1 - 32];
                        __nv_bfloat162 pr = __floats2bfloat162_rn(s0 <= t ? v0 : 0.0f,
                                                                  s0 + 1 <= t ? v1 : 0.0f);
                        w4[e] = *reinterpret_cast<uint32_t *>(&pr);
                    }
                    *reinterpret_cast<uint4 *>(Ps + t * 128 + ((chunk ^ (t & 7)) << 4)) =
                        make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            }
        }

        // ---- Lambda, reference m, V~ and V~'
        {
            float off = 0.0f, lc = 0.0f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float tw = TOT[w * 32 + lane];
                off += w < warp ? tw : 0.0f;
                lc += tw;
            }
            const float l0 = L0S[lane];
            const float m = 0.5f * (l0 + lc);
            if (warp == 0 && !(l0 - lc <= kMaxSpread)) hg_report(LR_ERR_RANGE);
            // 2^(Lambda_C - Lambda) = 2^(m - Lambda) 2^(Lambda_C - m); both factors stay
            // inside fp32 range because |Lambda - m| and |Lambda_C - m| are at most 80
            const float cm = ex2_approx(lc - m);
            uint32_t vt[8], vtp[8];  // bf16 pairs of this lane's row, columns 16w .. 16w+15
#pragma unroll
            for (int u = 0; u < 16; u += 2) {
                const int t = 16 * warp + u;
                const float lam0 = loc[u] + off, lam1 = loc[u + 1] + off;
                LAM[lam_index(t, lane)] = ex2_approx(lam0 - m);
                LAM[lam_index(t + 1, lane)] = ex2_approx(lam1 - m);
                const float v0 = __bfloat162float(sV[t * RB + lane]);
                const float v1 = __bfloat162float(sV[(t + 1) * RB + lane]);
                const float w0 = ex2_approx(m - lam0) * v0, w1 = ex2_approx(m - lam1) * v1;
                __nv_bfloat162 a = __floats2bfloat162_rn(w0, w1);
                __nv_bfloat162 bq = __floats2bfloat162_rn(w0 * cm, w1 * cm);
                vt[u / 2] = *reinterpret_cast<uint32_t *>(&a);
                vtp[u / 2] = *reinterpret_cast<uint32_t *>(&bq);
            }
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {   // two 16-byte chunks: columns 16w + 8*h8 ..
                const uint32_t off8 = sw128_offset(lane, 16 * warp + 8 * h8);
                *reinterpret_cast<uint4 *>(VT + off8) =
                    make_uint4(vt[4 * h8], vt[4 * h8 + 1], vt[4 * h8 + 2], vt[4 * h8 + 3]);
                *reinterpret_cast<uint4 *>(VTP + off8) =
                    make_uint4(vtp[4 * h8], vtp[4 * h8 + 1], vtp[4 * h8 + 2], vtp[4 * h8 + 3]);
            }
            if (warp == 0) {
                MS[lane] = ex2_approx(m);
                LCS[lane] = ex2_approx(lc);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) {
            if (tid == 0) hg_report(LR_ERR_TIMEOUT);
            break;
        }
        if (tid == 0) {
            tc_fence_after();
            // dS^T = K^T V~'  (K tile read MN-major: 64-column halves 8 KB apart)
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                umma_bf16(tmem + T_S, umma_smem_desc(sK + kk * 2048, 8192, 1024),
                          umma_smem_desc(smem_u32(VTP) + kk * 32, 16, 1024), IDESC_S, kk > 0);
            // OI = tril(P) V~
#pragma unroll
            for (int kk = 0; kk < C / 16; ++kk)
                umma_bf16(tmem + T_OI, umma_smem_desc(smem_u32(Ps) + kk * 32, 16, 1024),
                          umma_smem_desc(smem_u32(VT) + kk * 32, 16, 1024), IDESC_O, kk > 0);
            umma_commit(bar_o);
        }
        ok = mbar_wait_bounded(bar_o, c & 1, timeout_ns);
        tc_fence_after();
        {   // ---- output rows: o_t = 2^(Lambda_t - m) (OI_t + 2^m OX_t)
            const uint32_t lw = uint32_t(warp * 32) << 16;
            const int t = 16 * warp + lane;
            float oi[32], ox[32];
            tmem_ld32_nowait(tmem + T_OI + lw, oi);
            tmem_ld32_nowait(tmem + T_OX + lw, ox);
            tmem_ld_wait();
            if (lane < 16 && t0 + t < L) {
                uint4 w4[4];
                uint32_t *wp = reinterpret_cast<uint32_t *>(w4);
#pragma unroll
                for (int i = 0; i < RB; i += 4) {
                    const float4 e1 = *reinterpret_cast<const float4 *>(LAM + lam_index(t, i));
                    const float4 em = *reinterpret_cast<const float4 *>(MS + i);
                    const float r0 = fmaf(em.x, ox[i], oi[i]) * e1.x;
                    const float r1 = fmaf(em.y, ox[i + 1], oi[i + 1]) * e1.y;
                    const float r2 = fmaf(em.z, ox[i + 2], oi[i + 2]) * e1.z;
                    const float r3 = fmaf(em.w, ox[i + 3], oi[i + 3]) * e1.w;
                    __nv_bfloat162 p0 = __floats2bfloat162_rn(r0, r1);
                    __nv_bfloat162 p1 = __floats2bfloat162_rn(r2, r3);
                    wp[i / 2] = *reinterpret_cast<uint32_t *>(&p0);
                    wp[i / 2 + 1] = *reinterpret_cast<uint32_t *>(&p1);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(o + (size_t(b) * L + t0 + t) * HV + vcol);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = w4[q];
            }
        }
        {   // ---- state: S = diag(2^Lambda_C) S + dS, and its bf16 copy for the next chunk
            const uint32_t ta = tmem + T_S + (uint32_t(warp * 32) << 16);
            float ds[32];
            tmem_ld32_nowait(ta, ds);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < RB; ++i) S[i] = fmaf(LCS[i], S[i], ds[i]);
            write_state_bf16();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) {
            if (tid == 0) hg_report(LR_ERR_TIMEOUT);
            break;
        }
        if (tid == 0) {
            if (c + 2 < n_chunks) issue(c + 2, st);
            if (c + 1 < n_chunks &&
                mbar_wait_bounded(&full[(c + 1) & 1], ((c + 1) >> 1) & 1, timeout_ns)) {
                tc_fence_after();
                issue_p_ox((c + 1) & 1);
            }
        }
    }

    if (S_final != nullptr) {
#pragma unroll
        for (int i = 0; i < RB; ++i) S_final[(srow0 + i) * DK + tid] = S[i];
    }
    tc_fence_before();
    __syncthreads();
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

bool hg_setup_once() {
    static std::once_flag once;
    static bool ok = false;
    std::call_once(once, [] {
        ok = cudaFuncSetAttribute(hgrn2_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(hg::SMEM)) == cudaSuccess;
    });
    return ok;
}

}  // namespace

int hgrn2_workspace(int64_t, int64_t, int64_t, size_t *bytes) {
    *bytes = 0;
    return LR_OK;
}

int hgrn2_launch(const void *q, const void *k, const void *v, const void *g, const float *S0,
                 void *o, float *S_final, int64_t B, int64_t L, int64_t H, void *,
                 cudaStream_t stream) {
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
    hgrn2_chunk_kernel<<<static_cast<unsigned>(grid), hg::THREADS, hg::SMEM, stream>>>(
        mq, mk, mv, mg, S0, S_final, static_cast<__nv_bfloat16 *>(o), static_cast<int>(L),
        static_cast<int>(H), n_chunks, timeout);
    return cudaGetLastError() == cudaSuccess ? LR_OK : LR_ERR_CUDA;
}

int hgrn2_status_read_and_clear(int *status) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_hgrn2_status, sizeof(int)) != cudaSuccess) return LR_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_hgrn2_status, &zero, sizeof(int)) != cudaSuccess)
            return LR_ERR_CUDA;
    }
    *status = v;
    return LR_OK;
}

}  // namespace lr
