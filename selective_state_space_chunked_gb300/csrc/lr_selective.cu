// lr_selective.cu -- host side of the selective SSM scan: the work plan, the
// workspace layout and the launch ([SSM] cortexnet 3.2.1, cortexnet/ssm.py,
// MultiScaleSSM._selective_scan).  The kernel and its design notes are in
// lr_selective.cuh; its variants are compiled in lr_sel_*.cu.
#include "lr_selective.cuh"

namespace lr {
namespace {

template <typename IO>
using HostCfg = SelCfg<IO, cpl_of<IO>()>;

// The compiled variants of one I/O type: (z gate, softplus on dt) -> entry points.
struct VariantFns {
    int (*launch)(const CUtensorMap *, const SelArgs &, int, cudaStream_t);
    int (*blocks)(int);
};
const VariantFns &variant_of(bool bf16, bool hz, bool sp) {
    static const VariantFns t[8] = {
        {sel::launch_f32_noz_nosp, sel::blocks_f32_noz_nosp},    {sel::launch_f32_noz_sp, sel::blocks_f32_noz_sp},
        {sel::launch_f32_z_nosp, sel::blocks_f32_z_nosp},        {sel::launch_f32_z_sp, sel::blocks_f32_z_sp},
        {sel::launch_bf16_noz_nosp, sel::blocks_bf16_noz_nosp},  {sel::launch_bf16_noz_sp, sel::blocks_bf16_noz_sp},
        {sel::launch_bf16_z_nosp, sel::blocks_bf16_z_nosp},      {sel::launch_bf16_z_sp, sel::blocks_bf16_z_sp}};
    return t[(bf16 ? 4 : 0) + (hz ? 2 : 0) + (sp ? 1 : 0)];
}

// Resident blocks per SM over the four variants of an I/O type (they share
// block size and shared memory).
int resident_blocks(bool bf16, int dev) {
    int n = 1 << 30;
    for (int v = 0; v < 4; ++v) {
        const int k = variant_of(bf16, v & 2, v & 1).blocks(dev);
        n = k < n ? k : n;
    }
    return n;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

struct SelLayout {
    size_t ticket, ticket2, flags, defer, ctl, agg, incl, total;
};

SelLayout sel_layout(int W, int wch) {
    SelLayout s{};
    s.ticket = kStatusBytes;
    s.ticket2 = s.ticket + 4;
    s.flags = s.ticket + 8;
    s.defer = s.flags + size_t(W) * 4;
    s.ctl = (s.defer + size_t(W) * 4 + 7) & ~size_t(7);
    s.agg = align256(s.ctl + size_t(W) * 8);
    s.incl = s.agg + align256(size_t(W) * (kN + 1) * wch * sizeof(float));
    s.total = s.incl + align256(size_t(W) * kN * wch * sizeof(float));
    return s;
}

template <typename IO, bool ACC>
int launch_t(const void *x, const void *dt, const void *z, const void *Bm, const void *Cm, const float *A_log,
             const float *Dskip, const float *h0, void *y, float *h_final, int64_t B, int64_t L, int64_t D,
             int dt_softplus, const DiagPlan &p, void *workspace, cudaStream_t stream) {
    constexpr uint32_t wch = HostCfg<IO>::WCH;
    const auto tt = Io<IO>::kTmType;
    CUtensorMap mp[6];
    if (!encode_map_3d(&mp[0], x, tt, sizeof(IO), D, L, B, wch, kT, 1) ||
        !encode_map_3d(&mp[1], dt, tt, sizeof(IO), D, L, B, wch, kT, 1) ||
        !encode_map_3d(&mp[2], z != nullptr ? z : x, tt, sizeof(IO), D, L, B, wch, kT, 1) ||
        !encode_map_3d(&mp[3], Bm, tt, sizeof(IO), kN, L, B, kN, kT, 1) ||
        !encode_map_3d(&mp[4], Cm, tt, sizeof(IO), kN, L, B, kN, kT, 1) ||
        !encode_map_3d(&mp[5], y, tt, sizeof(IO), D, L, B, wch, kT, 1))
        return LR_ERR_CUDA;
    const SelLayout lay = sel_layout(p.warps, wch);
    char *ws = static_cast<char *>(workspace);
    if (cudaMemsetAsync(ws + lay.ticket, 0, lay.agg - lay.ticket, stream) != cudaSuccess) return LR_ERR_CUDA;
    SelArgs a{};
    a.A_log = A_log;
    a.Dskip = Dskip;
    a.h0 = h0;
    a.y = y;
    a.h_final = h_final;
    a.B = static_cast<int>(B);
    a.L = static_cast<int>(L);
    a.D = static_cast<int>(D);
    a.ntt = p.n_tiles;
    a.F = static_cast<long long>(p.n_cb) * p.n_tiles;
    a.W = p.warps;
    a.ticket = reinterpret_cast<uint32_t *>(ws + lay.ticket);
    a.ticket2 = reinterpret_cast<uint32_t *>(ws + lay.ticket2);
    a.defer = reinterpret_cast<uint32_t *>(ws + lay.defer);
    a.ctl = reinterpret_cast<unsigned long long *>(ws + lay.ctl);
    a.flags = reinterpret_cast<uint32_t *>(ws + lay.flags);
    a.agg = reinterpret_cast<float *>(ws + lay.agg);
    a.incl = reinterpret_cast<float *>(ws + lay.incl);
    a.st = call_status(workspace);
    a.withheld = g_withheld_split;
    // automatic: warm-ups for bf16 outputs (a 2^-10 horizon, a few hundred
    // steps on the pages' layers); look-back for fp32 outputs, whose 2^-32
    // horizon runs about as long as the sequences themselves
    const int64_t wsteps = g_selective_warmup_steps >= 0 ? g_selective_warmup_steps : (sizeof(IO) == 2 ? 2048 : 0);
    a.warmup_tiles = static_cast<int>(wsteps / kT);
    // ranges with stealing: warm-up mode, flat tile indices within 32 bits,
    // no withheld carry (that test hook needs the static shares)
    a.steal = a.warmup_tiles > 0 && a.F < (1ll << 31) - kClaim * 4ll && g_withheld_split < 0;
    a.timeout_ns = g_withheld_split >= 1 ? uint64_t(g_withheld_timeout_ms) * 1000000ull : kDefaultTimeoutNs;
    return variant_of(sizeof(IO) == 2, z != nullptr, dt_softplus != 0).launch(mp, a, p.grid, stream);
}

}  // namespace

int selective_plan(int64_t B, int64_t L, int64_t D, lr_dtype io, DiagPlan *p) {
    int sms = 0, dev = 0;
    if (device_sm_count(&sms) != LR_OK || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return LR_ERR_CUDA;
    *p = DiagPlan{};
    const int wch = io == LR_BF16 ? HostCfg<__nv_bfloat16>::WCH : HostCfg<float>::WCH;
    p->dc = wch;
    p->tile_t = kT;
    p->n_cb = B * ((D + wch - 1) / wch);   // chains
    p->n_tiles = static_cast<int>((L + kT - 1) / kT);
    const int per_sm = resident_blocks(io == LR_BF16, dev);
    if (per_sm <= 0) return LR_ERR_CUDA;
    const long long F = static_cast<long long>(p->n_cb) * p->n_tiles;
    long long W;
    if (g_split_override > 0) {
        W = static_cast<long long>(p->n_cb) * g_split_override;   // about that many pieces per chain
    } else {
        W = static_cast<long long>(sms) * per_sm * kWpb;           // one resident wave
        const long long by_len = F / kMinTiles;
        if (by_len < W) W = by_len;
    }
    if (W > F) W = F;
    if (W < 1) W = 1;
    if (W > (1 << 24)) W = 1 << 24;
    p->warps = static_cast<int>(W);
    p->grid = static_cast<int>((W + kWpb - 1) / kWpb);
    p->S = 1;
    p->tps = p->n_tiles;
    p->ctrl_bytes = 0;
    p->ws_bytes = sel_layout(p->warps, wch).total;
    return LR_OK;
}

int selective_launch(const void *x, const void *dt, const void *z, const void *Bm, const void *Cm,
                     const float *A_log, const float *Dskip, const float *h0, void *y, float *h_final,
                     int64_t B, int64_t L, int64_t D, lr_dtype io, int dt_softplus, const DiagPlan &p,
                     void *workspace, cudaStream_t stream) {
    if (io == LR_BF16)
        return launch_t<__nv_bfloat16, false>(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final, B, L, D,
                                              dt_softplus, p, workspace, stream);
    return launch_t<float, true>(x, dt, z, Bm, Cm, A_log, Dskip, h0, y, h_final, B, L, D, dt_softplus, p,
                                 workspace, stream);
}

}  // namespace lr
