// C-ABI of the dgrad library: validation, planning, TMA descriptors, launches.
//
// The plan turns one Conv2d dgrad shape into the parameter block of a single
// persistent kernel launch:
//   * P, Q from the floor convention of the forward convolution;
//   * the stride^2 phase sub-convolutions of a strided dgrad (apache/tvm PR
//     #10110, "[CUTLASS] Conv2d dgrad", benchmark comment: the "strided dgrad"
//     case): dX pixel (h, w) with h = stride*i + ph, w = stride*j + pw receives
//     exactly the taps (r, s) with ph + pad - r*dil = 0 (mod stride) and
//     likewise for s, reading dY at p = i + (ph + pad - r*dil)/stride;
//   * the operand mode: 1x1 pad-0 filters read dY rows as a plain 2-D matrix,
//     everything else reads 4-D (channel, column, row, image) boxes per tap,
//     or one halo box per tile for all taps with the weights resident when
//     the filter fits; the TMA unit fills out-of-range parts with zeros;
//   * the issue variant: CTA pairs (2-SM MMA) for long 256-channel tiles,
//     two MMA warps for N tiles of up to 128 channels;
//   * the tile shape, pipeline depth and work list (phases ordered by tap
//     count, longest first, then M tiles, then N tiles; equal phases
//     interleaved round by round).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/cdg.h"
#include "cdg_params.h"

namespace {

constexpr int kMaxSmem = CDG_MAX_DYN_SMEM;
constexpr int kMaxStages = 8;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

int floor_mod(int a, int m)
{
    int r = a % m;
    return r < 0 ? r + m : r;
}

}  // namespace

// Planner choices that can be overridden (environment variables, or the
// candidates cdg_autotune times); -1 leaves the choice to the planner.
struct PlanOpts {
    int halo = -1;        // 0 off, 1 halo boxes wherever the geometry allows
    int pair = -1;        // 0 never, 1 whenever BN >= 128
    int dual = -1;        // 0 one MMA warp
    int interleave = -1;  // 0 phases one after another
    int max_bn = 256;     // 128 caps the N tile
    int bn = 0;           // > 0: this N tile (a multiple of 64, or of 128 with the packed mask), if it fits C
    int nacc = 2;         // halo plans: accumulators in flight (2 or 4)
    int prefetch = 0;     // 1: L2 prefetch of operand and gate tiles ahead of their loads (measured slower)
    int gate_bufs = 4;    // gated by the saved activation: staging buffers (4; 6 measured slower)
    int pdl = 1;          // 0 plain launches
    int max_grid = 0;     // > 0: at most this many CTAs (tests: many work items per CTA on small problems)
};

struct cdg_plan_st {
    int N, H, W, C, K, R, S, stride, pad, dil, dtype, epi;
    PlanOpts opts;
    int P, Q;
    bool host_only;
    int device;
    int num_sms;
    int out_type, in_type;
    bool mask;       // gated epilogue (x or packed bits)
    bool mask_bits;  // the gate reads a packed bit mask
    size_t smem;
    int grid;
    int *d_status;
    CdgParams prm;  // tensor maps and pointers are filled per call
    const void *cached_dY, *cached_Wp;
    void *cached_dX;
    const void *cached_mask;
    int il_phases, il_items;  // interleaving the planner would use, before the grid is known
    bool noalloc_grid_checked;  // host plan: pair grid checked against the device (cdg_dgrad_noalloc)
    cdg_plan_info_t info;
};

namespace {

// Choose the 4-D halo box (box_w x box_h x box_n dX pixels of one phase
// sub-grid, at most 128) that covers the phases' sub-grids with the fewest
// tiles; ties prefer wider boxes (longer contiguous rows in dY and dX).
void choose_box(const std::vector<CdgPhase> &phases, int N, int &bw, int &bh, int &bn)
{
    int hmax = 0, wmax = 0;
    for (const CdgPhase &ph : phases)
        if (ph.tap_count > 0) {
            hmax = std::max(hmax, ph.hph);
            wmax = std::max(wmax, ph.wph);
        }
    long long best = -1;
    bw = bh = bn = 1;
    for (int w = 1; w <= std::min(wmax, CDG_BM); ++w)
        for (int h = 1; h <= std::min(hmax, CDG_BM / w); ++h) {
            int n = 1;
            if (w >= wmax && h >= hmax) n = std::max(1, std::min(N, CDG_BM / (w * h)));
            long long tiles = 0;
            for (const CdgPhase &ph : phases)
                if (ph.tap_count > 0)
                    tiles += 1LL * ceil_div(ph.wph, w) * ceil_div(ph.hph, h) * ceil_div(N, n);
            const bool better = best < 0 || tiles < best || (tiles == best && w > bw) ||
                                (tiles == best && w == bw && h > bh);
            if (better) {
                best = tiles;
                bw = w;
                bh = h;
                bn = n;
            }
        }
}

// GEMM N tile.  C <= 256: one tile covering C (a multiple of 16, the UMMA N
// granule).  C > 256: several tiles, each a multiple of 64 so that the
// epilogue's 64-channel store boxes never reach into the neighbouring tile;
// least padding wins, larger tiles on ties.
int choose_bn(int C, int max_bn, int step)
{
    if (C <= max_bn) return ((C + 15) / 16) * 16;
    int best = max_bn;
    long long best_waste = -1;
    for (int bn = max_bn; bn >= step; bn -= step) {
        const long long waste = 1LL * ceil_div(C, bn) * bn - C;
        if (best_waste < 0 || waste < best_waste) {
            best_waste = waste;
            best = bn;
        }
    }
    return best;
}

// Set the persistent grid and the interleaving that goes with it: every
// scheduling round of G items (G = CTAs, or CTA pairs) must hold whole groups
// of `il_phases` items, else the phases run one after another.
void apply_grid(cdg_plan_st *h, int grid)
{
    CdgParams &p = h->prm;
    if (h->opts.max_grid > 0) grid = std::min(grid, std::max(p.pair ? 2 : 1, p.pair ? h->opts.max_grid & ~1 : h->opts.max_grid));
    h->grid = grid;
    h->info.grid = grid;
    const int G = p.pair ? grid / 2 : grid;
    const bool ok = h->il_phases > 0 && G % h->il_phases == 0 && 1LL * h->il_phases * h->il_items >= G;
    p.interleave = ok ? h->il_phases : 0;
    p.il_items = ok ? h->il_items : 0;
    p.il_round = G;
    p.div_il = cdg_make_div(static_cast<uint32_t>(std::max(1, p.interleave)));
    p.div_il_round = cdg_make_div(static_cast<uint32_t>(std::max(1, G)));
}

PlanOpts opts_from_env()
{
    PlanOpts o;
    auto flag = [](const char *name) -> int {
        const char *v = std::getenv(name);
        if (!v || !v[0]) return -1;
        return v[0] == '0' ? 0 : (v[0] == '1' ? 1 : -1);
    };
    o.halo = flag("CDG_HALO");
    o.pair = flag("CDG_PAIR");
    o.dual = flag("CDG_DUAL");
    o.interleave = flag("CDG_INTERLEAVE") == 0 ? 0 : -1;
    const char *bn = std::getenv("CDG_MAX_BN");
    o.max_bn = (bn && std::atoi(bn) == 128) ? 128 : 256;
    const char *fbn = std::getenv("CDG_BN");
    o.bn = fbn ? std::atoi(fbn) : 0;
    o.prefetch = flag("CDG_PREFETCH") == 1 ? 1 : 0;
    const char *gb = std::getenv("CDG_GATE_BUFS");
    o.gate_bufs = (gb && std::atoi(gb) == 6) ? 6 : 4;
    const char *na = std::getenv("CDG_NACC");
    o.nacc = (na && std::atoi(na) == 4) ? 4 : 2;
    o.pdl = flag("CDG_PDL") == 0 ? 0 : 1;
    const char *mg = std::getenv("CDG_MAX_GRID");
    o.max_grid = mg ? std::max(0, std::atoi(mg)) : 0;
    return o;
}

int make_plan(int N, int H, int W, int C, int K, int R, int S, int stride, int pad, int dil, int dtype, int epilogue,
              int num_sms, bool host_only, const PlanOpts &opt, cdg_handle_t *out)
{
    if (!out) return CDG_ERR_INVALID_ARG;
    *out = nullptr;
    if (N < 1 || H < 1 || W < 1 || C < 1 || K < 1 || R < 1 || S < 1 || stride < 1 || pad < 0 || dil < 1)
        return CDG_ERR_INVALID_ARG;
    if (dtype != CDG_F16 && dtype != CDG_BF16) return CDG_ERR_INVALID_ARG;
    if (epilogue & ~(CDG_EPI_RELU_BWD | CDG_EPI_OUT_F32 | CDG_EPI_RELU_BWD_BITS | CDG_EPI_SUM | CDG_EPI_SUM_X |
                     CDG_EPI_GELU_BWD | CDG_EPI_SILU_BWD))
        return CDG_ERR_INVALID_ARG;
    const int gates = ((epilogue & CDG_EPI_RELU_BWD) != 0) + ((epilogue & CDG_EPI_RELU_BWD_BITS) != 0) +
                      ((epilogue & CDG_EPI_GELU_BWD) != 0) + ((epilogue & CDG_EPI_SILU_BWD) != 0);
    if (gates > 1) return CDG_ERR_INVALID_ARG;
    if ((epilogue & CDG_EPI_SUM_X) && !(epilogue & CDG_EPI_RELU_BWD)) return CDG_ERR_INVALID_ARG;
    const long long spanH = 1LL * H + 2LL * pad - 1LL * dil * (R - 1) - 1;
    const long long spanW = 1LL * W + 2LL * pad - 1LL * dil * (S - 1) - 1;
    if (spanH < 0 || spanW < 0) return CDG_ERR_INVALID_ARG;
    const int P = static_cast<int>(spanH / stride + 1), Q = static_cast<int>(spanW / stride + 1);
    if (C % 8 || K % 8) return CDG_ERR_UNSUPPORTED;
    if (stride > 4 || R * S > CDG_MAX_TAPS) return CDG_ERR_UNSUPPORTED;
    // TMA: dimensions < 2^32, strides < 2^40 bytes; keep every index in int32
    if (1LL * N * P * Q * K >= (1LL << 31) || 1LL * N * H * W * C >= (1LL << 31) ||
        1LL * R * S * C * K >= (1LL << 31) || P > 65535 || Q > 65535)
        return CDG_ERR_UNSUPPORTED;
    // tap offsets (pad - r*dil)/stride are kept as int16
    if (pad + 1LL * dil * (std::max(R, S) - 1) > 32767) return CDG_ERR_UNSUPPORTED;

    cdg_plan_st *h = new (std::nothrow) cdg_plan_st();
    if (!h) return CDG_ERR_INVALID_ARG;
    h->N = N; h->H = H; h->W = W; h->C = C; h->K = K; h->R = R; h->S = S;
    h->stride = stride; h->pad = pad; h->dil = dil; h->dtype = dtype; h->epi = epilogue;
    h->P = P; h->Q = Q;
    h->host_only = host_only;
    h->num_sms = num_sms;
    h->opts = opt;
    h->in_type = dtype == CDG_F16 ? CDG_T_F16 : CDG_T_BF16;
    h->out_type = (epilogue & CDG_EPI_OUT_F32) ? CDG_T_F32 : h->in_type;
    h->mask = (epilogue & (CDG_EPI_RELU_BWD | CDG_EPI_RELU_BWD_BITS | CDG_EPI_GELU_BWD | CDG_EPI_SILU_BWD)) != 0;
    h->mask_bits = (epilogue & CDG_EPI_RELU_BWD_BITS) != 0;
    const int nsum = (epilogue & CDG_EPI_SUM_X) ? 2 : ((epilogue & CDG_EPI_SUM) ? 1 : 0);

    // ---- phases and their taps
    std::vector<CdgPhase> phases;
    std::vector<CdgTap> taps;
    int phase_taps_by_index[16] = {0};
    for (int ph = 0; ph < stride; ++ph)
        for (int pw = 0; pw < stride; ++pw) {
            CdgPhase f;
            std::memset(&f, 0, sizeof f);
            f.ph = ph;
            f.pw = pw;
            f.hph = ph < H ? (H - ph + stride - 1) / stride : 0;
            f.wph = pw < W ? (W - pw + stride - 1) / stride : 0;
            std::vector<CdgTap> mine;
            for (int r = 0; r < R; ++r) {
                const int th = ph + pad - r * dil;
                if (floor_mod(th, stride)) continue;
                for (int s = 0; s < S; ++s) {
                    const int tw = pw + pad - s * dil;
                    if (floor_mod(tw, stride)) continue;
                    CdgTap t;
                    t.dr = static_cast<int16_t>(th / stride);  // exact: th is a multiple of stride
                    t.ds = static_cast<int16_t>(tw / stride);
                    t.t = static_cast<int16_t>(r * S + s);
                    t.hoff = 0;
                    mine.push_back(t);
                }
            }
            f.tap_count = static_cast<int16_t>(mine.size());
            phase_taps_by_index[ph * stride + pw] = f.tap_count;
            if (f.hph == 0 || f.wph == 0) continue;  // no dX pixel in this residue class
            f.tap_begin = static_cast<int16_t>(taps.size());
            if (!mine.empty()) {
                f.dr_min = mine[0].dr;
                f.ds_min = mine[0].ds;
                for (const CdgTap &t : mine) {
                    f.dr_min = std::min(f.dr_min, t.dr);
                    f.ds_min = std::min(f.ds_min, t.ds);
                }
            }
            taps.insert(taps.end(), mine.begin(), mine.end());
            phases.push_back(f);
        }
    // longest phases first (static schedule, largest work items in the first wave)
    std::stable_sort(phases.begin(), phases.end(),
                     [](const CdgPhase &a, const CdgPhase &b) { return a.tap_count > b.tap_count; });

    // ---- operand and store modes, tiles
    // 1x1 pad-0 filters read dY as a plain matrix of rows.  At stride 1 a tile
    // is 128 consecutive dX pixels; at stride s > 1 (only phase (0,0) has a
    // tap) a tile is whole rows of the phase sub-grid, which the store map can
    // address as one box when H is a multiple of s.  Everything else uses 4-D
    // halo boxes over the phase sub-grids.
    int d_mode = CDG_D_BOX4, rpt = 0, m_step = CDG_BM;
    if (R == 1 && S == 1 && pad == 0) {
        if (stride == 1) {
            d_mode = CDG_D_LINEAR;
        } else if (H % stride == 0 && Q <= CDG_BM) {
            d_mode = CDG_D_ROWS;
            rpt = CDG_BM / Q;
            m_step = rpt * Q;
        }
    }
    const bool flat = d_mode != CDG_D_BOX4;
    int bw = 0, bh = 0, bnb = 0;
    if (!flat) choose_box(phases, N, bw, bh, bnb);
    // N tile: all of C up to 256 channels, else the multiple of 64 up to 256
    // with the least padding (max_bn 128 caps it at 128).  With the packed mask
    // a tile's mask bytes must start on a 16-byte unit: multiples of 128.
    const int bn_step = h->mask_bits ? 128 : 64;
    int BN = choose_bn(C, opt.max_bn == 128 ? 128 : 256, bn_step);
    if (opt.bn > 0 && opt.bn % bn_step == 0 && opt.bn <= (opt.max_bn == 128 ? 128 : 256) &&
        opt.bn < ((C + 15) / 16) * 16)
        BN = opt.bn;
    const int tiles_n = ceil_div(C, BN);
    // per-channel sums: the epilogue warps' partials of a chunk, after the tail
    // and the CTA's per-channel accumulators ([sum][C] fp32)
    const int red_bytes = nsum ? CDG_SMEM_RED + ((nsum * C * 4 + 127) / 128) * 128 : 0;
    // output staging; gated by the activation: four buffers, its chunks land
    // in them two chunks ahead of use (six, four ahead, with CDG_GATE_BUFS=6:
    // measured slower, the ring loses a stage); by the packed mask: a ring of
    // mask tiles besides
    const int gate_bufs = (h->mask && !h->mask_bits) ? (opt.gate_bufs == 6 ? 6 : 4) : 0;
    const int staging =
        CDG_SMEM_STAGING + (h->mask ? (h->mask_bits ? CDG_GATE_RING : (gate_bufs - 2) * (CDG_SMEM_STAGING / 2)) : 0);
    const int ring_budget = kMaxSmem - 1024 - staging - CDG_SMEM_TAIL - red_bytes;

    // ---- halo operand mode: a tile is halo_bh full-width rows of one image's
    // phase sub-grid; one TMA box of (width + tap span) x (rows + tap span)
    // positions of dY serves every tap of the phase, each tap's operand
    // starting hoff rows into it.  Tile row a*halo_wb + b is output (a, b);
    // rows with b >= halo_wt are padding.  With the weights resident (the
    // whole filter of a single N tile fits beside the halo stages) a tile
    // costs one pipeline handshake for all its taps, which measured faster
    // than per-tap boxes on GB300 (ResNet-50 3x3 64->64: 76 vs 84 us), so the
    // planner picks it by default.  With streamed weights it measured slower
    // (one weight handshake per tap, as in per-tap mode, on top of the halo
    // stage), so that form is used only when asked (CDG_HALO=1), wherever the
    // geometry allows; CDG_HALO=0 turns halo mode off.
    bool halo = false, b_res = false, halo_pair = false;
    int hwb = 0, hwt = 0, hbh = 0, hhb = 0, hrows = 0, a_stages = 0, b_stages = 0, b_res_bytes = 0, halo_tg = 1;
    const bool halo_forced = opt.halo == 1;
    // Halo boxes with CTA pairs: each CTA of a pair holds its own tile's halo
    // box and half of every weight tile, so twice the filter fits resident,
    // and each SM reads half of B per MMA.  Taken when both are asked for
    // (CDG_HALO=1 CDG_PAIR=1; CDG_HALO=1 alone keeps single CTAs), and by
    // default, tried first, for stride-1 layers whose filter is resident as
    // halves (measured on GB300, ResNet-50
    // 3x3 128 -> 128 at 28x28: 45.6 us against 57.3 us with per-tap boxes; 3x3
    // 64 -> 64 at 56x56, both with two MMA warps: 53.4 us against 56.8 in
    // single CTAs; the strided and streamed-weight cases measured slower).
    const bool pair_ok = BN >= 64 && BN % 16 == 0 && num_sms >= 2;
    const bool pair_forced = halo_forced && opt.pair == 1 && pair_ok;
    const bool pair_auto = !halo_forced && opt.halo != 0 && opt.pair != 0 && stride == 1 && pair_ok;
    // Gated by the saved activation, plans with per-tap or row boxes let a
    // loader warp issue the activation tiles (the kernels' gate issuer), and
    // halo plans do not; measured on GB300 the x-gated 3x3 64 -> 64 layer runs
    // 99.7 us with per-tap boxes (two MMA warps) against 110.9 with halo boxes,
    // so such plans take halo boxes only when asked (CDG_HALO=1).
    const bool xgate = h->mask && !h->mask_bits;
    // The exception: ReLU-gated stride-1 plans with 128-channel N tiles take
    // halo boxes in CTA pairs, with weight halves resident or streamed
    // (measured on GB300, x-gated 3x3 128 -> 128 at 28x28: 55.3 us against
    // 65.1 with per-tap boxes and two MMA warps; at 64 channels 105.8 against
    // 95.7, at 256 channels 52.9 against 52.2 (14x14) and 89.9 against 50.3
    // (7x7)).  With GELU or SiLU backward, or the per-channel sums, the
    // epilogue has the most work and issues the activation loads itself in a
    // halo plan; those stay with per-tap boxes (the 28x28 layer: GELU 115.7
    // against 131.1 us, SiLU 75.8 against 86.5, both sums 94 against 111).
    const bool heavy_epi = (epilogue & (CDG_EPI_GELU_BWD | CDG_EPI_SILU_BWD | CDG_EPI_SUM | CDG_EPI_SUM_X)) != 0;
    const bool xg_pair = xgate && !heavy_epi && !halo_forced && opt.halo != 0 && opt.pair != 0 && stride == 1 &&
                         BN == 128 && pair_ok;
    const bool halo_allowed = opt.halo != 0 && (!xgate || halo_forced || xg_pair);
    // attempts: resident halves in CTA pairs first where pairs may be taken,
    // then a single CTA (forced pairs, and the gated pairs above: the pair
    // attempt only)
    const bool pair_only = pair_forced || xg_pair;
    const int n_attempts = pair_only ? 1 : (pair_auto ? 2 : 1);
    for (int attempt = 0; attempt < n_attempts && !halo && !flat && halo_allowed; ++attempt) {
        const bool pw = pair_only || (pair_auto && attempt == 0);  // half of the weight rows per CTA
        const int b_rows = pw ? BN / 2 : BN;  // weight rows one CTA holds
        int span_r = 0, span_s = 0, wt = 0, hmax = 0, maxtaps = 0;
        for (const CdgPhase &f : phases) {
            if (f.tap_count == 0) continue;
            int dr_max = f.dr_min, ds_max = f.ds_min;
            for (int t = f.tap_begin; t < f.tap_begin + f.tap_count; ++t) {
                dr_max = std::max<int>(dr_max, taps[t].dr);
                ds_max = std::max<int>(ds_max, taps[t].ds);
            }
            span_r = std::max(span_r, dr_max - f.dr_min);
            span_s = std::max(span_s, ds_max - f.ds_min);
            wt = std::max(wt, f.wph);
            hmax = std::max(hmax, f.hph);
            maxtaps = std::max<int>(maxtaps, f.tap_count);
        }
        const int wb = wt + span_s;
        if (maxtaps < 2 || wb > CDG_BM) break;
        const int rows_per_tile = std::min(hmax, CDG_BM / wb);
        const int hb = rows_per_tile + span_r;
        const int off_max = span_r * wb + span_s;
        const int rows = ((std::max(wb * hb, off_max + CDG_BM) + 7) / 8) * 8;
        const int a_bytes = rows * 128, b_bytes = b_rows * 128;
        // streamed weights: stages of tg taps, one handshake per group; the
        // largest tg (up to 4, and at most the longest phase's taps) that
        // leaves at least two halo and three weight stages
        int tg = 1;
        for (int t = std::min(4, maxtaps); t >= 1; --t)
            if (2 * a_bytes + 3 * t * b_bytes <= ring_budget) {
                tg = t;
                break;
            }
        int as = (3 * a_bytes + 4 * tg * b_bytes <= ring_budget) ? 3 : 2;
        int bs = std::min(std::min(kMaxStages, CDG_MAX_STAGES_TOTAL - as), (ring_budget - as * a_bytes) / (tg * b_bytes));
        // the whole packed filter of a single N tile fits next to at least
        // two halo stages: load it once per CTA and keep it resident, so a
        // tile needs one pipeline handshake (its halo box) for all taps
        bool res = false;
        int res_int = 0;
        const long long res_bytes = 1LL * static_cast<long long>(taps.size()) * ceil_div(K, CDG_BK) * b_rows * 128;
        if (tiles_n == 1 && res_bytes + 2LL * a_bytes <= ring_budget) {
            res = true;
            res_int = static_cast<int>(res_bytes);
            as = std::min<int>(CDG_MAX_STAGES_TOTAL - 1, (ring_budget - res_int) / a_bytes);
            bs = 1;  // one barrier: the resident weights have landed
            tg = 1;
        }
        // streamed weights only when asked (by default pairs only with resident
        // halves; a single CTA falls back to streamed weights only when asked)
        const bool take = pw && !pair_only ? res : (res || halo_forced || xg_pair);
        if (hb <= 256 && bs >= (res ? 1 : 2) && take) {
            halo = true;
            halo_pair = pw;
            b_res = res;
            b_res_bytes = res_int;
            hwb = wb;
            hwt = wt;
            hbh = rows_per_tile;
            hhb = hb;
            hrows = rows;
            a_stages = as;
            b_stages = bs;
            halo_tg = tg;
            for (CdgPhase &f : phases)
                for (int t = f.tap_begin; t < f.tap_begin + f.tap_count; ++t)
                    taps[t].hoff = static_cast<int16_t>((taps[t].dr - f.dr_min) * wb + (taps[t].ds - f.ds_min));
            bw = hwt;
            bh = hbh;
            bnb = 1;
        }
    }
    const int b_rows = halo_pair ? BN / 2 : BN;  // weight rows one CTA holds (halo mode)

    if (!halo) b_res = false;

    // ---- CTA pairs: two CTAs (a cluster) share each 256-row tile through the
    // 2-SM MMA, each holding its 128 rows of dY and half of the weight tile.
    // Measured on GB300 over the ResNet-50 layers: pairs win for 256-channel
    // N tiles whose tiles run at least 4 pipeline stages (1x1 1024 -> 512 at
    // 14x14, 8 stages: 51.4 -> 43.5 us; 512 -> 256 at 28x28, 4 stages: 61.7 ->
    // 58.5 us), and lose with 1 or 2 (1x1 512 -> 128 at 28x28: 46.2 -> 49.1
    // us: the short tiles couple two SMs' epilogues); 192-channel tiles
    // (below) behave alike.
    int tap_phases = 0, tap_sum = 0;
    for (const CdgPhase &f : phases)
        if (f.tap_count > 0) {
            ++tap_phases;
            tap_sum += f.tap_count;
        }
    const double stages_per_tile = tap_phases ? double(tap_sum) / tap_phases * ceil_div(K, CDG_BK) : 0.0;
    bool pair = halo ? halo_pair : (BN >= 192 && num_sms >= 2 && stages_per_tile >= 4.0);
    if (opt.pair == 0) pair = false;
    if (opt.pair == 1) pair = halo ? halo_pair : (BN >= 128 && num_sms >= 2);

    int items = 0;
    for (CdgPhase &f : phases) {
        if (f.tap_count == 0) {
            // zero-filled with TMA stores of a zeroed 128-row staging buffer:
            // boxes of up to 128 sub-grid positions, whole rows where possible
            f.zbw = static_cast<int16_t>(std::min(f.wph, CDG_BM));
            f.zbh = static_cast<int16_t>(std::min(f.hph, std::max(1, CDG_BM / f.zbw)));
            f.tiles_w = ceil_div(f.wph, f.zbw);
            f.tiles_h = ceil_div(f.hph, f.zbh);
            f.tiles_m = f.tiles_w * f.tiles_h * N;
        } else if (flat) {
            f.tiles_w = f.tiles_h = 1;
            f.tiles_m = ceil_div(1LL * N * P * Q, m_step);
        } else {
            f.tiles_w = ceil_div(f.wph, bw);
            f.tiles_h = ceil_div(f.hph, bh);
            f.tiles_m = f.tiles_w * f.tiles_h * ceil_div(N, bnb);
        }
        // a pair takes M tiles 2t and 2t + 1 (an odd last tile's partner reads
        // and writes only out-of-range coordinates, which TMA fills and drops)
        f.items = (pair ? (f.tiles_m + 1) / 2 : f.tiles_m) * tiles_n;
        items += f.items;
    }
    const int stage_bytes = CDG_BM * 128 + (pair ? BN / 2 : BN) * 128;
    const int max_stages = halo ? a_stages + b_stages : std::min(kMaxStages, ring_budget / stage_bytes);
    // ---- dual issue: for N tiles of up to 128 channels two MMA warps take
    // alternate work items, each with half of the stages and two accumulators
    // of its own.  One warp alone stalls on its per-stage barrier handshake
    // (measured on GB300: ~350 cycles per 64-channel stage against ~200 of
    // tensor work); with two, the other warp's MMAs fill that gap.  Tiles of
    // fewer than four stages gain nothing (the epilogue dominates them).
    // (gated by the activation, dual issue leaves no warp for the gate issuer:
    // it pays only for long tiles, where one MMA warp's stage hand-offs are
    // the bound; the x-gated 3x3 s2 128-channel layer runs 112.7 us with one
    // MMA warp and the issuer against 141.2 with two, the 1x1 128 -> 512 layer
    // with eight stages a tile 58.9 against 62.4, the 3x3 64-channel layer
    // with nine stages a tile 140.9 against 99.7)
    bool dual = !halo && !pair && BN <= 128 && max_stages >= 4 && stages_per_tile >= (xgate ? 9.0 : 4.0);
    // Halo boxes with resident weights: two MMA warps take alternate items
    // from the one halo ring, so that one warp's per-tile hand-offs (commits,
    // item bookkeeping, barrier waits: ~1,400 cycles a tile, measured with a
    // cycle-counter trace) overlap the other's MMAs.  Measured on GB300: the
    // 3x3 64 -> 64 layer at 56x56 79.7 -> 57.8 us; the 128-channel layer in
    // CTA pairs unchanged.  (Each warp has full barriers of its own for the
    // halo stages: at most six halo stages keep every barrier within the
    // kernel's 384-byte area.)
    if (halo && b_res && BN <= 128 && a_stages >= 2 && opt.dual != 0) {
        dual = true;
        a_stages = std::min(a_stages, 6);
    }
    if (opt.dual == 0) dual = false;
    const int stages = dual && !halo ? (max_stages / 2) * 2 : (halo ? a_stages + b_stages : max_stages);
    const int ring_bytes = halo ? a_stages * hrows * 128 + (b_res ? b_res_bytes : b_stages * halo_tg * b_rows * 128)
                                : stages * stage_bytes;
    // two accumulators per MMA warp, each at least as wide as the 64-column
    // chunks the epilogue reads
    // (four only while they fit the 512 TMEM columns: N tiles up to 128)
    const int acc_cols = ((BN + 63) / 64) * 64;
    const int n_acc = dual ? 4 : (halo && opt.nacc == 4 && 4 * acc_cols <= 512 ? 4 : 2);
    int tmem_cols = 32;
    while (tmem_cols < n_acc * acc_cols) tmem_cols *= 2;
    if (tmem_cols > 512) return CDG_ERR_UNSUPPORTED;  // not reached: BN <= 256, two accumulators

    CdgParams &p = h->prm;
    std::memset(&p, 0, sizeof p);
    p.N = N; p.H = H; p.W = W; p.C = C; p.K = K; p.P = P; p.Q = Q; p.stride = stride;
    p.BN = BN;
    p.KB = ceil_div(K, CDG_BK);
    p.stages = stages;
    p.tiles_n = tiles_n;
    p.nphases = static_cast<int>(phases.size());
    p.ntaps = static_cast<int>(taps.size());
    p.total_items = items;
    p.a_flat = flat ? 1 : 0;
    p.box_w = bw; p.box_h = bh; p.box_n = bnb;
    p.d_mode = d_mode;
    p.m_step = m_step;
    p.rows_per_tile = rpt;
    p.halo = halo ? 1 : 0;
    p.halo_wb = hwb;
    p.halo_wt = hwt;
    p.halo_bh = hbh;
    p.a_stages = halo ? a_stages : stages;
    p.b_stages = b_stages;
    p.a_stage_bytes = static_cast<uint32_t>(halo ? hrows * 128 : stage_bytes);
    p.halo_hb = hhb;
    p.b_res = b_res ? 1 : 0;
    p.halo_tg = halo_tg;
    p.b_res_bytes = static_cast<uint32_t>(b_res_bytes);
    p.tx_a = static_cast<uint32_t>(hwb * hhb * 128);
    p.tx_b = static_cast<uint32_t>(b_rows * 128);
    const uint32_t ab = dtype == CDG_BF16 ? 1u : 0u;
    const int mma_m = pair ? 2 * CDG_BM : CDG_BM;
    p.idesc = (1u << 4) | (ab << 7) | (ab << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
              (static_cast<uint32_t>(mma_m >> 4) << 24);
    // bytes one stage's full barrier waits for (a pair's leader: both CTAs' copies)
    const int a_bytes = (flat ? CDG_BM : bw * bh * bnb) * 128;
    p.tx_bytes = static_cast<uint32_t>(pair ? 2 * (a_bytes + (BN / 2) * 128) : a_bytes + BN * 128);
    p.pair = pair ? 1 : 0;
    // Programmatic dependent launch: the kernel's set-up overlaps the end of the
    // previous kernel in the stream ("0" turns it off).
    p.pdl = opt.pdl == 0 ? 0 : 1;
    p.prefetch = opt.prefetch == 1 ? 1 : 0;
    p.wait_limit_ns = CDG_WAIT_LIMIT_NS;
    p.withhold_stage = -1;
    p.mask_bits = h->mask_bits ? 1 : 0;
    p.gate_bufs = gate_bufs;
    p.act = (epilogue & CDG_EPI_GELU_BWD) ? 1 : ((epilogue & CDG_EPI_SILU_BWD) ? 2 : 0);
    // gate loads take the dX store box: its rows x the activation chunk's bytes
    // (64 channels; 32 with fp32 output) or the item's mask bytes per row
    {
        const int box_rows = d_mode == CDG_D_BOX4 ? bw * bh * bnb : m_step;
        const int mask_row = tiles_n == 1 ? 16 * ceil_div(C, 128) : BN / 8;
        p.gate_row_bytes = h->mask_bits ? mask_row : (h->out_type == CDG_T_F32 ? 64 : 128);
        p.gate_tx = h->mask ? static_cast<uint32_t>(box_rows * p.gate_row_bytes) : 0u;
    }
    p.dual = dual ? 1 : 0;
    // phases with taps (sorted first) of equal item counts are interleaved item
    // by item, so that their tiles over the same dY run close together (a
    // strided 3x3 layer's four phases otherwise read dY from DRAM once each)
    {
        int ntp = 0;
        while (ntp < static_cast<int>(phases.size()) && phases[ntp].tap_count > 0) ++ntp;
        bool equal = ntp >= 2;
        for (int i = 1; i < ntp; ++i) equal = equal && phases[i].items == phases[0].items;
        if (opt.interleave == 0) equal = false;
        p.interleave = equal ? ntp : 0;
        p.il_items = equal ? phases[0].items : 0;
    }  // p.il_round is set once the grid is final (below)
    p.tmem_cols = static_cast<uint32_t>(tmem_cols);
    p.acc_stride = static_cast<uint32_t>(tmem_cols / n_acc);
    p.acc_ring = dual ? 2u : static_cast<uint32_t>(n_acc);
    for (size_t i = 0; i < phases.size(); ++i) {
        p.phase[i] = phases[i];
        p.div_tiles_w[i] = cdg_make_div(static_cast<uint32_t>(std::max(1, phases[i].tiles_w)));
        p.div_tiles_h[i] = cdg_make_div(static_cast<uint32_t>(std::max(1, phases[i].tiles_h)));
    }
    p.div_tiles_n = cdg_make_div(static_cast<uint32_t>(std::max(1, tiles_n)));
    for (size_t i = 0; i < taps.size(); ++i) p.tap[i] = taps[i];

    h->smem = static_cast<size_t>(1024 + ring_bytes + staging + CDG_SMEM_TAIL + red_bytes);
    p.nsum = nsum;
    p.red_ws = nullptr;
    h->grid = pair ? 2 * std::max(1, std::min(num_sms / 2, items)) : std::max(1, std::min(num_sms, items));

    h->il_phases = p.interleave;
    h->il_items = p.il_items;
    apply_grid(h, h->grid);

    cdg_plan_info_t &inf = h->info;
    std::memset(&inf, 0, sizeof inf);
    inf.P = P; inf.Q = Q;
    inf.num_phases = stride * stride;
    for (int i = 0; i < stride * stride; ++i) inf.phase_taps[i] = phase_taps_by_index[i];
    inf.tile_m = CDG_BM; inf.tile_n = BN; inf.tile_k = CDG_BK;
    inf.a_mode = halo ? (b_res ? 3 : 2) : (flat ? 1 : 0);
    inf.box_w = bw; inf.box_h = bh; inf.box_n = bnb;
    inf.stages = stages;
    inf.work_items = items;
    inf.grid = h->grid;
    inf.smem_bytes = static_cast<int>(h->smem);
    inf.tmem_cols = tmem_cols;
    inf.cta_pair = pair ? 1 : 0;
    inf.mma_warps = dual ? 2 : 1;

    if (!host_only && pair) {
        // pairs must be co-resident on one GPC: size the persistent grid by
        // how many the device can hold at once, not by the SM count alone
        if (cdg_prepare_dgrad(h->out_type, h->in_type, h->mask, h->smem) != cudaSuccess) {
            delete h;
            return CDG_ERR_CUDA;
        }
        const int pairs = cdg_max_active_pairs(h->out_type, h->in_type, h->mask, h->smem);
        if (pairs >= 1) apply_grid(h, 2 * std::max(1, std::min(pairs, items)));
    }
    if (!host_only) {
        if (cudaGetDevice(&h->device) != cudaSuccess ||
            cdg_prepare_dgrad(h->out_type, h->in_type, h->mask, h->smem) != cudaSuccess ||
            cudaMalloc(&h->d_status, sizeof(int)) != cudaSuccess ||
            cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess) {
            if (h->d_status) cudaFree(h->d_status);
            delete h;
            return CDG_ERR_CUDA;
        }
    }
    *out = h;
    return CDG_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + nb && pb < pa + na;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bytes of a packed mask row: a pixel's C bits in whole 16-byte units.
long long mask_row_bytes(int C) { return 16LL * ((C + 127) / 128); }

// Bytes of the gate's input: x (2 bytes per element) or the packed mask.
size_t mask_bytes(const cdg_plan_st *h)
{
    const size_t pixels = static_cast<size_t>(h->N) * h->H * h->W;
    return h->mask_bits ? pixels * mask_row_bytes(h->C) : 2 * pixels * h->C;
}

CUtensorMapDataType tmap_type(int dtype)
{
    return dtype == CDG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

int encode_operand_maps(cdg_plan_st *h, const void *dY, const void *Wp)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return CDG_ERR_CUDA;
    CdgParams &p = h->prm;
    const cuuint32_t ones[5] = {1, 1, 1, 1, 1};
    const CUtensorMapDataType dt = tmap_type(h->dtype);
    CUresult r;
    if (p.a_flat) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(h->K), static_cast<cuuint64_t>(1LL * h->N * h->P * h->Q)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(h->K) * 2};
        const cuuint32_t box[2] = {CDG_BK, CDG_BM};
        r = enc(&p.tmA, dt, 2, const_cast<void *>(dY), dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(h->K), static_cast<cuuint64_t>(h->Q),
                                    static_cast<cuuint64_t>(h->P), static_cast<cuuint64_t>(h->N)};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(h->K) * 2, static_cast<cuuint64_t>(h->Q) * h->K * 2,
                                       static_cast<cuuint64_t>(h->P) * h->Q * h->K * 2};
        const cuuint32_t box[4] = {CDG_BK, static_cast<cuuint32_t>(p.halo ? p.halo_wb : p.box_w),
                                   static_cast<cuuint32_t>(p.halo ? p.halo_hb : p.box_h),
                                   static_cast<cuuint32_t>(p.halo ? 1 : p.box_n)};
        r = enc(&p.tmA, dt, 4, const_cast<void *>(dY), dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return CDG_ERR_CUDA;
    const cuuint64_t bdims[3] = {static_cast<cuuint64_t>(h->K), static_cast<cuuint64_t>(h->C),
                                 static_cast<cuuint64_t>(h->R) * h->S};
    const cuuint64_t bstrides[2] = {static_cast<cuuint64_t>(h->K) * 2, static_cast<cuuint64_t>(h->C) * h->K * 2};
    const cuuint32_t bbox[3] = {CDG_BK, static_cast<cuuint32_t>(p.pair ? p.BN / 2 : p.BN), 1};
    r = enc(&p.tmB, dt, 3, const_cast<void *>(Wp), bdims, bstrides, bbox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return CDG_ERR_CUDA;
    h->cached_dY = dY;
    h->cached_Wp = Wp;
    return CDG_OK;
}

// Store maps for dX: one per phase slot that has taps (zero phases are
// written with plain stores).  Each covers 128-byte rows (64 fp16/bf16 or 32
// fp32 channels) with the 128-byte swizzle the epilogue's staging uses.
int encode_store_maps(cdg_plan_st *h, void *dX)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return CDG_ERR_CUDA;
    CdgParams &p = h->prm;
    const cuuint32_t ones[4] = {1, 1, 1, 1};
    const bool f32 = h->out_type == CDG_T_F32;
    const cuuint64_t osz = f32 ? 4 : 2;
    const cuuint32_t ch = static_cast<cuuint32_t>(128 / osz);
    const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : tmap_type(h->dtype);
    const cuuint64_t C = h->C, W = h->W, H = h->H, s = h->stride;
    for (int i = 0; i < p.nphases; ++i) {
        const CdgPhase &f = p.phase[i];
        CUresult r;
        if (f.tap_count == 0 || p.d_mode == CDG_D_BOX4) {
            // phase sub-grid {C, wph, hph, N} of dX, starting at pixel (ph, pw)
            char *base = static_cast<char *>(dX) + (static_cast<cuuint64_t>(f.ph) * W + f.pw) * C * osz;
            const cuuint64_t dims[4] = {C, static_cast<cuuint64_t>(f.wph), static_cast<cuuint64_t>(f.hph),
                                        static_cast<cuuint64_t>(h->N)};
            const cuuint64_t strides[3] = {s * C * osz, s * W * C * osz, H * W * C * osz};
            const bool zero = f.tap_count == 0;
            const cuuint32_t box[4] = {ch, static_cast<cuuint32_t>(zero ? f.zbw : p.box_w),
                                       static_cast<cuuint32_t>(zero ? f.zbh : p.box_h),
                                       static_cast<cuuint32_t>(zero ? 1 : p.box_n)};
            r = enc(&p.tmD[i], dt, 4, base, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else if (p.d_mode == CDG_D_LINEAR) {
            const cuuint64_t dims[2] = {C, static_cast<cuuint64_t>(h->N) * H * W};
            const cuuint64_t strides[1] = {C * osz};
            const cuuint32_t box[2] = {ch, CDG_BM};
            r = enc(&p.tmD[i], dt, 2, dX, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else {
            // phase (0,0): rows n*hph + i are s*W*C elements apart because H = s*hph
            const cuuint64_t dims[3] = {C, static_cast<cuuint64_t>(f.wph),
                                        static_cast<cuuint64_t>(h->N) * static_cast<cuuint64_t>(f.hph)};
            const cuuint64_t strides[2] = {s * C * osz, s * W * C * osz};
            const cuuint32_t box[3] = {ch, static_cast<cuuint32_t>(f.wph), static_cast<cuuint32_t>(p.rows_per_tile)};
            r = enc(&p.tmD[i], dt, 3, dX, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
        if (r != CUDA_SUCCESS) return CDG_ERR_CUDA;
    }
    h->cached_dX = dX;
    return CDG_OK;
}

// Gate load maps: the dX store maps' geometry over the saved activation (the
// input type; 64-channel boxes with the staging's 128-byte swizzle, or plain
// 32-channel boxes of 64-byte rows for fp32 output) or over the packed mask
// (bytes; rows of mask_row_bytes(C) per pixel; boxes of gate_row_bytes).
// Phases without taps need none.
int encode_gate_maps(cdg_plan_st *h, const void *gate)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return CDG_ERR_CUDA;
    CdgParams &p = h->prm;
    const cuuint32_t ones[4] = {1, 1, 1, 1};
    const bool bits = h->mask_bits;
    const cuuint64_t esz = bits ? 1 : 2;
    const cuuint64_t row = bits ? static_cast<cuuint64_t>(mask_row_bytes(h->C)) : static_cast<cuuint64_t>(h->C);
    const cuuint32_t inner = static_cast<cuuint32_t>(bits ? p.gate_row_bytes : p.gate_row_bytes / 2);
    const CUtensorMapDataType dt = bits ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : tmap_type(h->dtype);
    const CUtensorMapSwizzle sw =
        (!bits && h->out_type != CDG_T_F32) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
    const cuuint64_t W = h->W, H = h->H, s = h->stride;
    char *base0 = static_cast<char *>(const_cast<void *>(gate));
    for (int i = 0; i < p.nphases; ++i) {
        const CdgPhase &f = p.phase[i];
        if (f.tap_count == 0) continue;
        CUresult r;
        if (p.d_mode == CDG_D_BOX4) {
            char *base = base0 + (static_cast<cuuint64_t>(f.ph) * W + f.pw) * row * esz;
            const cuuint64_t dims[4] = {row, static_cast<cuuint64_t>(f.wph), static_cast<cuuint64_t>(f.hph),
                                        static_cast<cuuint64_t>(h->N)};
            const cuuint64_t strides[3] = {s * row * esz, s * W * row * esz, H * W * row * esz};
            const cuuint32_t box[4] = {inner, static_cast<cuuint32_t>(p.box_w), static_cast<cuuint32_t>(p.box_h),
                                       static_cast<cuuint32_t>(p.box_n)};
            r = enc(&p.tmG[i], dt, 4, base, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else if (p.d_mode == CDG_D_LINEAR) {
            const cuuint64_t dims[2] = {row, static_cast<cuuint64_t>(h->N) * H * W};
            const cuuint64_t strides[1] = {row * esz};
            const cuuint32_t box[2] = {inner, CDG_BM};
            r = enc(&p.tmG[i], dt, 2, base0, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        } else {
            const cuuint64_t dims[3] = {row, static_cast<cuuint64_t>(f.wph),
                                        static_cast<cuuint64_t>(h->N) * static_cast<cuuint64_t>(f.hph)};
            const cuuint64_t strides[2] = {s * row * esz, s * W * row * esz};
            const cuuint32_t box[3] = {inner, static_cast<cuuint32_t>(f.wph), static_cast<cuuint32_t>(p.rows_per_tile)};
            r = enc(&p.tmG[i], dt, 3, base0, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
        if (r != CUDA_SUCCESS) return CDG_ERR_CUDA;
    }
    h->cached_mask = gate;
    return CDG_OK;
}

// Validate the tensors of one dgrad, refresh the cached tensor maps and
// launch the kernel (red_ws: the per-channel sums workspace, or NULL).
int launch_plan(cdg_handle_t h, const void *dY, const void *Wpacked, void *dX, const void *relu_mask, float *red_ws,
                cdg_stream_t stream)
{
    if (!h || !dY || !Wpacked || !dX) return CDG_ERR_INVALID_ARG;
    if (h->mask != (relu_mask != nullptr)) return CDG_ERR_INVALID_ARG;
    if (h->host_only) return CDG_ERR_NO_DEVICE;
    if (!aligned16(dY) || !aligned16(Wpacked) || !aligned16(dX) || (relu_mask && !aligned16(relu_mask)))
        return CDG_ERR_ALIGNMENT;
    const size_t dx_bytes = static_cast<size_t>(h->N) * h->H * h->W * h->C * (h->out_type == CDG_T_F32 ? 4 : 2);
    const size_t dy_bytes = static_cast<size_t>(h->N) * h->P * h->Q * h->K * 2;
    if (overlaps(dX, dx_bytes, dY, dy_bytes) || overlaps(dX, dx_bytes, Wpacked, cdg_packed_weight_bytes(h)) ||
        (relu_mask && overlaps(dX, dx_bytes, relu_mask, mask_bytes(h))))
        return CDG_ERR_ALIAS;
    if (dY != h->cached_dY || Wpacked != h->cached_Wp) {
        const int rc = encode_operand_maps(h, dY, Wpacked);
        if (rc != CDG_OK) return rc;
    }
    if (dX != h->cached_dX) {
        const int rc = encode_store_maps(h, dX);
        if (rc != CDG_OK) return rc;
    }
    if (relu_mask && relu_mask != h->cached_mask) {
        const int rc = encode_gate_maps(h, relu_mask);
        if (rc != CDG_OK) return rc;
    }
    CdgParams &p = h->prm;
    p.dX = dX;
    p.mask = relu_mask;
    p.status = h->d_status;
    p.red_ws = red_ws;
    if (cdg_launch_dgrad(p, h->out_type, h->in_type, h->mask, h->grid, h->smem, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return CDG_ERR_CUDA;
    return CDG_OK;
}

// The planner's N tile for C > 256 channels is 256 (or the multiple of 64 with
// the least padding).  192-channel tiles, which fill the last scheduling round
// of the 1x1 512 -> 2048 channel layer at 7x7 better (147 pair items, 1.93
// rounds, against 98, 1.29 rounds), measured faster once (31.9 -> 27.0 us)
// but slower since the CTA pairs' accumulator hand-back got cheaper (29.5 us
// with 256, 30.8 with 192), so the planner no longer picks them by itself:
// CDG_BN=192 asks for them, and cdg_autotune times them.
int choose_plan_bn(int, int, int, int, int, int, int, int, int, int, int, int, int, const PlanOpts &opt)
{
    return opt.bn;
}

}  // namespace

extern "C" {

int cdg_plan(int N, int H, int W, int C, int K, int R, int S, int stride, int pad, int dil, int dtype, int epilogue,
             cdg_handle_t *out)
{
    if (out) *out = nullptr;
    int dev = 0, sms = 0;
    // validate first so that argument errors never depend on a device
    cdg_handle_t probe = nullptr;
    PlanOpts opt = opts_from_env();
    int rc = make_plan(N, H, W, C, K, R, S, stride, pad, dil, dtype, epilogue, 1, true, opt, &probe);
    if (rc != CDG_OK) return rc;
    cdg_destroy(probe);
    if (cudaGetDevice(&dev) != cudaSuccess) return CDG_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return CDG_ERR_CUDA;
    opt.bn = choose_plan_bn(N, H, W, C, K, R, S, stride, pad, dil, dtype, epilogue, sms, opt);
    return make_plan(N, H, W, C, K, R, S, stride, pad, dil, dtype, epilogue, sms, false, opt, out);
}

int cdg_plan_host(int N, int H, int W, int C, int K, int R, int S, int stride, int pad, int dil, int dtype,
                  int epilogue, int num_sms, cdg_handle_t *out)
{
    if (num_sms < 1) {
        if (out) *out = nullptr;
        return CDG_ERR_INVALID_ARG;
    }
    PlanOpts opt = opts_from_env();
    opt.bn = choose_plan_bn(N, H, W, C, K, R, S, stride, pad, dil, dtype, epilogue, num_sms, opt);
    return make_plan(N, H, W, C, K, R, S, stride, pad, dil, dtype, epilogue, num_sms, true, opt, out);
}

void cdg_destroy(cdg_handle_t h)
{
    if (!h) return;
    if (h->d_status) cudaFree(h->d_status);
    delete h;
}

int cdg_get_output_dims(cdg_handle_t h, int *P, int *Q)
{
    if (!h || !P || !Q) return CDG_ERR_INVALID_ARG;
    *P = h->P;
    *Q = h->Q;
    return CDG_OK;
}

size_t cdg_packed_weight_bytes(cdg_handle_t h)
{
    if (!h) return 0;
    return static_cast<size_t>(h->R) * h->S * h->C * h->K * 2;
}

int cdg_plan_get_info(cdg_handle_t h, cdg_plan_info_t *info)
{
    if (!h || !info) return CDG_ERR_INVALID_ARG;
    *info = h->info;
    return CDG_OK;
}

int cdg_prepack_weights(cdg_handle_t h, const void *W_krsc, void *Wpacked, cdg_stream_t stream)
{
    if (!h || !W_krsc || !Wpacked) return CDG_ERR_INVALID_ARG;
    if (h->host_only) return CDG_ERR_NO_DEVICE;
    if (!aligned16(W_krsc) || !aligned16(Wpacked)) return CDG_ERR_ALIGNMENT;
    const size_t nb = cdg_packed_weight_bytes(h);
    if (overlaps(W_krsc, nb, Wpacked, nb)) return CDG_ERR_ALIAS;
    if (cdg_launch_prepack(W_krsc, Wpacked, h->K, h->R * h->S, h->C, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return CDG_ERR_CUDA;
    return CDG_OK;
}

int cdg_dgrad(cdg_handle_t h, const void *dY, const void *Wpacked, void *dX, const void *relu_mask,
              cdg_stream_t stream)
{
    if (h && h->prm.nsum) return CDG_ERR_INVALID_ARG;  // such plans run through cdg_dgrad_sums
    return launch_plan(h, dY, Wpacked, dX, relu_mask, nullptr, stream);
}

size_t cdg_sums_workspace_bytes(cdg_handle_t h)
{
    if (!h) return 0;
    // one row per CTA; no plan of this handle (autotuned ones included) has
    // more CTAs than the device has SMs
    return static_cast<size_t>(h->num_sms) * h->prm.nsum * h->C * sizeof(float);
}

int cdg_dgrad_sums(cdg_handle_t h, const void *dY, const void *Wpacked, void *dX, const void *relu_mask, float *sums,
                   void *workspace, cdg_stream_t stream)
{
    if (!h || !sums || !workspace || !h->prm.nsum) return CDG_ERR_INVALID_ARG;
    if (!aligned16(sums) || !aligned16(workspace)) return CDG_ERR_ALIGNMENT;
    const size_t sb = static_cast<size_t>(h->prm.nsum) * h->C * sizeof(float);
    const size_t wb = cdg_sums_workspace_bytes(h);
    const size_t dx_bytes = static_cast<size_t>(h->N) * h->H * h->W * h->C * (h->out_type == CDG_T_F32 ? 4 : 2);
    const size_t dy_bytes = static_cast<size_t>(h->N) * h->P * h->Q * h->K * 2;
    const void *outs[3] = {dX, sums, workspace};
    const size_t outb[3] = {dx_bytes, sb, wb};
    const void *ins[3] = {dY, Wpacked, relu_mask};
    const size_t inb[3] = {dy_bytes, cdg_packed_weight_bytes(h), relu_mask ? mask_bytes(h) : 0};
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 3; ++j)
            if (ins[j] && outs[i] && overlaps(outs[i], outb[i], ins[j], inb[j])) return CDG_ERR_ALIAS;
        for (int j = i + 1; j < 3; ++j)
            if (overlaps(outs[i], outb[i], outs[j], outb[j])) return CDG_ERR_ALIAS;
    }
    int rc = launch_plan(h, dY, Wpacked, dX, relu_mask, static_cast<float *>(workspace), stream);
    if (rc != CDG_OK) return rc;
    if (cdg_launch_channel_sums(static_cast<const float *>(workspace), h->grid, h->prm.nsum, h->C, sums,
                                static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CDG_ERR_CUDA;
    return CDG_OK;
}

// Plan-time autotuning: the planner's candidate configurations for this
// shape, each timed on the caller's tensors; the fastest replaces the plan.
int cdg_autotune(cdg_handle_t h, const void *dY, const void *Wpacked, void *dX, const void *relu_mask,
                 cdg_stream_t stream, int reps, float *best_ms)
{
    if (!h || !dY || !Wpacked || !dX || reps < 1 || reps > 1000) return CDG_ERR_INVALID_ARG;
    if (h->mask != (relu_mask != nullptr)) return CDG_ERR_INVALID_ARG;
    if (h->host_only) return CDG_ERR_NO_DEVICE;
    if (h->prm.nsum) return CDG_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    std::vector<PlanOpts> cands;
    const PlanOpts base = h->opts;
    cands.push_back(base);
    auto variant = [&](int pair, int dual, int halo, int interleave, int max_bn, int bn = -1) {
        PlanOpts o = base;
        if (pair != -2) o.pair = pair;
        if (dual != -2) o.dual = dual;
        if (halo != -2) o.halo = halo;
        if (interleave != -2) o.interleave = interleave;
        if (max_bn) o.max_bn = max_bn;
        if (bn >= 0) o.bn = bn;
        cands.push_back(o);
    };
    variant(0, -2, -2, -2, 0);    // no CTA pairs
    variant(1, -2, -2, -2, 0);    // CTA pairs wherever BN >= 128
    variant(-2, 0, -2, -2, 0);    // one MMA warp
    variant(-2, -2, 0, -2, 0);    // no halo boxes
    variant(-2, -2, 1, -2, 0);    // halo boxes wherever the geometry allows
    variant(1, -2, 1, -2, 0);     // halo boxes with CTA pairs (half of the weights per CTA)
    variant(-2, -2, -2, 0, 0);    // phases one after another
    variant(-2, -2, -2, -2, 128); // 128-channel N tiles
    variant(1, -2, -2, -2, 128);
    variant(-2, 0, -2, -2, 128);
    variant(-2, -2, -2, -2, 0, 0);    // the default N tile (256 channels when C > 256)
    variant(-2, -2, -2, -2, 0, 192);  // 192-channel N tiles

    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        return CDG_ERR_CUDA;
    }
    // each timed launch follows a write of twice the L2 size, so every
    // candidate starts with cold caches, as a layer inside a network step does
    int l2 = 0;
    size_t flush_bytes = 0;
    void *flush = nullptr;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, h->device) == cudaSuccess && l2 > 0) {
        flush_bytes = 2 * static_cast<size_t>(l2);
        if (cudaMalloc(&flush, flush_bytes) != cudaSuccess) {
            flush = nullptr;
            cudaGetLastError();  // clear the failed allocation; time without flushing
        }
    }
    // plans that come out identical are timed once
    struct Sig {
        int a_mode, pair, warps, bn, stages, box_w, box_h, box_n, interleave, tg, pdl;
        bool operator==(const Sig &o) const { return std::memcmp(this, &o, sizeof *this) == 0; }
    };
    std::vector<Sig> seen;
    cdg_plan_st *best = nullptr;
    bool best_is_default = false;
    float best_t = 0.0f;
    int rc = CDG_OK;
    for (const PlanOpts &o : cands) {
        cdg_handle_t c = nullptr;
        if (make_plan(h->N, h->H, h->W, h->C, h->K, h->R, h->S, h->stride, h->pad, h->dil, h->dtype, h->epi,
                      h->num_sms, false, o, &c) != CDG_OK)
            continue;
        Sig sig;
        std::memset(&sig, 0, sizeof sig);
        sig = Sig{c->info.a_mode, c->info.cta_pair, c->info.mma_warps, c->info.tile_n, c->info.stages,
                  c->info.box_w, c->info.box_h, c->info.box_n, c->prm.interleave, c->prm.halo_tg, c->prm.pdl};
        if (std::find(seen.begin(), seen.end(), sig) != seen.end()) {
            cdg_destroy(c);
            continue;
        }
        seen.push_back(sig);
        // one untimed launch (it also encodes the tensor maps), then reps timed
        rc = cdg_dgrad(c, dY, Wpacked, dX, relu_mask, stream);
        float ms = 0.0f;
        for (int i = 0; rc == CDG_OK && i < reps; ++i) {
            float one = 0.0f;
            if (flush && cudaMemsetAsync(flush, i & 0xff, flush_bytes, s) != cudaSuccess) rc = CDG_ERR_CUDA;
            if (rc == CDG_OK && cudaEventRecord(e0, s) != cudaSuccess) rc = CDG_ERR_CUDA;
            if (rc == CDG_OK) rc = cdg_dgrad(c, dY, Wpacked, dX, relu_mask, stream);
            if (rc == CDG_OK && (cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                                 cudaEventElapsedTime(&one, e0, e1) != cudaSuccess))
                rc = CDG_ERR_CUDA;
            ms += one;
        }
        if (rc == CDG_OK) rc = cdg_device_status(c, stream);
        if (rc != CDG_OK) {  // a failed launch or a device timeout ends the search
            cdg_destroy(c);
            break;
        }
        ms /= static_cast<float>(reps);
        // the planner's own choice (the first candidate) is kept unless another
        // is at least 2 % faster: closer timings are within launch-to-launch noise
        const float margin = best_is_default ? 0.98f : 1.0f;
        if (!best || ms < best_t * margin) {
            if (best) cdg_destroy(best);
            best_is_default = &o == &cands[0];
            best = c;
            best_t = ms;
        } else {
            cdg_destroy(c);
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (flush) cudaFree(flush);
    if (rc != CDG_OK || !best) {
        if (best) cdg_destroy(best);
        return rc != CDG_OK ? rc : CDG_ERR_UNSUPPORTED;
    }
    // the handle takes the best plan (and keeps its own status word)
    int *status = h->d_status;
    *h = *best;
    h->d_status = status;
    h->info.tuned = 1;
    cdg_destroy(best);
    if (best_ms) *best_ms = best_t;
    return CDG_OK;
}

int cdg_plan_set_wait_limit(cdg_handle_t h, unsigned long long ns)
{
    if (!h || ns < 100000ull || ns > 60000000000ull) return CDG_ERR_INVALID_ARG;
    h->prm.wait_limit_ns = ns;
    return CDG_OK;
}

int cdg_plan_withhold_load_for_test(cdg_handle_t h, int stage)
{
    if (!h || stage < -1) return CDG_ERR_INVALID_ARG;
    // only the per-tap / row loaders of single CTAs honour it
    if (stage >= 0 && (h->prm.halo || h->prm.pair)) return CDG_ERR_UNSUPPORTED;
    h->prm.withhold_stage = stage;
    return CDG_OK;
}

int cdg_device_status(cdg_handle_t h, cdg_stream_t stream)
{
    if (!h) return CDG_ERR_INVALID_ARG;
    if (h->host_only) return CDG_ERR_NO_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, h->d_status, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return CDG_ERR_CUDA;
    if (v != 0) {
        if (cudaMemsetAsync(h->d_status, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
            return CDG_ERR_CUDA;
    }
    return v;
}

long long cdg_relu_mask_bytes(long long pixels, int C)
{
    if (pixels < 0 || C <= 0 || C % 8 != 0) return -1;
    return pixels * mask_row_bytes(C);
}

int cdg_pack_relu_mask(const void *x, void *bits, long long pixels, int C, int dtype, cdg_stream_t stream)
{
    if (!x || !bits || pixels < 0 || C <= 0 || C % 8 != 0) return CDG_ERR_INVALID_ARG;
    if (dtype != CDG_F16 && dtype != CDG_BF16) return CDG_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(bits)) return CDG_ERR_ALIGNMENT;
    if (overlaps(x, static_cast<size_t>(pixels) * C * 2, bits, static_cast<size_t>(pixels * mask_row_bytes(C))))
        return CDG_ERR_ALIAS;
    if (cdg_launch_pack_mask(x, bits, pixels, C, dtype == CDG_F16 ? CDG_T_F16 : CDG_T_BF16,
                             static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CDG_ERR_CUDA;
    return CDG_OK;
}

const char *cdg_status_string(int status)
{
    switch (status) {
    case CDG_OK: return "ok";
    case CDG_ERR_INVALID_ARG: return "invalid argument";
    case CDG_ERR_UNSUPPORTED: return "unsupported shape (C and K must be multiples of 8, stride <= 4, R*S <= 128)";
    case CDG_ERR_ALIGNMENT: return "tensor pointer not 16-byte aligned";
    case CDG_ERR_ALIAS: return "dX overlaps an input tensor";
    case CDG_ERR_CUDA: return "CUDA runtime or launch error";
    case CDG_ERR_TIMEOUT: return "device pipeline wait timed out";
    case CDG_ERR_NO_DEVICE: return "handle was planned without a device";
    case CDG_ERR_SCRATCH_TOO_SMALL:
        return "packed weights exceed the 8 MiB scratch of cdg_dgrad_noalloc (R*S*C*K must be <= 4194304)";
    default: return "unknown status";
    }
}

}  // extern "C"

// ------------------------------------------------------------------ allocation-free entry point
// Scratch for cdg_dgrad_noalloc: [0, 256) the kernel's status word, then the
// packed weights.  Device code could name it directly; host code needs its
// device address, which cudaGetSymbolAddress returns per device.
#define CDG_NOALLOC_STATUS_BYTES 256
static __device__ __align__(256) unsigned char cdg_noalloc_scratch[CDG_NOALLOC_STATUS_BYTES + CDG_NOALLOC_MAX_WEIGHT_BYTES];

#include <mutex>

namespace {

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mutex;
unsigned char *g_noalloc_addr[kNoallocMaxDevices];  // device address of the scratch, per device
unsigned g_noalloc_prepared[kNoallocMaxDevices];     // kernels whose shared-memory limit was raised

// Once per device (with that device current): the scratch's device address,
// and the dynamic shared-memory opt-in of the kernel instantiation `key`.
int noalloc_address(int dev, unsigned char **scratch)
{
    if (!g_noalloc_addr[dev]) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, cdg_noalloc_scratch) != cudaSuccess || !addr) return CDG_ERR_CUDA;
        g_noalloc_addr[dev] = static_cast<unsigned char *>(addr);
    }
    *scratch = g_noalloc_addr[dev];
    return CDG_OK;
}

int noalloc_setup(int dev, cdg_plan_st *h, unsigned char **scratch)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    const int rc = noalloc_address(dev, scratch);
    if (rc != CDG_OK) return rc;
    const unsigned key = 1u << (h->out_type * 4 + h->in_type * 2 + (h->mask ? 1 : 0));
    if (!(g_noalloc_prepared[dev] & key)) {
        if (cdg_prepare_dgrad(h->out_type, h->in_type, h->mask, h->smem) != cudaSuccess) return CDG_ERR_CUDA;
        g_noalloc_prepared[dev] |= key;
    }
    // A plan made without a device sized a CTA-pair grid from the SM count
    // alone; on this device only as many pairs as fit at once run per round.
    if (h->host_only && h->prm.pair && !h->noalloc_grid_checked) {
        const int pairs = cdg_max_active_pairs(h->out_type, h->in_type, h->mask, h->smem);
        if (pairs >= 1 && 2 * pairs < h->grid) apply_grid(h, 2 * pairs);
        h->noalloc_grid_checked = true;
    }
    return CDG_OK;
}

}  // namespace

extern "C" int cdg_dgrad_noalloc(cdg_handle_t h, const void *dY, const void *W_krsc, void *dX,
                                 const void *relu_mask, cdg_stream_t stream)
{
    if (!h || !dY || !W_krsc || !dX || h->prm.nsum) return CDG_ERR_INVALID_ARG;
    if (h->mask != (relu_mask != nullptr)) return CDG_ERR_INVALID_ARG;
    const size_t wbytes = cdg_packed_weight_bytes(h);
    if (wbytes > CDG_NOALLOC_MAX_WEIGHT_BYTES) return CDG_ERR_SCRATCH_TOO_SMALL;
    if (!aligned16(dY) || !aligned16(W_krsc) || !aligned16(dX) || (relu_mask && !aligned16(relu_mask)))
        return CDG_ERR_ALIGNMENT;
    const size_t dx_bytes = static_cast<size_t>(h->N) * h->H * h->W * h->C * (h->out_type == CDG_T_F32 ? 4 : 2);
    const size_t dy_bytes = static_cast<size_t>(h->N) * h->P * h->Q * h->K * 2;
    if (overlaps(dX, dx_bytes, dY, dy_bytes) || overlaps(dX, dx_bytes, W_krsc, wbytes) ||
        (relu_mask && overlaps(dX, dx_bytes, relu_mask, mask_bytes(h))))
        return CDG_ERR_ALIAS;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CDG_ERR_CUDA;
    if (dev < 0 || dev >= kNoallocMaxDevices) return CDG_ERR_UNSUPPORTED;
    unsigned char *scratch = nullptr;
    const int rc = noalloc_setup(dev, h, &scratch);
    if (rc != CDG_OK) return rc;
    int *status = reinterpret_cast<int *>(scratch);
    void *Wp = scratch + CDG_NOALLOC_STATUS_BYTES;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return CDG_ERR_CUDA;
    if (cdg_launch_prepack(W_krsc, Wp, h->K, h->R * h->S, h->C, s) != cudaSuccess) return CDG_ERR_CUDA;
    if (dY != h->cached_dY || Wp != h->cached_Wp) {
        const int e = encode_operand_maps(h, dY, Wp);
        if (e != CDG_OK) return e;
    }
    if (dX != h->cached_dX) {
        const int e = encode_store_maps(h, dX);
        if (e != CDG_OK) return e;
    }
    if (relu_mask && relu_mask != h->cached_mask) {
        const int e = encode_gate_maps(h, relu_mask);
        if (e != CDG_OK) return e;
    }
    CdgParams &p = h->prm;
    p.dX = dX;
    p.mask = relu_mask;
    p.status = status;
    p.red_ws = nullptr;
    if (cdg_launch_dgrad(p, h->out_type, h->in_type, h->mask, h->grid, h->smem, s) != cudaSuccess)
        return CDG_ERR_CUDA;
    return CDG_OK;
}

extern "C" int cdg_dgrad_noalloc_status(cdg_stream_t stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CDG_ERR_CUDA;
    if (dev < 0 || dev >= kNoallocMaxDevices) return CDG_ERR_UNSUPPORTED;
    unsigned char *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        const int rc = noalloc_address(dev, &scratch);
        if (rc != CDG_OK) return rc;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, scratch, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return CDG_ERR_CUDA;
    if (v != 0) {
        if (cudaMemsetAsync(scratch, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
            return CDG_ERR_CUDA;
    }
    return v;
}

// ------------------------------------------------------------------ back-to-back fusion
struct cdg_fused_st {
    cdg_plan_st *g;  // GEMM 1: the first dgrad (stride 1, halo operand mode, resident weights)
    int C1, BN2;     // dX1 channels and GEMM 2's N tile
    bool write_g;
    size_t smem;
    const void *cached_W1p;
    void *cached_dX1;
};

namespace {

int fused_make(int N, int H, int W, int C1, int C2, int K2, int R2, int S2, int pad2, int dil2, int dtype, int flags,
               int num_sms, bool host_only, cdg_fused_t *out)
{
    if (!out) return CDG_ERR_INVALID_ARG;
    *out = nullptr;
    const int gates = CDG_EPI_RELU_BWD | CDG_EPI_GELU_BWD | CDG_EPI_SILU_BWD;
    if (flags & ~(gates | CDG_FUSED_WRITE_G)) return CDG_ERR_INVALID_ARG;
    if (C1 < 1) return CDG_ERR_INVALID_ARG;
    if (C2 != 64 || C1 % 8 || C1 > 256) return CDG_ERR_UNSUPPORTED;
    PlanOpts opt = opts_from_env();
    opt.halo = 1;
    opt.bn = 0;
    opt.gate_bufs = 4;  // the fused kernel lays out its own shared memory
    opt.dual = 0;       // and issues its MMAs from one warp,
    opt.pair = 0;       // in single CTAs
    cdg_handle_t g = nullptr;
    int rc = make_plan(N, H, W, C2, K2, R2, S2, 1, pad2, dil2, dtype, flags & gates, num_sms, host_only, opt, &g);
    if (rc != CDG_OK) return rc;
    CdgParams &p = g->prm;
    // the first dgrad must be one phase in halo mode with its whole filter resident
    if (!p.halo || !p.b_res || p.tiles_n != 1 || p.BN != 64 || p.nphases != 1 || p.phase[0].tap_count < 1) {
        cdg_destroy(g);
        return CDG_ERR_UNSUPPORTED;
    }
    const bool gated = (flags & gates) != 0;
    const int BN2 = ((C1 + 15) / 16) * 16;
    const int w1_bytes = BN2 * 128;
    const int fixed = 1024 + static_cast<int>(p.b_res_bytes) + w1_bytes + (gated ? CDG_FUSED_X2_BYTES : 0) +
                      CDG_SMEM_STAGING + CDG_SMEM_TAIL;
    const int as = std::min(3, (kMaxSmem - fixed) / static_cast<int>(p.a_stage_bytes));
    if (as < 2) {
        cdg_destroy(g);
        return CDG_ERR_UNSUPPORTED;
    }
    p.a_stages = as;
    p.stages = as;
    p.C1 = C1;
    p.BN2 = BN2;
    p.w1_bytes = static_cast<uint32_t>(w1_bytes);
    p.write_g = (flags & CDG_FUSED_WRITE_G) ? 1 : 0;
    const uint32_t ab = dtype == CDG_BF16 ? 1u : 0u;
    p.idesc2 = (1u << 4) | (ab << 7) | (ab << 10) | (static_cast<uint32_t>(BN2 >> 3) << 17) | (static_cast<uint32_t>(CDG_BM >> 4) << 24);
    cdg_fused_st *f = new (std::nothrow) cdg_fused_st();
    if (!f) {
        cdg_destroy(g);
        return CDG_ERR_INVALID_ARG;
    }
    f->g = g;
    f->C1 = C1;
    f->BN2 = BN2;
    f->write_g = p.write_g != 0;
    f->smem = static_cast<size_t>(fixed + as * static_cast<int>(p.a_stage_bytes));
    if (!host_only && cdg_prepare_fused(g->in_type, gated ? p.act : -1) != cudaSuccess) {
        cdg_destroy(g);
        delete f;
        return CDG_ERR_CUDA;
    }
    *out = f;
    return CDG_OK;
}

int encode_fused_maps(cdg_fused_st *f, const void *W1p, void *dX1)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return CDG_ERR_CUDA;
    const cdg_plan_st *g = f->g;
    CdgParams &p = f->g->prm;
    const CUtensorMapDataType dt = tmap_type(g->dtype);
    const cuuint32_t ones[4] = {1, 1, 1, 1};
    const cuuint64_t C1 = f->C1, C2 = g->C;
    const cuuint64_t wdims[3] = {C2, C1, 1};
    const cuuint64_t wstrides[2] = {C2 * 2, C1 * C2 * 2};
    const cuuint32_t wbox[3] = {CDG_BK, static_cast<cuuint32_t>(f->BN2), 1};
    if (enc(&p.tmW1, dt, 3, const_cast<void *>(W1p), wdims, wstrides, wbox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
        return CDG_ERR_CUDA;
    const cuuint64_t Wd = g->W, Hd = g->H;
    const cuuint64_t xdims[4] = {C1, Wd, Hd, static_cast<cuuint64_t>(g->N)};
    const cuuint64_t xstrides[3] = {C1 * 2, Wd * C1 * 2, Hd * Wd * C1 * 2};
    const cuuint32_t xbox[4] = {64, static_cast<cuuint32_t>(p.halo_wt), static_cast<cuuint32_t>(p.halo_bh), 1};
    if (enc(&p.tmX1, dt, 4, dX1, xdims, xstrides, xbox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return CDG_ERR_CUDA;
    f->cached_W1p = W1p;
    f->cached_dX1 = dX1;
    return CDG_OK;
}

}  // namespace

extern "C" {

int cdg_fused_plan(int N, int H, int W, int C1, int C2, int K2, int R2, int S2, int pad2, int dil2, int dtype,
                   int flags, cdg_fused_t *out)
{
    if (out) *out = nullptr;
    cdg_fused_t probe = nullptr;
    int rc = fused_make(N, H, W, C1, C2, K2, R2, S2, pad2, dil2, dtype, flags, 1, true, &probe);
    if (rc != CDG_OK) return rc;
    cdg_fused_destroy(probe);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CDG_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return CDG_ERR_CUDA;
    return fused_make(N, H, W, C1, C2, K2, R2, S2, pad2, dil2, dtype, flags, sms, false, out);
}

int cdg_fused_plan_host(int N, int H, int W, int C1, int C2, int K2, int R2, int S2, int pad2, int dil2, int dtype,
                        int flags, int num_sms, cdg_fused_t *out)
{
    if (num_sms < 1) {
        if (out) *out = nullptr;
        return CDG_ERR_INVALID_ARG;
    }
    return fused_make(N, H, W, C1, C2, K2, R2, S2, pad2, dil2, dtype, flags, num_sms, true, out);
}

void cdg_fused_destroy(cdg_fused_t f)
{
    if (!f) return;
    cdg_destroy(f->g);
    delete f;
}

int cdg_fused_packed_weight_bytes(cdg_fused_t f, size_t *w2_bytes, size_t *w1_bytes)
{
    if (!f || !w2_bytes || !w1_bytes) return CDG_ERR_INVALID_ARG;
    *w2_bytes = cdg_packed_weight_bytes(f->g);
    *w1_bytes = static_cast<size_t>(f->C1) * f->g->C * 2;
    return CDG_OK;
}

int cdg_fused_prepack_weights(cdg_fused_t f, const void *W2_krsc, const void *W1_krsc, void *W2p, void *W1p,
                              cdg_stream_t stream)
{
    if (!f || !W2_krsc || !W1_krsc || !W2p || !W1p) return CDG_ERR_INVALID_ARG;
    if (f->g->host_only) return CDG_ERR_NO_DEVICE;
    if (!aligned16(W1_krsc) || !aligned16(W1p)) return CDG_ERR_ALIGNMENT;
    size_t b2 = 0, b1 = 0;
    cdg_fused_packed_weight_bytes(f, &b2, &b1);
    if (overlaps(W1_krsc, b1, W1p, b1) || overlaps(W1p, b1, W2p, b2) || overlaps(W1p, b1, W2_krsc, b2) ||
        overlaps(W2p, b2, W1_krsc, b1))
        return CDG_ERR_ALIAS;
    const int rc = cdg_prepack_weights(f->g, W2_krsc, W2p, stream);
    if (rc != CDG_OK) return rc;
    // the 1x1 layer: W1 [C2][1][1][C1] -> [1][C1][C2], its dgrad's B operand
    if (cdg_launch_prepack(W1_krsc, W1p, f->g->C, 1, f->C1, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CDG_ERR_CUDA;
    return CDG_OK;
}

int cdg_dgrad_fused(cdg_fused_t f, const void *dY2, const void *W2p, const void *x2, const void *W1p, void *g,
                    void *dX1, cdg_stream_t stream)
{
    if (!f || !dY2 || !W2p || !W1p || !dX1) return CDG_ERR_INVALID_ARG;
    cdg_plan_st *h = f->g;
    if (h->mask != (x2 != nullptr) || f->write_g != (g != nullptr)) return CDG_ERR_INVALID_ARG;
    if (h->host_only) return CDG_ERR_NO_DEVICE;
    if (!aligned16(dY2) || !aligned16(W2p) || !aligned16(W1p) || !aligned16(dX1) || (x2 && !aligned16(x2)) ||
        (g && !aligned16(g)))
        return CDG_ERR_ALIGNMENT;
    size_t b2 = 0, b1 = 0;
    cdg_fused_packed_weight_bytes(f, &b2, &b1);
    const size_t px = static_cast<size_t>(h->N) * h->H * h->W;
    const size_t dy_bytes = static_cast<size_t>(h->N) * h->P * h->Q * h->K * 2;
    const void *ins[4] = {dY2, W2p, x2, W1p};
    const size_t inb[4] = {dy_bytes, b2, x2 ? px * h->C * 2 : 0, b1};
    void *outs[2] = {dX1, g};
    const size_t outb[2] = {px * f->C1 * 2, g ? px * h->C * 2 : 0};
    for (int i = 0; i < 2; ++i) {
        if (!outs[i]) continue;
        for (int j = 0; j < 4; ++j)
            if (ins[j] && overlaps(outs[i], outb[i], ins[j], inb[j])) return CDG_ERR_ALIAS;
    }
    if (g && overlaps(dX1, outb[0], g, outb[1])) return CDG_ERR_ALIAS;
    if (dY2 != h->cached_dY || W2p != h->cached_Wp) {
        const int rc = encode_operand_maps(h, dY2, W2p);
        if (rc != CDG_OK) return rc;
    }
    if (g && g != h->cached_dX) {
        const int rc = encode_store_maps(h, g);
        if (rc != CDG_OK) return rc;
    }
    if (x2 && x2 != h->cached_mask) {
        const int rc = encode_gate_maps(h, x2);
        if (rc != CDG_OK) return rc;
    }
    if (W1p != f->cached_W1p || dX1 != f->cached_dX1) {
        const int rc = encode_fused_maps(f, W1p, dX1);
        if (rc != CDG_OK) return rc;
    }
    CdgParams &p = h->prm;
    p.dX = g;
    p.mask = x2;
    p.status = h->d_status;
    p.red_ws = nullptr;
    if (cdg_launch_fused(p, h->in_type, h->mask ? p.act : -1, h->grid, f->smem, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return CDG_ERR_CUDA;
    return CDG_OK;
}

int cdg_fused_get_info(cdg_fused_t f, cdg_plan_info_t *info)
{
    if (!f || !info) return CDG_ERR_INVALID_ARG;
    *info = f->g->info;
    info->stages = f->g->prm.a_stages;
    info->smem_bytes = static_cast<int>(f->smem);
    info->tmem_cols = 512;
    return CDG_OK;
}

int cdg_fused_device_status(cdg_fused_t f, cdg_stream_t stream)
{
    if (!f) return CDG_ERR_INVALID_ARG;
    return cdg_device_status(f->g, stream);
}

}  // extern "C"
