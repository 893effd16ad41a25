// Implicit-GEMM Conv2d dgrad for sm_103a (GB300): the device code (role
// functions, kernels as templates), shared by the translation units that
// instantiate the kernels.
//
// GEMM view (apache/tvm PR #10110, "[CUTLASS] Conv2d dgrad": the dgrad the page
// benchmarks runs as an implicit GEMM): for one phase sub-convolution,
//   M = dX pixels of the phase sub-grid, N = C, K = (taps of the phase) x K.
// A[m, (tap, k)] = dY[n, i + dr, j + ds, k]  (zero outside dY),
// B[(tap, k), c] = W[k, r, s, c]             (packed as [tap][c][k]).
// A stride-s problem runs as its s^2 phase sub-convolutions (the "strided
// dgrad" case of the same page) inside one persistent launch, so no
// zero-inserted multiply is ever issued; phases that no tap reaches are
// written as zeros by the epilogue.
//
// CTA layout (256 threads, one CTA per SM, persistent over work items,
// launched with programmatic stream serialization):
//   warps 0, 2, 3  TMA loaders: per (tap, 64-channel block of K) one dY box
//                  and one weight box into a ring of stages (mbarrier
//                  full/empty), stages taken round-robin;
//   warp 1         owns TMEM; one elected lane issues tcgen05.mma (M=128,
//                  N=BN, K=16) into one of two fp32 accumulators and commits
//                  stages back;
//   warps 4-7      epilogue: tcgen05.ld of the accumulator, optional
//                  ReLU-backward gate, RNE conversion into a swizzled staging
//                  buffer, TMA bulk stores into NHWC dX.
// Modes (MODE below): halo boxes (one dY box per tile and K block for all
// taps, weights resident or streamed), CTA pairs (2-SM MMA over 256-row
// tiles), dual issue (warps 1 and 3 issue MMAs for alternate items, each fed
// by its own loader warp 0 or 2 and ring half, with two accumulators each).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "cdg_params.h"
#include "ptx.cuh"
#include "wait.cuh"

namespace cdg {

// n / d for 0 <= n < 2^31 with d's precomputed multiplier and shift (CdgDiv).
__device__ __forceinline__ int fdiv(int n, CdgDiv d)
{
    return static_cast<int>((__umulhi(static_cast<uint32_t>(n), d.mul) + static_cast<uint32_t>(n)) >> d.shr);
}

// Walk over this CTA's work items g = start, start + step, ... as (phase,
// index within the phase), phases read from the shared-memory copy.  The
// first `il` phases (il >= 2, all with il_items items) are interleaved: the
// items of scheduling round r (G consecutive items, one per CTA or CTA pair;
// G a multiple of il) are tiles r*G/il .. (r+1)*G/il - 1 of every one of those
// phases, so the phases' tiles over the same region of dY run together and
// share it through L2; position pos = il*a + b of the round is tile
// r*G/il + a of phase (b + r) mod il, which rotates each CTA through the
// phases (their tap counts differ) from round to round.  The remaining phases
// follow one after another.
struct ItemWalk {
    const CdgPhase *tab;
    int nph, step, il, il_items, il_round, per_round;
    CdgDiv div_il, div_round;
    int g, phase, local;
    // items start, start + step, ...: one CTA's (step = gridDim.x) or one CTA
    // pair's (step = number of pairs) share of the work list
    __device__ __forceinline__ ItemWalk(const CdgPhase *t, const CdgParams &p, int start, int stp)
        : tab(t), nph(p.nphases), step(stp), il(p.interleave), il_items(p.il_items), il_round(p.il_round),
          per_round(0), div_il(p.div_il), div_round(p.div_il_round), g(start), phase(0), local(0)
    {
        if (il > 0) per_round = fdiv(il_round, div_il);  // tiles of each phase per round
        settle();
    }
    __device__ __forceinline__ void settle()
    {
        if (il > 0 && g < il * il_items) {
            const int r = fdiv(g, div_round);
            const int pos = g - r * il_round;
            const int a = fdiv(pos, div_il);
            const int b = pos - a * il;
            const int rr = r - fdiv(r, div_il) * il;  // r mod il
            phase = b + rr >= il ? b + rr - il : b + rr;
            local = r * per_round + a;
            return;
        }
        phase = il;
        local = g - il * il_items;
        while (phase < nph && local >= tab[phase].items) {
            local -= tab[phase].items;
            ++phase;
        }
    }
    __device__ __forceinline__ bool valid() const { return phase < nph; }
    __device__ __forceinline__ void next()
    {
        g += step;
        settle();
    }
};

// Work distribution: which items this CTA walks, and (pairs) its M tile in a pair.
struct Sched {
    int start, step;
    int pair;   // 1: CTA pairs share each item (M tiles 2*t and 2*t + 1)
    int rank;   // rank in the pair (0 = leader, issues the MMAs)
    __device__ __forceinline__ int m_tile(int local, int tiles_n, CdgDiv div_tiles_n) const
    {
        const int t = tiles_n == 1 ? local : fdiv(local, div_tiles_n);
        return pair ? 2 * t + rank : t;
    }
};

// Origin (j0, i0, n0) of 4-D box tile mt of phase `phase` (tiles_w x tiles_h
// boxes per image).
__device__ __forceinline__ void box_origin(const CdgParams &p, const CdgPhase &ph, int phase, int mt, int bw, int bh,
                                           int bn, int &j0, int &i0, int &n0)
{
    const int rest = fdiv(mt, p.div_tiles_w[phase]);
    const int tj = mt - rest * ph.tiles_w;
    const int tn = fdiv(rest, p.div_tiles_h[phase]);
    const int ti = rest - tn * ph.tiles_h;
    j0 = tj * bw;
    i0 = ti * bh;
    n0 = tn * bn;
}

struct Ring {
    int stages;            // stages of this ring (dual issue: each MMA warp has a ring of its own)
    uint32_t a0;           // shared address of stage 0's A tile (1024-aligned)
    uint32_t stage_bytes;  // A tile + B tile (halo mode: one halo box stage)
    uint32_t b0;           // halo mode: first weight stage
    uint32_t b_bytes;      // halo mode: bytes of one weight stage
    uint32_t out0;         // first of the 16 KB output staging buffers (two; four when gated by the activation)
    uint32_t full0, empty0;
    uint32_t acc_full0, acc_empty0, drain;
    uint32_t gfull0;       // gate loads: eight mbarriers
    uint32_t gfree0;       // activation gate issued by a loader warp: eight "staging buffer free" mbarriers
    uint32_t gate0;        // packed-mask ring (four CDG_GATE_SLOT slots)
    uint32_t red0;         // per-channel sums: the warps' partials of one chunk, [sum][warp][64] fp32
};

// ------------------------------------------------------------------ loaders
// nloaders warps walk the same (item, tap, k-block) sequence; the loader
// with index li issues the stages whose global counter is li modulo
// nloaders.  The whole warp runs the loop; one elected lane issues.  The parity of
// each slot's latest load is recorded in shared memory for the abort drain.
template <bool PAIR>
__device__ __forceinline__ void run_loader(const CdgParams &p, const Ring &R, const CdgPhase *tab,
                                           const CdgTap *taps, Ctl ctl, int li, int nloaders, bool leader,
                                           volatile uint32_t *slot_parity, Sched S)
{
    const uint64_t mapA = reinterpret_cast<uint64_t>(&p.tmA);
    const uint64_t mapB = reinterpret_cast<uint64_t>(&p.tmB);
    if (leader) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(mapA) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(mapB) : "memory");
    }
    const int KB = p.KB, stages = R.stages, tiles_n = p.tiles_n, BN = p.BN, m_step = p.m_step;
    const int bw = p.box_w, bh = p.box_h, bn = p.box_n;
    const bool flat = p.a_flat != 0;
    const uint32_t tx = p.tx_bytes;
    const uint32_t a0 = R.a0, sbytes = R.stage_bytes, full0 = R.full0, empty0 = R.empty0;
    const uint32_t lead_full0 = PAIR ? mapa_shared(full0, 0) : full0;

    int stage = 0;
    uint32_t parity = 0;
    int owner = 0;  // loader index of the current global stage
    int seq = 0;    // sequence number of the current stage (all loaders count every stage)
    const int withhold = p.withhold_stage;
    // Row-matrix operands (1x1 filters), with p.prefetch: the dY rows of the
    // stage kPrefetchStages ahead are prefetched into L2 by the owner of the
    // current stage, so that the ring's loads find them there.  Measured on
    // GB300 this makes the 1x1 layers slower (the ring already covers the
    // latency), so plans leave it off unless asked.
    constexpr int kPrefetchStages = 8;
    ItemWalk pw(tab, p, S.start, S.step);
    int pkb = 0;
    auto pf_advance = [&]() {
        if (!pw.valid()) return;
        if (++pkb == KB) {
            pkb = 0;
            pw.next();
        }
    };
    const bool prefetch = flat && p.prefetch;
    if (prefetch)
        for (int i = 0; i < kPrefetchStages; ++i) pf_advance();
    bool ok = true;
    for (ItemWalk w(tab, p, S.start, S.step); ok && w.valid(); w.next()) {
        const CdgPhase &ph = tab[w.phase];
        const int ntap = ph.tap_count;
        if (ntap == 0) continue;
        const int tq = tiles_n == 1 ? w.local : fdiv(w.local, p.div_tiles_n);
        const int nt = w.local - tq * tiles_n;
        const int mt = S.m_tile(w.local, tiles_n, p.div_tiles_n);
        int j0 = 0, i0 = 0, n0 = 0;
        if (!flat) box_origin(p, ph, w.phase, mt, bw, bh, bn, j0, i0, n0);
        // a pair splits the N tile's weight rows: this CTA loads its half
        const int c0 = nt * BN + (PAIR ? S.rank * (BN / 2) : 0);
        const int m0 = mt * m_step;
        for (int tt = 0; ok && tt < ntap; ++tt) {
            const CdgTap tap = taps[ph.tap_begin + tt];
            const int y = j0 + tap.ds, z = i0 + tap.dr, t = tap.t;
            for (int kb = 0; kb < KB; ++kb) {
                if (owner == li) {
                    const uint32_t full = full0 + 8u * stage;
                    if (!wait_bar(empty0 + 8u * stage, parity ^ 1u, ctl)) {
                        ok = false;
                        break;
                    }
                    if (prefetch && leader && pw.valid() && tab[pw.phase].tap_count > 0)
                        tma_prefetch_2d(mapA, pkb * CDG_BK, S.m_tile(pw.local, tiles_n, p.div_tiles_n) * m_step);
                    // (test only) a withheld stage gets neither its copies nor
                    // their byte count, and is not recorded for the abort drain:
                    // its full barrier never completes, so the consumer's
                    // bounded wait runs out and the launch aborts
                    if (leader && seq != withhold) {
                        slot_parity[stage] = parity | 2u;  // bit 1: slot used
                        const uint32_t sa = a0 + stage * sbytes;
                        if (PAIR) {
                            // both CTAs' copies complete on the leader's barrier,
                            // which expects the bytes of both
                            const uint32_t lead = lead_full0 + 8u * stage;
                            if (S.rank == 0) mbar_arrive_expect_tx(full, tx);
                            if (flat)
                                tma_load_2d_pair(sa, mapA, lead, kb * CDG_BK, m0);
                            else
                                tma_load_4d_pair(sa, mapA, lead, kb * CDG_BK, y, z, n0);
                            tma_load_3d_pair(sa + CDG_BM * 128, mapB, lead, kb * CDG_BK, c0, t);
                        } else {
                            mbar_arrive_expect_tx(full, tx);
                            if (flat)
                                tma_load_2d(sa, mapA, full, kb * CDG_BK, m0);
                            else
                                tma_load_4d(sa, mapA, full, kb * CDG_BK, y, z, n0);
                            tma_load_3d(sa + CDG_BM * 128, mapB, full, kb * CDG_BK, c0, t);
                        }
                    }
                    __syncwarp();
                }
                if (++owner == nloaders) owner = 0;
                ++seq;
                if (prefetch) pf_advance();
                if (++stage == stages) {
                    stage = 0;
                    parity ^= 1u;
                }
            }
        }
    }
}

// After an abort: wait (bounded) until the latest load of every used slot has
// landed, so that no TMA still writes shared memory when the CTA exits.  On
// the normal path the MMA warp has already waited for every load.
__device__ __forceinline__ void drain_loads(const Ring &R, int stages, int *status, uint64_t limit,
                                            const volatile uint32_t *slot_parity)
{
    volatile uint32_t no_abort = 0;
    const Ctl drain_ctl{&no_abort, status, limit};
    for (int s = 0; s < stages; ++s) {
        const uint32_t v = slot_parity[s];
        if (v & 2u) wait_bar(R.full0 + 8u * s, v & 1u, drain_ctl);
    }
}

// ------------------------------------------------------------------ halo-mode loaders
// Loader 0 streams one dY halo box per (tile, K block) into the A ring;
// loaders 1.. stream the weight tiles, up to tg taps per stage, into the B
// ring round-robin (or loader 1 loads every weight tile once, when resident).
// CTA pairs (PAIR): each CTA loads the halo box of its own M tile and its half
// of every weight tile's rows, and all of them complete on the leader's
// barriers, which expect the bytes of both CTAs.
// Two MMA warps (DUALH): the halo box of the n-th item with taps completes on
// the full barrier of its stage for MMA warp n % 2: stage s for warp 0,
// a_stages + b_stages + s for warp 1.
template <bool PAIR, bool DUALH = false>
__device__ __forceinline__ void run_loader_halo(const CdgParams &p, const Ring &R, const CdgPhase *tab,
                                                const CdgTap *taps, Ctl ctl, int li, bool leader,
                                                volatile uint32_t *slot_parity, Sched S)
{
    const uint32_t lead_full0 = PAIR ? mapa_shared(R.full0, 0) : R.full0;
    const uint32_t pair_mul = PAIR ? 2u : 1u;  // the leader's barriers count both CTAs' bytes
    const int b_row0 = PAIR ? S.rank * (p.BN / 2) : 0;
    const uint64_t mapA = reinterpret_cast<uint64_t>(&p.tmA);
    const uint64_t mapB = reinterpret_cast<uint64_t>(&p.tmB);
    if (leader) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(mapA) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(mapB) : "memory");
    }
    const int KB = p.KB, tiles_n = p.tiles_n, BN = p.BN;
    const int as = p.a_stages, bs = p.b_stages, bh = p.halo_bh, wt = p.halo_wt, tg = p.halo_tg;
    const uint32_t tx_a = p.tx_a;
    const uint32_t gstride = static_cast<uint32_t>(tg) * R.b_bytes;  // bytes of one weight stage
    int a_stage = 0, b_stage = 0, owner = 1;
    uint32_t a_par = 0, b_par = 0;
    bool ok = true;
    // with p.prefetch (off unless asked: measured slower), loader 0 prefetches
    // into L2 the halo box kPrefetchBoxes (tile, K block) steps ahead of the
    // one it loads
    constexpr int kPrefetchBoxes = 4;
    ItemWalk pw(tab, p, S.start, S.step);
    int pkb = 0;
    auto pf_advance = [&]() {
        if (!pw.valid()) return;
        if (++pkb == KB) {
            pkb = 0;
            pw.next();
        }
    };
    if (li == 0)
        for (int i = 0; i < kPrefetchBoxes; ++i) pf_advance();
    if (p.b_res && li == 1) {
        // every (tap, K block) weight tile of the single N tile, in the order of
        // the tap table (phase by phase), completing on the one weight barrier
        const uint32_t full = R.full0 + 8u * as;
        if (leader) {
            slot_parity[as] = 2u;
            if (!PAIR || S.rank == 0) mbar_arrive_expect_tx(full, pair_mul * p.b_res_bytes);
            for (int q = 0; q < p.ntaps; ++q)
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t dst = R.b0 + static_cast<uint32_t>(q * KB + kb) * R.b_bytes;
                    if (PAIR)
                        tma_load_3d_pair(dst, mapB, lead_full0 + 8u * as, kb * CDG_BK, b_row0, taps[q].t);
                    else
                        tma_load_3d(dst, mapB, full, kb * CDG_BK, 0, taps[q].t);
                }
        }
        __syncwarp();
    }
    uint32_t n_item = 0;             // items with taps so far (two MMA warps: item n is warp n % 2's)
    uint32_t wpar[2] = {0u, 0u};     // two MMA warps: parity bit per stage of each warp's full barriers
    for (ItemWalk w(tab, p, S.start, S.step); ok && w.valid(); w.next()) {
        const CdgPhase &ph = tab[w.phase];
        const int ntap = ph.tap_count;
        if (ntap == 0) continue;
        const int mt = S.m_tile(w.local, tiles_n, p.div_tiles_n);
        const int nt = w.local - (tiles_n == 1 ? w.local : fdiv(w.local, p.div_tiles_n)) * tiles_n;
        int j0, i0, n0;
        box_origin(p, ph, w.phase, mt, wt, bh, 1, j0, i0, n0);
        const int c0 = nt * BN;
        const uint32_t wj = DUALH ? (n_item & 1u) : 0u;
        ++n_item;
        for (int kb = 0; ok && kb < KB; ++kb) {
            if (li == 0) {
                // this stage's full barrier (two MMA warps: the item's warp's own)
                const int fidx = wj ? as + bs + a_stage : a_stage;
                const uint32_t fpar = DUALH ? (wpar[wj] >> a_stage) & 1u : a_par;
                if (DUALH) wpar[wj] ^= 1u << a_stage;
                const uint32_t full = R.full0 + 8u * fidx;
                if (!wait_bar(R.empty0 + 8u * a_stage, a_par ^ 1u, ctl)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    slot_parity[fidx] = fpar | 2u;
                    if (!PAIR || S.rank == 0) mbar_arrive_expect_tx(full, pair_mul * tx_a);
                    if (PAIR)
                        tma_load_4d_pair(R.a0 + a_stage * R.stage_bytes, mapA, lead_full0 + 8u * fidx, kb * CDG_BK,
                                         j0 + ph.ds_min, i0 + ph.dr_min, n0);
                    else
                        tma_load_4d(R.a0 + a_stage * R.stage_bytes, mapA, full, kb * CDG_BK, j0 + ph.ds_min,
                                    i0 + ph.dr_min, n0);
                    if (p.prefetch && pw.valid() && tab[pw.phase].tap_count > 0) {
                        const CdgPhase &pph = tab[pw.phase];
                        int pj, pi, pn;
                        box_origin(p, pph, pw.phase, S.m_tile(pw.local, tiles_n, p.div_tiles_n), wt, bh, 1, pj, pi, pn);
                        tma_prefetch_4d(mapA, pkb * CDG_BK, pj + pph.ds_min, pi + pph.dr_min, pn);
                    }
                }
                __syncwarp();
                pf_advance();
                if (++a_stage == as) {
                    a_stage = 0;
                    a_par ^= 1u;
                }
            } else if (p.b_res) {
                // resident weights: loaded once, before the first tile (above)
            } else {
                // weight stages of up to tg taps each: one handshake per group
                for (int g0 = 0; g0 < ntap; g0 += tg) {
                    const int n_in = min(tg, ntap - g0);
                    if (owner == li) {
                        const int slot = as + b_stage;
                        const uint32_t full = R.full0 + 8u * slot;
                        if (!wait_bar(R.empty0 + 8u * slot, b_par ^ 1u, ctl)) {
                            ok = false;
                            break;
                        }
                        if (leader) {
                            slot_parity[slot] = b_par | 2u;
                            if (!PAIR || S.rank == 0)
                                mbar_arrive_expect_tx(full, pair_mul * static_cast<uint32_t>(n_in) * R.b_bytes);
                            for (int i = 0; i < n_in; ++i) {
                                const uint32_t dst = R.b0 + b_stage * gstride + static_cast<uint32_t>(i) * R.b_bytes;
                                if (PAIR)
                                    tma_load_3d_pair(dst, mapB, lead_full0 + 8u * slot, kb * CDG_BK, c0 + b_row0,
                                                     taps[ph.tap_begin + g0 + i].t);
                                else
                                    tma_load_3d(dst, mapB, full, kb * CDG_BK, c0, taps[ph.tap_begin + g0 + i].t);
                            }
                        }
                        __syncwarp();
                    }
                    if (++owner == CDG_LOADERS) owner = 1;
                    if (++b_stage == bs) {
                        b_stage = 0;
                        b_par ^= 1u;
                    }
                }
            }
        }
    }
}

// Halo-mode MMA issuer: per K block one halo stage; per group of up to tg taps
// one weight stage (or the resident weights), and per tap four MMAs whose A
// operand starts at the tap's row of the halo box.  With CTA pairs (PAIR) the
// leader issues 2-SM MMAs over both CTAs' halo boxes (the same layout, so the
// same descriptors) and weight halves, and its commits reach both CTAs.
// With two MMA warps (DUALH; resident weights only) warp j takes the items
// at positions j, j + 2, ... of the CTA's walk (S as given), and the halo
// stages of those items: the ring is filled in item order by one loader, so
// stage n (n = item position x KB + K block) is the warp's when its item is.
template <bool PAIR, bool DUALH = false>
__device__ __forceinline__ void run_mma_halo(const CdgParams &p, const Ring &R, const CdgPhase *tab,
                                             const CdgTap *taps, Ctl ctl, uint32_t tmem_base, bool leader, Sched S,
                                             int j = 0)
{
    auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
        if (PAIR)
            umma_f16_pair(d, a, b, p.idesc, acc);
        else
            umma_f16(d, a, b, p.idesc, acc);
    };
    auto commit = [&](uint32_t bar) {
        if (PAIR)
            umma_commit_pair(bar);
        else
            umma_commit(bar);
    };
    const int KB = p.KB, as = p.a_stages, bs = p.b_stages, tg = p.halo_tg;
    const uint32_t acc_stride = p.acc_stride;
    const uint64_t adesc0 = sdesc_k128_sw128(R.a0);
    const uint64_t bdesc0 = sdesc_k128_sw128(R.b0);
    const uint32_t astep = R.stage_bytes >> 4;  // descriptor units per halo stage
    int a_stage = 0, b_stage = 0;
    uint32_t a_par = 0, b_par = 0, acc_count = 0;
    // advance the halo-stage cursor by n stages
    auto a_skip = [&](int n) {
        for (int i = 0; i < n; ++i)
            if (++a_stage == as) {
                a_stage = 0;
                a_par ^= 1u;
            }
    };
    if (DUALH) a_skip(j * KB);  // warp 1's first item is the CTA's second
    // two MMA warps: this warp's full barriers (stage s: s, or a_stages +
    // b_stages + s for warp 1) and their parities, one bit per stage
    const uint32_t full_w = R.full0 + (DUALH && j ? 8u * static_cast<uint32_t>(as + bs) : 0u);
    uint32_t wpar = 0u;
    bool ok = true;
    bool b_ready = false;  // full barrier of the current weight stage already seen complete
    const bool res = p.b_res != 0;
    if (res && !wait_bar(R.full0 + 8u * as, 0, ctl)) ok = false;  // resident weights landed
    for (ItemWalk w(tab, p, S.start, S.step); ok && w.valid(); w.next()) {
        const CdgPhase &ph = tab[w.phase];
        const int ntap = ph.tap_count;
        if (ntap == 0) continue;
        // halo plans may keep up to four accumulators in flight (p.acc_ring)
        const uint32_t acc = acc_count & (p.acc_ring - 1u);
        const uint32_t acc_parity = (acc_count >> (p.acc_ring == 4u ? 2 : 1)) & 1u;
        if (!wait_bar(R.acc_empty0 + 8u * acc, acc_parity ^ 1u, ctl)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * acc_stride;
        for (int kb = 0; ok && kb < KB; ++kb) {
            const uint32_t fpar = DUALH ? (wpar >> a_stage) & 1u : a_par;
            if (DUALH) wpar ^= 1u << a_stage;
            if (!wait_bar(full_w + 8u * a_stage, fpar, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t abase = adesc0 + static_cast<uint64_t>(a_stage * astep);
            const CdgTap *ptap = taps + ph.tap_begin;
            int hoff = ptap[0].hoff;  // loaded a stage ahead: its latency overlaps MMA issue
            if (res) {
                // all taps of this K block back to back: one handshake per halo box
                const uint32_t bunit = R.b_bytes >> 4;  // descriptor units per weight tile
                const int tbase = ph.tap_begin * KB + kb;
                for (int tt = 0; tt < ntap; ++tt) {
                    if (leader) {
                        const uint64_t adesc = abase + 8u * static_cast<uint32_t>(hoff);
                        const uint64_t bdesc =
                            bdesc0 + static_cast<uint64_t>(static_cast<uint32_t>(tbase + tt * KB) * bunit);
#pragma unroll
                        for (int k = 0; k < CDG_BK / 16; ++k)
                            mma(d_tmem, adesc + 2u * k, bdesc + 2u * k, (kb | tt | k) != 0);
                    }
                    __syncwarp();
                    // the next tap's row offset is read only once this tap's MMAs
                    // are queued: an outstanding shared-memory load delays MMA issue
                    if (tt + 1 < ntap) hoff = ptap[tt + 1].hoff;
                }
            } else {
                const uint32_t bunit = R.b_bytes >> 4;  // descriptor units per weight tile
                for (int g0 = 0; g0 < ntap; g0 += tg) {
                    const int n_in = min(tg, ntap - g0);
                    const int slot = as + b_stage;
                    if (!b_ready && !wait_bar(R.full0 + 8u * slot, b_par, ctl)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int i = 0; i < n_in; ++i) {
                        const int tt = g0 + i;
                        if (leader) {
                            // 128-byte rows: a row offset of hoff is 8*hoff descriptor units
                            const uint64_t adesc = abase + 8u * static_cast<uint32_t>(hoff);
                            const uint64_t bdesc =
                                bdesc0 + static_cast<uint64_t>(static_cast<uint32_t>(b_stage * tg + i) * bunit);
#pragma unroll
                            for (int k = 0; k < CDG_BK / 16; ++k)
                                mma(d_tmem, adesc + 2u * k, bdesc + 2u * k, (kb | tt | k) != 0);
                        }
                        __syncwarp();
                        // the next tap's row offset is read only once this tap's MMAs
                        // are queued: an outstanding shared-memory load delays MMA issue
                        if (tt + 1 < ntap) hoff = ptap[tt + 1].hoff;
                    }
                    if (leader) commit(R.empty0 + 8u * slot);
                    __syncwarp();
                    if (++b_stage == bs) {
                        b_stage = 0;
                        b_par ^= 1u;
                    }
                    {  // test the next weight stage (its latency overlaps the queued MMAs)
                        b_ready = mbar_test_wait(R.full0 + 8u * (as + b_stage), b_par);
                    }
                }
            }
            if (!ok) break;
            if (leader) commit(R.empty0 + 8u * a_stage);
            __syncwarp();
            if (++a_stage == as) {
                a_stage = 0;
                a_par ^= 1u;
            }
        }
        if (!ok) break;
        if (leader) commit(R.acc_full0 + 8u * acc);
        __syncwarp();
        ++acc_count;
        if (DUALH) a_skip(KB);  // the other warp's item
    }
    if (leader) commit(R.drain);
    __syncwarp();
    volatile uint32_t no_abort = 0;
    const Ctl drain_ctl{&no_abort, ctl.status, ctl.limit};
    wait_bar(R.drain, 0, drain_ctl);
}

// ------------------------------------------------------------------ MMA issuer
// Whole warp runs the loop; one elected lane issues tcgen05.mma / tcgen05.commit.
template <bool PAIR>
__device__ __forceinline__ void run_mma(const CdgParams &p, const Ring &R, const CdgPhase *tab, Ctl ctl,
                                        uint32_t tmem_base, bool leader, Sched S)
{
    const int KB = p.KB, stages = R.stages;
    const uint32_t idesc = p.idesc, acc_stride = p.acc_stride;
    const uint64_t adesc0 = sdesc_k128_sw128(R.a0);
    const uint64_t bdesc0 = sdesc_k128_sw128(R.a0 + CDG_BM * 128);
    const uint32_t dstep = R.stage_bytes >> 4;  // descriptor units per stage
    const uint32_t full0 = R.full0, empty0 = R.empty0;

    int stage = 0;
    uint32_t parity = 0;
    uint32_t acc_count = 0;
    bool ok = true;
    bool ready = false;  // full barrier of `stage` already seen complete
    for (ItemWalk w(tab, p, S.start, S.step); ok && w.valid(); w.next()) {
        const int ntap = tab[w.phase].tap_count;
        if (ntap == 0) continue;
        const uint32_t acc = acc_count & 1u;
        const uint32_t acc_parity = (acc_count >> 1) & 1u;
        if (!wait_bar(R.acc_empty0 + 8u * acc, acc_parity ^ 1u, ctl)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * acc_stride;
        const int nk = ntap * KB;
        for (int kk = 0; kk < nk; ++kk) {
            if (!ready && !wait_bar(full0 + 8u * stage, parity, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            int next = stage + 1;
            uint32_t next_parity = parity;
            if (next == stages) {
                next = 0;
                next_parity ^= 1u;
            }
            // Test the next stage now, so that the test's latency overlaps this
            // stage's MMAs instead of idling the tensor pipe between stages.
            ready = mbar_test_wait(full0 + 8u * next, next_parity);
            if (leader) {
                const uint64_t adesc = adesc0 + static_cast<uint64_t>(stage * dstep);
                const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(stage * dstep);
#pragma unroll
                for (int k = 0; k < CDG_BK / 16; ++k) {  // 16 elements = 32 bytes = 2 descriptor units
                    if (PAIR)
                        umma_f16_pair(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kk | k) != 0);
                    else
                        umma_f16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kk | k) != 0);
                }
                if (PAIR)
                    umma_commit_pair(empty0 + 8u * stage);  // frees the slot in both CTAs
                else
                    umma_commit(empty0 + 8u * stage);
            }
            __syncwarp();
            stage = next;
            parity = next_parity;
        }
        if (!ok) break;
        if (leader) {
            if (PAIR)
                umma_commit_pair(R.acc_full0 + 8u * acc);
            else
                umma_commit(R.acc_full0 + 8u * acc);
        }
        __syncwarp();
        ++acc_count;
    }
    // All MMAs issued by this warp complete before TMEM is released.
    if (leader) {
        if (PAIR)
            umma_commit_pair(R.drain);
        else
            umma_commit(R.drain);
    }
    __syncwarp();
    volatile uint32_t no_abort = 0;
    const Ctl drain_ctl{&no_abort, ctl.status, ctl.limit};
    wait_bar(R.drain, 0, drain_ctl);
}

// ------------------------------------------------------------------ epilogue
template <int IN_T>
__device__ __forceinline__ float gate_value(uint16_t bits)
{
    if (IN_T == CDG_T_BF16) return __uint_as_float(static_cast<uint32_t>(bits) << 16);
    return __half2float(__ushort_as_half(bits));
}

__device__ __forceinline__ uint32_t pack2(float a, float b, int out_t)
{
    if (out_t == CDG_T_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void ld_shared_v2(uint32_t addr, uint32_t (&v)[2])
{
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "r"(addr) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t (&v)[4])
{
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "r"(addr)
                 : "memory");
}

// The gate's lookahead: a position in this CTA's sequence of gate loads, one
// per output chunk (CH channels of a work item with taps: saved activation) or
// one per such item (packed mask).  Items without taps come after all items
// with taps in every CTA's walk (the planner sorts those phases last and
// interleaves only phases with taps), so the sequence ends at the first one.
struct GateCursor {
    ItemWalk w;
    int cc;  // channel offset of the chunk within the item's N tile
    __device__ __forceinline__ bool valid() const { return w.valid() && w.tab[w.phase].tap_count > 0; }
    __device__ __forceinline__ void next(int step, int BN)
    {
        cc += step;
        if (cc >= BN) {
            cc = 0;
            w.next();
        }
    }
};

// Issue the TMA load of the cursor's gate tile: the dX store box of that chunk
// or item, read from the saved activation (the chunk's channels, laid out as
// the chunk's output staging) or from the packed mask (the item's bytes of each
// pixel row).  Completion lands on `bar` (expecting p.gate_tx bytes).
// With PREFETCH the same box is only prefetched into L2 (no destination, no
// barrier), further ahead than the loads.
template <bool PREFETCH>
__device__ __forceinline__ void gate_issue(const CdgParams &p, const GateCursor &gc, const Sched &S, uint32_t dst,
                                           uint32_t bar)
{
    const CdgPhase &ph = gc.w.tab[gc.w.phase];
    const int mt = S.m_tile(gc.w.local, p.tiles_n, p.div_tiles_n);
    const int nt = gc.w.local - (p.tiles_n == 1 ? gc.w.local : fdiv(gc.w.local, p.div_tiles_n)) * p.tiles_n;
    const int x0 = p.mask_bits ? (p.tiles_n == 1 ? 0 : nt * (p.BN / 8)) : nt * p.BN + gc.cc;
    const uint64_t map = reinterpret_cast<uint64_t>(&p.tmG[gc.w.phase]);
    if (!PREFETCH) mbar_arrive_expect_tx(bar, p.gate_tx);
    if (p.d_mode == CDG_D_BOX4) {
        int j0, i0, n0;
        box_origin(p, ph, gc.w.phase, mt, max(p.box_w, 1), max(p.box_h, 1), max(p.box_n, 1), j0, i0, n0);
        if (PREFETCH)
            tma_prefetch_4d(map, x0, j0, i0, n0);
        else
            tma_load_4d(dst, map, bar, x0, j0, i0, n0);
    } else if (p.d_mode == CDG_D_LINEAR) {
        if (PREFETCH)
            tma_prefetch_2d(map, x0, mt * p.m_step);
        else
            tma_load_2d(dst, map, bar, x0, mt * p.m_step);
    } else {
        if (PREFETCH)
            tma_prefetch_3d(map, x0, 0, mt * p.rows_per_tile);
        else
            tma_load_3d(dst, map, bar, x0, 0, mt * p.rows_per_tile);
    }
}

// With p.prefetch (off unless asked: measured slower on GB300), gate tiles
// are prefetched into L2 this many loads ahead of their loads into shared
// memory.
constexpr int kGatePrefetchChunks = 6;
constexpr int kGatePrefetchItems = 3;

// Derivative of the activation at its saved input x.  GELU in its erf form,
// f'(x) = Phi(x) + x phi(x) with Phi(x) = (1 + erf(x / sqrt 2)) / 2 and
// phi(x) = exp(-x^2 / 2) / sqrt(2 pi); erf from Abramowitz and Stegun,
// Handbook of Mathematical Functions, formula 7.1.26: for z >= 0,
// erf(z) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2) with
// t = 1 / (1 + p z), absolute error at most 1.5e-7, and with z = |x| / sqrt 2
// its exp(-z^2) is phi's exponential, so one exponential serves both (the
// erff of CUDA's math library cost the epilogue twice the time of the ReLU
// gate).  SiLU, f'(x) = s (1 + x (1 - s)) with s = 1 / (1 + exp(-x)).  The
// hardware exponential (__expf) and the fast division are accurate to a few
// ulp of fp32: far below the 16-bit output's rounding.
template <int ACT>
__device__ __forceinline__ float act_grad(float x)
{
    if (ACT == 1) {
        const float e = __expf(-0.5f * x * x);  // exp(-z^2) = sqrt(2 pi) phi(x)
        const float t = __fdividef(1.0f, fmaf(0.3275911f * 0.70710678118654752f, fabsf(x), 1.0f));
        float poly = fmaf(t, 1.061405429f, -1.453152027f);
        poly = fmaf(t, poly, 1.421413741f);
        poly = fmaf(t, poly, -0.284496736f);
        poly = fmaf(t, poly, 0.254829592f);
        poly *= t;
        const float erf_abs = fmaf(-poly, e, 1.0f);  // erf(|x| / sqrt 2)
        const float Phi = 0.5f + copysignf(0.5f * erf_abs, x);
        return fmaf(x, 0.39894228040143268f * e, Phi);
    }
    const float sg = __fdividef(1.0f, 1.0f + __expf(-x));
    return sg * fmaf(x, 1.0f - sg, 1.0f);
}

// Backward of the activation whose saved input is x, on PER consecutive
// values.  ReLU (ACT 0): v = (x > 0) ? v : +0.0 (a select, so masked outputs
// are +0.0 whatever the accumulator holds), and xp receives v * x where the
// gate passes, +0.0 elsewhere (the terms of the per-channel sum of dX * x).
// GELU (ACT 1) and SiLU (ACT 2): v = v * f'(x).
template <int IN_T, int PER, int ACT>
__device__ __forceinline__ void gate_x(float *v, const uint32_t *w, float *xp)
{
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        const float x = gate_value<IN_T>(static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1))));
        if (ACT == 0) {
            const bool pass = x > 0.0f;
            v[e] = pass ? v[e] : 0.0f;
            xp[e] = pass ? v[e] * x : 0.0f;
        } else {
            v[e] *= act_grad<ACT>(x);
        }
    }
}

// ReLU-backward gate on PER consecutive values: v = (x > 0) ? v : +0.0 (the
// plain kernels' compact form of gate_x with act 0 and no products).
template <int IN_T, int PER>
__device__ __forceinline__ void gate_relu(float *v, const uint32_t *w)
{
#pragma unroll
    for (int e = 0; e < PER / 2; ++e) {
        if (!(gate_value<IN_T>(static_cast<uint16_t>(w[e] & 0xFFFFu)) > 0.0f)) v[2 * e] = 0.0f;
        if (!(gate_value<IN_T>(static_cast<uint16_t>(w[e] >> 16)) > 0.0f)) v[2 * e + 1] = 0.0f;
    }
}

// Column sums of a warp's 32 rows: each lane holds N values (one row), and
// afterwards lane l holds in a[0 .. N/32) the warp's totals of values
// (N/32)*l + j.  Five exchange steps with the lane at distance d = 16, 8, 4,
// 2, 1: a lane keeps the upper half of its current values when its lane bit
// d is set, the lower half otherwise, and adds the partner's copy of that
// half.  Each step's N/2, N/4, ... exchanges are independent of one another.
template <int N>
__device__ __forceinline__ void warp_transpose_sum(float (&a)[N], int lane)
{
    static_assert(N == 32 || N == 64, "a chunk holds 32 or 64 channels");
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int d = 16 >> step;
        const int h = N >> (step + 1);
        const bool upper = (lane & d) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = upper ? a[i] : a[i + h];
            const float keep = upper ? a[i + h] : a[i];
            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
        }
    }
}

template <int PER>
__device__ __forceinline__ void gate_mask(float *v, uint32_t bits)
{
#pragma unroll
    for (int e = 0; e < PER; ++e)
        if (!((bits >> e) & 1u)) v[e] = 0.0f;
}

// EPI, the epilogue variant: 0 plain (the ReLU gate or none), 1 with the
// per-channel sums, 2 GELU backward, 3 SiLU backward (these two with or
// without the sums).  Each is its own kernel, so that no variant's code
// enlarges another's unrolled per-element loop.
template <int OUT_T, bool MASK, int IN_T, bool HALO, bool PAIR, bool DUAL, int EPI>
__device__ __forceinline__ void run_epilogue(const CdgParams &p, const Ring &R, const CdgPhase *tab, Ctl ctl,
                                             uint32_t tmem_base, Sched S, volatile uint32_t *gate_used_sh)
{
    constexpr int OSZ = OUT_T == CDG_T_F32 ? 4 : 2;
    constexpr int CH = 128 / OSZ;  // channels per 128-byte staging row
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool elected = elect_one_sync();  // this warp's issuing lane for stores and arrivals
    const int quad = warp & 3;  // this warp may read TMEM lanes [32*quad, 32*quad + 32)
    const int row = quad * 32 + lane;
    const int ew = warp - CDG_EPI_WARP0;  // epilogue warp 0..3
    const int tiles_n = p.tiles_n, BN = p.BN, C = p.C;
    // box dims are 0 in the linear operand modes; keep the divisions defined
    const int bw = max(p.box_w, 1), bh = max(p.box_h, 1), bn = max(p.box_n, 1);
    const int d_mode = p.d_mode, m_step = p.m_step, rpt = max(p.rows_per_tile, 1);
    const uint32_t acc_stride = p.acc_stride;
    const bool mask_bits = p.mask_bits != 0;
    // staging buffers: p.gate_bufs (6 or 4) when the activation's chunks land
    // in them ahead of use (two outputs in flight, the rest gate tiles ahead),
    // else two
    const uint32_t nbuf = (MASK && !mask_bits) ? static_cast<uint32_t>(p.gate_bufs) : 2u;
    // tile row -> box position, and the staging row it fills (halo mode: row
    // a*halo_wb + b is output (a, b); padding rows b >= halo_wt are dropped)
    int jl, il, nl, srow;
    if (HALO) {
        const int a = row / p.halo_wb, b = row - (row / p.halo_wb) * p.halo_wb;
        jl = b;
        il = a;
        nl = (b < p.halo_wt && a < p.halo_bh) ? 0 : 1;
        srow = nl == 0 ? a * p.halo_wt + b : -1;
    } else {
        jl = row % bw;
        il = (row / bw) % bh;
        nl = row / (bw * bh);
        srow = row;
    }
    const uint32_t srow_off = static_cast<uint32_t>(max(srow, 0)) * 128u;
    const uint32_t sw = static_cast<uint32_t>(srow & 7);
    const uint32_t zero_buf = R.out0;  // staging buffer 0 doubles as the zero source
    bool zero_ready = false;

    // Per-channel sums (p.nsum > 0): this CTA adds each chunk's column sums
    // into its own accumulators in shared memory, [sum][C] fp32, and writes
    // them to its row of the workspace, [CTA][sum][C], once at the end.
    // Channel c is always handled by epilogue thread c % CH (N tiles are
    // multiples of CH channels, or a single tile from channel 0), which zeroes,
    // adds and writes it, so nothing needs atomics or a barrier, and the sums
    // keep one order from run to run.
    const int nsum = EPI != 0 ? p.nsum : 0;
    constexpr int ACT = EPI >= 2 ? EPI - 1 : 0;  // activation of the x gate (0 ReLU, 1 GELU, 2 SiLU)
    const int ethread = ew * 32 + lane;
    const uint32_t red_acc0 = R.red0 + CDG_SMEM_RED;
    if (nsum && ethread < CH)
        for (int c = ethread; c < C; c += CH)
            for (int k = 0; k < nsum; ++k) st_shared_f32(red_acc0 + 4u * static_cast<uint32_t>(k * C + c), 0.0f);

    // TMA stores are spread over the four warps' elected lanes (an issue holds its
    // thread for a few hundred cycles): chunk k is stored by epilogue warp k % 4.
    // accumulators filled so far by each MMA warp (dual issue: items alternate
    // between two MMA warps, each with two accumulators of its own)
    uint32_t acc_count[2] = {0u, 0u}, chunk_count = 0;
    uint32_t item_index = 0;
    // Gate inputs arrive by TMA ahead of use: chunk k's activation tile into
    // staging buffer k % 6 while chunk k - 4 is processed (its load is issued
    // once chunk k - 4's own tile has landed and store k - 6, the buffer's
    // previous user, has finished reading it; with four buffers, k % 4 and
    // k - 2); the mask tile of the i-th item
    // with taps into ring slot i % 4 three items ahead.  Load n is issued by
    // epilogue warp n % 4 (an issue holds its thread for a few hundred cycles,
    // so one warp issuing them all would pace the epilogue); every epilogue
    // thread walks the cursor in step.  (Four chunks of lookahead, six
    // buffers, measured slower on GB300: the operand ring loses a stage.)
    GateCursor gc{ItemWalk(tab, p, S.start, S.step), 0};
    const int gstep = mask_bits ? BN : CH;
    const uint32_t gring = mask_bits ? R.gate0 : R.out0;
    const uint32_t gslot = mask_bits ? static_cast<uint32_t>(CDG_GATE_SLOT) : 128u * 128u;
    const uint32_t grow = static_cast<uint32_t>(p.gate_row_bytes);
    uint32_t g_issued = 0, g_used = 0;  // gate loads issued and waited for (the same count in every thread)
    uint32_t gated_items = 0;
    // the prefetch cursor runs ahead of gc by the loads' lookahead plus
    // kGatePrefetch* loads; its issues rotate over the warps like the loads'
    GateCursor pf{ItemWalk(tab, p, S.start, S.step), 0};
    uint32_t pf_issued = 0;
    auto gate_prefetch = [&]() {
        if (!p.prefetch || !pf.valid()) return;
        const uint32_t n = pf_issued++;
        if (elected && static_cast<uint32_t>(ew) == (n & 3u)) gate_issue<true>(p, pf, S, 0u, 0u);
        pf.next(mask_bits ? BN : CH, BN);
    };
    // Gate tiles are loaded by this CTA and always land, so their waits do not
    // give up when another role aborts (only after the time limit): the four
    // warps then never disagree about a gate wait.  The accumulator wait can
    // legitimately fail (the MMA warp aborted); its outcome is agreed by all
    // 128 epilogue threads in a reducing barrier before anyone leaves, because
    // a thread that left while others went on to the next named barrier would
    // leave them waiting there for good.
    volatile uint32_t gate_no_abort = 0;
    const Ctl gate_ctl{&gate_no_abort, ctl.status, ctl.limit};
    // Gate load n: the packed mask's tile into ring slot n % 4 on barrier
    // n % 4; the activation's chunk into staging buffer n % 6 on barrier n % 8
    // (phase n / 8), so that no barrier is re-armed before its last load was
    // waited for.
    auto gate_ahead = [&]() {
        if (!gc.valid()) return;
        const uint32_t n = g_issued++;
        const uint32_t slot = mask_bits ? (n & 3u) : (n % nbuf);
        const uint32_t bar = mask_bits ? (n & 3u) : (n & 7u);
        if (elected && static_cast<uint32_t>(ew) == (n & 3u))
            gate_issue<false>(p, gc, S, gring + slot * gslot, R.gfull0 + 8u * bar);
        gc.next(gstep, BN);
        gate_prefetch();
    };
    // Per-tap and row plans gated by the activation: loader warp 3 issues the
    // activation tiles (run_gate_issuer), so no epilogue thread is held by a
    // TMA issue; the epilogue only signals, on R.gfree0, each staging buffer
    // that its store has finished reading.
    const bool xg_ext = MASK && !HALO && !DUAL && !mask_bits;
    if (MASK && !xg_ext) {
        const int ahead = mask_bits ? 3 : static_cast<int>(nbuf) - 2;
        // skip the prefetch cursor past the loads issued at once, then run it
        // kGatePrefetch* loads further
        for (int j = 0; j < ahead; ++j) pf.next(mask_bits ? BN : CH, BN);
        for (int j = 0; j < (mask_bits ? kGatePrefetchItems : kGatePrefetchChunks); ++j) gate_prefetch();
        for (int j = 0; j < ahead; ++j) gate_ahead();
    }
    bool ok = true;
    for (ItemWalk w(tab, p, S.start, S.step); w.valid(); w.next(), ++item_index) {
        const CdgPhase &ph = tab[w.phase];
        const int mt = S.m_tile(w.local, tiles_n, p.div_tiles_n);
        const int nt = w.local - (tiles_n == 1 ? w.local : fdiv(w.local, p.div_tiles_n)) * tiles_n;
        const int c_begin = nt * BN;
        const int c_end = min(C, c_begin + BN);
        const uint64_t mapD = reinterpret_cast<uint64_t>(&p.tmD[w.phase]);

        if (ph.tap_count == 0) {
            // No tap reaches this phase: dX = +0.0, stored box by box from a
            // zeroed staging buffer.
            if (!zero_ready) {
                if (elected) bulk_wait_group_read<0>();  // no store may still read the buffer
                named_bar_sync(1, 128);
#pragma unroll
                for (int q = 0; q < 8; ++q) st_shared_v4(zero_buf + static_cast<uint32_t>(row) * 128u + (q << 4), 0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
                named_bar_sync(1, 128);
                zero_ready = true;
            }
            int j0, i0, n0;
            box_origin(p, ph, w.phase, mt, ph.zbw, ph.zbh, 1, j0, i0, n0);
            const int nchunks = (c_end - c_begin + CH - 1) / CH;
            if (elected)
                for (int q = ew; q < nchunks; q += 4) {
                    tma_store_4d(mapD, zero_buf, c_begin + q * CH, j0, i0, n0);
                    bulk_commit_group();
                }
            continue;
        }

        if (zero_ready) {
            // back from zero-fill items (the planner orders them last, so this
            // is only a safeguard): every zero store must have read its source
            if (elected) bulk_wait_group_read<0>();
            named_bar_sync(1, 128);
            zero_ready = false;
        }
        // tile origin in the store map's coordinates
        int j0 = 0, i0 = 0, n0 = 0;
        if (d_mode == CDG_D_BOX4) box_origin(p, ph, w.phase, mt, bw, bh, bn, j0, i0, n0);
        // does this thread's tile row hold a dX pixel of the item?  (rows past
        // the sub-grid's edges, halo padding rows and the tail of the last
        // tile are computed but never stored; the sums must skip them too)
        bool row_ok = false;
        if (nsum) {
            if (d_mode == CDG_D_BOX4)
                row_ok = srow >= 0 && nl < bn && j0 + jl < ph.wph && i0 + il < ph.hph && n0 + nl < p.N;
            else if (d_mode == CDG_D_LINEAR)
                row_ok = mt * m_step + row < p.N * p.H * p.W;
            else
                row_ok = row < m_step && mt * rpt + row / ph.wph < p.N * ph.hph;
        }
        uint32_t mrow = 0;  // packed mask: this row's bytes in the item's mask tile
        if (MASK && mask_bits) {
            gate_ahead();  // into the slot the previous item's tile has left
            const uint32_t n = gated_items++;
            if (!wait_bar(R.gfull0 + 8u * (n & 3u), (n >> 2) & 1u, gate_ctl)) break;
            ++g_used;
            mrow = R.gate0 + (n & 3u) * static_cast<uint32_t>(CDG_GATE_SLOT) + static_cast<uint32_t>(max(srow, 0)) * grow;
        }

        const uint32_t issuer = DUAL ? (item_index & 1u) : 0u;
        const uint32_t n_acc = acc_count[issuer]++;
        // accumulator slot: two per MMA warp with dual issue, else p.acc_ring (2 or 4)
        const uint32_t acc = DUAL ? 2u * issuer + (n_acc & 1u) : (n_acc & (p.acc_ring - 1u));
        const uint32_t acc_parity = (n_acc >> (!DUAL && p.acc_ring == 4u ? 2 : 1)) & 1u;
        const bool acc_ok = wait_bar(R.acc_full0 + 8u * acc, acc_parity, ctl);
        if (named_bar_red_or(1, 128, !acc_ok)) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + acc * acc_stride + (static_cast<uint32_t>(quad * 32) << 16);
        for (int cc = 0; cc < BN; cc += CH) {
            const uint32_t k = chunk_count++;
            const uint32_t buf = R.out0 + (nbuf == 2u ? (k & 1u) : (k % nbuf)) * (128u * 128u);
            // the store of chunk k-2 (issued by warp (k-2) % 4) must be done
            // reading its buffer: with two buffers that is this chunk's, with
            // nbuf it is the one chunk k + nbuf - 2's gate goes into
            if (k >= 2 && elected && static_cast<uint32_t>(ew) == ((k - 2) & 3u)) {
                bulk_wait_group_read<0>();
                // staging buffer (k - 2) % nbuf is free: gate load k - 2 + nbuf may land in it
                if (xg_ext) mbar_arrive(R.gfree0 + 8u * ((k - 2u) & 7u));
            }
            named_bar_sync(1, 128);
            uint32_t gw[2] = {0u, 0u};  // packed mask: the chunk's bits 0-31 and 32-63
            uint32_t xf[OSZ == 4 ? 16 : 1];  // fp32 output: the chunk's 32 activation values
            if (MASK && mask_bits && srow >= 0) {
                if (OSZ == 2) {
                    ld_shared_v2(mrow + static_cast<uint32_t>(cc >> 3), gw);
                } else {
                    gw[0] = ld_shared_u32(mrow + static_cast<uint32_t>(cc >> 3));
                }
            } else if (MASK && !mask_bits) {
                if (!wait_bar(R.gfull0 + 8u * (k & 7u), (k >> 3) & 1u, gate_ctl)) {
                    ok = false;
                    break;
                }
                ++g_used;
                if (!xg_ext) gate_ahead();  // chunk k + nbuf - 2 into the buffer store k - 2 has finished reading
                if (OSZ == 4) {
                    // fp32 output: the activation tile holds 64-byte rows; read this
                    // row before any thread writes the wider output over the buffer
                    if (srow >= 0)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ld_shared_v4(buf + static_cast<uint32_t>(srow) * 64u + 16u * q,
                                         *reinterpret_cast<uint32_t(*)[4]>(&xf[(4 * q) % (OSZ == 4 ? 16 : 1)]));
                    named_bar_sync(1, 128);
                }
            }
            uint32_t r[CH];
            float xs[EPI != 0 ? CH : 1];  // the chunk's terms of the sum of dX * x (sums plans)
#pragma unroll
            for (int q = 0; q < CH / 16; ++q)
                tmem_ld_32x32b_x16(taddr + cc + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&r[16 * q]));
            tmem_ld_wait();
            if (cc + CH >= BN) {  // last read of this accumulator: hand it back to the MMA warp
                tc_fence_before();
                __syncwarp();
                if (elected) {
                    if (PAIR && S.rank != 0)  // the pair's MMA warp lives in the leader CTA
                        mbar_arrive_cluster(mapa_shared(R.acc_empty0 + 8u * acc, 0));
                    else
                        mbar_arrive(R.acc_empty0 + 8u * acc);
                }
            }
            // 16-bit output gated by the saved activation: this row's eight
            // activation pieces, all read before any output piece is written
            // over them (volatile shared-memory reads and writes interleaved
            // piece by piece would pay the read latency eight times a chunk)
            uint32_t xwa[(MASK && OSZ == 2) ? 8 : 1][4];
            if (MASK && OSZ == 2 && !mask_bits && srow >= 0) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    ld_shared_v4(buf + srow_off + ((static_cast<uint32_t>(q) ^ sw) << 4), xwa[q % ((MASK && OSZ == 2) ? 8 : 1)]);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {  // 16-byte pieces of this row
                constexpr int PER = 16 / OSZ;  // values per piece
                float v[PER], xp[PER];
#pragma unroll
                for (int e = 0; e < PER; ++e) {
                    v[e] = __uint_as_float(r[PER * q + e]);
                    xp[e] = 0.0f;
                }
                if (MASK && srow >= 0) {
                    if (mask_bits) {
                        gate_mask<PER>(v, gw[(PER * q) >> 5] >> ((PER * q) & 31));
                    } else if (OSZ == 2) {  // x piece q sat where output piece q goes
                        const uint32_t *xw = xwa[q % ((MASK && OSZ == 2) ? 8 : 1)];
                        if (EPI != 0)
                            gate_x<IN_T, PER, ACT>(v, xw, xp);
                        else
                            gate_relu<IN_T, PER>(v, xw);
                    } else {  // fp32 output: values 4q .. 4q+3 of the chunk
                        if (EPI != 0)
                            gate_x<IN_T, PER, ACT>(v, &xf[(2 * q) % (OSZ == 4 ? 16 : 1)], xp);
                        else
                            gate_relu<IN_T, PER>(v, &xf[(2 * q) % (OSZ == 4 ? 16 : 1)]);
                    }
                }
                if (nsum) {
                    // keep the chunk's gated values (and their products with x)
                    // for the column sums below; r[] is not read again
#pragma unroll
                    for (int e = 0; e < PER; ++e) {
                        r[PER * q + e] = __float_as_uint(row_ok ? v[e] : 0.0f);
                        if constexpr (EPI != 0) xs[PER * q + e] = row_ok ? xp[e] : 0.0f;
                    }
                }
                uint32_t wv[4];
                if (OUT_T == CDG_T_F32) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) wv[e] = __float_as_uint(v[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) wv[e] = pack2(v[2 * e], v[2 * e + 1], OUT_T);
                }
                if (srow >= 0)
                    st_shared_v4(buf + srow_off + ((static_cast<uint32_t>(q) ^ sw) << 4), wv[0], wv[1], wv[2], wv[3]);
            }
            if constexpr (EPI != 0) if (nsum) {
                // the chunk's column sums over this warp's 32 rows into the
                // warp's slot of the partials: lane l ends with channels
                // (CH/32)*l + j
                float t[CH];
#pragma unroll
                for (int i = 0; i < CH; ++i) t[i] = __uint_as_float(r[i]);
                warp_transpose_sum<CH>(t, lane);
#pragma unroll
                for (int j = 0; j < CH / 32; ++j)
                    st_shared_f32(R.red0 + static_cast<uint32_t>(ew * 64 + (CH / 32) * lane + j) * 4u, t[j]);
                if (nsum == 2) {
                    warp_transpose_sum<CH>(xs, lane);
#pragma unroll
                    for (int j = 0; j < CH / 32; ++j)
                        st_shared_f32(R.red0 + 4u * 64u * 4u + static_cast<uint32_t>(ew * 64 + (CH / 32) * lane + j) * 4u,
                                      xs[j]);
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (elected && static_cast<uint32_t>(ew) == (k & 3u)) {
                const int c = c_begin + cc;
                if (d_mode == CDG_D_BOX4)
                    tma_store_4d(mapD, buf, c, j0, i0, n0);
                else if (d_mode == CDG_D_LINEAR)
                    tma_store_2d(mapD, buf, c, mt * m_step);
                else
                    tma_store_3d(mapD, buf, c, 0, mt * rpt);
                bulk_commit_group();
            }
            if (nsum && ethread < CH) {
                // the chunk's column sums: the four warps' partials in warp
                // order, added to this CTA's row (the next chunk overwrites the
                // partials only after its first named barrier, which every
                // thread reaches after this read)
                const int c = c_begin + cc + ethread;
                if (c < c_end) {
                    const uint32_t col = static_cast<uint32_t>(ethread) * 4u;
                    for (int k2 = 0; k2 < nsum; ++k2) {
                        const uint32_t base = R.red0 + static_cast<uint32_t>(k2) * (4u * 64u * 4u) + col;
                        const float t = ((ld_shared_f32(base) + ld_shared_f32(base + 256u)) + ld_shared_f32(base + 512u)) +
                                        ld_shared_f32(base + 768u);
                        const uint32_t a = red_acc0 + 4u * static_cast<uint32_t>(k2 * C + c);
                        st_shared_f32(a, ld_shared_f32(a) + t);
                    }
                }
            }
        }
        if (!ok) break;
    }
    if (nsum && ethread < CH) {
        // this thread's channels, added by it alone, to the CTA's workspace row
        float *const row_out = p.red_ws + static_cast<size_t>(blockIdx.x) * nsum * C;
        for (int c = ethread; c < C; c += CH)
            for (int k = 0; k < nsum; ++k) row_out[k * C + c] = ld_shared_f32(red_acc0 + 4u * static_cast<uint32_t>(k * C + c));
    }
    if (xg_ext && ew == 0 && elected) *gate_used_sh = g_used;  // for the abort drain
    if (MASK && ew == 0 && elected && g_used != g_issued) {
        // aborted: let the gate loads still in flight land before the CTA exits
        volatile uint32_t no_abort = 0;
        const Ctl drain_ctl{&no_abort, ctl.status, ctl.limit};
        for (uint32_t n = g_used; n < g_issued; ++n) {
            if (mask_bits)
                wait_bar(R.gfull0 + 8u * (n & 3u), (n >> 2) & 1u, drain_ctl);
            else
                wait_bar(R.gfull0 + 8u * (n & 7u), (n >> 3) & 1u, drain_ctl);
        }
    }
    if (elected) bulk_wait_group_all();
}

// Gate issuer (per-tap and row plans gated by the saved activation): loader
// warp 3 walks the chunk sequence of the epilogue and loads chunk n's
// activation tile into staging buffer n % nbuf on gate barrier n % 8, once
// the epilogue has signalled (R.gfree0, barrier (n - nbuf) % 8) that store
// n - nbuf, the buffer's previous user, has finished reading it.  The count
// of issued loads goes to *issued_sh for the abort drain.
__device__ __forceinline__ void run_gate_issuer(const CdgParams &p, const Ring &R, const CdgPhase *tab, Ctl ctl,
                                                Sched S, int ch, volatile uint32_t *issued_sh)
{
    const bool leader = elect_one_sync();
    const uint32_t nbuf = static_cast<uint32_t>(p.gate_bufs);
    GateCursor gc{ItemWalk(tab, p, S.start, S.step), 0};
    uint32_t n = 0;
    for (; gc.valid(); ++n) {
        if (n >= nbuf) {
            const uint32_t f = n - nbuf;
            if (!wait_bar(R.gfree0 + 8u * (f & 7u), (f >> 3) & 1u, ctl)) break;
        }
        if (leader) gate_issue<false>(p, gc, S, R.out0 + (n % nbuf) * (128u * 128u), R.gfull0 + 8u * (n & 7u));
        __syncwarp();
        gc.next(ch, p.BN);
    }
    if (leader) *issued_sh = n;
}

// ------------------------------------------------------------------ kernel
// MODE: 0 per-tap operand boxes (or row boxes for 1x1 filters), one CTA per
//         tile, one MMA warp;
//       1 halo operand mode (weights resident when they fit, else streamed);
//       4 the halo operand mode with CTA pairs (2-SM MMAs over two halo tiles);
//       2 per-tap or row boxes, CTA pairs (cluster of 2) sharing 256-row tiles
//         through tcgen05.mma.cta_group::2: each CTA holds its own 128 rows of
//         A and half of the weight tile, which halves the B bytes every SM's
//         shared memory takes in and hands to the tensor core;
//       3 per-tap or row boxes, two MMA warps (dual issue) for N tiles of up to
//         128 channels;
//       5 the halo operand mode with resident weights and two MMA warps taking
//         alternate items from the one halo ring; 6 the same with CTA pairs.
template <int OUT_T, bool MASK, int IN_T, int MODE, int EPI>
__global__ void __launch_bounds__(CDG_THREADS, 1) dgrad_kernel(const __grid_constant__ CdgParams p)
{
    constexpr bool HALO = MODE == 1 || MODE == 4 || MODE == 5 || MODE == 6;
    constexpr bool PAIR = MODE == 2 || MODE == 4 || MODE == 6;
    // two MMA warps, each with two accumulators (and, without halo boxes, its own ring)
    constexpr bool DUAL = MODE == 3 || MODE == 5 || MODE == 6;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    // shared memory: operand ring(s) | 2 x 16 KB output staging | gate buffers | mbarriers, flags | phase and tap tables
    const int stages = HALO ? p.a_stages + p.b_stages : p.stages;  // mbarrier pairs
    Ring R;
    R.stages = stages;
    R.a0 = base;
    R.stage_bytes = p.a_stage_bytes;
    R.b0 = base + p.a_stages * R.stage_bytes;
    R.b_bytes = (PAIR ? p.BN / 2 : p.BN) * 128;  // halo mode: this CTA's rows of one weight tile
    R.out0 = HALO ? R.b0 + (p.b_res ? p.b_res_bytes : p.b_stages * p.halo_tg * R.b_bytes) : base + stages * R.stage_bytes;
    // gated by the activation: p.gate_bufs staging buffers; by the packed mask: two and the mask ring
    R.gate0 = R.out0 + CDG_SMEM_STAGING;
    const uint32_t bars =
        R.out0 + CDG_SMEM_STAGING +
        (MASK ? (p.mask_bits ? CDG_GATE_RING : static_cast<uint32_t>(p.gate_bufs - 2) * (CDG_SMEM_STAGING / 2)) : 0u);
    // mbarriers: full[nfull], empty[stages], acc_full[4], acc_empty[4], drain[2], gate[8].
    // With two MMA warps over the one halo ring, each warp waits on full
    // barriers of its own (a_stages more after the stage ones): a stage
    // alternates between the warps when the ring has an odd number of stages,
    // and a shared barrier could then be waited on two phases ahead, whose
    // parity test would pass on the older phase.
    const int nfull = (HALO && DUAL) ? stages + p.a_stages : stages;
    // per-tap and row kernels with a gate: eight more barriers, on which the
    // epilogue frees staging buffers for the gate issuer (activation gate);
    // such plans have at most eight stages, so all fits the 384-byte area
    constexpr int kGfree = (MASK && !HALO && !DUAL) ? 8 : 0;
    R.full0 = bars;
    R.empty0 = bars + 8u * nfull;
    R.acc_full0 = bars + 8u * (nfull + stages);
    R.acc_empty0 = R.acc_full0 + 32u;
    R.drain = R.acc_full0 + 64u;
    R.gfull0 = R.acc_full0 + 80u;
    R.gfree0 = R.gfull0 + 64u;
    R.red0 = bars + CDG_SMEM_TAIL;  // only plans with per-channel sums reserve it
    uint8_t *const tail = smem_raw + (bars - raw);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tail + 8 * (nfull + stages + 18 + kGfree));
    volatile uint32_t *abort_flag = tmem_slot + 1;
    volatile uint32_t *slot_parity = tmem_slot + 2;  // [nfull]: the planner keeps all of it within the tables' offset
    volatile uint32_t *gate_counts = slot_parity + nfull;  // gate loads issued, consumed (activation gate issuer)
    CdgPhase *tab = reinterpret_cast<CdgPhase *>(tail + CDG_SMEM_TABLES);
    CdgTap *taps = reinterpret_cast<CdgTap *>(tab + CDG_MAX_PHASES);
    static_assert(8 * (2 * CDG_MAX_STAGES_TOTAL + 18) + 8 + 4 * CDG_MAX_STAGES_TOTAL + 8 <= CDG_SMEM_TABLES,
                  "mbarrier area overflows");
    // per-tap and row plans have at most eight stages (kMaxStages in the planner)
    static_assert(8 * (2 * 8 + 18 + 8) + 8 + 4 * 8 + 8 <= CDG_SMEM_TABLES, "gate-issuer barriers overflow");
    static_assert(CDG_SMEM_TABLES + CDG_MAX_PHASES * sizeof(CdgPhase) + CDG_MAX_TAPS * sizeof(CdgTap) <=
                      CDG_SMEM_TAIL,
                  "phase and tap tables overflow the shared-memory tail");
    const int warp = threadIdx.x / 32;
    Sched S;
    if (PAIR) {
        uint32_t cid, ncl;
        asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(cid));
        asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(ncl));
        S.start = static_cast<int>(cid);
        S.step = static_cast<int>(ncl);
        S.pair = 1;
        S.rank = static_cast<int>(cluster_ctarank());
    } else {
        S.start = blockIdx.x;
        S.step = gridDim.x;
        S.pair = 0;
        S.rank = 0;
    }
    // The next kernel in the stream may be scheduled now: with one CTA per SM
    // its CTAs take SMs only as this grid's CTAs exit.
    grid_dep_launch_dependents();
    for (int i = threadIdx.x; i < p.nphases; i += blockDim.x) tab[i] = p.phase[i];
    for (int i = threadIdx.x; i < p.ntaps; i += blockDim.x) taps[i] = p.tap[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < nfull; ++s) mbar_init(R.full0 + 8u * s, 1);
        for (int s = 0; s < stages; ++s) mbar_init(R.empty0 + 8u * s, 1);
        for (int a = 0; a < 4; ++a) {
            mbar_init(R.acc_full0 + 8u * a, 1);
            // one arrival per epilogue warp (in a pair, the leader's counts both CTAs' warps)
            mbar_init(R.acc_empty0 + 8u * a, PAIR && S.rank == 0 ? 8 : 4);
        }
        mbar_init(R.drain, 1);
        mbar_init(R.drain + 8u, 1);
        for (int g = 0; g < 8; ++g) mbar_init(R.gfull0 + 8u * g, 1);
        for (int g = 0; g < kGfree; ++g) mbar_init(R.gfree0 + 8u * g, 1);
        *abort_flag = 0u;
        for (int s = 0; s < nfull; ++s) slot_parity[s] = 0u;
        gate_counts[0] = 0u;
        gate_counts[1] = 0u;
        fence_mbar_init();
    }
    // Everything above touches only shared memory and kernel parameters.  Global
    // memory (dY, W, x, dX, the status word) and tensor memory are used only
    // after the kernels this launch depends on have completed; allocating TMEM
    // after the wait means a waiting CTA never holds TMEM another kernel needs.
    grid_dep_wait();
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), p.tmem_cols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // both CTAs' barriers exist before any copy or arrive crosses over
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Ctl ctl{abort_flag, p.status, p.wait_limit_ns};

    // dual issue: MMA warp j (warp 1 + 2j) and loader warp j (warp 2j) serve the
    // items at odd/even positions of this CTA's walk, through ring j (half of
    // the stages) and accumulator slots 2j, 2j + 1
    auto ring_of = [&](int j) {
        Ring Rj = R;
        Rj.stages = stages / 2;
        Rj.a0 = R.a0 + static_cast<uint32_t>(j * Rj.stages) * R.stage_bytes;
        Rj.full0 = R.full0 + 8u * static_cast<uint32_t>(j * Rj.stages);
        Rj.empty0 = R.empty0 + 8u * static_cast<uint32_t>(j * Rj.stages);
        Rj.acc_full0 = R.acc_full0 + 16u * j;
        Rj.acc_empty0 = R.acc_empty0 + 16u * j;
        Rj.drain = R.drain + 8u * j;
        return Rj;
    };
    auto sched_of = [&](int j) {
        Sched Sj = S;
        Sj.start = S.start + j * S.step;
        Sj.step = 2 * S.step;
        return Sj;
    };
    if (DUAL && HALO) {
        // warps 1 and 3 issue the MMAs of alternate items from the one halo
        // ring (accumulator slots 2j, 2j + 1); warp 0 loads the halo boxes and
        // warp 2 the resident weights
        if (warp == 1 || warp == 3) {
            const int j = warp >> 1;
            Ring Rj = R;
            Rj.acc_full0 = R.acc_full0 + 16u * j;
            Rj.acc_empty0 = R.acc_empty0 + 16u * j;
            Rj.drain = R.drain + 8u * j;
            if (!PAIR || S.rank == 0) {
                run_mma_halo<PAIR, true>(p, Rj, tab, taps, ctl, tmem_base + 2u * j * p.acc_stride, elect_one_sync(),
                                         sched_of(j), j);
            } else {
                volatile uint32_t no_abort = 0;
                wait_bar(Rj.drain, 0, Ctl{&no_abort, p.status, p.wait_limit_ns});
            }
        } else if (warp >= CDG_EPI_WARP0) {
            run_epilogue<OUT_T, MASK, IN_T, HALO, PAIR, true, EPI>(p, R, tab, ctl, tmem_base, S, gate_counts + 1);
        } else {
            run_loader_halo<PAIR, true>(p, R, tab, taps, ctl, warp == 0 ? 0 : 1, elect_one_sync(), slot_parity, S);
        }
    } else if (DUAL) {
        if (warp == 1 || warp == 3) {
            const int j = warp >> 1;
            run_mma<false>(p, ring_of(j), tab, ctl, tmem_base + 2u * j * p.acc_stride, elect_one_sync(), sched_of(j));
        } else if (warp >= CDG_EPI_WARP0) {
            run_epilogue<OUT_T, MASK, IN_T, false, false, true, EPI>(p, R, tab, ctl, tmem_base, S, gate_counts + 1);
        } else {
            const int j = warp >> 1;  // warps 0 and 2
            run_loader<false>(p, ring_of(j), tab, taps, ctl, 0, 1, elect_one_sync(),
                              slot_parity + j * (stages / 2), sched_of(j));
        }
    } else if (warp == 1) {
        if (HALO && (!PAIR || S.rank == 0)) {
            run_mma_halo<PAIR>(p, R, tab, taps, ctl, tmem_base, elect_one_sync(), S);
        } else if (!HALO && (!PAIR || S.rank == 0)) {
            run_mma<PAIR>(p, R, tab, ctl, tmem_base, elect_one_sync(), S);
        } else {
            // the leader issues the pair's MMAs; wait until they are all done
            // with this CTA's tensor memory
            volatile uint32_t no_abort = 0;
            wait_bar(R.drain, 0, Ctl{&no_abort, p.status, p.wait_limit_ns});
        }
    } else if (warp >= CDG_EPI_WARP0) {
        run_epilogue<OUT_T, MASK, IN_T, HALO, PAIR, false, EPI>(p, R, tab, ctl, tmem_base, S, gate_counts + 1);
    } else if (HALO) {
        run_loader_halo<PAIR>(p, R, tab, taps, ctl, warp == 0 ? 0 : warp - 1, elect_one_sync(), slot_parity, S);
    } else if (kGfree && !p.mask_bits) {
        // gated by the saved activation: warps 0 and 2 load the operands,
        // warp 3 the activation tiles
        if (warp == 3)
            run_gate_issuer(p, R, tab, ctl, S, OUT_T == CDG_T_F32 ? 32 : 64, gate_counts);
        else
            run_loader<PAIR>(p, R, tab, taps, ctl, warp == 0 ? 0 : 1, 2, elect_one_sync(), slot_parity, S);
    } else {
        run_loader<PAIR>(p, R, tab, taps, ctl, warp == 0 ? 0 : warp - 1, CDG_LOADERS, elect_one_sync(), slot_parity,
                         S);
    }

    __syncthreads();
    if (kGfree && !p.mask_bits && *abort_flag && threadIdx.x == 0) {
        // activation tiles the issuer loaded and the epilogue never waited for
        volatile uint32_t no_abort = 0;
        const Ctl drain_ctl{&no_abort, p.status, p.wait_limit_ns};
        for (uint32_t n = gate_counts[1]; n < gate_counts[0]; ++n)
            wait_bar(R.gfull0 + 8u * (n & 7u), (n >> 3) & 1u, drain_ctl);
    }
    if (*abort_flag && threadIdx.x == 0) {
        if (!PAIR || S.rank == 0) {
            drain_loads(R, nfull, p.status, p.wait_limit_ns, slot_parity);
        } else {
            // this CTA's copies complete on the leader's barriers; give any
            // still in flight time to land before the pair may exit
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < 200000ull) {
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();  // neither CTA leaves while the other may still signal it
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, p.tmem_cols);
        else
            tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// ------------------------------------------------------------------ back-to-back fusion
// Persistent fusion of two dgrads (the persistent kernel fusion of the Bolt
// reading notes, with threadblock residence): GEMM 1 is a stride-1 dgrad in
// the halo operand mode with resident weights (a 3x3 layer, C2 = 64 output
// channels: the whole channel count in one N tile), GEMM 2 the 1x1 dgrad of
// GEMM 1's gated output g, g = act_bwd(dgrad(dY2, W2), x2), into dX1 with
// C1 <= 256 channels.  A tile of g never leaves the CTA: the epilogue reads
// GEMM 1's accumulator, applies the gate, rounds to the input type and writes
// the tile into tensor memory, where it is GEMM 2's A operand (tcgen05.mma
// reads A from TMEM); W1 stays resident in shared memory.  Only dX1 (and, if
// asked, g) goes to HBM.
//
// Tensor memory (512 columns): GEMM-1 accumulators at columns 0 and 64, the
// two g tiles (64 bf16 = 32 columns each) at 128 and 160, the GEMM-2
// accumulator at 256.  Items alternate between the two GEMM-1 accumulators
// and the two g tiles.  The MMA warp issues GEMM 1 of item i before GEMM 2 of
// item i - 1, so the epilogue's gate of item i - 1 overlaps GEMM 1 of item i.
constexpr uint32_t kFusedAcc1 = 64;   // columns of one GEMM-1 accumulator
constexpr uint32_t kFusedA2 = 128;    // first g tile
constexpr uint32_t kFusedAcc2 = 256;  // GEMM-2 accumulator

struct FusedBars {
    uint32_t acc1_full0, acc1_empty0;  // [2] each
    uint32_t a2_full0, a2_empty0;      // [2] each: g tile written (4 epilogue warps) / consumed (MMA commit)
    uint32_t acc2_full, acc2_empty;
    uint32_t w1_full, gate_full, drain;
};

__device__ __forceinline__ void run_mma_fused(const CdgParams &p, const Ring &R, const FusedBars &B,
                                              const CdgPhase *tab, const CdgTap *taps, Ctl ctl, uint32_t tmem_base,
                                              bool leader, Sched S, uint32_t w1_smem)
{
    const int KB = p.KB, as = p.a_stages;
    const uint32_t idesc = p.idesc, idesc2 = p.idesc2;
    const uint64_t adesc0 = sdesc_k128_sw128(R.a0);
    const uint64_t bdesc0 = sdesc_k128_sw128(R.b0);
    const uint64_t w1desc = sdesc_k128_sw128(w1_smem);
    const uint32_t astep = R.stage_bytes >> 4;  // descriptor units per halo stage
    const uint32_t bunit = R.b_bytes >> 4;      // descriptor units per weight tile
    int a_stage = 0;
    uint32_t a_par = 0, n = 0;
    // both weight sets are resident: GEMM-1 weights (loader 1), GEMM-2 weights (warp 3)
    bool ok = wait_bar(R.full0 + 8u * as, 0, ctl) && wait_bar(B.w1_full, 0, ctl);
    // GEMM 2 of item j: dX1 tile (acc2) = g tile j (TMEM) x W1^T, K = 64 channels of g
    auto gemm2 = [&](uint32_t j) -> bool {
        if (!wait_bar(B.a2_full0 + 8u * (j & 1u), (j >> 1) & 1u, ctl)) return false;
        if (!wait_bar(B.acc2_empty, (j & 1u) ^ 1u, ctl)) return false;
        tc_fence_after();
        if (leader) {
            const uint32_t a = tmem_base + kFusedA2 + 32u * (j & 1u);
#pragma unroll
            for (int k = 0; k < CDG_BK / 16; ++k)  // 16 values = 8 TMEM columns of A, 32 B of B
                umma_f16_ts(tmem_base + kFusedAcc2, a + 8u * k, w1desc + 2u * k, idesc2, k != 0);
            umma_commit(B.acc2_full);
            umma_commit(B.a2_empty0 + 8u * (j & 1u));
        }
        __syncwarp();
        return true;
    };
    for (ItemWalk w(tab, p, S.start, S.step); ok && w.valid(); w.next()) {
        const CdgPhase &ph = tab[w.phase];
        const int ntap = ph.tap_count;
        const uint32_t acc = n & 1u;
        if (!wait_bar(B.acc1_empty0 + 8u * acc, ((n >> 1) & 1u) ^ 1u, ctl)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kFusedAcc1;
        for (int kb = 0; ok && kb < KB; ++kb) {
            if (!wait_bar(R.full0 + 8u * a_stage, a_par, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t abase = adesc0 + static_cast<uint64_t>(a_stage * astep);
            const CdgTap *ptap = taps + ph.tap_begin;
            const int tbase = ph.tap_begin * KB + kb;
            int hoff = ptap[0].hoff;
            for (int tt = 0; tt < ntap; ++tt) {
                if (leader) {
                    const uint64_t adesc = abase + 8u * static_cast<uint32_t>(hoff);
                    const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(static_cast<uint32_t>(tbase + tt * KB) * bunit);
#pragma unroll
                    for (int k = 0; k < CDG_BK / 16; ++k)
                        umma_f16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kb | tt | k) != 0);
                }
                __syncwarp();
                if (tt + 1 < ntap) hoff = ptap[tt + 1].hoff;
            }
            if (leader) umma_commit(R.empty0 + 8u * a_stage);
            __syncwarp();
            if (++a_stage == as) {
                a_stage = 0;
                a_par ^= 1u;
            }
        }
        if (!ok) break;
        if (leader) umma_commit(B.acc1_full0 + 8u * acc);
        __syncwarp();
        if (n >= 1 && !gemm2(n - 1)) {
            ok = false;
            break;
        }
        ++n;
    }
    if (ok && n >= 1) gemm2(n - 1);
    if (leader) umma_commit(B.drain);
    __syncwarp();
    volatile uint32_t no_abort = 0;
    wait_bar(B.drain, 0, Ctl{&no_abort, ctl.status, ctl.limit});
}

template <int IN_T, int ACT>
__device__ __forceinline__ void run_epilogue_fused(const CdgParams &p, const Ring &R, const FusedBars &B,
                                                   const CdgPhase *tab, Ctl ctl, uint32_t tmem_base, Sched S,
                                                   uint32_t x2_smem)
{
    constexpr bool GATE = ACT >= 0;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool elected = elect_one_sync();
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int ew = warp - CDG_EPI_WARP0;
    // tile row a*halo_wb + b is output (a, b) of the halo tile; the store box
    // (and the gate tile) holds the valid rows compacted, a*halo_wt + b
    const int ha = row / p.halo_wb, hb = row - (row / p.halo_wb) * p.halo_wb;
    const int srow = (hb < p.halo_wt && ha < p.halo_bh) ? ha * p.halo_wt + hb : -1;
    const uint32_t srow_off = static_cast<uint32_t>(max(srow, 0)) * 128u;
    const uint32_t sw = static_cast<uint32_t>(srow & 7);
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint64_t mapX1 = reinterpret_cast<uint64_t>(&p.tmX1);
    const uint64_t mapG = reinterpret_cast<uint64_t>(&p.tmD[0]);
    const uint64_t mapGate = reinterpret_cast<uint64_t>(&p.tmG[0]);
    volatile uint32_t gate_no_abort = 0;
    const Ctl gate_ctl{&gate_no_abort, ctl.status, ctl.limit};
    // the gate tile of the next item is loaded into the one gate buffer as
    // soon as every thread has read the current one (issued by warp 0)
    ItemWalk nx(tab, p, S.start, S.step);
    // and the tile two items beyond that is prefetched into L2 meanwhile
    ItemWalk px(tab, p, S.start, S.step);
    px.next();
    px.next();
    uint32_t g_issued = 0, g_used = 0;
    auto gate_issue = [&]() {
        if (!GATE || !nx.valid()) return;
        ++g_issued;
        if (ew == 0 && elected) {
            int j0, i0, n0;
            box_origin(p, tab[nx.phase], nx.phase, S.m_tile(nx.local, 1, p.div_tiles_n), p.halo_wt, p.halo_bh, 1, j0, i0, n0);
            mbar_arrive_expect_tx(B.gate_full, p.gate_tx);
            tma_load_4d(x2_smem, mapGate, B.gate_full, 0, j0, i0, n0);
            if (p.prefetch && px.valid()) {
                box_origin(p, tab[px.phase], px.phase, S.m_tile(px.local, 1, p.div_tiles_n), p.halo_wt, p.halo_bh, 1, j0, i0, n0);
                tma_prefetch_4d(mapGate, 0, j0, i0, n0);
            }
        }
        nx.next();
        px.next();
    };
    gate_issue();
    uint32_t chunk = 0;
    // one 16 KB output chunk through staging buffer chunk % 2 (the same
    // hand-over as the plain epilogue); each thread writes its row
    auto store_chunk = [&](uint64_t map, int c, int j0, int i0, int n0, const uint32_t (&pk)[32]) {
        const uint32_t k = chunk++;
        const uint32_t buf = R.out0 + (k & 1u) * (128u * 128u);
        if (k >= 2 && elected && static_cast<uint32_t>(ew) == ((k - 2) & 3u)) bulk_wait_group_read<0>();
        named_bar_sync(1, 128);
        if (srow >= 0)
#pragma unroll
            for (int q = 0; q < 8; ++q)
                st_shared_v4(buf + srow_off + ((static_cast<uint32_t>(q) ^ sw) << 4), pk[4 * q], pk[4 * q + 1],
                             pk[4 * q + 2], pk[4 * q + 3]);
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (elected && static_cast<uint32_t>(ew) == (k & 3u)) {
            tma_store_4d(map, buf, c, j0, i0, n0);
            bulk_commit_group();
        }
    };
    // dX1 of item j: GEMM 2's accumulator in 64-channel chunks; false if the
    // launch is giving up
    auto stage_b = [&](uint32_t j, int j0, int i0, int n0) -> bool {
        const bool okw = wait_bar(B.acc2_full, j & 1u, ctl);
        if (named_bar_red_or(1, 128, !okw)) return false;
        tc_fence_after();
        for (int cc = 0; cc < p.BN2; cc += 64) {
            uint32_t o[64], pk[32];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                tmem_ld_32x32b_x16(tmem_base + kFusedAcc2 + lane_base + static_cast<uint32_t>(cc) + 16u * q,
                                   *reinterpret_cast<uint32_t(*)[16]>(&o[16 * q]));
            tmem_ld_wait();
            if (cc + 64 >= p.BN2) {  // last read of the accumulator: GEMM 2 of the next item may start
                tc_fence_before();
                __syncwarp();
                if (elected) mbar_arrive(B.acc2_empty);
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) pk[e] = pack2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1]), IN_T);
            store_chunk(mapX1, cc, j0, i0, n0, pk);
        }
        return true;
    };
    // Order: g of item n, then dX1 of item n - 1.  GEMM 2 of item n - 1 runs on
    // the tensor pipe while this thread makes g of item n, so dX1's chunks
    // never wait for it, and the stores (the bound) keep flowing.
    uint32_t n = 0;
    int pj0 = 0, pi0 = 0, pn0 = 0;  // the previous item's tile origin
    bool ok = true;
    for (ItemWalk w(tab, p, S.start, S.step); w.valid(); w.next(), ++n) {
        const CdgPhase &ph = tab[w.phase];
        int j0, i0, n0;
        box_origin(p, ph, w.phase, S.m_tile(w.local, 1, p.div_tiles_n), p.halo_wt, p.halo_bh, 1, j0, i0, n0);
        // ---- g = gate(GEMM 1): accumulator -> registers -> tensor memory (GEMM 2's A)
        bool okw = wait_bar(B.acc1_full0 + 8u * (n & 1u), (n >> 1) & 1u, ctl);
        okw = okw && wait_bar(B.a2_empty0 + 8u * (n & 1u), ((n >> 1) & 1u) ^ 1u, ctl);
        if (named_bar_red_or(1, 128, !okw)) {
            ok = false;
            break;
        }
        tc_fence_after();
        uint32_t xr[32];
        if (GATE) {
            wait_bar(B.gate_full, g_used & 1u, gate_ctl);
            ++g_used;
            if (srow >= 0) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    ld_shared_v4(x2_smem + srow_off + ((static_cast<uint32_t>(q) ^ sw) << 4),
                                 *reinterpret_cast<uint32_t(*)[4]>(&xr[4 * q]));
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) xr[e] = 0u;
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 128);  // every row read: the gate buffer takes the next tile
            gate_issue();
        }
        uint32_t r[64];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            tmem_ld_32x32b_x16(tmem_base + (n & 1u) * kFusedAcc1 + lane_base + 16u * q,
                               *reinterpret_cast<uint32_t(*)[16]>(&r[16 * q]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (elected) mbar_arrive(B.acc1_empty0 + 8u * (n & 1u));
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            float v[2] = {__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])};
            if (GATE) {
                float xp[2];
                gate_x<IN_T, 2, (ACT < 0 ? 0 : ACT)>(v, &xr[e], xp);
            }
            pk[e] = pack2(v[0], v[1], IN_T);
        }
        tmem_st_32x32b_x32(tmem_base + kFusedA2 + 32u * (n & 1u) + lane_base, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (elected) mbar_arrive(B.a2_full0 + 8u * (n & 1u));
        if (p.write_g) store_chunk(mapG, 0, j0, i0, n0, pk);
        // ---- dX1 of the previous item
        if (n >= 1 && !stage_b(n - 1, pj0, pi0, pn0)) {
            ok = false;
            break;
        }
        pj0 = j0;
        pi0 = i0;
        pn0 = n0;
    }
    if (ok && n >= 1) stage_b(n - 1, pj0, pi0, pn0);
    if (GATE && ew == 0 && elected && g_used != g_issued) {
        // left early: let the gate tile still in flight land before the CTA exits
        volatile uint32_t no_abort = 0;
        const Ctl drain_ctl{&no_abort, ctl.status, ctl.limit};
        for (uint32_t k = g_used; k < g_issued; ++k) wait_bar(B.gate_full, k & 1u, drain_ctl);
    }
    if (elected) bulk_wait_group_all();
}

// Shared memory: halo ring | W2 (resident) | W1 (resident) | gate tile | 2 x
// 16 KB staging | mbarriers, flags | phase and tap tables.
template <int IN_T, int ACT>
__global__ void __launch_bounds__(CDG_THREADS, 1) fused_kernel(const __grid_constant__ CdgParams p)
{
    constexpr bool GATE = ACT >= 0;  // ACT: -1 no activation, 0 ReLU, 1 GELU, 2 SiLU
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int stages = p.a_stages + 1;  // halo stages and the resident-weights barrier
    Ring R;
    R.stages = stages;
    R.a0 = base;
    R.stage_bytes = p.a_stage_bytes;
    R.b0 = base + p.a_stages * R.stage_bytes;
    R.b_bytes = p.BN * 128;
    const uint32_t w1_smem = R.b0 + p.b_res_bytes;
    const uint32_t x2_smem = w1_smem + p.w1_bytes;
    R.out0 = x2_smem + (GATE ? CDG_FUSED_X2_BYTES : 0u);
    const uint32_t bars = R.out0 + CDG_SMEM_STAGING;
    R.full0 = bars;
    R.empty0 = bars + 8u * stages;
    FusedBars B;
    B.acc1_full0 = bars + 16u * stages;
    B.acc1_empty0 = B.acc1_full0 + 16u;
    B.a2_full0 = B.acc1_full0 + 32u;
    B.a2_empty0 = B.acc1_full0 + 48u;
    B.acc2_full = B.acc1_full0 + 64u;
    B.acc2_empty = B.acc1_full0 + 72u;
    B.w1_full = B.acc1_full0 + 80u;
    B.gate_full = B.acc1_full0 + 88u;
    B.drain = B.acc1_full0 + 96u;
    uint8_t *const tail = smem_raw + (bars - raw);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tail + 16 * stages + 104);
    volatile uint32_t *abort_flag = tmem_slot + 1;
    volatile uint32_t *slot_parity = tmem_slot + 2;  // [stages]
    CdgPhase *tab = reinterpret_cast<CdgPhase *>(tail + CDG_SMEM_TABLES);
    CdgTap *taps = reinterpret_cast<CdgTap *>(tab + CDG_MAX_PHASES);
    static_assert(16 * 4 + 104 + 8 + 4 * 4 <= CDG_SMEM_TABLES, "fused mbarrier area overflows");
    const int warp = threadIdx.x / 32;
    Sched S;
    S.start = blockIdx.x;
    S.step = gridDim.x;
    S.pair = 0;
    S.rank = 0;
    grid_dep_launch_dependents();
    for (int i = threadIdx.x; i < p.nphases; i += blockDim.x) tab[i] = p.phase[i];
    for (int i = threadIdx.x; i < p.ntaps; i += blockDim.x) taps[i] = p.tap[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(R.full0 + 8u * s, 1);
            mbar_init(R.empty0 + 8u * s, 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(B.acc1_full0 + 8u * j, 1);
            mbar_init(B.acc1_empty0 + 8u * j, 4);  // one arrival per epilogue warp
            mbar_init(B.a2_full0 + 8u * j, 4);
            mbar_init(B.a2_empty0 + 8u * j, 1);
        }
        mbar_init(B.acc2_full, 1);
        mbar_init(B.acc2_empty, 4);
        mbar_init(B.w1_full, 1);
        mbar_init(B.gate_full, 1);
        mbar_init(B.drain, 1);
        *abort_flag = 0u;
        for (int s = 0; s < stages; ++s) slot_parity[s] = 0u;
        fence_mbar_init();
    }
    grid_dep_wait();
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Ctl ctl{abort_flag, p.status, p.wait_limit_ns};
    if (warp == 1) {
        run_mma_fused(p, R, B, tab, taps, ctl, tmem_base, elect_one_sync(), S, w1_smem);
    } else if (warp >= CDG_EPI_WARP0) {
        run_epilogue_fused<IN_T, ACT>(p, R, B, tab, ctl, tmem_base, S, x2_smem);
    } else if (warp == 3) {
        // the 1x1 weights, once per CTA: BN2 rows of 64 channels (128 B) of g
        if (elect_one_sync()) {
            const uint64_t mapW1 = reinterpret_cast<uint64_t>(&p.tmW1);
            mbar_arrive_expect_tx(B.w1_full, p.w1_bytes);
            tma_load_3d(w1_smem, mapW1, B.w1_full, 0, 0, 0);
        }
        __syncwarp();
    } else {
        run_loader_halo<false>(p, R, tab, taps, ctl, warp == 0 ? 0 : 1, elect_one_sync(), slot_parity, S);
    }
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        drain_loads(R, stages, p.status, p.wait_limit_ns, slot_parity);
        // the 1x1 weights' copy, if the launch gave up before the MMA warp saw it land
        volatile uint32_t no_abort = 0;
        wait_bar(B.w1_full, 0, Ctl{&no_abort, p.status, p.wait_limit_ns});
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace cdg
