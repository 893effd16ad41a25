// Launch parameters shared by the host planner (cdg_api.cu) and the sm_103a
// dgrad kernel (dgrad_sm103.cu).  Passed by value as one __grid_constant__
// kernel argument, so the TMA descriptors live in parameter space.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define CDG_MAX_PHASES 16   // stride <= 4
#define CDG_MAX_TAPS 128    // R * S <= 128
#define CDG_BM 128          // dX pixels per tile = TMEM lanes = UMMA M
#define CDG_BK 64           // dY channels per pipeline stage (128 B of fp16/bf16)
#define CDG_MAX_DYN_SMEM 232448  // sm_103 opt-in dynamic shared memory per CTA (227 KB)
// Warp roles: warps 0, 2, 3 load operands with TMA (pipeline stages taken
// round-robin: a TMA issue holds its thread for a few hundred cycles, so one
// issuing thread cannot keep the tensor core fed); warp 1 issues tcgen05.mma;
// warps 4-7 run the epilogue (warp w reads TMEM lanes 32*(w%4)..+31).
#define CDG_THREADS 256
#define CDG_LOADERS 3
#define CDG_EPI_WARP0 4
#define CDG_WAIT_LIMIT_NS 4000000000ull  // a pipeline wait gives up after 4 s (default)
// Shared memory after the operand ring: two 16 KB output staging buffers
// (128 rows x 128 B, the box a TMA store writes; four (or six) when the
// ReLU-backward gate reads the saved activation, whose chunks land in them
// ahead of use; two plus a 16 KB ring of mask tiles when it reads the packed
// mask), then mbarriers and flags (384 B), then the phase and tap tables
// copied out of the parameter block.
#define CDG_SMEM_STAGING (2 * 128 * 128)
#define CDG_GATE_SLOT 4096   // one item's packed-mask tile: 128 rows x up to 32 bytes
#define CDG_GATE_RING (4 * CDG_GATE_SLOT)
#define CDG_SMEM_TAIL 2048
#define CDG_SMEM_TABLES 384
// Per-channel output sums (plans with CDG_EPI_SUM): after the tail, the four
// epilogue warps' partial sums of one chunk, [sums][4 warps][64 channels]
// fp32, then the CTA's accumulators, [sums][C] fp32 (in 128-byte units).
#define CDG_SMEM_RED (2 * 4 * 64 * 4)
#define CDG_MAX_STAGES_TOTAL 10  // all ring stages together (their mbarriers live in the 384-byte area)

// Division by a divisor fixed for the launch as a multiply-high, an add and a
// shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994, the round-up method with N = 32): with
// shr = ceil(log2 d) and mul = floor(2^32 (2^shr - d) / d) + 1,
// n / d = (mulhi(n, mul) + n) >> shr for every 0 <= n < 2^31 and d >= 1.
// The kernels' item bookkeeping divides by tile counts; as plain integer
// divisions they cost the epilogue several hundred cycles per work item.
struct CdgDiv {
    uint32_t mul, shr;
};

static inline CdgDiv cdg_make_div(uint32_t d)
{
    uint32_t shr = 0;
    while ((1ull << shr) < d) ++shr;
    const unsigned long long m = ((1ull << 32) * ((1ull << shr) - d)) / d + 1ull;
    return CdgDiv{static_cast<uint32_t>(m), shr};
}

// One phase sub-convolution of a (possibly strided) dgrad.  The dX pixels with
// h = stride*i + ph, w = stride*j + pw (0 <= i < hph, 0 <= j < wph) form the
// phase sub-grid; the filter taps whose contributions land on it are
// tap[tap_begin .. tap_begin + tap_count), each reading dY at (i + dr, j + ds).
struct CdgPhase {
    int hph, wph;
    int tiles_w, tiles_h;  // box tiles along j and i (4-D halo boxes, or the zero-fill box)
    int tiles_m;           // M tiles of this phase
    int items;             // tiles_m * (N tiles): work items of this phase
    int16_t ph, pw;
    int16_t tap_begin, tap_count;
    int16_t zbw, zbh;        // phases without taps: box (zbw x zbh x 1 positions) of one zero-fill store
    int16_t dr_min, ds_min;  // halo operand mode: smallest tap offsets (origin of the halo box)
};

struct CdgTap {
    int16_t dr, ds;  // dY row/column offset relative to the phase sub-grid position
    int16_t t;       // tap index r*S + s into the packed weights
    int16_t hoff;    // halo operand mode: row of the halo box where this tap's operand starts
};

// How a tile's rows map onto dX and how the epilogue's TMA store addresses them.
enum {
    CDG_D_BOX4 = 0,   // per-phase 4-D map {C, wph, hph, N} over the phase sub-grid; tile = box
    CDG_D_LINEAR = 1, // 2-D map {C, N*H*W}; tile = 128 consecutive pixels (stride 1, 1x1, pad 0)
    CDG_D_ROWS = 2    // 3-D map {C, wph, N*hph} over phase (0,0); tile = whole sub-grid rows
};

struct CdgParams {  // CUtensorMap members carry their own (128-byte) alignment
    CUtensorMap tmA;  // dY: 4-D {K, Q, P, N} halo boxes, or 2-D {K, N*P*Q} rows
    CUtensorMap tmB;  // packed weights: 3-D {K, C, R*S}
    CUtensorMap tmD[CDG_MAX_PHASES];  // dX stores, one map per phase (index = phase slot)
    CUtensorMap tmG[CDG_MAX_PHASES];  // gate loads (saved activation or packed mask) in the stores' geometry
    // back-to-back fusion (cdg_dgrad_fused): this stride-1 dgrad (GEMM 1) feeds,
    // gated, a 1x1 dgrad (GEMM 2) whose A operand never leaves the CTA
    CUtensorMap tmW1;     // packed 1x1 weights [1][C1][C2]: 3-D {C2, C1, 1}, box {64, BN2, 1}
    CUtensorMap tmX1;     // dX1 stores: 4-D {C1, W, H, N}, the halo tile's store box, 64 channels
    void *dX;
    const void *mask;
    int *status;
    int N, H, W, C, K, P, Q, stride;
    int BN, KB, stages, tiles_n, nphases, ntaps, total_items;
    int a_flat, box_w, box_h, box_n;
    int d_mode;           // CDG_D_*
    int halo;             // 1: one dY halo box per (tile, K block) serves every tap (see dgrad_sm103.cu)
    int pair;             // 1: CTA pairs (clusters of 2) share 256-row tiles through 2-SM MMAs
    int pdl;              // 1: launch with programmatic stream serialization (host side only)
    int prefetch;         // 1: operand and gate tiles are prefetched into L2 ahead of their loads
                          // (opt-in, CDG_PREFETCH=1: measured slower on GB300)
    int mask_bits;        // 1: the gate reads the packed bit mask (rows of 16-byte units per pixel), not x
    int act;              // activation whose backward the gate applies with x: 0 ReLU (select),
                          // 1 GELU (erf form), 2 SiLU (out = dX * f'(x))
    int gate_row_bytes;   // bytes of one tile row of a gate load (activation chunk, or mask tile)
    int gate_bufs;        // gated by the activation: staging buffers (4: its chunks land two chunks
                          // ahead; 6 with CDG_GATE_BUFS=6: four ahead, measured slower)
    uint32_t gate_tx;     // bytes one gate load delivers (the store box's rows x gate_row_bytes)
    int dual;             // 1: two MMA warps, each with half of the stages and two accumulators
    int interleave;       // >= 2: the first `interleave` phases' items are interleaved (il_items each)
    int il_items;
    int il_round;         // items per scheduling round (CTAs, or CTA pairs), a multiple of interleave
    int halo_wb;          // halo box width = row pitch of the halo tile rows (tile width + tap span)
    int halo_wt, halo_bh; // output tile: halo_wt columns x halo_bh rows of one image
    int halo_hb;          // halo box height (halo_bh + tap span)
    int a_stages, b_stages;   // halo mode: separate rings for halo boxes and weight tiles
    int b_res;            // halo mode: every weight tile resident in shared memory, loaded once
    int halo_tg;          // halo mode, streamed weights: taps per weight stage (>= 1)
    uint32_t b_res_bytes; // bytes of the resident weights (taps x K blocks x BN rows x 128 B)
    uint32_t a_stage_bytes;   // halo mode: bytes of one halo stage (>= the box, room for every tap's 128 rows)
    uint32_t tx_a, tx_b;      // halo mode: bytes one halo stage / one weight stage receives
    int m_step;           // linear operand modes: dY rows per M tile (128, or whole sub-grid rows)
    int rows_per_tile;    // CDG_D_ROWS: sub-grid rows per tile
    uint32_t idesc;       // tcgen05 instruction descriptor (kind::f16, M=128, N=BN)
    uint32_t tx_bytes;    // bytes one pipeline stage receives (A box + B box)
    uint32_t tmem_cols;   // allocated TMEM columns (two accumulators)
    uint32_t acc_stride;  // column offset of the second accumulator
    uint32_t acc_ring;    // accumulators an MMA warp cycles through (2; 4 for halo plans that ask)
    float *red_ws;        // per-channel sums: this launch's [grid][nsum][C] fp32 partials (one row per CTA)
    int nsum;             // per-channel output sums the epilogue accumulates: 0, 1 (sum of dX) or
                          // 2 (also the sum of dX * x where the gate passes)
    int write_g;          // fused: also store the gated intermediate g (through tmD[0])
    int C1, BN2;          // fused: dX1 channels; GEMM-2 N tile (C1 rounded up to 16)
    uint32_t idesc2;      // fused: tcgen05 instruction descriptor of GEMM 2 (M = 128, N = BN2)
    uint32_t w1_bytes;    // fused: bytes of the resident 1x1 weights (BN2 rows x 128 B)
    unsigned long long wait_limit_ns;  // a pipeline wait gives up (status CDG_ERR_TIMEOUT) after this long
    int withhold_stage;   // test only: >= 0 makes every per-tap/row loader skip the load (and its
                          // transaction count) of its stage with this sequence number, so the MMA
                          // warp's wait for it runs out; -1 in normal use
    CdgDiv div_tiles_w[CDG_MAX_PHASES], div_tiles_h[CDG_MAX_PHASES];  // per phase: its box tiles along j and i
    CdgDiv div_tiles_n;   // N tiles
    CdgDiv div_il;        // interleaved phases (1 when none)
    CdgDiv div_il_round;  // items per scheduling round (il_round; 1 when unset)
    CdgPhase phase[CDG_MAX_PHASES];
    CdgTap tap[CDG_MAX_TAPS];
};

// Element types of dX and of the gate input, as kernel template arguments.
enum { CDG_T_F16 = 0, CDG_T_BF16 = 1, CDG_T_F32 = 2 };

// Launchers implemented in dgrad_sm103.cu.
cudaError_t cdg_launch_pack_mask(const void *x, void *bits, long long pixels, int C, int in_type,
                                 cudaStream_t stream);
cudaError_t cdg_launch_dgrad(const CdgParams &p, int out_type, int in_type, bool mask,
                             int grid, size_t smem, cudaStream_t stream);
cudaError_t cdg_prepare_dgrad(int out_type, int in_type, bool mask, size_t smem);
cudaError_t cdg_launch_prepack(const void *W, void *Wp, int K, int T, int C, cudaStream_t stream);
cudaError_t cdg_launch_channel_sums(const float *ws, int rows, int nsum, int C, float *out, cudaStream_t stream);
// Shared memory of the fused kernel beyond the halo ring, W2 and W1: the gate
// tile (16 KB, gated plans only), two 16 KB staging buffers, the tail.
#define CDG_FUSED_X2_BYTES (128 * 128)
int cdg_max_active_pairs(int out_type, int in_type, bool mask, size_t smem);
// One epilogue variant of the dgrad kernels (EPI: 0 plain, 1 per-channel
// sums, 2 GELU backward, 3 SiLU backward), each instantiated in a
// translation unit of its own.
template <int EPI>
cudaError_t cdg_dgrad_prepare_variant(int out_type, int in_type, bool mask);
template <int EPI>
cudaError_t cdg_dgrad_launch_variant(const CdgParams &p, int out_type, int in_type, bool mask, int grid, size_t smem,
                                     cudaStream_t stream);
template <int EPI>
int cdg_dgrad_max_pairs_variant(int out_type, int in_type, bool mask, size_t smem);
cudaError_t cdg_prepare_fused(int in_type, int act);
cudaError_t cdg_launch_fused(const CdgParams &p, int in_type, int act, int grid, size_t smem, cudaStream_t stream);
