// Launch parameters shared by the host planner (cdg_api.cu) and the sm_103a
// wgrad kernel (wgrad_sm103.cu).  Passed by value as one __grid_constant__
// kernel argument, so the TMA descriptors live in parameter space.
#pragma once

#include "cdg_params.h"

// Weight gradient of the cross-correlation Conv2d as a GEMM per filter tap t:
//   dW[k, t, c] = sum over positions (n, p, q) of dY[n,p,q,k] * x[n, h, w, c],
//   h = p*stride - pad + r*dil, w = q*stride - pad + s*dil (zero outside).
// M = 128 dY channels k, N = BN input channels c, the reduction runs over
// blocks of 64 positions (a qb x pb x nb box of (q, p, n)).  Both operands
// arrive position-major (channels contiguous), i.e. MN-major for the MMA.
// The reduction is split over `splits` ranges of blocks; every split writes
// its fp32 partial dW to a workspace, reduced in a fixed order afterwards.
struct CwgParams {
    CUtensorMap tmA;                   // dY: 4-D {K, Q, P, N}, boxes {64, qb, pb, nb}
    CUtensorMap tmB[CDG_MAX_PHASES];   // x per phase (h mod stride, w mod stride): 4-D
                                       // {C, wph, hph, N} over the phase sub-grid, boxes {64, qb, pb, nb}
    CUtensorMap tmW;                   // workspace: 4-D {C, T, K, splits} fp32, boxes {32, 1, 128, 1}
    CUtensorMap tmWx;                  // the same workspace, boxes {64, 1, 32, 1} (x-major tiles, below)
    int *status;
    int N, H, W, C, K, P, Q, stride;
    int T;                // filter taps R*S
    int BN;               // channels of x per tile and tap (multiple of 64, <= 256)
    int G;                // taps per work item: their B tiles side by side along N (G*BN <= 256)
    int ngroups;          // ceil(T / G)
    int tiles_m, tiles_n; // ceil(K/128), ceil(C/BN)
    int splits;           // reduction splits
    int qb, pb, nb;       // position box (qb*pb*nb = 64)
    int bq, bp;           // boxes along q and p (blocks are numbered q fastest, then p, then n)
    int nblk;             // position blocks in all
    int stages;
    int total_items;      // splits * ngroups * tiles_m * tiles_n
    uint32_t idesc;       // tcgen05 instruction descriptor (kind::f16, M=128, N=G*BN, both operands MN-major)
    uint32_t stage_bytes; // A (2 slices x 8 KB) + B (G*BN/64 slices x 8 KB)
    uint32_t tmem_cols;   // two accumulators
    uint32_t acc_stride;
    // x-major tiles (K <= 64, where a 128-row tile of dY channels would leave
    // half of its rows idle): M = two units of (tap t, 64-channel slice cs of
    // x), unit u = t * cslices + cs, units 2m and 2m + 1 in M tile m; N = the
    // dY channels (64, zero-filled past K); the accumulator holds dW^T rows
    // (t, c), stored transposed through shared memory
    int xm;
    int cslices, units;   // x-major: 64-channel slices of x, and T * cslices
    int16_t tap_phase[CDG_MAX_TAPS];  // phase index (ph*stride + pw) of tap t
    int16_t tap_di[CDG_MAX_TAPS];     // row offset of tap t in its phase sub-grid: h = stride*(p + di) + ph
    int16_t tap_dj[CDG_MAX_TAPS];     // column offset: w = stride*(q + dj) + pw
};

// Launchers implemented in wgrad_sm103.cu.
cudaError_t cwg_prepare(size_t smem);
cudaError_t cwg_launch(const CwgParams &p, int grid, size_t smem, cudaStream_t stream);
cudaError_t cwg_launch_reduce(const float *ws, void *dW, long long count, int splits, int out_type,
                              cudaStream_t stream);
