// Implicit-GEMM Conv2d dgrad for sm_103a (GB300).
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
// CTA layout (192 threads, one CTA per SM, persistent over work items):
//   warp 0     TMA producer: per (tap, 64-channel block) one dY box and one
//              weight box into a shared-memory ring, mbarrier full/empty.
//   warp 1     owns TMEM; one thread issues tcgen05.mma (M=128, N=BN, K=16)
//              into one of two fp32 accumulators and commits stages back.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator, optional ReLU-backward
//              gate, conversion, 16-byte stores into NHWC dX.
// Every wait is bounded: past CDG_WAIT_LIMIT_NS the kernel records
// CDG_ERR_TIMEOUT in the status word and all roles leave their loops.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "cdg_params.h"
#include "ptx.cuh"

namespace cdg {

constexpr int kTimeoutStatus = 6;  // CDG_ERR_TIMEOUT

struct SmemLayout {
    uint32_t base;        // 1024-aligned shared address of stage 0
    uint32_t stage_bytes;
    uint32_t bars;        // first mbarrier
    int stages;
    __device__ uint32_t a(int s) const { return base + s * stage_bytes; }
    __device__ uint32_t b(int s) const { return base + s * stage_bytes + CDG_BM * 128; }
    __device__ uint32_t full(int s) const { return bars + 8u * s; }
    __device__ uint32_t empty(int s) const { return bars + 8u * (stages + s); }
    __device__ uint32_t acc_full(int a) const { return bars + 8u * (2 * stages + a); }
    __device__ uint32_t acc_empty(int a) const { return bars + 8u * (2 * stages + 2 + a); }
    __device__ uint32_t drain() const { return bars + 8u * (2 * stages + 4); }
};

struct Ctl {
    volatile uint32_t *abort;
    int *status;
};

// Wait for phase `parity` of barrier `bar` to complete; false if this CTA is
// aborting (another role gave up, or this wait ran past the limit).
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Ctl &ctl)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0) {
            if (*ctl.abort) return false;
            if (global_timer_ns() - t0 > CDG_WAIT_LIMIT_NS) {
                *ctl.abort = 1u;
                atomicCAS(ctl.status, 0, kTimeoutStatus);
                return false;
            }
        }
    }
}

struct Item {
    int phase, mt, nt;
};

__device__ __forceinline__ Item decode_item(const CdgParams &p, int g)
{
    int ph = 0;
    while (ph + 1 < p.nphases && g >= p.phase[ph + 1].item_begin) ++ph;
    const int local = g - p.phase[ph].item_begin;
    return {ph, local / p.tiles_n, local % p.tiles_n};
}

// Origin (j0, i0, n0) of 4-D box tile mt of a phase.
__device__ __forceinline__ void box_origin(const CdgParams &p, const CdgPhase &ph, int mt, int &j0, int &i0,
                                           int &n0)
{
    const int tj = mt % ph.tiles_w;
    const int rest = mt / ph.tiles_w;
    const int ti = rest % ph.tiles_h;
    const int tn = rest / ph.tiles_h;
    j0 = tj * p.box_w;
    i0 = ti * p.box_h;
    n0 = tn * p.box_n;
}

// ------------------------------------------------------------------ producer
__device__ void run_producer(const CdgParams &p, const SmemLayout &L, const Ctl &ctl)
{
    int stage = 0;
    uint32_t parity = 0;
    uint32_t used_mask = 0, last_parity = 0;  // for the final drain
    bool ok = true;
    for (int g = blockIdx.x; ok && g < p.total_items; g += gridDim.x) {
        const Item it = decode_item(p, g);
        const CdgPhase &ph = p.phase[it.phase];
        if (ph.tap_count == 0) continue;
        int j0 = 0, i0 = 0, n0 = 0;
        if (!p.a_flat) box_origin(p, ph, it.mt, j0, i0, n0);
        const int c0 = it.nt * p.BN;
        for (int tt = 0; ok && tt < ph.tap_count; ++tt) {
            const CdgTap tap = p.tap[ph.tap_begin + tt];
            for (int kb = 0; kb < p.KB; ++kb) {
                if (!wait_bounded(L.empty(stage), parity ^ 1u, ctl)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(L.full(stage), p.tx_bytes);
                if (p.a_flat)
                    tma_load_2d(L.a(stage), &p.tmA, L.full(stage), kb * CDG_BK, it.mt * CDG_BM);
                else
                    tma_load_4d(L.a(stage), &p.tmA, L.full(stage), kb * CDG_BK, j0 + tap.ds, i0 + tap.dr, n0);
                tma_load_3d(L.b(stage), &p.tmB, L.full(stage), kb * CDG_BK, c0, tap.t);
                used_mask |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (parity << stage);
                if (++stage == p.stages) {
                    stage = 0;
                    parity ^= 1u;
                }
            }
        }
    }
    // Every copy this thread started must land before the CTA may exit.  On
    // the normal path they all have (the MMA warp waited for each) and this
    // returns at once; after an abort it waits, bounded, for copies in flight.
    volatile uint32_t no_abort = 0;
    const Ctl drain_ctl{&no_abort, ctl.status};
    for (int s = 0; s < p.stages; ++s)
        if (used_mask & (1u << s)) wait_bounded(L.full(s), (last_parity >> s) & 1u, drain_ctl);
}

// ------------------------------------------------------------------ MMA issuer
__device__ void run_mma(const CdgParams &p, const SmemLayout &L, const Ctl &ctl, uint32_t tmem_base)
{
    int stage = 0;
    uint32_t parity = 0;
    uint32_t acc_count = 0;
    bool ok = true;
    for (int g = blockIdx.x; ok && g < p.total_items; g += gridDim.x) {
        const Item it = decode_item(p, g);
        const CdgPhase &ph = p.phase[it.phase];
        if (ph.tap_count == 0) continue;
        const uint32_t acc = acc_count & 1u;
        const uint32_t acc_parity = (acc_count >> 1) & 1u;
        if (!wait_bounded(L.acc_empty(acc), acc_parity ^ 1u, ctl)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * p.acc_stride;
        const int nk = ph.tap_count * p.KB;
        for (int kk = 0; kk < nk; ++kk) {
            if (!wait_bounded(L.full(stage), parity, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t adesc = sdesc_k128_sw128(L.a(stage));
            const uint64_t bdesc = sdesc_k128_sw128(L.b(stage));
#pragma unroll
            for (int k = 0; k < CDG_BK / 16; ++k)  // 16 elements = 32 bytes = 2 descriptor units
                umma_f16(d_tmem, adesc + 2u * k, bdesc + 2u * k, p.idesc, (kk | k) != 0);
            umma_commit(L.empty(stage));
            if (++stage == p.stages) {
                stage = 0;
                parity ^= 1u;
            }
        }
        if (!ok) break;
        umma_commit(L.acc_full(acc));
        ++acc_count;
    }
    // All MMAs issued by this thread complete before TMEM is released.
    umma_commit(L.drain());
    volatile uint32_t no_abort = 0;
    Ctl drain_ctl{&no_abort, ctl.status};
    wait_bounded(L.drain(), 0, drain_ctl);
}

// ------------------------------------------------------------------ epilogue
template <int IN_T>
__device__ __forceinline__ float gate_value(uint16_t bits)
{
    if (IN_T == CDG_T_BF16) return __uint_as_float(static_cast<uint32_t>(bits) << 16);
    return __half2float(__ushort_as_half(bits));
}

// Store n (8 or 16) consecutive channel values of one pixel.
template <int OUT_T>
__device__ __forceinline__ void store_chunk(void *dst, const float *v, int n)
{
    if (OUT_T == CDG_T_F32) {
        float4 *d = reinterpret_cast<float4 *>(dst);
        for (int i = 0; i < n / 4; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        for (int i = 0; i < n / 8; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float a = v[8 * i + 2 * j], b = v[8 * i + 2 * j + 1];
                if (OUT_T == CDG_T_BF16) {
                    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
                    w[j] = *reinterpret_cast<uint32_t *>(&h);
                } else {
                    __half2 h = __floats2half2_rn(a, b);
                    w[j] = *reinterpret_cast<uint32_t *>(&h);
                }
            }
            d[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

template <int OUT_T, bool MASK, int IN_T>
__device__ void run_epilogue(const CdgParams &p, const SmemLayout &L, const Ctl &ctl, uint32_t tmem_base)
{
    constexpr int OSZ = OUT_T == CDG_T_F32 ? 4 : 2;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int quad = warp & 3;  // this warp may read TMEM lanes [32*quad, 32*quad + 32)
    const int row = quad * 32 + lane;
    uint32_t acc_count = 0;
    for (int g = blockIdx.x; g < p.total_items; g += gridDim.x) {
        const Item it = decode_item(p, g);
        const CdgPhase &ph = p.phase[it.phase];
        // dX pixel of this tile row
        int n, i, j;
        bool valid;
        if (ph.linear) {
            const long long m = static_cast<long long>(it.mt) * CDG_BM + row;
            const long long plane = static_cast<long long>(ph.hph) * ph.wph;
            valid = m < plane * p.N;
            n = static_cast<int>(m / plane);
            const int rem = static_cast<int>(m - static_cast<long long>(n) * plane);
            i = rem / ph.wph;
            j = rem - i * ph.wph;
        } else {
            int j0, i0, n0;
            box_origin(p, ph, it.mt, j0, i0, n0);
            const int jl = row % p.box_w;
            const int il = (row / p.box_w) % p.box_h;
            const int nl = row / (p.box_w * p.box_h);
            n = n0 + nl;
            i = i0 + il;
            j = j0 + jl;
            valid = nl < p.box_n && n < p.N && i < ph.hph && j < ph.wph;
        }
        const long long pix =
            valid ? (static_cast<long long>(n) * p.H + (p.stride * i + ph.ph)) * p.W + (p.stride * j + ph.pw) : 0;
        char *out_row = static_cast<char *>(p.dX) + pix * p.C * OSZ;
        const uint16_t *x_row = MASK ? static_cast<const uint16_t *>(p.mask) + pix * p.C : nullptr;
        const int c_begin = it.nt * p.BN;
        const int c_end = min(p.C, c_begin + p.BN);

        if (ph.tap_count == 0) {  // no tap reaches this phase: dX = +0.0
            if (valid) {
                uint4 *d = reinterpret_cast<uint4 *>(out_row + static_cast<long long>(c_begin) * OSZ);
                const int n16 = (c_end - c_begin) * OSZ / 16;
                for (int q = 0; q < n16; ++q) d[q] = make_uint4(0, 0, 0, 0);
            }
            continue;
        }

        const uint32_t acc = acc_count & 1u;
        const uint32_t acc_parity = (acc_count >> 1) & 1u;
        if (!wait_bounded(L.acc_full(acc), acc_parity, ctl)) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + acc * p.acc_stride + (static_cast<uint32_t>(quad * 32) << 16);
        for (int cc = 0; cc < p.BN; cc += 16) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(taddr + cc, r);
            tmem_ld_wait();
            const int c = c_begin + cc;
            if (valid && c < c_end) {
                const int nc = min(16, c_end - c);  // 16 or 8 (C is a multiple of 8)
                float v[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] = __uint_as_float(r[q]);
                if (MASK) {
                    uint16_t xb[16];
                    const uint4 *xs = reinterpret_cast<const uint4 *>(x_row + c);
                    for (int q = 0; q < nc / 8; ++q) {
                        const uint4 u = __ldg(xs + q);
                        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            xb[8 * q + 2 * e] = static_cast<uint16_t>(w4[e] & 0xFFFFu);
                            xb[8 * q + 2 * e + 1] = static_cast<uint16_t>(w4[e] >> 16);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (q < nc && !(gate_value<IN_T>(xb[q]) > 0.0f)) v[q] = 0.0f;
                }
                store_chunk<OUT_T>(out_row + static_cast<long long>(c) * OSZ, v, nc);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(L.acc_empty(acc));
        ++acc_count;
    }
}

// ------------------------------------------------------------------ kernel
template <int OUT_T, bool MASK, int IN_T>
__global__ void __launch_bounds__(CDG_THREADS, 1) dgrad_kernel(const __grid_constant__ CdgParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    SmemLayout L;
    L.base = (raw + 1023u) & ~1023u;
    L.stage_bytes = CDG_BM * 128 + p.BN * 128;
    L.stages = p.stages;
    L.bars = L.base + p.stages * L.stage_bytes;
    uint8_t *bars_generic = smem_raw + (L.bars - raw);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars_generic + 8 * (2 * p.stages + 5));
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(L.full(s), 1);
            mbar_init(L.empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(L.acc_full(a), 1);
            mbar_init(L.acc_empty(a), 4);  // one arrival per epilogue warp
        }
        mbar_init(L.drain(), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Ctl ctl{abort_flag, p.status};

    if (warp == 0) {
        if (lane == 0) run_producer(p, L, ctl);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) run_mma(p, L, ctl, tmem_base);
        __syncwarp();
    } else {
        run_epilogue<OUT_T, MASK, IN_T>(p, L, ctl, tmem_base);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// ------------------------------------------------------------------ prepack
// Wp[t][c][k] = W[k][t][c] for t = r*S + s: per tap, the C x K matrix with K
// contiguous that the kernel's B operand expects.  32x32 tiles through shared
// memory so both the read (along c) and the write (along k) are coalesced.
__global__ void prepack_kernel(const uint16_t *__restrict__ W, uint16_t *__restrict__ Wp, int K, int T, int C)
{
    __shared__ uint16_t tile[32][33];
    const int t = blockIdx.z;
    const int c0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
    for (int y = threadIdx.y; y < 32; y += blockDim.y) {
        const int k = k0 + y, c = c0 + threadIdx.x;
        if (k < K && c < C) tile[y][threadIdx.x] = W[(static_cast<size_t>(k) * T + t) * C + c];
    }
    __syncthreads();
    for (int y = threadIdx.y; y < 32; y += blockDim.y) {
        const int c = c0 + y, k = k0 + threadIdx.x;
        if (c < C && k < K) Wp[(static_cast<size_t>(t) * C + c) * K + k] = tile[threadIdx.x][y];
    }
}

}  // namespace cdg

// ------------------------------------------------------------------ launchers
namespace {

typedef void (*DgradFn)(CdgParams);

template <int OUT_T, bool MASK, int IN_T>
DgradFn pick() { return cdg::dgrad_kernel<OUT_T, MASK, IN_T>; }

DgradFn select_kernel(int out_type, int in_type, bool mask)
{
    if (in_type == CDG_T_F16) {
        if (out_type == CDG_T_F32) return mask ? pick<CDG_T_F32, true, CDG_T_F16>() : pick<CDG_T_F32, false, CDG_T_F16>();
        return mask ? pick<CDG_T_F16, true, CDG_T_F16>() : pick<CDG_T_F16, false, CDG_T_F16>();
    }
    if (out_type == CDG_T_F32) return mask ? pick<CDG_T_F32, true, CDG_T_BF16>() : pick<CDG_T_F32, false, CDG_T_BF16>();
    return mask ? pick<CDG_T_BF16, true, CDG_T_BF16>() : pick<CDG_T_BF16, false, CDG_T_BF16>();
}

}  // namespace

// The dynamic shared-memory opt-in is a property of the kernel function, shared
// by every plan that uses it: always raise it to the largest size any plan
// may request, never to one plan's own size (a smaller later plan would
// otherwise lower the limit under an earlier one).
cudaError_t cdg_prepare_dgrad(int out_type, int in_type, bool mask, size_t smem)
{
    if (smem > static_cast<size_t>(CDG_MAX_DYN_SMEM)) return cudaErrorInvalidValue;
    DgradFn fn = select_kernel(out_type, in_type, mask);
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                CDG_MAX_DYN_SMEM);
}

cudaError_t cdg_launch_dgrad(const CdgParams &p, int out_type, int in_type, bool mask, int grid, size_t smem,
                             cudaStream_t stream)
{
    DgradFn fn = select_kernel(out_type, in_type, mask);
    fn<<<grid, CDG_THREADS, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t cdg_launch_prepack(const void *W, void *Wp, int K, int T, int C, cudaStream_t stream)
{
    dim3 grid((C + 31) / 32, (K + 31) / 32, T), block(32, 8);
    cdg::prepack_kernel<<<grid, block, 0, stream>>>(static_cast<const uint16_t *>(W), static_cast<uint16_t *>(Wp),
                                                    K, T, C);
    return cudaGetLastError();
}
