// Conv2d weight gradient (wgrad) for sm_103a: the follow-up to dgrad that the
// apache/tvm PR #10110 page ("[CUTLASS] Conv2d dgrad") names, "wgrad +
// parallel split-k" (merge comment).  The page gives no kernel; this one
// restates the definition as one GEMM per filter tap t = (r, s):
//
//   dW[k, r, s, c] = sum over positions (n, p, q) of
//                    dY[n, p, q, k] * x[n, p*stride - pad + r*dil, q*stride - pad + s*dil, c]
//
// M = 128 dY channels, N = BN input channels, K (reduction) = the positions,
// in blocks of 64 (a qb x pb x nb box of (q, p, n)).  Both operands are NHWC,
// so a block arrives position-major: 64 rows of 128 bytes per 64-channel
// slice, which is the MN-major operand layout of the tensor core with the
// 128-byte swizzle (atoms of 64 channels x 8 positions; slices 8 KB apart).
// x is read through per-phase strided maps at the tap's offset, so padding
// and image edges come from TMA's zero fill, as in dgrad.
//
// Parallel split-K: the position blocks are divided into `splits` ranges and
// every (split, tap, M tile, N tile) is a work item of a persistent grid.  Each
// item's fp32 partial goes to its own slice of a workspace; a second kernel
// adds the slices in split order (deterministic) and converts to dW's type.
//
// Narrow layers (C <= 128) put G taps side by side along N: the dY block is
// the same for every tap, so one MMA of N = G*BN serves G taps' dW tiles.
//
// Roles per CTA (256 threads, one CTA per SM): warps 0, 2, 3 load the stages
// round-robin (2 + G*BN/64 TMA copies each); warp 1 issues the MMAs; warps
// 4-7 read the accumulator and store fp32 rows of 32 channels with TMA.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "cwg_params.h"
#include "ptx.cuh"
#include "wait.cuh"

namespace cdg {
namespace {

constexpr int kSlice = 64 * 128;  // one 64-channel slice of a 64-position block: 8 KB

// Shared-memory matrix descriptor of an MN-major operand in 128-byte-swizzled
// atoms (64 channels x 8 positions, 1 KB): leading-dimension offset = bytes
// between 64-channel slices along M/N, stride-dimension offset = bytes between
// groups of 8 positions along the reduction.  Bits as for the K-major form:
// [0,14) start >> 4; [16,30) LBO >> 4; [32,46) SBO >> 4; [46,48) version 1;
// [61,64) 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t lbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

struct WgRing {
    int stages;
    uint32_t s0;        // stage 0 (A slices, then B slices)
    uint32_t out0;      // two 16 KB staging buffers
    uint32_t full0, empty0, acc_full0, acc_empty0, drain;
};

// Work item g = ((split * ngroups + group) * tiles_m + mt) * tiles_n + nt;
// group covers taps t0 .. t0 + G - 1 (those below T).
struct WgItem {
    int split, t0, mt, nt;
    __device__ __forceinline__ WgItem(const CwgParams &p, int g)
    {
        nt = g % p.tiles_n;
        int r = g / p.tiles_n;
        mt = r % p.tiles_m;
        r /= p.tiles_m;
        t0 = (r % p.ngroups) * p.G;
        split = r / p.ngroups;
    }
};

// Position blocks [b0, b1) of a split: an even division of nblk.
__device__ __forceinline__ void split_range(const CwgParams &p, int split, int &b0, int &b1)
{
    b0 = static_cast<int>((static_cast<long long>(p.nblk) * split) / p.splits);
    b1 = static_cast<int>((static_cast<long long>(p.nblk) * (split + 1)) / p.splits);
}

__device__ __forceinline__ void run_wg_loader(const CwgParams &p, const WgRing &R, Ctl ctl, int li, bool leader,
                                              volatile uint32_t *slot_parity)
{
    const uint64_t mapA = reinterpret_cast<uint64_t>(&p.tmA);
    if (leader) asm volatile("prefetch.tensormap [%0];" ::"l"(mapA) : "memory");
    const int nbs = p.BN / 64;  // B slices per tap
    const uint32_t tx = p.stage_bytes;
    int stage = 0, owner = 0;
    uint32_t parity = 0;
    bool ok = true;
    for (int g = blockIdx.x; ok && g < p.total_items; g += gridDim.x) {
        const WgItem it(p, g);
        int b0, b1;
        split_range(p, it.split, b0, b1);
        const int k0 = it.mt * 128, c0 = it.nt * p.BN;
        for (int b = b0; b < b1; ++b) {
            if (owner == li) {
                if (!wait_bar(R.empty0 + 8u * stage, parity ^ 1u, ctl)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    slot_parity[stage] = parity | 2u;
                    const int bq = b % p.bq, rest = b / p.bq;
                    const int q0 = bq * p.qb, p0 = (rest % p.bp) * p.pb, n0 = (rest / p.bp) * p.nb;
                    const uint32_t full = R.full0 + 8u * stage;
                    const uint32_t sa = R.s0 + static_cast<uint32_t>(stage) * p.stage_bytes;
                    mbar_arrive_expect_tx(full, tx);
                    if (p.xm) {
                        // x-major: A = x slices of units 2 mt and 2 mt + 1 (a unit
                        // past the last loads a box wholly past the images: zeros,
                        // never stored), B = the dY slice
                        for (int hf = 0; hf < 2; ++hf) {
                            const int u = 2 * it.mt + hf;
                            const bool real = u < p.units;
                            const int t = real ? u / p.cslices : p.T - 1;
                            const int cs = real ? u - (u / p.cslices) * p.cslices : 0;
                            const uint64_t mapB = reinterpret_cast<uint64_t>(&p.tmB[p.tap_phase[t]]);
                            tma_load_4d(sa + static_cast<uint32_t>(hf) * kSlice, mapB, full, 64 * cs, q0 + p.tap_dj[t],
                                        p0 + p.tap_di[t], real ? n0 : n0 + p.N);
                        }
                        tma_load_4d(sa + 2 * kSlice, mapA, full, 0, q0, p0, n0);
                    } else {
                    tma_load_4d(sa, mapA, full, k0, q0, p0, n0);
                    tma_load_4d(sa + kSlice, mapA, full, k0 + 64, q0, p0, n0);
                    for (int u = 0; u < p.G; ++u) {
                        // tap t0 + u's x slices; a tap past T (short last group)
                        // loads a box wholly past the images: zeros, never stored
                        const int t = min(it.t0 + u, p.T - 1);
                        const int nz = it.t0 + u < p.T ? n0 : n0 + p.N;
                        const uint64_t mapB = reinterpret_cast<uint64_t>(&p.tmB[p.tap_phase[t]]);
                        for (int j = 0; j < nbs; ++j)
                            tma_load_4d(sa + static_cast<uint32_t>((2 + u * nbs + j) * kSlice), mapB, full, c0 + 64 * j,
                                        q0 + p.tap_dj[t], p0 + p.tap_di[t], nz);
                    }
                    }
                }
                __syncwarp();
            }
            if (++owner == CDG_LOADERS) owner = 0;
            if (++stage == R.stages) {
                stage = 0;
                parity ^= 1u;
            }
        }
    }
}

__device__ __forceinline__ void run_wg_mma(const CwgParams &p, const WgRing &R, Ctl ctl, uint32_t tmem_base,
                                           bool leader)
{
    const uint32_t idesc = p.idesc;
    int stage = 0;
    uint32_t parity = 0, acc_count = 0;
    bool ok = true;
    for (int g = blockIdx.x; ok && g < p.total_items; g += gridDim.x) {
        const WgItem it(p, g);
        int b0, b1;
        split_range(p, it.split, b0, b1);
        const uint32_t acc = acc_count & 1u;
        if (!wait_bar(R.acc_empty0 + 8u * acc, ((acc_count >> 1) & 1u) ^ 1u, ctl)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * p.acc_stride;
        for (int b = b0; b < b1; ++b) {
            if (!wait_bar(R.full0 + 8u * stage, parity, ctl)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (leader) {
                const uint32_t sa = R.s0 + static_cast<uint32_t>(stage) * p.stage_bytes;
                const uint64_t adesc = sdesc_mn_sw128(sa, kSlice);
                const uint64_t bdesc = sdesc_mn_sw128(sa + 2 * kSlice, kSlice);
#pragma unroll
                for (int k = 0; k < 4; ++k)  // 16 positions = 2 KB = 128 descriptor units
                    umma_f16(d_tmem, adesc + 128u * k, bdesc + 128u * k, idesc, (b != b0 || k != 0) ? 1u : 0u);
                umma_commit(R.empty0 + 8u * stage);
            }
            __syncwarp();
            if (++stage == R.stages) {
                stage = 0;
                parity ^= 1u;
            }
        }
        if (!ok) break;
        if (leader) umma_commit(R.acc_full0 + 8u * acc);
        __syncwarp();
        ++acc_count;
    }
    if (leader) umma_commit(R.drain);
    __syncwarp();
    volatile uint32_t no_abort = 0;
    wait_bar(R.drain, 0, Ctl{&no_abort, ctl.status});
}

// Accumulator rows (dY channels) -> fp32 workspace rows of 32 channels, through
// two 16 KB staging buffers in the TMA store's 128-byte swizzle.
__device__ __forceinline__ void run_wg_epilogue(const CwgParams &p, const WgRing &R, Ctl ctl, uint32_t tmem_base)
{
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool elected = elect_one_sync();
    const int quad = warp & 3, ew = warp - CDG_EPI_WARP0;
    const int row = quad * 32 + lane;
    const uint32_t srow_off = static_cast<uint32_t>(row) * 128u, sw = static_cast<uint32_t>(row & 7);
    const uint64_t mapW = reinterpret_cast<uint64_t>(&p.tmW);
    const uint64_t mapWx = reinterpret_cast<uint64_t>(&p.tmWx);
    uint32_t acc_count = 0, chunk = 0;
    for (int g = blockIdx.x; g < p.total_items; g += gridDim.x) {
        const WgItem it(p, g);
        const uint32_t acc = acc_count & 1u;
        if (!wait_bar(R.acc_full0 + 8u * acc, (acc_count >> 1) & 1u, ctl)) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + acc * p.acc_stride + (static_cast<uint32_t>(quad * 32) << 16);
        const int NW = p.G * p.BN;  // accumulator columns: G taps x BN channels
        for (int cc = 0; cc < NW; cc += 32) {
            const uint32_t k = chunk++;
            const uint32_t buf = R.out0 + (k & 1u) * (128u * 128u);
            if (k >= 2 && elected && static_cast<uint32_t>(ew) == ((k - 2) & 3u)) bulk_wait_group_read<0>();
            named_bar_sync(1, 128);
            uint32_t r[32];
            tmem_ld_32x32b_x16(taddr + cc, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
            tmem_ld_32x32b_x16(taddr + cc + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
            tmem_ld_wait();
            if (cc + 32 >= NW) {  // last read of this accumulator
                tc_fence_before();
                __syncwarp();
                if (elected) mbar_arrive(R.acc_empty0 + 8u * acc);
            }
            if (p.xm) {
                // x-major: row = (unit 2 mt + row / 64, x channel row % 64), columns
                // = dY channels cc .. cc + 31.  Transposed into [dY channel][x
                // channel] rows of 256 bytes, one 8 KB half per unit: a warp
                // writes one 128-byte run per dY channel.
                const uint32_t dst = buf + static_cast<uint32_t>(row / 64) * 8192u + static_cast<uint32_t>(row % 64) * 4u;
#pragma unroll
                for (int j = 0; j < 32; ++j) st_shared_f32(dst + static_cast<uint32_t>(j) * 256u, __uint_as_float(r[j]));
                fence_proxy_async_smem();
                named_bar_sync(1, 128);
                if (cc < p.K && elected && static_cast<uint32_t>(ew) == (k & 3u)) {  // dY channels cc.. exist
                    for (int hf = 0; hf < 2; ++hf) {
                        const int u = 2 * it.mt + hf;
                        if (u >= p.units) break;
                        const int t = u / p.cslices, cs = u - (u / p.cslices) * p.cslices;
                        tma_store_4d(mapWx, buf + static_cast<uint32_t>(hf) * 8192u, 64 * cs, t, cc, it.split);
                    }
                    bulk_commit_group();
                }
                continue;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q)
                st_shared_v4(buf + srow_off + ((static_cast<uint32_t>(q) ^ sw) << 4), r[4 * q], r[4 * q + 1],
                             r[4 * q + 2], r[4 * q + 3]);
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            const int u = cc / p.BN, t = it.t0 + u;
            if (t < p.T && elected && static_cast<uint32_t>(ew) == (k & 3u)) {
                tma_store_4d(mapW, buf, it.nt * p.BN + (cc - u * p.BN), t, it.mt * 128, it.split);
                bulk_commit_group();
            }
        }
        ++acc_count;
    }
    if (elected) bulk_wait_group_all();
}

__global__ void __launch_bounds__(CDG_THREADS, 1) wgrad_kernel(const __grid_constant__ CwgParams p)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    // shared memory: stages | 2 x 16 KB staging | mbarriers, flags
    WgRing R;
    R.stages = p.stages;
    R.s0 = base;
    R.out0 = base + static_cast<uint32_t>(p.stages) * p.stage_bytes;
    const uint32_t bars = R.out0 + CDG_SMEM_STAGING;
    R.full0 = bars;
    R.empty0 = bars + 8u * p.stages;
    R.acc_full0 = bars + 16u * p.stages;
    R.acc_empty0 = R.acc_full0 + 16u;
    R.drain = R.acc_empty0 + 16u;
    uint8_t *const tail = smem_raw + (bars - raw);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tail + 8 * (2 * p.stages + 5));
    volatile uint32_t *abort_flag = tmem_slot + 1;
    volatile uint32_t *slot_parity = tmem_slot + 2;
    static_assert(8 * (2 * 8 + 5) + 8 + 4 * 8 <= CDG_SMEM_TABLES, "wgrad mbarrier area overflows");
    const int warp = threadIdx.x / 32;
    grid_dep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(R.full0 + 8u * s, 1);
            mbar_init(R.empty0 + 8u * s, 1);
            slot_parity[s] = 0u;
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(R.acc_full0 + 8u * a, 1);
            mbar_init(R.acc_empty0 + 8u * a, 4);  // one arrival per epilogue warp
        }
        mbar_init(R.drain, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    grid_dep_wait();
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Ctl ctl{abort_flag, p.status};

    if (warp == 1) {
        run_wg_mma(p, R, ctl, tmem_base, elect_one_sync());
    } else if (warp >= CDG_EPI_WARP0) {
        run_wg_epilogue(p, R, ctl, tmem_base);
    } else {
        run_wg_loader(p, R, ctl, warp == 0 ? 0 : warp - 1, elect_one_sync(), slot_parity);
    }

    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // let the latest load of every used slot land before the CTA exits
        volatile uint32_t no_abort = 0;
        const Ctl drain_ctl{&no_abort, p.status};
        for (int s = 0; s < p.stages; ++s) {
            const uint32_t v = slot_parity[s];
            if (v & 2u) wait_bar(R.full0 + 8u * s, v & 1u, drain_ctl);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// dW = sum of the splits' partials in split order, converted to dW's type;
// four elements per thread (count is a multiple of 8).
template <int OUT_T>
__global__ void wgrad_reduce_kernel(const float4 *__restrict__ ws, void *__restrict__ dW, long long count4,
                                    int splits)
{
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= count4) return;
    float4 s = __ldg(ws + i);
    for (int j = 1; j < splits; ++j) {
        const float4 v = __ldg(ws + static_cast<long long>(j) * count4 + i);
        s.x += v.x;
        s.y += v.y;
        s.z += v.z;
        s.w += v.w;
    }
    if (OUT_T == CDG_T_F32) {
        reinterpret_cast<float4 *>(dW)[i] = s;
    } else if (OUT_T == CDG_T_BF16) {
        __nv_bfloat162 a = __floats2bfloat162_rn(s.x, s.y), b = __floats2bfloat162_rn(s.z, s.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&a);
        u.y = *reinterpret_cast<uint32_t *>(&b);
        reinterpret_cast<uint2 *>(dW)[i] = u;
    } else {
        __half2 a = __floats2half2_rn(s.x, s.y), b = __floats2half2_rn(s.z, s.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&a);
        u.y = *reinterpret_cast<uint32_t *>(&b);
        reinterpret_cast<uint2 *>(dW)[i] = u;
    }
}

}  // namespace
}  // namespace cdg

// The kernel's shared-memory limit is raised to the opt-in maximum once, not
// to one plan's size: a later plan with a smaller footprint must not lower
// the limit under an earlier plan that is still launched.
cudaError_t cwg_prepare(size_t smem)
{
    if (smem > static_cast<size_t>(CDG_MAX_DYN_SMEM)) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(cdg::wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CDG_MAX_DYN_SMEM);
}

cudaError_t cwg_launch(const CwgParams &p, int grid, size_t smem, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(CDG_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, cdg::wgrad_kernel, p);
}

cudaError_t cwg_launch_reduce(const float *ws, void *dW, long long count, int splits, int out_type,
                              cudaStream_t stream)
{
    const long long count4 = count / 4;
    if (count4 <= 0) return cudaSuccess;
    const unsigned blocks = static_cast<unsigned>((count4 + 255) / 256);
    const float4 *w4 = reinterpret_cast<const float4 *>(ws);
    if (out_type == CDG_T_F32)
        cdg::wgrad_reduce_kernel<CDG_T_F32><<<blocks, 256, 0, stream>>>(w4, dW, count4, splits);
    else if (out_type == CDG_T_BF16)
        cdg::wgrad_reduce_kernel<CDG_T_BF16><<<blocks, 256, 0, stream>>>(w4, dW, count4, splits);
    else
        cdg::wgrad_reduce_kernel<CDG_T_F16><<<blocks, 256, 0, stream>>>(w4, dW, count4, splits);
    return cudaGetLastError();
}
