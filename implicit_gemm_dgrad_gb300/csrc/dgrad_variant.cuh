// Kernel selection and launch for one epilogue variant of the dgrad kernels
// (EPI: 0 plain, 1 per-channel sums, 2 GELU backward, 3 SiLU backward).
// Variants are instantiated in translation units of their own
// (dgrad_plain_sm103.cu, dgrad_ext_sm103.cu, dgrad_act_sm103.cu), so that the
// kernel sets compile in parallel.
#pragma once

#include "dgrad_device.cuh"

namespace {

typedef void (*DgradFn)(CdgParams);

template <int OUT_T, bool MASK, int IN_T, int EPI>
DgradFn pick_mode(int mode)
{
    if (mode == 1) return cdg::dgrad_kernel<OUT_T, MASK, IN_T, 1, EPI>;
    if (mode == 2) return cdg::dgrad_kernel<OUT_T, MASK, IN_T, 2, EPI>;
    if (mode == 3) return cdg::dgrad_kernel<OUT_T, MASK, IN_T, 3, EPI>;
    if (mode == 4) return cdg::dgrad_kernel<OUT_T, MASK, IN_T, 4, EPI>;
    if (mode == 5) return cdg::dgrad_kernel<OUT_T, MASK, IN_T, 5, EPI>;
    if (mode == 6) return cdg::dgrad_kernel<OUT_T, MASK, IN_T, 6, EPI>;
    return cdg::dgrad_kernel<OUT_T, MASK, IN_T, 0, EPI>;
}

// The activation variants (EPI 2, 3) exist only with the gate, which reads
// the activation's saved input.
template <int OUT_T, int IN_T, int EPI>
DgradFn pick_gate(bool mask, int mode)
{
    if constexpr (EPI >= 2)
        return mask ? pick_mode<OUT_T, true, IN_T, EPI>(mode) : nullptr;
    else
        return mask ? pick_mode<OUT_T, true, IN_T, EPI>(mode) : pick_mode<OUT_T, false, IN_T, EPI>(mode);
}

template <int EPI>
DgradFn select_kernel(int out_type, int in_type, bool mask, int mode)
{
    if (in_type == CDG_T_F16)
        return out_type == CDG_T_F32 ? pick_gate<CDG_T_F32, CDG_T_F16, EPI>(mask, mode)
                                     : pick_gate<CDG_T_F16, CDG_T_F16, EPI>(mask, mode);
    return out_type == CDG_T_F32 ? pick_gate<CDG_T_F32, CDG_T_BF16, EPI>(mask, mode)
                                 : pick_gate<CDG_T_BF16, CDG_T_BF16, EPI>(mask, mode);
}

}  // namespace

// Raise the dynamic shared-memory limit of every kernel of this variant for
// the given types to the largest size any plan may request.
template <int EPI>
cudaError_t cdg_dgrad_prepare_variant(int out_type, int in_type, bool mask)
{
    for (int mode = 0; mode < 7; ++mode) {
        DgradFn fn = select_kernel<EPI>(out_type, in_type, mask, mode);
        if (!fn) return cudaSuccess;  // no such variant for these types (activation without gate)
        const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, CDG_MAX_DYN_SMEM);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int EPI>
cudaError_t cdg_dgrad_launch_variant(const CdgParams &p, int out_type, int in_type, bool mask, int grid, size_t smem,
                                     cudaStream_t stream)
{
    const int mode = p.halo ? (p.pair ? (p.dual ? 6 : 4) : (p.dual ? 5 : 1)) : (p.pair ? 2 : (p.dual ? 3 : 0));
    DgradFn fn = select_kernel<EPI>(out_type, in_type, mask, mode);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(CDG_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (p.pair) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (p.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

// Largest number of CTA pairs of this variant's pair kernel resident at once.
template <int EPI>
int cdg_dgrad_max_pairs_variant(int out_type, int in_type, bool mask, size_t smem)
{
    DgradFn fn = select_kernel<EPI>(out_type, in_type, mask, 2);
    if (!fn) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(CDG_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void *>(fn), &cfg) != cudaSuccess) return -1;
    return n;
}
