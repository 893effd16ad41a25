// The dgrad library's non-template kernels (weight prepack, ReLU-mask
// packing, the ordered reduction of per-channel sums), the back-to-back fused
// kernel's launch, and the dispatch of dgrad launches to the plain or the
// extended kernel variant.
#include "dgrad_device.cuh"

namespace cdg {

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

// Packed ReLU mask: each pixel's C channels as bits padded to whole 16-byte
// units (cb bytes a pixel), channel c of pixel p in bit c % 8 of byte
// p*cb + c/8, set when x[p][c] > 0.  One thread per byte: its eight channels in
// one 16-byte load; bytes past C are 0.
__global__ void pack_relu_mask_kernel(const uint16_t *__restrict__ x, uint8_t *__restrict__ bits, long long nbytes,
                                      int C, int cb, int in_type)
{
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= nbytes) return;
    const long long pix = i / cb;
    const int c0 = 8 * static_cast<int>(i - pix * cb);
    uint32_t byte = 0;
    if (c0 < C) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(x + pix * C + c0));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint16_t h = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
            const float v = in_type == CDG_T_BF16 ? gate_value<CDG_T_BF16>(h) : gate_value<CDG_T_F16>(h);
            if (v > 0.0f) byte |= 1u << e;
        }
    }
    bits[i] = static_cast<uint8_t>(byte);
}

// Per-channel sums: out[k][c] = sum over the workspace rows r = 0, 1, ... of
// ws[r][k][c], added in row order (one row per CTA of the dgrad launch), so
// the result does not depend on how the CTAs were scheduled.
__global__ void channel_sums_kernel(const float *__restrict__ ws, int rows, int nsum, int C, float *__restrict__ out)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nsum * C) return;
    const int k = i / C, c = i - k * C;
    float acc = 0.0f;
    for (int r = 0; r < rows; ++r) acc += ws[(static_cast<size_t>(r) * nsum + k) * C + c];
    out[i] = acc;
}

}  // namespace cdg

// ------------------------------------------------------------------ launchers
// The dynamic shared-memory opt-in is a property of the kernel function, shared
// by every plan that uses it: always raise it to the largest size any plan
// may request, never to one plan's own size (a smaller later plan would
// otherwise lower the limit under an earlier one).
cudaError_t cdg_prepare_dgrad(int out_type, int in_type, bool mask, size_t smem)
{
    if (smem > static_cast<size_t>(CDG_MAX_DYN_SMEM)) return cudaErrorInvalidValue;
    cudaError_t e = cdg_dgrad_prepare_variant<0>(out_type, in_type, mask);
    if (e == cudaSuccess) e = cdg_dgrad_prepare_variant<1>(out_type, in_type, mask);
    if (e == cudaSuccess) e = cdg_dgrad_prepare_variant<2>(out_type, in_type, mask);
    if (e == cudaSuccess) e = cdg_dgrad_prepare_variant<3>(out_type, in_type, mask);
    return e;
}

cudaError_t cdg_launch_dgrad(const CdgParams &p, int out_type, int in_type, bool mask, int grid, size_t smem,
                             cudaStream_t stream)
{
    // each epilogue variant only where a plan needs it
    if (p.act == 1) return cdg_dgrad_launch_variant<2>(p, out_type, in_type, mask, grid, smem, stream);
    if (p.act == 2) return cdg_dgrad_launch_variant<3>(p, out_type, in_type, mask, grid, smem, stream);
    if (p.nsum != 0) return cdg_dgrad_launch_variant<1>(p, out_type, in_type, mask, grid, smem, stream);
    return cdg_dgrad_launch_variant<0>(p, out_type, in_type, mask, grid, smem, stream);
}

int cdg_max_active_pairs(int out_type, int in_type, bool mask, size_t smem)
{
    return cdg_dgrad_max_pairs_variant<0>(out_type, in_type, mask, smem);
}

cudaError_t cdg_launch_pack_mask(const void *x, void *bits, long long pixels, int C, int in_type,
                                 cudaStream_t stream)
{
    const int cb = 16 * ((C + 127) / 128);
    const long long nbytes = pixels * cb;
    if (nbytes <= 0) return cudaSuccess;
    const long long blocks = (nbytes + 255) / 256;
    cdg::pack_relu_mask_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t *>(x), static_cast<uint8_t *>(bits), nbytes, C, cb, in_type);
    return cudaGetLastError();
}

cudaError_t cdg_launch_prepack(const void *W, void *Wp, int K, int T, int C, cudaStream_t stream)
{
    dim3 grid((C + 31) / 32, (K + 31) / 32, T), block(32, 8);
    cdg::prepack_kernel<<<grid, block, 0, stream>>>(static_cast<const uint16_t *>(W), static_cast<uint16_t *>(Wp),
                                                    K, T, C);
    return cudaGetLastError();
}

cudaError_t cdg_launch_channel_sums(const float *ws, int rows, int nsum, int C, float *out, cudaStream_t stream)
{
    const int n = nsum * C;
    if (n <= 0) return cudaSuccess;
    cdg::channel_sums_kernel<<<(n + 255) / 256, 256, 0, stream>>>(ws, rows, nsum, C, out);
    return cudaGetLastError();
}

namespace {

typedef void (*FusedFn)(CdgParams);

// act: -1 no activation between the two dgrads, 0 ReLU, 1 GELU, 2 SiLU
template <int IN_T>
FusedFn select_fused_t(int act)
{
    if (act == 0) return cdg::fused_kernel<IN_T, 0>;
    if (act == 1) return cdg::fused_kernel<IN_T, 1>;
    if (act == 2) return cdg::fused_kernel<IN_T, 2>;
    return cdg::fused_kernel<IN_T, -1>;
}

FusedFn select_fused(int in_type, int act)
{
    return in_type == CDG_T_F16 ? select_fused_t<CDG_T_F16>(act) : select_fused_t<CDG_T_BF16>(act);
}

}  // namespace

cudaError_t cdg_prepare_fused(int in_type, int act)
{
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(select_fused(in_type, act)),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, CDG_MAX_DYN_SMEM);
}

cudaError_t cdg_launch_fused(const CdgParams &p, int in_type, int act, int grid, size_t smem, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(CDG_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    unsigned n = 0;
    if (p.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, select_fused(in_type, act), p);
}
