// C-ABI of the wgrad path: the weight gradient of the same convolution (the
// apache/tvm PR #10110 page's announced follow-up to dgrad, "wgrad +
// parallel split-k"): one GEMM per filter tap (or per group of taps, side by
// side along N, for narrow layers) over blocks of 64 output positions, split
// over the positions, partials reduced in a fixed order.  Validation,
// planning, tensor maps and launches; the kernels are in wgrad_sm103.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>

#include "../../include/cdg.h"
#include "cwg_params.h"

namespace {

constexpr int kMaxSmem = CDG_MAX_DYN_SMEM;
constexpr int kMaxStages = 8;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda
// symbol needed at link time).
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

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
    return pa < pb + nb && pb < pa + na;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

CUtensorMapDataType tmap_type(int dtype)
{
    return dtype == CDG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

}  // namespace


struct cdg_wgrad_st {
    int N, H, W, C, K, R, S, stride, pad, dil, dtype, out_type;
    bool host_only;
    size_t smem;
    int grid;
    int *d_status;
    size_t ws_bytes;
    CwgParams prm;
    const void *cached_dY, *cached_x;
    void *cached_ws;
    cdg_wgrad_info_t info;
};

namespace {

// x channels per tile: all of C rounded up to 64 when C <= 256, else the
// multiple of 64 up to 256 with the least padding.
int wgrad_bn(int C)
{
    if (C <= 256) return ((C + 63) / 64) * 64;
    int best = 256;
    long long waste = -1;
    for (int bn = 256; bn >= 64; bn -= 64) {
        const long long w = 1LL * ceil_div(C, bn) * bn - C;
        if (waste < 0 || w < waste) {
            waste = w;
            best = bn;
        }
    }
    return best;
}

int make_wgrad_plan(int N, int H, int W, int C, int K, int R, int S, int stride, int pad, int dil, int dtype,
                    int out_f32, int splits_req, int num_sms, bool host_only, cdg_wgrad_t *out)
{
    if (!out) return CDG_ERR_INVALID_ARG;
    *out = nullptr;
    if (N < 1 || H < 1 || W < 1 || C < 1 || K < 1 || R < 1 || S < 1 || stride < 1 || pad < 0 || dil < 1 ||
        (dtype != CDG_F16 && dtype != CDG_BF16) || (out_f32 != 0 && out_f32 != 1) || splits_req < 0 ||
        num_sms < 1)
        return CDG_ERR_INVALID_ARG;
    const int P = (H + 2 * pad - dil * (R - 1) - 1) / stride + 1;
    const int Q = (W + 2 * pad - dil * (S - 1) - 1) / stride + 1;
    if (H + 2 * pad - dil * (R - 1) - 1 < 0 || W + 2 * pad - dil * (S - 1) - 1 < 0 || P < 1 || Q < 1)
        return CDG_ERR_INVALID_ARG;
    // every phase sub-grid of x must be non-empty (its tensor map needs extent)
    if (C % 8 != 0 || K % 8 != 0 || stride > 4 || R * S > CDG_MAX_TAPS || H < stride || W < stride)
        return CDG_ERR_UNSUPPORTED;

    cdg_wgrad_st *h = new (std::nothrow) cdg_wgrad_st();
    if (!h) return CDG_ERR_CUDA;
    h->N = N; h->H = H; h->W = W; h->C = C; h->K = K; h->R = R; h->S = S;
    h->stride = stride; h->pad = pad; h->dil = dil; h->dtype = dtype;
    h->out_type = out_f32 ? CDG_T_F32 : (dtype == CDG_BF16 ? CDG_T_BF16 : CDG_T_F16);
    h->host_only = host_only;

    CwgParams &p = h->prm;
    std::memset(&p, 0, sizeof p);
    p.N = N; p.H = H; p.W = W; p.C = C; p.K = K; p.P = P; p.Q = Q; p.stride = stride;
    p.T = R * S;
    p.BN = wgrad_bn(C);
    p.tiles_m = ceil_div(K, 128);
    p.tiles_n = ceil_div(C, p.BN);
    // position box of exactly 64 (q, p, n) positions with the fewest blocks
    // (the image count absorbs small planes: 7x7 takes 1 x 1 x 64 boxes)
    long long best = -1;
    for (int qb = 64; qb >= 1; qb /= 2)
        for (int pb = 64 / qb; pb >= 1; pb /= 2) {
            const int nb = 64 / (qb * pb);
            const long long blocks = 1LL * ceil_div(Q, qb) * ceil_div(P, pb) * ceil_div(N, nb);
            if (best < 0 || blocks < best) {
                best = blocks;
                p.qb = qb;
                p.pb = pb;
                p.nb = nb;
            }
        }
    p.bq = ceil_div(Q, p.qb);
    p.bp = ceil_div(P, p.pb);
    p.nblk = static_cast<int>(best);
    // taps side by side along N when a tap's tile is narrow: the most taps
    // per item that N <= 256 allows, spread evenly over the groups
    p.G = 1;
    if (p.tiles_n == 1 && p.BN < 256) {
        const int gmax = std::min(p.T, 256 / p.BN);
        const int ng = ceil_div(p.T, gmax);
        p.G = ceil_div(p.T, ng);
    }
    p.ngroups = ceil_div(p.T, p.G);
    // x-major tiles when the dY channels fill at most half of a 128-row M
    // tile, for 1x1 filters with at least two 64-channel slices of x to pair
    // (measured on GB300: the 1x1 256 -> 64 layer at 56x56 99.3 -> 92.5 us).
    // With taps paired along M every item reads its dY block again (the 3x3
    // 64 -> 64 layer: five items a split against three tap groups), and that
    // layer measured slower (113.0 -> 116.3 us), so filters with more taps
    // keep the dY-channel tiles.
    p.cslices = ceil_div(C, 64);
    p.units = p.T * p.cslices;
    p.xm = (K <= 64 && p.T == 1 && p.units >= 2) ? 1 : 0;
    if (p.xm) {
        p.BN = 64;
        p.G = 1;
        p.ngroups = 1;
        p.tiles_m = ceil_div(p.units, 2);
        p.tiles_n = 1;
    }
    const int tiles = p.ngroups * p.tiles_m * p.tiles_n;
    int splits = splits_req;
    // default: as many splits as fit in one wave of work items
    if (splits == 0) splits = std::max(1, num_sms / tiles);
    splits = std::max(1, std::min(splits, p.nblk));
    p.splits = splits;
    p.total_items = splits * tiles;
    // A: two 8 KB slices (dY channels, or x-major: two units of x); B: the x
    // slices of the item's taps (x-major: one dY slice)
    p.stage_bytes = static_cast<uint32_t>(2 * 64 * 128 + p.G * (p.BN / 64) * 64 * 128);
    p.stages = std::min(kMaxStages, (kMaxSmem - 1024 - CDG_SMEM_STAGING - CDG_SMEM_TAIL) / static_cast<int>(p.stage_bytes));
    const uint32_t ab = dtype == CDG_BF16 ? 1u : 0u;
    // f32 accumulate; A, B in the input type; both MN-major (bits 15, 16); N; M = 128
    const int nw = p.G * p.BN;  // MMA N: G taps x BN channels
    p.idesc = (1u << 4) | (ab << 7) | (ab << 10) | (1u << 15) | (1u << 16) |
              (static_cast<uint32_t>(nw >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
    uint32_t cols = 32;
    while (cols < 2u * static_cast<uint32_t>(nw)) cols *= 2;
    p.tmem_cols = cols;
    p.acc_stride = cols / 2;
    for (int r = 0; r < R; ++r)
        for (int s = 0; s < S; ++s) {
            const int t = r * S + s;
            const int oh = r * dil - pad, ow = s * dil - pad;
            const int ph = floor_mod(oh, stride), pw = floor_mod(ow, stride);
            p.tap_phase[t] = static_cast<int16_t>(ph * stride + pw);
            p.tap_di[t] = static_cast<int16_t>((oh - ph) / stride);
            p.tap_dj[t] = static_cast<int16_t>((ow - pw) / stride);
        }
    h->smem = static_cast<size_t>(1024 + p.stages * static_cast<int>(p.stage_bytes) + CDG_SMEM_STAGING + CDG_SMEM_TAIL);
    h->grid = std::max(1, std::min(num_sms, p.total_items));
    h->ws_bytes = static_cast<size_t>(splits) * K * p.T * C * 4;

    cdg_wgrad_info_t &inf = h->info;
    std::memset(&inf, 0, sizeof inf);
    inf.P = P; inf.Q = Q;
    inf.tile_m = 128; inf.tile_n = p.BN;
    inf.x_major = p.xm;
    inf.taps_per_item = p.G;
    inf.splits = splits;
    inf.pos_box[0] = p.qb; inf.pos_box[1] = p.pb; inf.pos_box[2] = p.nb;
    inf.blocks = p.nblk;
    inf.stages = p.stages;
    inf.work_items = p.total_items;
    inf.grid = h->grid;
    inf.smem_bytes = static_cast<int>(h->smem);
    inf.tmem_cols = static_cast<int>(cols);

    if (!host_only) {
        if (cwg_prepare(h->smem) != cudaSuccess || cudaMalloc(&h->d_status, sizeof(int)) != cudaSuccess ||
            cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess) {
            if (h->d_status) cudaFree(h->d_status);
            delete h;
            return CDG_ERR_CUDA;
        }
    }
    *out = h;
    return CDG_OK;
}

int encode_wgrad_maps(cdg_wgrad_st *h, const void *dY, const void *x, void *ws)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return CDG_ERR_CUDA;
    CwgParams &p = h->prm;
    const cuuint32_t ones[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = tmap_type(h->dtype);
    const cuuint64_t C = h->C, K = h->K, W = h->W, H = h->H, s = h->stride;
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(p.qb), static_cast<cuuint32_t>(p.pb),
                               static_cast<cuuint32_t>(p.nb)};
    {
        const cuuint64_t dims[4] = {K, static_cast<cuuint64_t>(p.Q), static_cast<cuuint64_t>(p.P),
                                    static_cast<cuuint64_t>(h->N)};
        const cuuint64_t strides[3] = {K * 2, p.Q * K * 2, p.P * p.Q * K * 2};
        if (enc(&p.tmA, dt, 4, const_cast<void *>(dY), dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CDG_ERR_CUDA;
    }
    for (int ph = 0; ph < h->stride; ++ph)
        for (int pw = 0; pw < h->stride; ++pw) {
            // the phase sub-grid {C, wph, hph, N} of x, starting at pixel (ph, pw)
            const cuuint64_t hph = (H - ph + s - 1) / s, wph = (W - pw + s - 1) / s;
            char *base = static_cast<char *>(const_cast<void *>(x)) + (static_cast<cuuint64_t>(ph) * W + pw) * C * 2;
            const cuuint64_t dims[4] = {C, wph, hph, static_cast<cuuint64_t>(h->N)};
            const cuuint64_t strides[3] = {s * C * 2, s * W * C * 2, H * W * C * 2};
            if (enc(&p.tmB[ph * h->stride + pw], dt, 4, base, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return CDG_ERR_CUDA;
        }
    {
        const cuuint64_t T = static_cast<cuuint64_t>(p.T);
        const cuuint64_t dims[4] = {C, T, K, static_cast<cuuint64_t>(p.splits)};
        const cuuint64_t strides[3] = {C * 4, T * C * 4, K * T * C * 4};
        const cuuint32_t wbox[4] = {32, 1, 128, 1};
        if (enc(&p.tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws, dims, strides, wbox, ones,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CDG_ERR_CUDA;
        // x-major tiles: 32 dY channels x one tap x 64 x channels, rows of 256 bytes
        const cuuint32_t xbox[4] = {64, 1, 32, 1};
        if (p.xm && enc(&p.tmWx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws, dims, strides, xbox, ones,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CDG_ERR_CUDA;
    }
    h->cached_dY = dY;
    h->cached_x = x;
    h->cached_ws = ws;
    return CDG_OK;
}

}  // namespace

extern "C" {

int cdg_wgrad_plan(int N, int H, int W, int C, int K, int R, int S, int stride, int pad, int dil, int dtype,
                   int out_f32, int splits, cdg_wgrad_t *out)
{
    if (out) *out = nullptr;
    cdg_wgrad_t probe = nullptr;
    const int rc = make_wgrad_plan(N, H, W, C, K, R, S, stride, pad, dil, dtype, out_f32, splits, 148, true, &probe);
    if (rc != CDG_OK) return rc;
    cdg_wgrad_destroy(probe);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return CDG_ERR_CUDA;
    return make_wgrad_plan(N, H, W, C, K, R, S, stride, pad, dil, dtype, out_f32, splits, sms, false, out);
}

int cdg_wgrad_plan_host(int N, int H, int W, int C, int K, int R, int S, int stride, int pad, int dil, int dtype,
                        int out_f32, int splits, int num_sms, cdg_wgrad_t *out)
{
    return make_wgrad_plan(N, H, W, C, K, R, S, stride, pad, dil, dtype, out_f32, splits, num_sms, true, out);
}

void cdg_wgrad_destroy(cdg_wgrad_t h)
{
    if (!h) return;
    if (h->d_status) cudaFree(h->d_status);
    delete h;
}

size_t cdg_wgrad_workspace_bytes(cdg_wgrad_t h) { return h ? h->ws_bytes : 0; }

int cdg_wgrad_get_info(cdg_wgrad_t h, cdg_wgrad_info_t *info)
{
    if (!h || !info) return CDG_ERR_INVALID_ARG;
    *info = h->info;
    return CDG_OK;
}

int cdg_wgrad(cdg_wgrad_t h, const void *dY, const void *x, void *dW, void *workspace, cdg_stream_t stream)
{
    if (!h || !dY || !x || !dW || !workspace) return CDG_ERR_INVALID_ARG;
    if (h->host_only) return CDG_ERR_NO_DEVICE;
    if (!aligned16(dY) || !aligned16(x) || !aligned16(dW) || !aligned16(workspace)) return CDG_ERR_ALIGNMENT;
    const CwgParams &p = h->prm;
    const size_t dy_bytes = static_cast<size_t>(h->N) * p.P * p.Q * h->K * 2;
    const size_t x_bytes = static_cast<size_t>(h->N) * h->H * h->W * h->C * 2;
    const size_t dw_bytes = static_cast<size_t>(h->K) * p.T * h->C * (h->out_type == CDG_T_F32 ? 4 : 2);
    if (overlaps(dW, dw_bytes, dY, dy_bytes) || overlaps(dW, dw_bytes, x, x_bytes) ||
        overlaps(dW, dw_bytes, workspace, h->ws_bytes) || overlaps(workspace, h->ws_bytes, dY, dy_bytes) ||
        overlaps(workspace, h->ws_bytes, x, x_bytes))
        return CDG_ERR_ALIAS;
    if (dY != h->cached_dY || x != h->cached_x || workspace != h->cached_ws) {
        const int rc = encode_wgrad_maps(h, dY, x, workspace);
        if (rc != CDG_OK) return rc;
    }
    h->prm.status = h->d_status;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cwg_launch(h->prm, h->grid, h->smem, s) != cudaSuccess) return CDG_ERR_CUDA;
    if (cwg_launch_reduce(static_cast<const float *>(workspace), dW, static_cast<long long>(h->K) * p.T * h->C,
                          p.splits, h->out_type, s) != cudaSuccess)
        return CDG_ERR_CUDA;
    return CDG_OK;
}

int cdg_wgrad_device_status(cdg_wgrad_t h, cdg_stream_t stream)
{
    if (!h) return CDG_ERR_INVALID_ARG;
    if (h->host_only) return CDG_ERR_NO_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaMemcpyAsync(&v, h->d_status, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return CDG_ERR_CUDA;
    if (v != 0 && (cudaMemsetAsync(h->d_status, 0, sizeof(int), s) != cudaSuccess ||
                   cudaStreamSynchronize(s) != cudaSuccess))
        return CDG_ERR_CUDA;
    return v;
}

}  // extern "C"
