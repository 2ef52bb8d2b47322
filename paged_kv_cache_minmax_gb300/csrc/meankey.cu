// meankey.cu -- each page's mean key, the page representative of KVDrive's
// index (KVDrive, "Method details": the KV cache is split into blocks and
// each page's mean key stands for it; higher-level centroids group similar
// pages).  page_score_topk_mean scores these rows against the query with the
// same kernel as the MinMax bounds, on half their bytes.
//
// One warp per page: lane l holds channels [l*D/32, (l+1)*D/32) and sums the
// page's keys below tok_end in fp32, in token order, then divides by their
// count and rounds to bf16 (nearest even).
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace kvmm {
namespace {

constexpr int kMeanWarps = 8;

template <int D>
__global__ void __launch_bounds__(kMeanWarps * 32) meankey_kernel(const MeanParams p)
{
    constexpr int kCh = D / 32;  // channels per lane
    pdl_wait_then_release();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int h = blockIdx.x, b = blockIdx.y;
    const int page = blockIdx.z * kMeanWarps + warp;
    const int cap = p.Pmax * p.T;
    int tb = p.tok_begin ? p.tok_begin[b] : 0, te = p.tok_end[b];
    if (tb < 0 || te < tb || te > cap) {
        if (h == 0 && page == 0 && lane == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
        tb = max(tb, 0);
        te = min(max(te, tb), cap);
    }
    if (te <= tb) return;
    const int first = tb / p.T, last = (te - 1) / p.T;
    if (page < first || page > last) return;
    const size_t uf = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
    const int32_t phys = p.block_table[uf * p.Pmax + page];
    if (phys < 0 || phys >= p.n_phys) {
        if (lane == 0) report(p.err, phys < 0 ? KVMM_ERR_NULL_BLOCK : KVMM_ERR_OUT_OF_RANGE);
        return;
    }
    const int nv = min(p.T, te - page * p.T);
    const kvmm_bf16* kpage = p.k_pool + static_cast<size_t>(phys) * p.T * D + lane * kCh;
    float acc[kCh];
#pragma unroll
    for (int c = 0; c < kCh; ++c) acc[c] = 0.f;
    for (int r = 0; r < nv; ++r) {
        const kvmm_bf16* row = kpage + static_cast<size_t>(r) * D;
#pragma unroll
        for (int c = 0; c < kCh; ++c) acc[c] += __uint_as_float(static_cast<uint32_t>(row[c]) << 16);
    }
    kvmm_bf16* out = p.mean + (uf * p.Pmax + page) * D + lane * kCh;
#pragma unroll
    for (int c = 0; c < kCh; ++c) {
        const float m = acc[c] / static_cast<float>(nv);
        out[c] = __bfloat16_as_ushort(__float2bfloat16_rn(m));
    }
}

}  // namespace

cudaError_t launch_meankey(const MeanParams& p, cudaStream_t stream)
{
    const dim3 grid(static_cast<unsigned>(p.Hkv), static_cast<unsigned>(p.B),
                    static_cast<unsigned>((p.Pmax + kMeanWarps - 1) / kMeanWarps));
    if (p.D == 128) return launch_pdl(meankey_kernel<128>, grid, dim3(kMeanWarps * 32), 0, stream, p);
    return launch_pdl(meankey_kernel<64>, grid, dim3(kMeanWarps * 32), 0, stream, p);
}

}  // namespace kvmm
