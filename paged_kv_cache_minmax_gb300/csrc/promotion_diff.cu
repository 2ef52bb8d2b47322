// promotion_diff.cu -- pages entering and leaving each rescored unit's top-K.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 3. Periodic reranking and
// incremental promotion": after a rerank only (current top-K minus previous
// top-K) is transferred; "System design, head-level block table": the
// physical blocks of evicted pages are handed to promoted pages, which the
// evicted list (previous minus current) serves.
//
// One CTA per (batch, KV head) of the layer.  Both lists are ascending, so
// membership is a binary search in the other list; hits are compacted in
// order with warp ballots and a block prefix over the warp totals.
#include "common.cuh"
#include "kernels.h"

namespace kvmm {
namespace {

constexpr int kDiffThreads = 128;
constexpr int kDiffWarps = kDiffThreads / 32;

__device__ __forceinline__ bool contains(const int32_t* list, int n, int32_t x)
{
    int lo = 0, hi = n;  // search [lo, hi)
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const int32_t v = list[mid];
        if (v == x) return true;
        if (v < x)
            lo = mid + 1;
        else
            hi = mid;
    }
    return false;
}

// out <- elements of a[0..na) absent from b[0..nb), in order; returns the count
__device__ int ordered_difference(const int32_t* a, int na, const int32_t* b, int nb, int32_t* out,
                                  int* warp_tot)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    int base = 0;
    for (int t0 = 0; t0 < na; t0 += kDiffThreads) {
        const int i = t0 + tid;
        const bool keep = i < na && !contains(b, nb, a[i]);
        const unsigned bal = __ballot_sync(kFullMask, keep);
        if (lane == 0) warp_tot[warp] = __popc(bal);
        __syncthreads();
        int off = base, all = 0;
#pragma unroll
        for (int w = 0; w < kDiffWarps; ++w) {
            if (w < warp) off += warp_tot[w];
            all += warp_tot[w];
        }
        if (keep && out) out[off + __popc(bal & lt)] = a[i];
        base += all;
        __syncthreads();
    }
    return base;
}

__global__ void __launch_bounds__(kDiffThreads) promotion_diff_kernel(const DiffParams p)
{
    __shared__ int warp_tot[kDiffWarps];
    const int h = blockIdx.x;
    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    const size_t unit = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
    pdl_wait_then_release();  // the current selection comes from the preceding kernels

    if (p.rescore_mask != nullptr && p.rescore_mask[p.layer * p.Hkv + h] == 0) {
        if (tid == 0) {
            p.promoted_cnt[unit] = 0;
            if (p.evicted_cnt) p.evicted_cnt[unit] = 0;
        }
        return;
    }

    const int32_t* prev = p.prev_idx + unit * p.Kmax;
    const int32_t* cur = p.cur_idx + unit * p.Kmax;
    const int np = p.prev_cnt[unit];
    const int nc = p.cur_cnt[unit];
    bool bad = np < 0 || np > p.Kmax || nc < 0 || nc > p.Kmax;
    if (!bad) {
        bool local = false;
        for (int i = tid; i + 1 < np; i += kDiffThreads) local |= prev[i] >= prev[i + 1];
        for (int i = tid; i + 1 < nc; i += kDiffThreads) local |= cur[i] >= cur[i + 1];
        bad = __syncthreads_or(local) != 0;
    }
    if (bad) {
        if (tid == 0) {
            report(p.err, KVMM_ERR_OUT_OF_RANGE);
            p.promoted_cnt[unit] = 0;
            if (p.evicted_cnt) p.evicted_cnt[unit] = 0;
        }
        return;
    }

    const int n_prom = ordered_difference(cur, nc, prev, np, p.promoted + unit * p.Kmax, warp_tot);
    int n_evic = 0;
    if (p.evicted_cnt) n_evic = ordered_difference(prev, np, cur, nc, p.evicted ? p.evicted + unit * p.Kmax : nullptr, warp_tot);
    if (tid == 0) {
        p.promoted_cnt[unit] = n_prom;
        if (p.evicted_cnt) p.evicted_cnt[unit] = n_evic;
        if (p.total_promoted && n_prom) atomicAdd(p.total_promoted, n_prom);
    }
    if (p.commit) {
        __syncthreads();  // both differences have read prev
        int32_t* prev_w = p.prev_idx + unit * p.Kmax;
        for (int i = tid; i < nc; i += kDiffThreads) prev_w[i] = cur[i];
        if (tid == 0) p.prev_cnt[unit] = nc;
    }
}

}  // namespace

cudaError_t launch_promotion_diff(const DiffParams& p, cudaStream_t stream)
{
    return launch_pdl(promotion_diff_kernel, dim3(p.Hkv, p.B), dim3(kDiffThreads), 0, stream, p);
}

}  // namespace kvmm
