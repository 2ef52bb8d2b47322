// promote.cu -- promoted pages from the host KV store into the physical
// blocks of evicted pages, and the block-table rewrite.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 3. Periodic reranking
// and incremental promotion" (after a rerank only the promoted pages are
// transferred), "Core method, 4. Overlapping transfer and compute" (a UVA
// kernel reads the pinned host KV directly instead of a CPU gather, with a
// bounded grid so that it leaves the SMs to decoding) and "System design,
// head-level block table" (physical block reuse: the blocks of evicted pages
// are handed to promoted pages; an evicted entry keeps its place and points
// at the null block).
//
// A bounded grid (max_ctas CTAs of 256 threads, 16 by default) walks the
// layer's units.  Per unit: the evicted entries are read and nulled, their
// blocks paired in order with the promoted pages and written to the table;
// then the CTA copies the promoted pages from host memory, addressed through
// the unified address space (NVLink-C2C on GB300): 16-byte loads, sixteen in
// flight per thread before their stores (eight reached 0.65 of a contiguous
// host-to-device copy's rate at the default grid of 16 CTAs, sixteen 0.71; at
// 32 CTAs and more the kernel runs at that copy's rate).
#include "common.cuh"
#include "kernels.h"

namespace kvmm {
namespace {

constexpr int kPromoteThreads = 256;
constexpr int kPromoteBatch = 16;

__global__ void __launch_bounds__(kPromoteThreads) promote_kernel(const PromoteParams p)
{
    pdl_wait_then_release();
    extern __shared__ int32_t pm[];
    int32_t* phys_s = pm;            // [Kmax] block of pair i (-1: the pair moves nothing)
    int32_t* page_s = pm + p.Kmax;   // [Kmax] promoted page of pair i
    __shared__ int wsum[kPromoteThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t page_elems = static_cast<size_t>(p.T) * p.D;
    const int cpp = p.T * p.D / 4;  // 16-byte chunks of a page's keys and values together (a power of two)
    const int cpp_shift = __ffs(cpp) - 1;
    const int chunks = cpp / 2;     // 16-byte chunks of the keys (or of the values)
    const int U = p.B * p.Hkv;
    for (int unit = blockIdx.x; unit < U; unit += gridDim.x) {
        const int b = unit / p.Hkv, h = unit - (unit / p.Hkv) * p.Hkv;
        const size_t uf = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
        const bool rescored = p.rescore_mask == nullptr || p.rescore_mask[p.layer * p.Hkv + h] != 0;
        if (!rescored) {
            if (tid == 0) {
                if (p.moved) p.moved[uf] = 0;
                if (p.freed_cnt) p.freed_cnt[uf] = 0;
            }
            continue;
        }
        int np = p.promoted_cnt[uf], ne = p.evicted_cnt[uf];
        if (np < 0 || np > p.Kmax || ne < 0 || ne > p.Kmax) {
            if (tid == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
            np = min(max(np, 0), p.Kmax);
            ne = min(max(ne, 0), p.Kmax);
        }
        const int m = min(np, ne);
        int32_t* bt = p.block_table + uf * p.Pmax;

        // 1. evicted entries: null them; their blocks go to the pairs i < m, or are freed
        for (int i = tid; i < ne; i += kPromoteThreads) {
            const int32_t ev = p.evicted[uf * p.Kmax + i];
            int32_t ph = -1;
            if (ev < 0 || ev >= p.Pmax) {
                report(p.err, KVMM_ERR_OUT_OF_RANGE);
            } else {
                ph = bt[ev];
                if (ph < 0 || ph >= p.n_phys) {
                    report(p.err, ph < 0 ? KVMM_ERR_NULL_BLOCK : KVMM_ERR_OUT_OF_RANGE);
                    ph = -1;
                }
                bt[ev] = -1;
            }
            if (i < m)
                phys_s[i] = ph;
            else if (p.freed)
                p.freed[uf * p.Kmax + (i - m)] = ph;
        }
        if (tid == 0 && p.freed_cnt) p.freed_cnt[uf] = ne - m;
        __syncthreads();

        // 2. the promoted pages of the pairs take the blocks
        int mine = 0;
        for (int i = tid; i < m; i += kPromoteThreads) {
            const int32_t pr = p.promoted[uf * p.Kmax + i];
            if (pr < 0 || pr >= p.Pmax) {
                report(p.err, KVMM_ERR_OUT_OF_RANGE);
                phys_s[i] = -1;
            } else if (phys_s[i] >= 0) {
                bt[pr] = phys_s[i];
                ++mine;
            }
            page_s[i] = pr;
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mine += __shfl_xor_sync(kFullMask, mine, off);
        if (lane == 0) wsum[warp] = mine;
        __syncthreads();
        if (tid == 0 && p.moved) {
            int t = 0;
#pragma unroll
            for (int w = 0; w < kPromoteThreads / 32; ++w) t += wsum[w];
            p.moved[uf] = t;
        }

        // 3. copy the pairs' pages from the host store: flat index f = pair * cpp + chunk
        const int total = m * cpp;
        for (int f0 = tid; f0 < total; f0 += kPromoteThreads * kPromoteBatch) {
            uint4 v[kPromoteBatch];
#pragma unroll
            for (int k = 0; k < kPromoteBatch; ++k) {
                const int f = f0 + k * kPromoteThreads;
                v[k] = make_uint4(0u, 0u, 0u, 0u);
                if (f < total) {
                    const int i = f >> cpp_shift, c = f & (cpp - 1);
                    if (phys_s[i] >= 0) {
                        const bool val = c >= chunks;
                        const kvmm_bf16* src = (val ? p.host_v : p.host_k) +
                                               (uf * p.Pmax + page_s[i]) * page_elems + static_cast<size_t>(c - (val ? chunks : 0)) * 8;
                        v[k] = ld_stream_v4(src);
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kPromoteBatch; ++k) {
                const int f = f0 + k * kPromoteThreads;
                if (f < total) {
                    const int i = f >> cpp_shift, c = f & (cpp - 1);
                    if (phys_s[i] >= 0) {
                        const bool val = c >= chunks;
                        kvmm_bf16* dst = (val ? p.v_pool : p.k_pool) + static_cast<size_t>(phys_s[i]) * page_elems +
                                         static_cast<size_t>(c - (val ? chunks : 0)) * 8;
                        *reinterpret_cast<uint4*>(dst) = v[k];
                    }
                }
            }
        }
        __syncthreads();  // phys_s, page_s and wsum serve the next unit
    }
}

}  // namespace

cudaError_t launch_promote(const PromoteParams& p, int max_ctas, cudaStream_t stream)
{
    const int units = p.B * p.Hkv;
    const int grid = max(1, min(max_ctas > 0 ? max_ctas : 16, units));
    const size_t smem = 2 * static_cast<size_t>(p.Kmax) * sizeof(int32_t);
    static thread_local int dev_cache = -1;
    static thread_local size_t bytes_cache = 0;
    cudaError_t e = allow_smem(promote_kernel, smem, dev_cache, bytes_cache);
    if (e != cudaSuccess) return e;
    return launch_pdl(promote_kernel, dim3(static_cast<unsigned>(grid)), dim3(kPromoteThreads), smem, stream, p);
}

}  // namespace kvmm
