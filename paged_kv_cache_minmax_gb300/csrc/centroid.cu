// centroid.cu -- the centroid level of KVDrive's index over the pages' mean
// keys, and the two-level page selection it serves.
//
// KVDrive, "Method details": the KV cache is split into blocks, each page's
// mean key is its representative, and higher-level centroids group similar
// pages; "the trade-off between block size and centroid count": the centroid
// count is kept proportional to the context, and the similarity grouping
// needs half the centroids of a spatial blocking for the same accuracy.  The
// page names no clustering algorithm; the one built here is Lloyd's k-means
// per (batch, layer, KV head) unit, started from spatial blocks of R pages
// (n_c = ceil(P / R) centroids; no iteration = the spatial blocking):
//   - assignment (centroid_assign_kernel): a page joins the centroid of least
//     squared Euclidean distance, accumulated with fmaf(x, x, acc) in fp32 in
//     channel order, ties to the lower centroid -- a decision, taken in one
//     fixed precision and order, so the oracle takes the same one;
//   - update (centroid_update_kernel): the pages of each centroid in page
//     order (a stable counting sort: member_off / members), and the centroid
//     the bf16 rounding of their fp32 mean, summed in page order; a centroid
//     with no page keeps its value.
// The selection (centroid_select_kernel, one CTA per rescored unit) scores the
// centroids like pages (q . c over the query group, summed or maxed, fp32),
// keeps the M best exactly (block_topk), marks their pages in a bitmap,
// compacts them in page order, scores those pages by their mean keys and
// keeps the K best exactly, ties to the lower page, ascending.
//
// The build is an index build after prefill, off the decode step: its
// assignment runs on the CUDA cores in the oracle's order (a tensor-core
// distance would reorder the sums and move near-tie decisions).  The
// selection reads the centroid rows and the expanded pages' mean keys only.
#include <cfloat>

#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "topk_block.cuh"

namespace kvmm {
namespace {

constexpr int kUpdThreads = 256;
constexpr int kUpdWarps = kUpdThreads / 32;
constexpr int kAsgThreads = 128;  // one page a thread
constexpr int kAsgChunk = 32;     // centroids staged in shared memory at a time (fp32)
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// pages of sequence b, clamped to the table (reported when `report`)
__device__ __forceinline__ int centroid_unit_pages(const CentroidParams& p, int b, bool report_err)
{
    int seq = p.seq_len[b];
    const int cap = p.Pmax * p.T;
    if (seq < 0 || seq > cap) {
        if (report_err) report(p.err, KVMM_ERR_OUT_OF_RANGE);
        seq = seq < 0 ? 0 : cap;
    }
    return (seq + p.T - 1) / p.T;
}

// in-place inclusive scan of a[0 .. n) by the whole CTA (THREADS threads); wsum: THREADS / 32 ints
template <int THREADS>
__device__ void block_inclusive_scan(int32_t* a, int n, int32_t* wsum)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + THREADS - 1) / THREADS;
    const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
    int local = 0;
    for (int i = i0; i < i1; ++i) local += a[i];
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int x = __shfl_up_sync(kFullMask, incl, off);
        if (lane >= off) incl += x;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += wsum[w];
    for (int i = i0; i < i1; ++i) {
        run += a[i];
        a[i] = run;
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// update: member lists in page order, then each centroid's mean.  init: the spatial blocks (page p in
// centroid p / R), written to assign as well.
template <int D>
__global__ void __launch_bounds__(kUpdThreads) centroid_update_kernel(const CentroidParams p, int init)
{
    constexpr int kCh = D / 32;  // channels of a lane
    extern __shared__ __align__(16) int32_t usm[];
    __shared__ int32_t wsum[kUpdWarps];
    pdl_wait_then_release();
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t uf = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
    const int P = centroid_unit_pages(p, b, init && h == 0);
    const int n_c = (P + p.R - 1) / p.R;
    int32_t* cnt = usm;                                 // [n_c + 1]: counts, then offsets, then cursors
    int32_t* sa = usm + ((p.Cmax + 1 + 3) & ~3);        // [P]: each page's centroid
    int32_t* assign = p.assign + uf * p.Pmax;
    int32_t* off = p.member_off + uf * (p.Cmax + 1);
    int32_t* mem = p.members + uf * p.Pmax;

    for (int j = tid; j <= n_c; j += kUpdThreads) cnt[j] = 0;
    for (int pg = tid; pg < P; pg += kUpdThreads) {
        int a = init ? pg / p.R : assign[pg];
        if (a < 0 || a >= n_c) {  // not written by the assignment for this shape
            report(p.err, KVMM_ERR_OUT_OF_RANGE);
            a = 0;
        }
        sa[pg] = a;
        if (init) assign[pg] = a;
    }
    __syncthreads();
    for (int pg = tid; pg < P; pg += kUpdThreads) atomicAdd(&cnt[sa[pg] + 1], 1);
    __syncthreads();
    block_inclusive_scan<kUpdThreads>(cnt + 1, n_c, wsum);  // cnt[j] = pages of centroids below j
    for (int j = tid; j <= n_c; j += kUpdThreads) off[j] = cnt[j];
    __syncthreads();  // every offset is read before warp 0 moves the cursors
    // members, stable: warp 0 walks the pages in order, 32 at a time; pages of one centroid within those 32
    // take consecutive places in lane order after the ones before
    if (warp == 0) {
        for (int c0 = 0; c0 < P; c0 += 32) {
            const int pg = c0 + lane;
            const bool live = pg < P;
            const int a = live ? sa[pg] : -1 - lane;  // a value no other lane holds
            const unsigned peers = __match_any_sync(kFullMask, a);
            const int leader = __ffs(peers) - 1;
            int base = 0;
            if (live && lane == leader) base = cnt[a];
            base = __shfl_sync(kFullMask, base, leader);
            if (live) {
                mem[base + __popc(peers & ((1u << lane) - 1u))] = pg;
                if (lane == leader) cnt[a] = base + __popc(peers);
            }
            __syncwarp();
        }
    }
    __syncthreads();  // the member lists (global memory) are visible to the CTA
    // each centroid's mean: a warp a centroid, lane l sums channels [l*kCh, (l+1)*kCh) over the members in
    // page order, in fp32; an empty centroid keeps its value (at init every block has a page)
    for (int j = warp; j < n_c; j += kUpdWarps) {
        const int k0 = off[j], k1 = off[j + 1];
        if (k1 == k0) continue;
        float acc[kCh];
#pragma unroll
        for (int c = 0; c < kCh; ++c) acc[c] = 0.f;
        for (int k = k0; k < k1; k += 8) {
            int pgs[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) pgs[u] = k + u < k1 ? mem[k + u] : 0;
            uint32_t w[8][(kCh + 1) / 2];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const kvmm_bf16* row = p.mean + (uf * p.Pmax + pgs[u]) * D + lane * kCh;
                if constexpr (kCh == 4) {
                    const uint2 v = *reinterpret_cast<const uint2*>(row);
                    w[u][0] = v.x;
                    w[u][1] = v.y;
                } else {
                    w[u][0] = *reinterpret_cast<const uint32_t*>(row);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (k + u < k1) {
#pragma unroll
                    for (int c = 0; c < kCh; ++c) acc[c] += (c & 1) ? bf_hi(w[u][c >> 1]) : bf_lo(w[u][c >> 1]);
                }
            }
        }
        const float n = static_cast<float>(k1 - k0);
        kvmm_bf16* out = p.cent + (uf * p.Cmax + j) * D + lane * kCh;
#pragma unroll
        for (int c = 0; c < kCh; ++c) out[c] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[c] / n));
    }
}

// ---------------------------------------------------------------------------
// assignment: one page a thread; the unit's centroids pass through shared memory (fp32) kAsgChunk at a time
template <int D>
__global__ void __launch_bounds__(kAsgThreads) centroid_assign_kernel(const CentroidParams p)
{
    __shared__ __align__(16) float cs[kAsgChunk * D];
    pdl_wait_then_release();
    const int h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const size_t uf = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
    const int P = centroid_unit_pages(p, b, false);
    const int n_c = (P + p.R - 1) / p.R;
    if (static_cast<int>(blockIdx.x) * kAsgThreads >= P) return;  // the whole CTA: no page of this unit
    const int pg = blockIdx.x * kAsgThreads + tid;
    const bool live = pg < P;
    uint32_t m[D / 2];  // this page's mean key, bf16 pairs
    if (live) {
        const uint4* row = reinterpret_cast<const uint4*>(p.mean + (uf * p.Pmax + pg) * D);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            const uint4 v = row[i];
            m[4 * i] = v.x;
            m[4 * i + 1] = v.y;
            m[4 * i + 2] = v.z;
            m[4 * i + 3] = v.w;
        }
    }
    float best = 0.f;
    int arg = 0;
    const kvmm_bf16* cent = p.cent + uf * p.Cmax * D;
    for (int c0 = 0; c0 < n_c; c0 += kAsgChunk) {
        const int nc = min(kAsgChunk, n_c - c0);
        __syncthreads();  // the previous chunk is read
        for (int i = tid; i < nc * D / 2; i += kAsgThreads) {
            const uint32_t w = reinterpret_cast<const uint32_t*>(cent + static_cast<size_t>(c0) * D)[i];
            cs[2 * i] = bf_lo(w);
            cs[2 * i + 1] = bf_hi(w);
        }
        __syncthreads();
        if (!live) continue;
        int j = 0;
        for (; j + 4 <= nc; j += 4) {  // four centroids at once: independent chains, each in channel order
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const float* c = cs + j * D;
#pragma unroll
            for (int d2 = 0; d2 < D / 2; ++d2) {  // fully unrolled: m[] stays in registers
                const float x0 = bf_lo(m[d2]), x1 = bf_hi(m[d2]);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 cc = *reinterpret_cast<const float2*>(c + u * D + 2 * d2);
                    const float y0 = x0 - cc.x;
                    acc[u] = __fmaf_rn(y0, y0, acc[u]);
                    const float y1 = x1 - cc.y;
                    acc[u] = __fmaf_rn(y1, y1, acc[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if ((c0 + j + u) == 0 || acc[u] < best) {
                    best = acc[u];
                    arg = c0 + j + u;
                }
            }
        }
        for (; j < nc; ++j) {
            float acc = 0.f;
            const float* c = cs + j * D;
#pragma unroll
            for (int d2 = 0; d2 < D / 2; ++d2) {
                const float2 cc = *reinterpret_cast<const float2*>(c + 2 * d2);
                const float y0 = bf_lo(m[d2]) - cc.x;
                acc = __fmaf_rn(y0, y0, acc);
                const float y1 = bf_hi(m[d2]) - cc.y;
                acc = __fmaf_rn(y1, y1, acc);
            }
            if ((c0 + j) == 0 || acc < best) {
                best = acc;
                arg = c0 + j;
            }
        }
    }
    if (live) p.assign[uf * p.Pmax + pg] = arg;
}

// ---------------------------------------------------------------------------
// the two-level selection of one rescored unit
struct SelLayout {
    size_t qs, cscore, cbin, chosen, bits, wpre, cand, pscore, pbin, selpos, ts, total;
};
__host__ __device__ inline size_t c_align(size_t n) { return (n + 15) & ~static_cast<size_t>(15); }
__host__ __device__ inline SelLayout sel_layout(int D, int G, int Pmax, int Cmax, int K, int M)
{
    SelLayout l{};
    const int words = (Pmax + 31) / 32;
    l.qs = 0;
    l.cscore = c_align(l.qs + size_t(G) * D * 2);
    l.cbin = c_align(l.cscore + size_t(Cmax) * 4);
    l.chosen = c_align(l.cbin + size_t(Cmax) * 2);
    l.bits = c_align(l.chosen + size_t(M < Cmax ? M : Cmax) * 4);
    l.wpre = c_align(l.bits + size_t(words) * 4);
    l.cand = c_align(l.wpre + size_t(words) * 4);
    l.pscore = c_align(l.cand + size_t(Pmax) * 4);
    l.pbin = c_align(l.pscore + size_t(Pmax) * 4);
    l.selpos = c_align(l.pbin + size_t(Pmax) * 2);
    l.ts = c_align(l.selpos + size_t(K < Pmax ? K : Pmax) * 4);
    l.total = c_align(l.ts + sizeof(BlockTopkShared<kSelThreads>));
    return l;
}

// q_g . row over the group, reduced by sum (MODE 0) or max (MODE 1), by one warp: lane l takes channels
// [l*kCh, (l+1)*kCh); the row is D bf16 at `row` (global), the group G rows of D bf16 at `qs` (shared)
template <int D, int MODE>
__device__ __forceinline__ float warp_group_dot(const kvmm_bf16* row, const uint16_t* qs, int G, int lane)
{
    constexpr int kCh = D / 32;
    float r[kCh];
    if constexpr (kCh == 4) {
        const uint2 v = *reinterpret_cast<const uint2*>(row + lane * kCh);
        r[0] = bf_lo(v.x);
        r[1] = bf_hi(v.x);
        r[2] = bf_lo(v.y);
        r[3] = bf_hi(v.y);
    } else {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(row + lane * kCh);
        r[0] = bf_lo(v);
        r[1] = bf_hi(v);
    }
    float out = MODE == 0 ? 0.f : -FLT_MAX;
    for (int g = 0; g < G; ++g) {
        const uint16_t* qg = qs + g * D + lane * kCh;
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < kCh; ++c) s = fmaf(__uint_as_float(static_cast<uint32_t>(qg[c]) << 16), r[c], s);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(kFullMask, s, o);
        out = MODE == 0 ? out + s : fmaxf(out, s);
    }
    return out;
}

template <int D, int MODE>
__global__ void __launch_bounds__(kSelThreads) centroid_select_kernel(const CentroidParams p)
{
    extern __shared__ __align__(16) uint8_t ssm[];
    __shared__ int32_t wsum[kSelWarps];
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait_then_release();
    if (p.rescore_mask != nullptr && p.rescore_mask[p.layer * p.Hkv + h] == 0) return;  // keeps its selection
    const SelLayout lay = sel_layout(D, p.G, p.Pmax, p.Cmax, p.K, p.M);
    uint16_t* qs = reinterpret_cast<uint16_t*>(ssm + lay.qs);
    float* cscore = reinterpret_cast<float*>(ssm + lay.cscore);
    int16_t* cbin = reinterpret_cast<int16_t*>(ssm + lay.cbin);
    int32_t* chosen = reinterpret_cast<int32_t*>(ssm + lay.chosen);
    uint32_t* bits = reinterpret_cast<uint32_t*>(ssm + lay.bits);
    int32_t* wpre = reinterpret_cast<int32_t*>(ssm + lay.wpre);
    int32_t* cand = reinterpret_cast<int32_t*>(ssm + lay.cand);
    float* pscore = reinterpret_cast<float*>(ssm + lay.pscore);
    int16_t* pbin = reinterpret_cast<int16_t*>(ssm + lay.pbin);
    int32_t* selpos = reinterpret_cast<int32_t*>(ssm + lay.selpos);
    auto& ts = *reinterpret_cast<BlockTopkShared<kSelThreads>*>(ssm + lay.ts);

    const size_t uf = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
    const size_t ou = static_cast<size_t>(b) * p.Hkv + h;  // row of the [B][Hkv] outputs
    const int P = centroid_unit_pages(p, b, h == 0);
    const int n_c = (P + p.R - 1) / p.R;
    const int words = (P + 31) / 32;
    const int* off = p.member_off + uf * (p.Cmax + 1);
    const int* mem = p.members + uf * p.Pmax;

    // the query group, and an empty page bitmap
    const uint32_t* qsrc = reinterpret_cast<const uint32_t*>(p.q + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * p.G) * D);
    for (int i = tid; i < p.G * D / 2; i += kSelThreads) reinterpret_cast<uint32_t*>(qs)[i] = qsrc[i];
    for (int i = tid; i < words; i += kSelThreads) bits[i] = 0u;
    __syncthreads();
    // 1. the centroids' scores (a warp a centroid)
    for (int j = warp; j < n_c; j += kSelWarps) {
        const float s = warp_group_dot<D, MODE>(p.cent + (uf * p.Cmax + j) * D, qs, p.G, lane);
        if (lane == 0) {
            cscore[j] = s;
            if (p.centroid_scores_out) p.centroid_scores_out[ou * p.Cmax + j] = s;
        }
    }
    __syncthreads();
    // 2. the M best centroids, ascending
    const int nm = block_topk<kSelThreads>(nullptr, n_c, p.M, chosen, cscore, cbin, ts);
    // 3. their pages, marked in the bitmap, then compacted in page order
    for (int i = warp; i < nm; i += kSelWarps) {
        const int j = chosen[i];
        int k0 = off[j], k1 = off[j + 1];
        if (k0 < 0 || k1 < k0 || k1 > P) {  // not the member lists of this unit's build
            if (lane == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
            continue;
        }
        for (int k = k0 + lane; k < k1; k += 32) {
            const int pg = mem[k];
            if (pg >= 0 && pg < P)
                atomicOr(&bits[pg >> 5], 1u << (pg & 31));
            else
                report(p.err, KVMM_ERR_OUT_OF_RANGE);
        }
    }
    __syncthreads();
    for (int i = tid; i < words; i += kSelThreads) wpre[i] = __popc(bits[i]);
    __syncthreads();
    block_inclusive_scan<kSelThreads>(wpre, words, wsum);  // wpre[i] = candidates in words 0 .. i
    const int n = words ? wpre[words - 1] : 0;
    for (int i = tid; i < words; i += kSelThreads) {
        uint32_t w = bits[i];
        int at = wpre[i] - __popc(w);
        while (w) {
            const int bit = __ffs(w) - 1;
            cand[at++] = i * 32 + bit;
            w &= w - 1u;
        }
    }
    __syncthreads();
    // 4. the candidates' mean-key scores (a warp a page)
    for (int i = warp; i < n; i += kSelWarps) {
        const int pg = cand[i];
        const float s = warp_group_dot<D, MODE>(p.mean + (uf * p.Pmax + pg) * D, qs, p.G, lane);
        if (lane == 0) {
            pscore[i] = s;
            if (p.scores_out) p.scores_out[ou * p.Pmax + pg] = s;
        }
    }
    __syncthreads();
    // 5. the K best candidates (positions ascending = pages ascending)
    const int cnt = block_topk<kSelThreads>(nullptr, n, p.K, selpos, pscore, pbin, ts);
    for (int i = tid; i < cnt; i += kSelThreads) p.sel_idx[uf * p.Kmax + i] = cand[selpos[i]];
    if (tid == 0) p.sel_cnt[uf] = cnt;
}

template <int D>
cudaError_t build_for(const CentroidParams& p, int n_iter, cudaStream_t stream)
{
    static thread_local int dev_u = -1;
    static thread_local size_t bytes_u = 0;
    const size_t usmem = (static_cast<size_t>((p.Cmax + 1 + 3) & ~3) + p.Pmax) * sizeof(int32_t);
    cudaError_t e = allow_smem(centroid_update_kernel<D>, usmem, dev_u, bytes_u);
    if (e != cudaSuccess) return e;
    const dim3 ugrid(static_cast<unsigned>(p.Hkv), static_cast<unsigned>(p.B));
    const dim3 agrid(static_cast<unsigned>((p.Pmax + kAsgThreads - 1) / kAsgThreads), static_cast<unsigned>(p.Hkv),
                     static_cast<unsigned>(p.B));
    e = launch_pdl(centroid_update_kernel<D>, ugrid, dim3(kUpdThreads), usmem, stream, p, 1);
    for (int it = 0; it < n_iter && e == cudaSuccess; ++it) {
        e = launch_pdl(centroid_assign_kernel<D>, agrid, dim3(kAsgThreads), 0, stream, p);
        if (e == cudaSuccess) e = launch_pdl(centroid_update_kernel<D>, ugrid, dim3(kUpdThreads), usmem, stream, p, 0);
    }
    return e;
}

template <int D, int MODE>
cudaError_t select_for(const CentroidParams& p, cudaStream_t stream)
{
    static thread_local int dev_s = -1;
    static thread_local size_t bytes_s = 0;
    const size_t smem = sel_layout(D, p.G, p.Pmax, p.Cmax, p.K, p.M).total;
    cudaError_t e = allow_smem(centroid_select_kernel<D, MODE>, smem, dev_s, bytes_s);
    if (e != cudaSuccess) return e;
    return launch_pdl(centroid_select_kernel<D, MODE>, dim3(static_cast<unsigned>(p.Hkv), static_cast<unsigned>(p.B)),
                      dim3(kSelThreads), smem, stream, p);
}

}  // namespace

size_t centroid_select_smem(int D, int G, int Pmax, int Cmax, int K, int M)
{
    return sel_layout(D, G, Pmax, Cmax, K, M).total;
}

size_t centroid_update_smem(int Pmax, int Cmax)
{
    return (static_cast<size_t>((Cmax + 1 + 3) & ~3) + Pmax) * sizeof(int32_t);
}

cudaError_t launch_centroid_build(const CentroidParams& p, int n_iter, cudaStream_t stream)
{
    return p.D == 128 ? build_for<128>(p, n_iter, stream) : build_for<64>(p, n_iter, stream);
}

cudaError_t launch_centroid_select(const CentroidParams& p, int group_reduce, cudaStream_t stream)
{
    if (p.D == 128) return group_reduce ? select_for<128, 1>(p, stream) : select_for<128, 0>(p, stream);
    return group_reduce ? select_for<64, 1>(p, stream) : select_for<64, 0>(p, stream);
}

}  // namespace kvmm
