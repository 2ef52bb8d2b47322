// score_topk.cu -- MinMax page scoring and exact top-K page selection.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 2. MinMax-metadata page
// scoring": the query and each page's per-channel key bounds give the
// largest dot product the page can produce; the top-K pages are kept per
// (layer, KV head).  KVDrive, "Background and key observations": Quest
// multiplies the query with the channel-wise key min and max.
//
// Score of page p for query head g:  s_g(p) = sum_d max(q_gd*min_d, q_gd*max_d).
// Since max(q*m, q*M) = min(q,0)*m + max(q,0)*M, and min(q,0), max(q,0) are
// exact bf16 values, s_g(p) is the dot product of the page's [min | max] row
// (2D bf16) with the head's weight row [min(q_g,0) | max(q_g,0)] (2D bf16):
// bf16 x bf16 products are exact in fp32.  For 16 pages and the G <= 8 heads
// of a KV head that is one [16 x 2D] x [2D x 8] product on the tensor cores
// (mma.sync m16n8k16, fp32 accumulate); the unit's score is the sum (or, with
// group_reduce = 1, the max) over the real heads of each row.
//
// page_score_topk runs two kernels:
//  1. score_pages_kernel -- a persistent, warp-specialised stream over the
//     metadata (HBM bound, 2D*2 bytes per page).  Work items are chunks of
//     kChunk pages of one unit; each CTA takes a contiguous run of items, so
//     it rebuilds a unit's weight fragments only when the unit changes.  A
//     producer warp keeps kStages chunks (and the unit's query group) in
//     flight with 1-D bulk copies (TMA) on full/empty mbarriers; each
//     consumer warp scores 16 pages of a chunk.
//  2. select_topk_kernel -- one 512-thread CTA per rescored unit selects the
//     top K of the unit's P scores exactly (block_topk, topk_block.cuh: a
//     binned pass with an exact rank of the threshold bin, or a radix
//     select for degenerate inputs) and writes them in ascending page order.
// Both are launched with programmatic dependent launch so each is scheduled
// while its predecessor drains.
#include <cfloat>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "topk_block.cuh"

namespace kvmm {
namespace {

#ifndef KVMM_SCORE_WARPS
#define KVMM_SCORE_WARPS 4
#endif
#ifndef KVMM_SCORE_STAGES
#define KVMM_SCORE_STAGES 3
#endif

constexpr int kConsumerWarps = KVMM_SCORE_WARPS;
constexpr int kScoreThreads = kConsumerWarps * 32 + 32;  // + one producer warp
constexpr int kChunk = 16 * kConsumerWarps;               // pages per work item, 16 per consumer warp
constexpr int kStages = KVMM_SCORE_STAGES;
constexpr int kQBytes = 8 * 128 * 2;                      // largest query group (G <= 8, D <= 128)

constexpr int kTopkThreads = 512;

__host__ __device__ constexpr int stage_meta_bytes(int D) { return kChunk * 4 * D; }
__host__ __device__ constexpr int stage_bytes(int D) { return stage_meta_bytes(D) + kQBytes; }


// per 16-bit half: keep negative values (min(x, 0)) or positive ones (max(x, 0))
__device__ __forceinline__ uint32_t bf16x2_min0(uint32_t w)
{
    const uint32_t neg = ((w >> 15) & 0x00010001u) * 0xffffu;
    return w & neg;
}
__device__ __forceinline__ uint32_t bf16x2_max0(uint32_t w)
{
    const uint32_t neg = ((w >> 15) & 0x00010001u) * 0xffffu;
    return w & ~neg;
}

// pages of sequence `seq_len[b]` clamped to the table, reporting overflow once
__device__ __forceinline__ int unit_pages(const ScoreParams& p, int b, bool report_overflow)
{
    int seq = p.seq_len[b];
    const int cap = p.Pmax * p.T;
    if (seq < 0 || seq > cap) {
        if (report_overflow) report(p.err, KVMM_ERR_OUT_OF_RANGE);
        seq = seq < 0 ? 0 : cap;
    }
    return (seq + p.T - 1) / p.T;
}

// ---------------------------------------------------------------------------
// KIND 0: a page's row is its [min | max] key bounds (2D channels), weighted by [min(q,0) | max(q,0)];
// KIND 1: a page's row is its mean key (D channels), weighted by q (KVDrive's mean-key representative).
template <int D, int MODE, int KIND>
__global__ void __launch_bounds__(kScoreThreads) score_pages_kernel(const ScoreParams p)
{
    constexpr int kRowCh = KIND == 0 ? 2 * D : D;  // channels of a page's row
    constexpr int kRowBytes = 2 * kRowCh;
    constexpr int kRowChunks = kRowCh / 8;         // 16-byte chunks in a row
    constexpr int kR = kRowChunks / 4;             // chunk groups: lane tig takes chunk 4r + tig
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full_bar[kStages];
    __shared__ uint64_t empty_bar[kStages];
    __shared__ int4 info[kStages];  // {workspace unit, first page, pages (0 = skip), -}

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int gid = lane >> 2, tig = lane & 3;
    const int units = p.B * p.Hkv;
    const int chunks = (p.Pmax + kChunk - 1) / kChunk;
    const long long total = static_cast<long long>(units) * chunks;
    const int item0 = static_cast<int>(total * blockIdx.x / gridDim.x);
    const int item1 = static_cast<int>(total * (blockIdx.x + 1) / gridDim.x);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait_then_release();  // metadata and queries may come from the previous kernel

    if (warp == kConsumerWarps) {
        // ---- producer ------------------------------------------------------
        if (lane == 0) {
            for (int item = item0, k = 0; item < item1; ++item, ++k) {
                const int s = k % kStages;
                if (k >= kStages && !mbar_wait_bounded(&empty_bar[s], ((k / kStages) - 1) & 1))
                    report(p.err, KVMM_ERR_TIMEOUT);
                const int wunit = item / chunks;
                const int chunk = item - wunit * chunks;
                const int b = wunit / p.Hkv, h = wunit - b * p.Hkv;
                const int page0 = chunk * kChunk;
                int npg = 0;
                if (p.rescore_mask == nullptr || p.rescore_mask[p.layer * p.Hkv + h] != 0) {
                    const int P = unit_pages(p, b, chunk == 0 && h == 0);
                    npg = min(kChunk, P - page0);
                    if (npg < 0) npg = 0;
                }
                info[s] = make_int4(wunit, page0, npg, 0);
                if (npg > 0) {
                    uint8_t* st = smem + static_cast<size_t>(s) * stage_bytes(D);
                    const size_t unit = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
                    const uint32_t mbytes = static_cast<uint32_t>(npg) * kRowBytes;
                    const uint32_t qbytes = static_cast<uint32_t>(p.G) * D * 2;
                    mbar_arrive_expect_tx(&full_bar[s], mbytes + qbytes);
                    bulk_copy_g2s(st, p.meta + (unit * p.Pmax + page0) * kRowCh, mbytes, &full_bar[s]);
                    bulk_copy_g2s(st + stage_meta_bytes(D),
                                  p.q + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * p.G) * D,
                                  qbytes, &full_bar[s]);
                } else {
                    mbar_arrive(&full_bar[s]);  // nothing to copy: consumers skip the item
                }
            }
        }
        return;
    }

    // ---- consumers: warp w scores pages [16w, 16w + 16) of each chunk ------
    uint32_t wf[kR][4];  // weight B fragments of head gid: chunk 4r + tig of [min(q,0) | max(q,0)]
    int cached_unit = -1;
    const bool real_head = gid < p.G;
    for (int item = item0, k = 0; item < item1; ++item, ++k) {
        const int s = k % kStages;
        if (!mbar_wait_bounded(&full_bar[s], (k / kStages) & 1) && lane == 0) report(p.err, KVMM_ERR_TIMEOUT);
        const int4 inf = info[s];
        const int npg = inf.z;
        const uint8_t* st = smem + static_cast<size_t>(s) * stage_bytes(D);
        if (npg > 0 && inf.x != cached_unit) {
            const uint8_t* qs = st + stage_meta_bytes(D) + gid * (2 * D);
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const int cc = 4 * r + tig;                 // chunk of the row
                const int qc = cc % (D / 8);                // source chunk of q
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (real_head) v = ld_shared_v4(qs + 16 * qc);
                if (KIND == 1) {  // mean key: the query itself
                    wf[r][0] = v.x;
                    wf[r][1] = v.y;
                    wf[r][2] = v.z;
                    wf[r][3] = v.w;
                } else {
                    const bool is_max = cc >= D / 8;
                    wf[r][0] = is_max ? bf16x2_max0(v.x) : bf16x2_min0(v.x);
                    wf[r][1] = is_max ? bf16x2_max0(v.y) : bf16x2_min0(v.y);
                    wf[r][2] = is_max ? bf16x2_max0(v.z) : bf16x2_min0(v.z);
                    wf[r][3] = is_max ? bf16x2_max0(v.w) : bf16x2_min0(v.w);
                }
            }
            cached_unit = inf.x;
        }
        const int pg0 = warp * 16;
        if (pg0 < npg) {
            // C[page][head] over this warp's 16 pages: rows gid and gid + 8
            const uint8_t* ra = st + static_cast<size_t>(pg0 + gid) * kRowBytes;
            const uint8_t* rb = ra + 8 * kRowBytes;
            // four independent accumulation chains (even / odd r, low / high half of the chunk); the scoring
            // kernels of every path sum them in this same order, so their scores agree bit for bit
            float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
            float c3[4] = {0.f, 0.f, 0.f, 0.f}, c4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const uint4 ka = ld_shared_v4(ra + 16 * (4 * r + tig));
                const uint4 kb = ld_shared_v4(rb + 16 * (4 * r + tig));
                mma_bf16_16816((r & 1) ? c3 : c, ka.x, kb.x, ka.y, kb.y, wf[r][0], wf[r][1]);
                mma_bf16_16816((r & 1) ? c4 : c2, ka.z, kb.z, ka.w, kb.w, wf[r][2], wf[r][3]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) c[i] = (c[i] + c3[i]) + (c2[i] + c4[i]);
            // c: [page gid][head 2tig], [gid][2tig+1], [gid+8][2tig], [gid+8][2tig+1]
            float s_lo, s_hi;
            if (MODE == 0) {
                s_lo = c[0] + c[1];
                s_hi = c[2] + c[3];
                s_lo += __shfl_xor_sync(kFullMask, s_lo, 1);
                s_hi += __shfl_xor_sync(kFullMask, s_hi, 1);
                s_lo += __shfl_xor_sync(kFullMask, s_lo, 2);
                s_hi += __shfl_xor_sync(kFullMask, s_hi, 2);
            } else {
                const bool h0 = 2 * tig < p.G, h1 = 2 * tig + 1 < p.G;
                s_lo = fmaxf(h0 ? c[0] : -FLT_MAX, h1 ? c[1] : -FLT_MAX);
                s_hi = fmaxf(h0 ? c[2] : -FLT_MAX, h1 ? c[3] : -FLT_MAX);
                s_lo = fmaxf(s_lo, __shfl_xor_sync(kFullMask, s_lo, 1));
                s_hi = fmaxf(s_hi, __shfl_xor_sync(kFullMask, s_hi, 1));
                s_lo = fmaxf(s_lo, __shfl_xor_sync(kFullMask, s_lo, 2));
                s_hi = fmaxf(s_hi, __shfl_xor_sync(kFullMask, s_hi, 2));
            }
            if (tig == 0) {
                const size_t base = static_cast<size_t>(inf.x) * p.Pmax + inf.y + pg0;
                if (pg0 + gid < npg) {
                    p.scores_ws[base + gid] = s_lo;
                    if (p.scores_out) p.scores_out[base + gid] = s_lo;
                }
                if (pg0 + gid + 8 < npg) {
                    p.scores_ws[base + gid + 8] = s_hi;
                    if (p.scores_out) p.scores_out[base + gid + 8] = s_hi;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);  // the stage may be refilled
    }
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTopkThreads) select_topk_kernel(const ScoreParams p)
{
    extern __shared__ __align__(16) uint8_t tsm[];
    __shared__ BlockTopkShared<kTopkThreads> ts;
    const int h = blockIdx.x;
    const int b = blockIdx.y;
    pdl_wait_then_release();  // the scores are written by the scoring kernel

    if (p.rescore_mask != nullptr && p.rescore_mask[p.layer * p.Hkv + h] == 0) return;
    const int P = unit_pages(p, b, false);
    const size_t unit = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
    float* sc = reinterpret_cast<float*>(tsm);                                           // [P]
    int16_t* bin = reinterpret_cast<int16_t*>(tsm + static_cast<size_t>(p.Pmax) * 4);  // [P]
    const int n = block_topk<kTopkThreads>(p.scores_ws + static_cast<size_t>(b * p.Hkv + h) * p.Pmax, P, p.K,
                                           p.sel_idx + unit * p.Kmax, sc, bin, ts);
    if (threadIdx.x == 0) p.sel_cnt[unit] = n;
}

// one opt-in cache for the (single) selection kernel, shared by every launcher
cudaError_t allow_topk_smem(size_t bytes)
{
    static thread_local int dev_cache = -1;
    static thread_local size_t bytes_cache = 0;
    return allow_smem(select_topk_kernel, bytes, dev_cache, bytes_cache);
}

template <int D, int MODE, int KIND = 0>
cudaError_t launch_score(const ScoreParams& p, cudaStream_t stream, bool with_select)
{
    static thread_local int dev_a = -1;
    static thread_local size_t bytes_a = 0;
    const size_t smem = static_cast<size_t>(kStages) * stage_bytes(D);
    cudaError_t e = allow_smem(score_pages_kernel<D, MODE, KIND>, smem, dev_a, bytes_a);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148, per_sm = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, score_pages_kernel<D, MODE, KIND>, kScoreThreads, smem);
    if (per_sm < 1) per_sm = 1;
    const long long items = static_cast<long long>(p.B) * p.Hkv * ((p.Pmax + kChunk - 1) / kChunk);
    const long long slots = static_cast<long long>(sms) * per_sm;
    const long long grid = items < slots ? items : slots;
    e = launch_pdl(score_pages_kernel<D, MODE, KIND>, dim3(static_cast<unsigned>(grid)), dim3(kScoreThreads), smem,
                   stream, p);
    if (e != cudaSuccess || !with_select) return e;
    const size_t ksmem = static_cast<size_t>(p.Pmax) * (sizeof(float) + sizeof(int16_t));
    e = allow_topk_smem(ksmem);
    if (e != cudaSuccess) return e;
    return launch_pdl(select_topk_kernel, dim3(p.Hkv, p.B), dim3(kTopkThreads), ksmem, stream, p);
}

}  // namespace

cudaError_t launch_score_topk(const ScoreParams& p, int group_reduce, cudaStream_t stream)
{
    if (p.D == 128)
        return group_reduce ? launch_score<128, 1>(p, stream, true) : launch_score<128, 0>(p, stream, true);
    return group_reduce ? launch_score<64, 1>(p, stream, true) : launch_score<64, 0>(p, stream, true);
}

cudaError_t launch_score_topk_mean(const ScoreParams& p, int group_reduce, cudaStream_t stream)
{
    if (p.D == 128)
        return group_reduce ? launch_score<128, 1, 1>(p, stream, true) : launch_score<128, 0, 1>(p, stream, true);
    return group_reduce ? launch_score<64, 1, 1>(p, stream, true) : launch_score<64, 0, 1>(p, stream, true);
}

cudaError_t launch_score_only(const ScoreParams& p, int group_reduce, cudaStream_t stream)
{
    if (p.D == 128)
        return group_reduce ? launch_score<128, 1>(p, stream, false) : launch_score<128, 0>(p, stream, false);
    return group_reduce ? launch_score<64, 1>(p, stream, false) : launch_score<64, 0>(p, stream, false);
}

// ---------------------------------------------------------------------------
// Library-owned scratch for page_score_topk_static_scratch: a fixed array in
// the module's device memory, so that call needs no workspace from its
// caller and allocates nothing.  Every GPU that loads the library holds these
// bytes until the process exits.  Layout as for a caller workspace: the
// scores of every unit of the layer.
namespace {
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
void* g_static_ptr[kMaxDevices] = {};
}  // namespace

cudaError_t static_scratch_for_current_device(void** ptr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (g_static_ptr[dev] == nullptr) {
        // first call on this device: resolve the array's device address (the
        // host-side name is only a stand-in for it)
        void* addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_static_ptr[dev] = addr;
    }
    *ptr = g_static_ptr[dev];
    return cudaSuccess;
}

}  // namespace kvmm
