// score_topk.cu -- MinMax page scoring and exact top-K page selection.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 2. MinMax-metadata page
// scoring": the query and each page's per-channel key bounds give the
// largest dot product the page can produce; the top-K pages are kept per
// (layer, KV head).  KVDrive, "Background and key observations": Quest
// multiplies the query with the channel-wise key min and max.
//
// Score of page p for query head g:  s_g(p) = sum_d max(q_gd*min_d, q_gd*max_d).
// Since max(q*m, q*M) = max(q,0)*M + min(q,0)*m, the group SUM is a single
// dot product of the page's [min | max] row (2D bf16) with the fixed weight
// row [sum_g min(q_g,0) | sum_g max(q_g,0)] (fp32): one FMA per bf16 read,
// the same real number as the definition up to fp32 rounding.  The MAX
// group mode keeps one weight row per query head.
//
// Work split (HBM bound, 2D*2 bytes of metadata per page): one CTA scores a
// chunk of kChunk pages of one unit, staged into shared memory by one
// bulk copy (TMA) on an mbarrier; a warp reduces 4 pages at a time with a
// transposed butterfly (6 shuffles per 4 pages).  Scores go to the
// workspace; the last CTA of a unit (atomic ticket, no spinning) selects the
// top-K with an exact 4-pass radix select on order-preserving keys and
// writes the pages in ascending order, ties resolved to the lower index.
#include <cfloat>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace kvmm {
namespace {

constexpr int kScoreThreads = 128;
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kChunk = 64;  // pages per CTA

__host__ __device__ constexpr int chunk_bytes(int D) { return kChunk * 4 * D; }

// float -> unsigned key with the same order
__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float dot8(const uint4& v, const float (&w)[8])
{
    float s = bf16_lo(v.x) * w[0];
    s = fmaf(bf16_hi(v.x), w[1], s);
    s = fmaf(bf16_lo(v.y), w[2], s);
    s = fmaf(bf16_hi(v.y), w[3], s);
    s = fmaf(bf16_lo(v.z), w[4], s);
    s = fmaf(bf16_hi(v.z), w[5], s);
    s = fmaf(bf16_lo(v.w), w[6], s);
    s = fmaf(bf16_hi(v.w), w[7], s);
    return s;
}

// Sum four per-lane partials (one per page load j) over groups of LPP lanes.
// Afterwards lane l holds the total of load j = 2*bit(LPP/2) + bit(LPP/4)
// of its group; it is valid where (l % (LPP/4)) == 0.
template <int LPP>
__device__ __forceinline__ float reduce4(const float (&v)[4], int lane)
{
    const bool up1 = lane & (LPP / 2);
    float k0 = up1 ? v[2] : v[0];
    float k1 = up1 ? v[3] : v[1];
    const float s0 = up1 ? v[0] : v[2];
    const float s1 = up1 ? v[1] : v[3];
    k0 += __shfl_xor_sync(kFullMask, s0, LPP / 2);
    k1 += __shfl_xor_sync(kFullMask, s1, LPP / 2);
    const bool up2 = lane & (LPP / 4);
    float k = up2 ? k1 : k0;
    const float s = up2 ? k0 : k1;
    k += __shfl_xor_sync(kFullMask, s, LPP / 4);
#pragma unroll
    for (int off = LPP / 8; off >= 1; off >>= 1) k += __shfl_xor_sync(kFullMask, k, off);
    return k;
}

struct TopkShared {
    int hist[256];
    int warp_tot[2][kScoreWarps];
    int digit;
    int remaining;
    int last;
};

template <int D, int MODE>
__global__ void __launch_bounds__(kScoreThreads) score_topk_kernel(const ScoreParams p)
{
    constexpr int LPP = D / 4;      // lanes per page (16 bytes each)
    constexpr int PPL = 32 / LPP;   // pages per warp-wide load
    constexpr int kWRows = MODE == 0 ? 1 : 8;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t bar;
    __shared__ __align__(16) float w_s[kWRows][2 * D];
    __shared__ TopkShared ts;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int chunk = blockIdx.x;
    const int h = blockIdx.y;
    const int b = blockIdx.z;

    if (p.rescore_mask != nullptr && p.rescore_mask[p.layer * p.Hkv + h] == 0) return;

    int seq = p.seq_len[b];
    const int cap = p.Pmax * p.T;
    if (seq > cap || seq < 0) {
        if (chunk == 0 && tid == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
        seq = seq < 0 ? 0 : cap;
    }
    const int P = (seq + p.T - 1) / p.T;
    const int n_chunks = (P + kChunk - 1) / kChunk;
    const size_t unit = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;  // table / meta / sel
    const int wunit = b * p.Hkv + h;                                            // workspace slot

    if (P == 0) {  // empty sequence: empty selection
        if (chunk == 0 && tid == 0) p.sel_cnt[unit] = 0;
        return;
    }
    if (chunk >= n_chunks) return;

    const int page0 = chunk * kChunk;
    const int npg = min(kChunk, P - page0);
    const kvmm_bf16* src = p.meta + (unit * p.Pmax + page0) * 2 * D;

    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {
        const uint32_t bytes = static_cast<uint32_t>(npg) * 4 * D;
        mbar_arrive_expect_tx(&bar, bytes);
        bulk_copy_g2s(smem, src, bytes, &bar);
    }

    // weight rows while the copy is in flight
    const kvmm_bf16* qb = p.q + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * p.G) * D;
    for (int d = tid; d < D; d += kScoreThreads) {
        if (MODE == 0) {
            float wn = 0.f, wx = 0.f;
            for (int g = 0; g < p.G; ++g) {
                const float x = __uint_as_float(static_cast<uint32_t>(qb[g * D + d]) << 16);
                wn += fminf(x, 0.f);
                wx += fmaxf(x, 0.f);
            }
            w_s[0][d] = wn;
            w_s[0][D + d] = wx;
        } else {
            for (int g = 0; g < kWRows; ++g) {
                const float x = g < p.G ? __uint_as_float(static_cast<uint32_t>(qb[g * D + d]) << 16) : 0.f;
                w_s[g][d] = fminf(x, 0.f);
                w_s[g][D + d] = fmaxf(x, 0.f);
            }
        }
    }
    __syncthreads();

    const int sub = lane % LPP;  // 16-byte column of the page row: [min | max]
    float w[kWRows][8];
#pragma unroll
    for (int g = 0; g < kWRows; ++g)
#pragma unroll
        for (int i = 0; i < 8; ++i) w[g][i] = w_s[g][8 * sub + i];

    const bool ok = __syncthreads_and(mbar_wait_bounded(&bar, 0)) != 0;  // block-uniform
    if (!ok && tid == 0) report(p.err, KVMM_ERR_TIMEOUT);

    float* scores_ws = p.scores_ws + static_cast<size_t>(wunit) * p.Pmax;
    float* scores_out = p.scores_out ? p.scores_out + static_cast<size_t>(wunit) * p.Pmax : nullptr;
    if (ok) {
        constexpr int kPagesPerIter = 4 * PPL;
        for (int base = warp * kPagesPerIter; base < npg; base += kScoreWarps * kPagesPerIter) {
            float part[kWRows][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int pg = base + j * PPL + lane / LPP;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (pg < npg) v = ld_shared_v4(smem + static_cast<size_t>(pg) * 4 * D + 16 * sub);
#pragma unroll
                for (int g = 0; g < kWRows; ++g) part[g][j] = dot8(v, w[g]);
            }
            float score;
            if (MODE == 0) {
                score = reduce4<LPP>(part[0], lane);
            } else {
                score = -FLT_MAX;
#pragma unroll
                for (int g = 0; g < kWRows; ++g) {
                    const float sg = reduce4<LPP>(part[g], lane);
                    if (g < p.G) score = fmaxf(score, sg);
                }
            }
            const int j = 2 * ((lane / (LPP / 2)) & 1) + ((lane / (LPP / 4)) & 1);
            const int pg = base + j * PPL + lane / LPP;
            if ((lane % (LPP / 4)) == 0 && pg < npg) {
                scores_ws[page0 + pg] = score;
                if (scores_out) scores_out[page0 + pg] = score;
            }
        }
    }

    // ---- last CTA of the unit selects -----------------------------------
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int ticket = atomicAdd(p.counters + wunit, 1);
        ts.last = (ticket == n_chunks - 1);
        if (ts.last) p.counters[wunit] = 0;  // ready for the next call
    }
    __syncthreads();
    if (!ts.last) return;
    __threadfence();

    int32_t* sel = p.sel_idx + unit * p.Kmax;
    const int K = p.K;
    if (K >= P) {
        for (int i = tid; i < P; i += kScoreThreads) sel[i] = i;
        if (tid == 0) p.sel_cnt[unit] = P;
        return;
    }

    // keys in shared memory when they fit the staging buffer, else re-read from L2
    const bool keys_in_smem = static_cast<size_t>(P) * 4 <= static_cast<size_t>(chunk_bytes(D));
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
    if (keys_in_smem) {
        for (int i = tid; i < P; i += kScoreThreads) keys[i] = order_key(__ldcg(scores_ws + i));
        __syncthreads();
    }
    auto key_at = [&](int i) -> uint32_t {
        return keys_in_smem ? keys[i] : order_key(__ldcg(scores_ws + i));
    };

    // radix select of the K-th largest key, 8 bits per pass from the top
    uint32_t prefix = 0, pmask = 0;
    int remaining = K;
    const int P_round = (P + kScoreThreads - 1) / kScoreThreads * kScoreThreads;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kScoreThreads) ts.hist[i] = 0;
        __syncthreads();
        for (int i = tid; i < P_round; i += kScoreThreads) {
            const uint32_t k = i < P ? key_at(i) : 0u;
            const bool cand = i < P && (k & pmask) == prefix;
            const unsigned active = __ballot_sync(kFullMask, cand);
            if (cand) {
                const uint32_t digit = (k >> shift) & 255u;
                const unsigned peers = __match_any_sync(active, digit);
                if (lane == __ffs(peers) - 1) atomicAdd(&ts.hist[digit], __popc(peers));
            }
        }
        __syncthreads();
        if (warp == 0) {
            // lane l covers bins 255-8l .. 248-8l, scanned from the top
            int c[8];
            int tot = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = ts.hist[255 - 8 * lane - j];
                tot += c[j];
            }
            int incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(kFullMask, incl, off);
                if (lane >= off) incl += v;
            }
            const int excl = incl - tot;
            const bool here = excl < remaining && remaining <= incl;
            if (here) {
                int acc = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (acc + c[j] >= remaining) {
                        ts.digit = 255 - 8 * lane - j;
                        ts.remaining = remaining - acc;
                        break;
                    }
                    acc += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(ts.digit) << shift;
        pmask |= 255u << shift;
        remaining = ts.remaining;
        __syncthreads();
    }
    const uint32_t thr = prefix;  // the K-th largest key; `remaining` of its ties are taken

    // emit in ascending page order: every key > thr, and the first `remaining` keys == thr
    int out_base = 0, eq_base = 0;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int t0 = 0; t0 < P; t0 += kScoreThreads) {
        const int i = t0 + tid;
        const uint32_t k = i < P ? key_at(i) : 0u;
        const bool gt = i < P && k > thr;
        const bool eq = i < P && k == thr;
        const unsigned eqb = __ballot_sync(kFullMask, eq);
        if (lane == 0) ts.warp_tot[0][warp] = __popc(eqb);
        __syncthreads();
        int eq_off = eq_base, eq_all = 0;
#pragma unroll
        for (int w2 = 0; w2 < kScoreWarps; ++w2) {
            const int t = ts.warp_tot[0][w2];
            if (w2 < warp) eq_off += t;
            eq_all += t;
        }
        const bool take = gt || (eq && eq_off + __popc(eqb & lt_mask) < remaining);
        const unsigned tb = __ballot_sync(kFullMask, take);
        if (lane == 0) ts.warp_tot[1][warp] = __popc(tb);
        __syncthreads();
        int out_off = out_base, out_all = 0;
#pragma unroll
        for (int w2 = 0; w2 < kScoreWarps; ++w2) {
            const int t = ts.warp_tot[1][w2];
            if (w2 < warp) out_off += t;
            out_all += t;
        }
        if (take) sel[out_off + __popc(tb & lt_mask)] = i;
        out_base += out_all;
        eq_base += eq_all;
        __syncthreads();
    }
    if (tid == 0) p.sel_cnt[unit] = K;
}

template <int D, int MODE>
cudaError_t launch_one(const ScoreParams& p, cudaStream_t stream)
{
    const int smem = chunk_bytes(D);
    const dim3 grid((p.Pmax + kChunk - 1) / kChunk, p.Hkv, p.B);
    score_topk_kernel<D, MODE><<<grid, kScoreThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_topk(const ScoreParams& p, int group_reduce, cudaStream_t stream)
{
    if (p.D == 128) return group_reduce ? launch_one<128, 1>(p, stream) : launch_one<128, 0>(p, stream);
    return group_reduce ? launch_one<64, 1>(p, stream) : launch_one<64, 0>(p, stream);
}

// ---------------------------------------------------------------------------
// Library-owned scratch for page_score_topk_static_scratch: a fixed array in
// the module's device memory, so that call needs no workspace from its
// caller and allocates nothing.  Every GPU that loads the library holds these
// bytes until the process exits.  Layout as for a caller workspace: the
// per-unit counters first, then the scores.
namespace {
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
void* g_static_ptr[kMaxDevices] = {};
}  // namespace

cudaError_t static_scratch_for_current_device(void** ptr, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (g_static_ptr[dev] == nullptr) {
        // first call on this device: resolve the array's device address (the
        // host-side name is only a stand-in) and zero the counters, which
        // every later call leaves at zero again
        void* addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_static_scratch);
        if (e != cudaSuccess) return e;
        e = cudaMemsetAsync(addr, 0, kStaticScratchCounterBytes, stream);
        if (e != cudaSuccess) return e;
        g_static_ptr[dev] = addr;
    }
    *ptr = g_static_ptr[dev];
    return cudaSuccess;
}

}  // namespace kvmm
