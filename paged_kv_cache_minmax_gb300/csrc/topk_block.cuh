// topk_block.cuh -- exact top-K page selection by one thread block.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 2. MinMax-metadata page
// scoring": the K highest-scoring pages of a (layer, KV head) are kept.
// Ties go to the lower page index; the K pages are emitted in ascending
// page order (the layout of sel_idx).
//
// One pass buckets the unit's P scores into kTopkBins bins between their
// minimum and maximum (the bin is monotone in the score), a suffix scan
// finds the bin holding the K-th largest score, the few scores in that bin
// are ranked exactly (value descending, page ascending), and an ordered
// compaction writes the winners; when every thread can hold its share of the
// scores in registers, all of this runs on registers (block_topk_reg).
// Degenerate inputs (a crowded threshold bin, a non-finite range) take an
// exact 4-pass radix select over order-preserving keys.  The selections are out-of-line
// functions: called once per unit, they would otherwise share register
// allocation and scheduling with the caller's streaming loops.  Used with 512 threads by the selection kernel and
// with the attention CTA's 128 threads when attention selects its own pages.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace kvmm {

constexpr int kTopkBins = 2048;
constexpr int kTopkCandMax = 1024;

template <int THREADS>
struct BlockTopkShared {
    static_assert(THREADS % 32 == 0 && kTopkBins % THREADS == 0 && THREADS <= kTopkBins,
                  "the bins are split evenly over the block's threads");
    static constexpr int kWarps = THREADS / 32;
    alignas(16) int hist[kTopkBins];
    int cand[kTopkCandMax];
    float wmin[kWarps];
    float wmax[kWarps];
    alignas(16) int wsum[kWarps];  // read whole, 16 bytes at a time, when kWarps is a multiple of 4
    int rhist[256];
    int ncand;
    int tb;
    int need;
    int cbin;
    int digit;
    int remaining;
};

// the sum of the per-warp counts ts.wsum[w] over the warps w with lo <= w < hi, every count read in one pass
// (16-byte loads when the warp count allows) instead of one dependent load a warp
template <int WARPS>
__device__ __forceinline__ int topk_wsum_range(const int* wsum, int lo, int hi)
{
    int s = 0;
    if constexpr (WARPS % 4 == 0) {
#pragma unroll
        for (int w = 0; w < WARPS; w += 4) {
            const int4 c = *reinterpret_cast<const int4*>(wsum + w);
            s += (w >= lo && w < hi ? c.x : 0) + (w + 1 >= lo && w + 1 < hi ? c.y : 0) +
                 (w + 2 >= lo && w + 2 < hi ? c.z : 0) + (w + 3 >= lo && w + 3 < hi ? c.w : 0);
        }
    } else {
#pragma unroll
        for (int w = 0; w < WARPS; ++w) s += w >= lo && w < hi ? wsum[w] : 0;
    }
    return s;
}

// The threads that run one selection: the whole CTA, or a group of N threads
// (whole warps) starting at thread FIRST that synchronises on named barrier BAR.
struct CtaGroup {
    static constexpr int kFirst = 0;
    __device__ static void sync() { __syncthreads(); }
};
template <int BAR, int FIRST, int N>
struct WarpGroup {
    static_assert(FIRST % 32 == 0 && N % 32 == 0, "whole warps");
    static constexpr int kFirst = FIRST;
    __device__ static void sync() { asm volatile("bar.sync %0, %1;" ::"r"(BAR), "r"(N) : "memory"); }
};

// float -> unsigned key with the same order
__device__ __forceinline__ uint32_t topk_order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// bin of score v in [0, kTopkBins): floor((v - mn) * scale), monotone in v.  The clamps make every
// input defined: a NaN score (unsupported input) lands in bin 0, where the ranking keeps the selection a
// valid one (K distinct pages), with no promise on which of the tied or NaN pages win.
__device__ __forceinline__ int topk_bin(float v, float mn, float scale)
{
    const float x = fminf(fmaxf((v - mn) * scale, 0.f), static_cast<float>(kTopkBins - 1));
    return static_cast<int>(x);
}

// the sum of N consecutive histogram bins from `h` (16-byte aligned when N is a multiple of 4: then in
// 16-byte loads, free of the bank conflicts a thread stride of N words gives 4-byte loads)
template <int N>
__device__ __forceinline__ int topk_bin_sum(const int* h)
{
    int sum = 0;
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int j = 0; j < N; j += 4) {
            const int4 w = *reinterpret_cast<const int4*>(h + j);
            sum += (w.x + w.y) + (w.z + w.w);
        }
    } else {
#pragma unroll
        for (int j = 0; j < N; ++j) sum += h[j];
    }
    return sum;
}

// the float of an order key
__device__ __forceinline__ float topk_key_float(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Clears what block_topk(..., range) expects cleared: the histogram, the winner bitmask and the
// candidate count.  A caller that knows the scores' range ahead calls it before the scores are
// complete (every thread of the group); the group syncs at its end.
template <int THREADS, class Group = CtaGroup>
__device__ __forceinline__ void block_topk_prepare(BlockTopkShared<THREADS>& ts)
{
    const int tid = static_cast<int>(threadIdx.x) - Group::kFirst;
    for (int i = tid; i < kTopkBins; i += THREADS) ts.hist[i] = 0;
    for (int i = tid; i < 256; i += THREADS) ts.rhist[i] = 0;
    if (tid == 0) ts.ncand = 0;
    Group::sync();
}

// Exact top-K over the P scores in sc[] by 4 radix passes; writes sel[0..K) ascending.
template <int THREADS, class Group = CtaGroup>
__device__ __noinline__ void block_radix_topk(const float* sc, int P, int K, int32_t* sel, BlockTopkShared<THREADS>& ts)
{
    constexpr int kWarps = THREADS / 32;
    const int tid = static_cast<int>(threadIdx.x) - Group::kFirst, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0, pmask = 0;
    int remaining = K;
    const int P_round = (P + THREADS - 1) / THREADS * THREADS;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += THREADS) ts.rhist[i] = 0;
        Group::sync();
        for (int i = tid; i < P_round; i += THREADS) {
            const uint32_t key = i < P ? topk_order_key(sc[i]) : 0u;
            const bool cand = i < P && (key & pmask) == prefix;
            const unsigned active = __ballot_sync(kFullMask, cand);
            if (cand) {
                const uint32_t digit = (key >> shift) & 255u;
                const unsigned peers = __match_any_sync(active, digit);
                if (lane == __ffs(peers) - 1) atomicAdd(&ts.rhist[digit], __popc(peers));
            }
        }
        Group::sync();
        if (warp == 0) {
            int c[8];
            int tot = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = ts.rhist[255 - 8 * lane - j];
                tot += c[j];
            }
            int incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int v = __shfl_up_sync(kFullMask, incl, off);
                if (lane >= off) incl += v;
            }
            const int excl = incl - tot;
            if (excl < remaining && remaining <= incl) {
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
        Group::sync();
        prefix |= static_cast<uint32_t>(ts.digit) << shift;
        pmask |= 255u << shift;
        remaining = ts.remaining;
        Group::sync();
    }
    const uint32_t thr = prefix;
    int out_base = 0, eq_base = 0;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int t0 = 0; t0 < P; t0 += THREADS) {
        const int i = t0 + tid;
        const uint32_t key = i < P ? topk_order_key(sc[i]) : 0u;
        const bool gt = i < P && key > thr;
        const bool eq = i < P && key == thr;
        const unsigned eqb = __ballot_sync(kFullMask, eq);
        if (lane == 0) ts.wsum[warp] = __popc(eqb);
        Group::sync();
        int eq_off = eq_base, eq_all = 0;
        for (int w2 = 0; w2 < kWarps; ++w2) {
            const int t = ts.wsum[w2];
            if (w2 < warp) eq_off += t;
            eq_all += t;
        }
        Group::sync();
        const bool take = gt || (eq && eq_off + __popc(eqb & lt_mask) < remaining);
        const unsigned tb = __ballot_sync(kFullMask, take);
        if (lane == 0) ts.wsum[warp] = __popc(tb);
        Group::sync();
        int out_off = out_base, out_all = 0;
        for (int w2 = 0; w2 < kWarps; ++w2) {
            const int t = ts.wsum[w2];
            if (w2 < warp) out_off += t;
            out_all += t;
        }
        if (take) sel[out_off + __popc(tb & lt_mask)] = i;
        out_base += out_all;
        eq_base += eq_all;
        Group::sync();
    }
}

// The same selection when every thread can hold its share of the scores in
// registers (P <= 8 * THREADS): thread t owns pages [8t, 8t + 8), reads them
// once, bins them and emits its winners in order itself.  The threshold bin's
// pages are ranked one per thread, as in block_topk, and marked in a bitmask
// (the radix histogram's space) that their owners read back.  Same bins, same
// threshold, same result.
template <int THREADS, class Group = CtaGroup>
__device__ __forceinline__ int block_topk_reg_body(const float* scores, int P, int K, int32_t* sel, float* sc,
                                                   BlockTopkShared<THREADS>& ts, const uint32_t* range)
{
    constexpr int kPer = 8;
    constexpr int kWarps = THREADS / 32;
    const int tid = static_cast<int>(threadIdx.x) - Group::kFirst;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int i0 = kPer * tid;

    // 1. this thread's scores, their range, an empty histogram.  From shared memory a thread's 8 consecutive
    //    scores are two 16-byte loads when they are aligned (eight 4-byte loads at a 32-byte stride would
    //    hit the same four banks 8 times)
    float v[kPer];
    if (scores == nullptr && i0 + kPer <= P && (reinterpret_cast<uintptr_t>(sc) & 15u) == 0u) {
        const float4 a = *reinterpret_cast<const float4*>(sc + i0);
        const float4 c = *reinterpret_cast<const float4*>(sc + i0 + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
    } else {
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int i = i0 + e;
            v[e] = i < P ? (scores != nullptr ? __ldcg(scores + i) : sc[i]) : 0.f;
        }
    }
    uint32_t* winbits = reinterpret_cast<uint32_t*>(ts.rhist);  // bit i: page i of the threshold bin wins
    static_assert(8 * THREADS / 32 <= 256, "the winner bitmask fits the radix histogram");
    float mn, mx;
    if (range != nullptr) {  // known range; block_topk_prepare has cleared the histogram and the bitmask
        mn = topk_key_float(range[0]);
        mx = topk_key_float(range[1]);
    } else {
        float lo = FLT_MAX, hi = -FLT_MAX;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            if (i0 + e < P) {
                if (scores != nullptr) sc[i0 + e] = v[e];  // the ranking and the radix path read them here
                lo = fminf(lo, v[e]);
                hi = fmaxf(hi, v[e]);
            }
        }
        for (int i = tid; i < kTopkBins; i += THREADS) ts.hist[i] = 0;
        for (int i = tid; i < 8 * THREADS / 32; i += THREADS) winbits[i] = 0u;
        if (tid == 0) ts.ncand = 0;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            lo = fminf(lo, __shfl_xor_sync(kFullMask, lo, off));
            hi = fmaxf(hi, __shfl_xor_sync(kFullMask, hi, off));
        }
        if (lane == 0) {
            ts.wmin[warp] = lo;
            ts.wmax[warp] = hi;
        }
        Group::sync();
        mn = ts.wmin[0];
        mx = ts.wmax[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            mn = fminf(mn, ts.wmin[w]);
            mx = fmaxf(mx, ts.wmax[w]);
        }
    }
    if (!(mx > mn)) {  // every score equal: the K lowest pages win the ties
        for (int i = tid; i < K; i += THREADS) sel[i] = i;
        Group::sync();
        return K;
    }
    const float scale = static_cast<float>(kTopkBins) / (mx - mn);
    if (!(scale < FLT_MAX)) {
        block_radix_topk<THREADS, Group>(sc, P, K, sel, ts);
        return K;
    }

    // 2. bins, monotone in the score
    int b[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
        b[e] = -1;
        if (i0 + e < P) {
            b[e] = topk_bin(v[e], mn, scale);
            atomicAdd(&ts.hist[b[e]], 1);
        }
    }
    Group::sync();

    // 3. the bin holding the K-th largest score: suffix sums over bins (a thread's bins stay in registers
    //    for the search)
    constexpr int kBinsPerThread = kTopkBins / THREADS;
    static_assert(kBinsPerThread % 4 == 0, "a thread's bins are whole 16-byte words");
    int hb[kBinsPerThread];
    int local = 0;
#pragma unroll
    for (int j = 0; j < kBinsPerThread; j += 4) {
        const int4 h4 = *reinterpret_cast<const int4*>(&ts.hist[kBinsPerThread * tid + j]);
        hb[j] = h4.x;
        hb[j + 1] = h4.y;
        hb[j + 2] = h4.z;
        hb[j + 3] = h4.w;
        local += (h4.x + h4.y) + (h4.z + h4.w);
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int x = __shfl_down_sync(kFullMask, incl, off);
        if (lane + off < 32) incl += x;
    }
    if (lane == 0) ts.wsum[warp] = incl;
    Group::sync();
    const int above = incl - local + topk_wsum_range<kWarps>(ts.wsum, warp + 1, kWarps);
    if (above < K && K <= above + local) {
        // the K-th largest score lies in this thread's bins: the highest bin j whose count together with the
        // counts above it reaches K (suffix sums, then predicated selects: no early exit, no indexing)
        int suf = above;  // scores in bins above j
        int tj = 0, tneed = 0, tcnt = 0;
#pragma unroll
        for (int j = kBinsPerThread - 1; j >= 0; --j) {
            if (suf < K && suf + hb[j] >= K) {
                tj = j;
                tneed = K - suf;
                tcnt = hb[j];
            }
            suf += hb[j];
        }
        ts.tb = kBinsPerThread * tid + tj;
        ts.need = tneed;
        ts.cbin = tcnt;
    }
    Group::sync();
    const int tb = ts.tb, need = ts.need, cbin = ts.cbin;
    if (cbin > kTopkCandMax) {  // crowded threshold bin: exact radix path
        block_radix_topk<THREADS, Group>(sc, P, K, sel, ts);
        return K;
    }

    uint32_t win = 0u;
    if (need == cbin) {
        // every score of the threshold bin wins (the common case: about one score a bin near the K-th): no
        // ranking
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            if (b[e] >= tb) win |= 1u << e;
    } else {
        // 4. rank the threshold bin's pages exactly (value descending, page ascending), one per thread
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            if (b[e] == tb) ts.cand[atomicAdd(&ts.ncand, 1)] = i0 + e;
        Group::sync();
        for (int t = tid; t < cbin; t += THREADS) {
            const int i = ts.cand[t];
            const float s = sc[i];
            int rank = 0;
            for (int j = 0; j < cbin; ++j) {
                const int i2 = ts.cand[j];
                const float s2 = sc[i2];
                rank += (s2 > s) || (s2 == s && i2 < i);
            }
            if (rank < need) atomicOr(&winbits[i >> 5], 1u << (i & 31));
        }
        Group::sync();
        const uint32_t tw = winbits[i0 >> 5] >> (i0 & 31);  // this thread's 8 pages share one word
#pragma unroll
        for (int e = 0; e < kPer; ++e)
            if (b[e] > tb || (b[e] == tb && ((tw >> e) & 1u))) win |= 1u << e;
    }

    // 5. ordered compaction: thread t's winners follow those of threads below t
    const int mine = __popc(win);
    int pre = mine;  // inclusive prefix within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int x = __shfl_up_sync(kFullMask, pre, off);
        if (lane >= off) pre += x;
    }
    if (lane == 31) ts.wsum[warp] = pre;
    Group::sync();
    int pos = pre - mine + topk_wsum_range<kWarps>(ts.wsum, 0, warp);
#pragma unroll
    for (int e = 0; e < kPer; ++e)
        if ((win >> e) & 1u) sel[pos++] = i0 + e;
    Group::sync();
    return K;
}

// the register path as a call (one copy of its code, however many call sites)
template <int THREADS, class Group = CtaGroup>
__device__ __noinline__ int block_topk_reg(const float* scores, int P, int K, int32_t* sel, float* sc,
                                           BlockTopkShared<THREADS>& ts, const uint32_t* range)
{
    return block_topk_reg_body<THREADS, Group>(scores, P, K, sel, sc, ts, range);
}

// Selects the top K of the P scores at `scores` (global memory, read through
// L2; or null when sc[] already holds them) into sel[] (shared or global
// memory) and returns the count, min(K, P).  sc (P floats) and bin (P int16)
// are shared-memory scratch.  Every thread of the group must call it; sel[]
// is complete for every thread of the group on return.  `range`, if not
// null, holds the order keys (topk_order_key) of the scores' minimum and
// maximum, and block_topk_prepare ran before: the selection then skips its
// own range pass.
template <int THREADS, class Group = CtaGroup>
__device__ __noinline__ int block_topk(const float* scores, int P, int K, int32_t* sel, float* sc, int16_t* bin,
                          BlockTopkShared<THREADS>& ts, const uint32_t* range = nullptr)
{
    constexpr int kWarps = THREADS / 32;
    const int tid = static_cast<int>(threadIdx.x) - Group::kFirst;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    if (K >= P) {
        for (int i = tid; i < P; i += THREADS) sel[i] = i;
        Group::sync();
        return P;
    }
    if (P <= 8 * THREADS) return block_topk_reg<THREADS, Group>(scores, P, K, sel, sc, ts, range);

    // 1. scores to shared memory (16 loads in flight per thread), their range, an empty histogram (a known
    //    range: block_topk_prepare has emptied it, and the scores are in sc[] already)
    constexpr int kBatch = 16;
    float lo = FLT_MAX, hi = -FLT_MAX;
    float mn, mx;
    if (range != nullptr && scores == nullptr) {
        mn = topk_key_float(range[0]);
        mx = topk_key_float(range[1]);
    } else {
        if (scores == nullptr) {
            for (int i = tid; i < P; i += THREADS) {
                lo = fminf(lo, sc[i]);
                hi = fmaxf(hi, sc[i]);
            }
        }
        for (int c0 = 0; scores != nullptr && c0 < P; c0 += THREADS * kBatch) {
            float v[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = c0 + j * THREADS + tid;
                v[j] = i < P ? __ldcg(scores + i) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int i = c0 + j * THREADS + tid;
                if (i < P) {
                    sc[i] = v[j];
                    lo = fminf(lo, v[j]);
                    hi = fmaxf(hi, v[j]);
                }
            }
        }
        for (int i = tid; i < kTopkBins; i += THREADS) ts.hist[i] = 0;
        if (tid == 0) ts.ncand = 0;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            lo = fminf(lo, __shfl_xor_sync(kFullMask, lo, off));
            hi = fmaxf(hi, __shfl_xor_sync(kFullMask, hi, off));
        }
        if (lane == 0) {
            ts.wmin[warp] = lo;
            ts.wmax[warp] = hi;
        }
        Group::sync();
        mn = ts.wmin[0];
        mx = ts.wmax[0];
        for (int w = 1; w < kWarps; ++w) {
            mn = fminf(mn, ts.wmin[w]);
            mx = fmaxf(mx, ts.wmax[w]);
        }
    }
    if (!(mx > mn)) {  // every score equal: the K lowest pages win the ties
        for (int i = tid; i < K; i += THREADS) sel[i] = i;
        Group::sync();
        return K;
    }
    const float scale = static_cast<float>(kTopkBins) / (mx - mn);
    if (!(scale < FLT_MAX)) {
        block_radix_topk<THREADS, Group>(sc, P, K, sel, ts);
        return K;
    }

    // 2. bucket every score: bin(s) = floor((s - mn) * scale) is monotone in s
    for (int i = tid; i < P; i += THREADS) {
        const int bi = topk_bin(sc[i], mn, scale);
        bin[i] = static_cast<int16_t>(bi);
        atomicAdd(&ts.hist[bi], 1);
    }
    Group::sync();

    // 3. the bin holding the K-th largest score: suffix sums over bins
    constexpr int kBinsPerThread = kTopkBins / THREADS;
    const int local = topk_bin_sum<kBinsPerThread>(ts.hist + kBinsPerThread * tid);
    int incl = local;  // inclusive suffix within the warp (lanes >= this one)
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_down_sync(kFullMask, incl, off);
        if (lane + off < 32) incl += v;
    }
    if (lane == 0) ts.wsum[warp] = incl;
    Group::sync();
    const int above = incl - local + topk_wsum_range<kWarps>(ts.wsum, warp + 1, kWarps);
    if (above < K && K <= above + local) {
        int acc = above;
        for (int j = kBinsPerThread - 1; j >= 0; --j) {
            const int bj = kBinsPerThread * tid + j;
            if (acc + ts.hist[bj] >= K) {
                ts.tb = bj;
                ts.need = K - acc;
                ts.cbin = ts.hist[bj];
                break;
            }
            acc += ts.hist[bj];
        }
    }
    Group::sync();
    const int tb = ts.tb, need = ts.need, cbin = ts.cbin;
    if (cbin > kTopkCandMax) {  // crowded threshold bin: exact radix path
        block_radix_topk<THREADS, Group>(sc, P, K, sel, ts);
        return K;
    }

    // 4. rank the threshold bin's scores exactly; mark the winners above every bin
    for (int i = tid; i < P; i += THREADS)
        if (bin[i] == tb) ts.cand[atomicAdd(&ts.ncand, 1)] = i;
    Group::sync();
    for (int t = tid; t < cbin; t += THREADS) {
        const int i = ts.cand[t];
        const float s = sc[i];
        int rank = 0;
        for (int j = 0; j < cbin; ++j) {
            const int i2 = ts.cand[j];
            const float s2 = sc[i2];
            rank += (s2 > s) || (s2 == s && i2 < i);
        }
        if (rank < need) bin[i] = static_cast<int16_t>(kTopkBins);
    }
    Group::sync();

    // 5. ordered compaction: thread t emits the winners among pages [t*m, t*m + m)
    const int m = (P + THREADS - 1) / THREADS;
    const int i0 = min(P, tid * m), i1 = min(P, i0 + m);
    int mine = 0;
    for (int i = i0; i < i1; ++i) mine += bin[i] > tb;
    int pre = mine;  // inclusive prefix within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(kFullMask, pre, off);
        if (lane >= off) pre += v;
    }
    if (lane == 31) ts.wsum[warp] = pre;
    Group::sync();
    int pos = pre - mine + topk_wsum_range<kWarps>(ts.wsum, 0, warp);
    for (int i = i0; i < i1; ++i)
        if (bin[i] > tb) sel[pos++] = i;
    Group::sync();
    return K;
}

// block_topk with its register path inlined at the call site (the general path stays a call): for a caller
// with a single call site on a latency-critical path, where the two calls' overhead shows
template <int THREADS, class Group = CtaGroup>
__device__ __forceinline__ int block_topk_inline(const float* scores, int P, int K, int32_t* sel, float* sc,
                                                 int16_t* bin, BlockTopkShared<THREADS>& ts,
                                                 const uint32_t* range = nullptr)
{
    if (K < P && P <= 8 * THREADS) return block_topk_reg_body<THREADS, Group>(scores, P, K, sel, sc, ts, range);
    return block_topk<THREADS, Group>(scores, P, K, sel, sc, bin, ts, range);
}

}  // namespace kvmm
