// fused_decode.cu -- one launch per layer: MinMax page scoring, exact top-K
// page selection and sparse GQA decode attention over the selected pages.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 2. MinMax-metadata page
// scoring": the query and each page's per-channel key bounds give an upper
// bound of the page's attention logits, and the top-K pages of every
// (layer, KV head) are kept; "Core method, 1. Stability-differentiated
// placement": decode attention then runs over those pages only;
// "System design, head-level block table": pages are found through
// [batch, layer, head, logical_block] and null entries are never read.
// The result equals page_score_topk followed by sparse_paged_decode_attn.
//
// Why one launch.  Per unit (batch, KV head) the three steps are a chain:
// all page scores, then the selection, then the attention over the chosen
// pages.  Run as separate kernels, every link of the chain drains and
// refills the whole GPU.  Here the chains of different units overlap.
//
// Design (sm_103a, one persistent CTA per SM, 6 warps), as a dataflow over
// three global queues in the workspace:
//   - Producer warp: takes score items (128 pages of one unit's [min | max]
//     metadata rows, units one after another) from a work counter, then
//     attention items (one of `splits` equal shares of one unit's selected
//     pages) from the ready queue, in the order units became ready.  It
//     stages the unit's query group and the item's bytes into per-consumer
//     rings with 1-D bulk copies (TMA) on full/empty mbarriers: a score
//     item gives each consumer warp one 32-page slot; an attention item's
//     pages are resolved through the selection and the block table, its
//     32-token steps go round robin to the consumer warps, and one merge
//     marker per warp closes it.
//   - 4 consumer warps: score slots on the tensor cores (mma.sync
//     m16n8k16, [16 pages x 2D] x [2D x 8 heads]); attention steps as
//     S^T = K Q^T, online softmax, O^T += V^T P^T (P as bf16 hi + lo).  At a
//     merge marker the four warps combine their softmax partials in shared
//     memory and write the item's partial (m, l, O) to the workspace; the
//     CTA that writes a unit's last partial (a ticket counter) combines all
//     of the unit's partials into out and lse.  The warp that scores a
//     unit's last piece (a ticket counter) puts the unit on the select queue.
//   - Selector warp: takes units from the select queue (any CTA's selector
//     takes the next unit), selects the top K of the unit's scores exactly
//     (the scores in registers as order-preserving keys, the K-th largest
//     found bit by bit), writes sel_idx / sel_cnt and puts the unit's
//     attention items on the ready queue.  Units that are not rescored put
//     theirs there when the producer meets their first score item.
//   Nothing waits on work that has not been handed out: a producer blocks
//   on the ready queue only after every score item is taken, and every
//   taken score item is scored without waiting on anything.  Every wait is
//   still bounded; on expiry the kernel sets KVMM_ERR_TIMEOUT, stops taking
//   work and leaves.  The last CTA to finish resets the queue counters, so
//   a workspace serves any number of launches without host-side resets.
//   One-launch path: up to 2048 pages per unit (64 keys per selector lane).
#include <cfloat>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace kvmm {
namespace {

constexpr int kCons = 4;                     // consumer warps
constexpr int kProdWarp = kCons;             // producer warp
constexpr int kSelWarp = kCons + 1;          // selector warp
constexpr int kPubWarp = kCons + 2;          // publisher warp
constexpr int kFThreads = (kCons + 3) * 32;
constexpr int kNotices = 32;                 // consumer -> publisher notice queue
constexpr int kRing = 3;                     // slots per consumer warp
constexpr int kQRing = 4;                    // staged query groups
constexpr int kPiece = 32;                   // score pages per slot
constexpr int kChunkPages = kPiece * kCons;  // pages per score item
constexpr int kStepTok = 32;                 // tokens per attention step
constexpr int kSelPer = 64;                  // selector keys per lane: up to 2048 pages
constexpr int kSelCand = 256;                // threshold candidates finished in shared memory

constexpr uint32_t kKindEnd = 0, kKindScore = 1, kKindAtt = 2, kKindMerge = 3;
constexpr uint32_t kFlagTicket = 4;

constexpr uint64_t kWaitNs = 1000000000ull;   // 1 s: far beyond any legitimate wait
constexpr uint64_t kAbortWaitNs = 1000000ull;  // once aborting, give up quickly

// control words of the workspace (after them: score tickets [U], attention
// tickets [U], select queue [U], ready queue [U * splits])
enum : int { kCtlScoreItems = 0, kCtlDone, kCtlSelHead, kCtlSelTail, kCtlRdyHead, kCtlRdyTail, kCtlAbort };

__host__ __device__ constexpr int slot_bytes(int D) { return 128 * D; }  // 32 rows of 4D bytes, or 32 tokens of K and V
__host__ __device__ constexpr int qentry_bytes(int D) { return 8 * D * 2; }
__host__ __device__ constexpr size_t fused_dyn_smem(int D)
{
    return size_t(kCons) * kRing * slot_bytes(D) + size_t(kQRing) * qentry_bytes(D) +
           size_t(kCons) * 8 * D * sizeof(float);
}

struct FusedShared {
    uint64_t full[kCons][kRing];
    uint64_t empty[kCons][kRing];
    uint64_t qfull[kQRing];
    uint64_t qempty[kQRing];
    uint64_t gbar;  // consumer-group barrier (kCons arrivals per use)
    int4 desc[kCons][kRing];
    float mm[kCons][8];
    float ml[kCons][8];
    float f[kCons][8];
    int abort_flag;
    int last;
    int nq[kNotices];  // notices to the publisher (0 = empty)
    int nq_head;
    int nq_tail;
    int cons_done;
    float pf[64][8];   // publisher: merge weights of a unit's partials
    int pphys[32];  // producer: compacted pages of an attention item
    int pnv[32];
    uint32_t cand[kSelCand];  // selector: keys sharing the threshold's high half
};

__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

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

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t keep_halves(uint32_t w, bool lo, bool hi)
{
    return w & ((lo ? 0x0000ffffu : 0u) | (hi ? 0xffff0000u : 0u));
}

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ int ld_volatile(const int* p) { return *reinterpret_cast<const volatile int*>(p); }
__device__ __forceinline__ void st_volatile(int* p, int v) { *reinterpret_cast<volatile int*>(p) = v; }

// pages of sequence b clamped to the table
__device__ __forceinline__ int seq_pages(const FusedParams& p, int b, int& seq, bool report_overflow)
{
    seq = p.seq_len[b];
    const int cap = p.Pmax * p.T;
    if (seq < 0 || seq > cap) {
        if (report_overflow) report(p.err, KVMM_ERR_OUT_OF_RANGE);
        seq = seq < 0 ? 0 : cap;
    }
    return (seq + p.T - 1) / p.T;
}

// wait (lane-level, bounded) until *q holds a non-zero entry; returns it, or 0 on time-out
__device__ __forceinline__ int wait_entry(const int32_t* q, const int* abort_flag)
{
    int e = ld_acquire_gpu(q);
    if (e != 0) return e;
    const uint64_t t0 = global_timer_ns();
    while ((e = ld_acquire_gpu(q)) == 0) {
        __nanosleep(100);
        if (global_timer_ns() - t0 > kWaitNs || ld_volatile(abort_flag) != 0) return 0;
    }
    return e;
}

// ---------------------------------------------------------------------------
// exact top-K of one unit's scores by one warp (selector)
//
// Lane l holds the order-preserving 32-bit keys of pages [64l, 64l + 64).
// The K-th largest key t is found bit by bit: first its high half, the
// largest h with count(key >= h << 16) >= K, by bisection over the
// registers; then its low half, by bisection over the keys whose high half
// is h, compacted into shared memory (over the registers again if there are
// more than kSelCand of them).  Every key above t and the first
// K - count(key > t) keys equal to t (lowest pages first) are written in
// ascending page order: pages are contiguous per lane, so an exclusive scan
// over the lanes places each lane's run.

__device__ __forceinline__ int warp_exclusive_scan(int v, int lane)
{
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(kFullMask, incl, off);
        if (lane >= off) incl += t;
    }
    return incl - v;
}

__device__ __forceinline__ int warp_sum(int v) { return static_cast<int>(__reduce_add_sync(kFullMask, static_cast<uint32_t>(v))); }

// count over the warp of the register keys >= c
__device__ __forceinline__ int count_ge(const uint32_t (&k)[kSelPer], uint32_t c)
{
    int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
    for (int j = 0; j < kSelPer; j += 4) {
        a0 += k[j] >= c ? 1 : 0;
        a1 += k[j + 1] >= c ? 1 : 0;
        a2 += k[j + 2] >= c ? 1 : 0;
        a3 += k[j + 3] >= c ? 1 : 0;
    }
    return warp_sum((a0 + a1) + (a2 + a3));
}

// sc: the unit's scores (16-byte aligned, readable up to P rounded up to 4)
__device__ int warp_topk(const float* sc, int P, int K, int32_t* sel, uint32_t* cand, int lane)
{
    if (K >= P) {
        for (int i = lane; i < P; i += 32) sel[i] = i;
        return P;
    }
    const int base = lane * kSelPer;
    uint32_t k[kSelPer];  // 0 past P: below the key of every finite score
#pragma unroll
    for (int j = 0; j < kSelPer / 4; ++j) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (base + 4 * j < P) v = __ldcg(reinterpret_cast<const float4*>(sc + base) + j);
        const int i = base + 4 * j;
        k[4 * j] = i < P ? order_key(v.x) : 0u;
        k[4 * j + 1] = i + 1 < P ? order_key(v.y) : 0u;
        k[4 * j + 2] = i + 2 < P ? order_key(v.z) : 0u;
        k[4 * j + 3] = i + 3 < P ? order_key(v.w) : 0u;
    }
    // bits above the highest one in which the smallest and largest key differ are common
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int j = 0; j < kSelPer; ++j) {
        hi = max(hi, k[j]);
        if (base + j < P) lo = min(lo, k[j]);
    }
    lo = __reduce_min_sync(kFullMask, lo);
    hi = __reduce_max_sync(kFullMask, hi);
    const uint32_t diff = (lo ^ hi) >> 16;
    int bit = diff == 0u ? -1 : 31 - __clz(diff);
    uint32_t th = bit < 0 ? (hi >> 16) : ((hi >> 16) & ~((2u << bit) - 1u));
    // 1. the high half of the K-th largest key
#pragma unroll 1
    for (; bit >= 0; --bit) {
        const uint32_t c = th | (1u << bit);
        if (count_ge(k, c << 16) >= K) th = c;
    }
    // 2. its low half, among the keys whose high half is th
    int above = 0, mine = 0;
#pragma unroll
    for (int j = 0; j < kSelPer; ++j) {
        above += (k[j] >> 16) > th ? 1 : 0;
        mine += (k[j] >> 16) == th ? 1 : 0;
    }
    above = warp_sum(above);
    const int ncand = warp_sum(mine);
    uint32_t tl = 0;
    if (ncand <= kSelCand) {
        int pos = warp_exclusive_scan(mine, lane);
#pragma unroll
        for (int j = 0; j < kSelPer; ++j)
            if ((k[j] >> 16) == th) cand[pos++] = k[j] & 0xffffu;
        __syncwarp();
#pragma unroll 1
        for (int b2 = 15; b2 >= 0; --b2) {
            const uint32_t c = tl | (1u << b2);
            int n = 0;
            for (int i = lane; i < ncand; i += 32) n += cand[i] >= c ? 1 : 0;
            if (above + warp_sum(n) >= K) tl = c;
        }
        __syncwarp();
    } else {
#pragma unroll 1
        for (int b2 = 15; b2 >= 0; --b2) {
            const uint32_t c = tl | (1u << b2);
            if (count_ge(k, (th << 16) | c) >= K) tl = c;
        }
    }
    const uint32_t thr = (th << 16) | tl;  // the K-th largest key
    // 3. every key above thr, then the first keys equal to it, in page order
    unsigned long long mgt = 0ull, meq = 0ull;
#pragma unroll
    for (int j = 0; j < kSelPer; ++j) {
        if (k[j] > thr) mgt |= 1ull << j;
        if (k[j] == thr) meq |= 1ull << j;
    }
    const int ngt = __popcll(mgt), neq = __popcll(meq);
    const int remaining = K - warp_sum(ngt);
    const int eq_before = warp_exclusive_scan(neq, lane);
    const int take_eq = max(0, min(neq, remaining - eq_before));
    int pos = warp_exclusive_scan(ngt + take_eq, lane);
    unsigned long long m = mgt | meq;
    int eq_taken = 0;
    while (m != 0ull) {
        const int j = __ffsll(static_cast<long long>(m)) - 1;
        m &= m - 1ull;
        if ((meq >> j) & 1ull) {
            if (eq_taken >= take_eq) continue;
            ++eq_taken;
        }
        if (pos < K) sel[pos] = base + j;
        ++pos;
    }
    return K;
}

// ---------------------------------------------------------------------------
template <int D, int T, int MODE>
__global__ void __launch_bounds__(kFThreads, 1) fused_decode_kernel(const FusedParams p)
{
    constexpr int kSlot = slot_bytes(D);
    constexpr int kPageBytes = T * D * 2;  // a page's K (or V) block
    constexpr int kPPS = kStepTok / T;     // pages per attention step
    constexpr int kMTiles = D / 16;
    constexpr int kR = (2 * D / 8) / 4;    // 16-byte chunk groups of a [min | max] row
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ FusedShared sh;

    uint8_t* rings = smem;
    uint8_t* qring = smem + size_t(kCons) * kRing * kSlot;
    float* mo = reinterpret_cast<float*>(qring + size_t(kQRing) * qentry_bytes(D));  // [kCons][8][D]

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int units = p.B * p.Hkv;
    const int S = p.splits;
    const int n_att = units * S;
    int32_t* ctl = p.ctrl;
    int32_t* score_cnt = p.ctrl + kCtrlHead;
    int32_t* att_cnt = score_cnt + units;
    int32_t* sel_q = att_cnt + units;  // units awaiting selection (unit + 1)
    int32_t* rdy_q = sel_q + units;    // attention items ready to run (item + 1)
    int32_t* sel_tail = ctl + kCtlSelTail;
    const size_t part_stride = 16 + 8 * size_t(D);

    if (tid == 0) {
        for (int w = 0; w < kCons; ++w)
            for (int s = 0; s < kRing; ++s) {
                mbar_init(&sh.full[w][s], 1);
                mbar_init(&sh.empty[w][s], 1);
            }
        for (int e = 0; e < kQRing; ++e) {
            mbar_init(&sh.qfull[e], 1);
            mbar_init(&sh.qempty[e], kCons);
        }
        mbar_init(&sh.gbar, kCons);
        sh.abort_flag = sh.last = 0;
        for (int i = 0; i < kNotices; ++i) sh.nq[i] = 0;
        sh.nq_head = sh.nq_tail = sh.cons_done = 0;
        fence_barrier_init();
    }
    pdl_launch_dependents();
    pdl_wait();  // every input may come from the preceding kernels
    __syncthreads();

    auto aborting = [&]() { return ld_volatile(&sh.abort_flag) != 0; };
    auto set_abort = [&]() {
        st_volatile(&sh.abort_flag, 1);
        report(p.err, KVMM_ERR_TIMEOUT);
    };
    // a wait by one lane
    auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
        if (mbar_wait_bounded(bar, parity, aborting() ? kAbortWaitNs : kWaitNs)) return true;
        set_abort();
        return false;
    };
    // a wait by every lane of a warp, with one outcome for the whole warp
    auto wait_bar_warp = [&](uint64_t* bar, uint32_t parity) {
        const bool ok = __all_sync(kFullMask, mbar_wait_bounded(bar, parity, aborting() ? kAbortWaitNs : kWaitNs));
        if (!ok && (threadIdx.x & 31) == 0) set_abort();
        return ok;
    };
    // the abort flag as one value for the whole warp
    auto aborting_warp = [&]() { return __shfl_sync(kFullMask, static_cast<int>(aborting()), 0) != 0; };
    // put the `S` attention items of unit wunit on the ready queue (one lane;
    // the caller has ordered the unit's selection before this point)
    auto publish_unit = [&](int wunit) {
        const int pos = atomicAdd(ctl + kCtlRdyTail, S);
        fence_acq_rel_gpu();
        for (int s = 0; s < S && pos + s < n_att; ++s) st_volatile(rdy_q + pos + s, wunit * S + s + 1);
    };
    // a consumer's notice to the publisher (one lane): +(unit + 1) for a scored
    // piece carrying a ticket, -(unit + 1) for an attention item's partial
    auto post_notice = [&](int code) {
        const int pos = atomicAdd(&sh.nq_tail, 1);
        const uint64_t t0 = global_timer_ns();
        while (pos - ld_volatile(&sh.nq_head) >= kNotices) {  // full: let the publisher drain
            __nanosleep(32);
            if (global_timer_ns() - t0 > kWaitNs || aborting()) {
                set_abort();
                return;
            }
        }
        __threadfence_block();
        st_volatile(&sh.nq[pos % kNotices], code);
    };

    if (warp == kProdWarp) {
        // ================= producer ========================================
        const int n_score = units * p.chunks;
        const int cw = lane >> 3;  // consumer warp this lane serves
        const int cc = lane & 7;   // its copy within a step: 0 K0, 1 V0, 2 K1, 3 V1
        const bool ctl_lane = cc == 0;  // the lane that posts warp cw's slots
        int kposted = 0;           // slots posted to warp cw
        int qseq = 0;
        const int G = p.G;
        const uint32_t qbytes = static_cast<uint32_t>(G) * D * 2;

        auto stage_q = [&](int b, int h, bool copy) {  // lane 0
            const int qe = qseq % kQRing;
            if (qseq >= kQRing) wait_bar(&sh.qempty[qe], ((qseq / kQRing) - 1) & 1);
            if (copy) {
                mbar_arrive_expect_tx(&sh.qfull[qe], qbytes);
                bulk_copy_g2s(qring + size_t(qe) * qentry_bytes(D),
                              p.q + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * G) * D, qbytes,
                              &sh.qfull[qe]);
            } else {
                mbar_arrive(&sh.qfull[qe]);
            }
        };
        // ctl lane: wait until warp cw's next slot is free; returns the slot
        auto take_slot = [&]() {
            const int s = kposted % kRing;
            if (kposted >= kRing) wait_bar(&sh.empty[cw][s], ((kposted / kRing) - 1) & 1);
            return s;
        };

        // ---- score items, from the work counter ----------------------------
        int item = 0;
        if (lane == 0) item = atomicAdd(ctl + kCtlScoreItems, 1);
        item = __shfl_sync(kFullMask, item, 0);
        while (item < n_score && !aborting_warp()) {
            int next = 0;
            if (lane == 0) next = atomicAdd(ctl + kCtlScoreItems, 1);  // used after this item: its latency overlaps
            const int wunit = item / p.chunks;
            const int chunk = item - wunit * p.chunks;
            const int b = wunit / p.Hkv, h = wunit - b * p.Hkv;
            const bool rescored = p.rescore_mask == nullptr || p.rescore_mask[p.layer * p.Hkv + h] != 0;
            int seq;
            const int P = seq_pages(p, b, seq, lane == 0 && chunk == 0 && h == 0);
            const int page0 = chunk * kChunkPages;
            if (!rescored) {
                // the unit keeps its selection: its attention can start now
                if (chunk == 0 && lane == 0) publish_unit(wunit);
            } else if (chunk == 0 || page0 < P) {  // chunk 0 always carries the unit's first ticket
                const size_t ufull = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
                if (lane == 0) stage_q(b, h, page0 < P);
                if (ctl_lane) {
                    const int pb = page0 + kPiece * cw;
                    int npg = min(kPiece, P - pb);
                    if (npg < 0) npg = 0;
                    const bool ticket = npg > 0 || (chunk == 0 && cw == 0);
                    const int s = take_slot();
                    sh.desc[cw][s] = make_int4(static_cast<int>(kKindScore | (ticket ? kFlagTicket : 0u)) | (qseq << 8),
                                               wunit, pb, npg | (P << 8));
                    if (npg > 0) {
                        const uint32_t bytes = static_cast<uint32_t>(npg) * 4 * D;
                        mbar_arrive_expect_tx(&sh.full[cw][s], bytes);
                        bulk_copy_g2s(rings + size_t(cw * kRing + s) * kSlot, p.meta + (ufull * p.Pmax + pb) * 2 * D,
                                      bytes, &sh.full[cw][s]);
                    } else {
                        mbar_arrive(&sh.full[cw][s]);
                    }
                }
                ++kposted;
                ++qseq;
            }
            item = __shfl_sync(kFullMask, next, 0);
        }

        // ---- attention items, from the ready queue ---------------------------
        while (!aborting_warp()) {
            int a = -1;
            if (lane == 0) {
                const int i = atomicAdd(ctl + kCtlRdyHead, 1);
                if (i < n_att) {
                    const int e = wait_entry(rdy_q + i, &sh.abort_flag);
                    if (e == 0) {
                        set_abort();
                    } else {
                        a = e - 1;
                        rdy_q[i] = 0;  // consumed: the queue is clean for the next launch
                    }
                }
            }
            a = __shfl_sync(kFullMask, a, 0);
            if (a < 0) break;
            __syncwarp();  // lane 0's acquire of the entry orders every lane's reads of the selection
            const int wunit = a / S;
            const int sp = a - wunit * S;
            const int b = wunit / p.Hkv, h = wunit - b * p.Hkv;
            int seq;
            const int P = seq_pages(p, b, seq, false);
            const size_t ufull = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
            int cnt = 0;
            if (lane == 0) {
                cnt = __ldcg(p.sel_cnt + ufull);
                if (cnt < 0 || cnt > p.Kmax) {
                    if (sp == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
                    cnt = cnt < 0 ? 0 : p.Kmax;
                }
            }
            cnt = __shfl_sync(kFullMask, cnt, 0);
            const int beg = static_cast<int>(static_cast<long long>(cnt) * sp / S);
            const int end = static_cast<int>(static_cast<long long>(cnt) * (sp + 1) / S);
            if (lane == 0) stage_q(b, h, end > beg);
            int gstep = 0;  // steps of this item posted so far
            for (int base = beg; base < end; base += 32) {
                // resolve up to 32 selected pages; keep the valid ones in order
                const int i = base + lane;
                int phys = -1, nv = 0;
                if (i < end) {
                    const int lp = __ldcg(p.sel_idx + ufull * p.Kmax + i);
                    if (lp < 0 || lp >= P) {
                        report(p.err, KVMM_ERR_OUT_OF_RANGE);
                    } else {
                        const int32_t ph = __ldg(p.block_table + ufull * p.Pmax + lp);
                        if (ph < 0) {
                            report(p.err, KVMM_ERR_NULL_BLOCK);
                        } else if (ph >= p.n_phys) {
                            report(p.err, KVMM_ERR_OUT_OF_RANGE);
                        } else {
                            nv = min(T, seq - lp * T);
                            if (nv > 0) phys = ph;
                        }
                    }
                }
                const unsigned bal = __ballot_sync(kFullMask, phys >= 0);
                const int nvalid = __popc(bal);
                if (phys >= 0) {
                    const int pos = __popc(bal & ((1u << lane) - 1u));
                    sh.pphys[pos] = phys;
                    sh.pnv[pos] = nv;
                }
                __syncwarp();
                const int cphys = lane < nvalid ? sh.pphys[lane] : 0;  // lane j: the j-th valid page
                const int cnv = lane < nvalid ? sh.pnv[lane] : 0;
                __syncwarp();
                const int nsteps = (nvalid + kPPS - 1) / kPPS;
                for (int r0 = 0; r0 < nsteps; r0 += kCons) {
                    // this round's steps r0 .. r0+3; step g of the item goes to warp g % kCons
                    const int j = (cw - ((gstep + r0) & (kCons - 1))) & (kCons - 1);
                    const int st = r0 + j;
                    const bool has = st < nsteps;
                    const int pg0 = min(st * kPPS, 31);
                    const int np = has ? min(kPPS, nvalid - st * kPPS) : 0;
                    const int ph = __shfl_sync(kFullMask, cphys, min(pg0 + (cc >> 1), 31));
                    const int nv0 = __shfl_sync(kFullMask, cnv, pg0);
                    const int nv1 = __shfl_sync(kFullMask, cnv, min(pg0 + 1, 31));
                    const int s = kposted % kRing;
                    if (has && ctl_lane) {
                        take_slot();
                        sh.desc[cw][s] = make_int4(static_cast<int>(kKindAtt) | (qseq << 8), wunit, nv0,
                                                   np > 1 ? nv1 : 0);
                        mbar_arrive_expect_tx(&sh.full[cw][s], static_cast<uint32_t>(np) * 2 * kPageBytes);
                    }
                    __syncwarp();
                    if (has && cc < 2 * np) {
                        uint8_t* slot = rings + size_t(cw * kRing + s) * kSlot;
                        const size_t off = static_cast<size_t>(ph) * T * D;
                        if (cc & 1)
                            bulk_copy_g2s(slot + kStepTok * D * 2 + (cc >> 1) * kPageBytes, p.v_pool + off,
                                          kPageBytes, &sh.full[cw][s]);
                        else
                            bulk_copy_g2s(slot + (cc >> 1) * kPageBytes, p.k_pool + off, kPageBytes,
                                          &sh.full[cw][s]);
                    }
                    if (has) ++kposted;
                }
                gstep += nsteps;
            }
            // one merge marker per consumer warp closes the item
            if (ctl_lane) {
                const int s = take_slot();
                sh.desc[cw][s] = make_int4(static_cast<int>(kKindMerge) | (qseq << 8), wunit, sp, 0);
                mbar_arrive(&sh.full[cw][s]);
            }
            ++kposted;
            ++qseq;
        }
        // no more work: an end marker for every consumer warp
        if (ctl_lane) {
            const int s = take_slot();
            sh.desc[cw][s] = make_int4(static_cast<int>(kKindEnd), 0, 0, 0);
            mbar_arrive(&sh.full[cw][s]);
        }
    } else if (warp == kSelWarp) {
        // ================= selector ========================================
        // units selected in this launch: the rescored ones
        int n_sel = units;
        if (p.rescore_mask != nullptr) {
            int c = 0;
            for (int h = lane; h < p.Hkv; h += 32) c += p.rescore_mask[p.layer * p.Hkv + h] != 0 ? 1 : 0;
            n_sel = p.B * warp_sum(c);
        }
        while (!aborting_warp()) {
            int wunit = -1;
            if (lane == 0) {
                const int i = atomicAdd(ctl + kCtlSelHead, 1);
                if (i < n_sel) {
                    const int e = wait_entry(sel_q + i, &sh.abort_flag);
                    if (e == 0) {
                        set_abort();
                    } else {
                        wunit = e - 1;
                        sel_q[i] = 0;  // consumed: the queue is clean for the next launch
                    }
                }
            }
            wunit = __shfl_sync(kFullMask, wunit, 0);
            if (wunit < 0) break;
            __syncwarp();
            fence_acq_rel_gpu();  // with the poster's release: the unit's scores from every CTA are visible
            const int b = wunit / p.Hkv, h = wunit - b * p.Hkv;
            const size_t ufull = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
            int seq;
            const int P = seq_pages(p, b, seq, false);
            const int n = warp_topk(p.scores + static_cast<size_t>(wunit) * p.pstride, P, p.K,
                                    p.sel_idx + ufull * p.Kmax, sh.cand, lane);
            if (lane == 0) p.sel_cnt[ufull] = n;
            __syncwarp();
            if (lane == 0) publish_unit(wunit);  // the selection, then its attention items
        }
    } else if (warp == kPubWarp) {
        // ================= publisher =======================================
        // Counts finished score pieces and attention items (notices from the
        // consumers) with one GPU-scope fence per batch: a unit's last score
        // piece puts it on the select queue; its last attention item has its
        // partials combined here into out and lse.
        int head = 0;
        uint64_t t_idle = global_timer_ns();
        while (true) {
            int code = 0;
            if (lane < kNotices) code = ld_volatile(&sh.nq[(head + lane) % kNotices]);
            const unsigned got = __ballot_sync(kFullMask, code != 0);
            const int n = __ffs(~got) - 1 < 0 ? 32 : __ffs(~got) - 1;  // leading run of posted notices
            if (n == 0) {
                int fin = 0;
                if (lane == 0)
                    fin = (ld_volatile(&sh.cons_done) == kCons && ld_volatile(&sh.nq_tail) == head) || aborting();
                if (__shfl_sync(kFullMask, fin, 0)) break;
                __nanosleep(64);
                if (lane == 0 && global_timer_ns() - t_idle > kWaitNs) set_abort();
                continue;
            }
            t_idle = global_timer_ns();
            const bool mine = lane < n;
            if (mine) st_volatile(&sh.nq[(head + lane) % kNotices], 0);
            __syncwarp();
            if (lane == 0) st_volatile(&sh.nq_head, head + n);
            head += n;
            fence_acq_rel_gpu();  // the notices' global writes (scores, partials) before their tickets
            bool last = false;
            int wunit = 0;
            if (mine) {
                if (code > 0) {  // a score piece
                    wunit = code - 1;
                    int seq;
                    const int P = seq_pages(p, wunit / p.Hkv, seq, false);
                    const int pieces = max(1, (P + kPiece - 1) / kPiece);
                    last = atomicAdd(score_cnt + wunit, 1) == pieces - 1;
                } else {  // an attention item
                    wunit = -code - 1;
                    last = atomicAdd(att_cnt + wunit, 1) == S - 1;
                }
            }
            const unsigned lasts = __ballot_sync(kFullMask, last);
            if (lasts == 0u) continue;
            fence_acq_rel_gpu();  // every counted write of those units, then what follows
            if (last && code > 0) {
                score_cnt[wunit] = 0;
                st_volatile(sel_q + atomicAdd(sel_tail, 1), wunit + 1);  // to the selectors
            }
            // units whose attention items are all in: combine their partials
            unsigned todo = __ballot_sync(kFullMask, last && code < 0);
            while (todo != 0u) {
                const int src = __ffs(todo) - 1;
                todo &= todo - 1u;
                const int u = __shfl_sync(kFullMask, wunit, src);
                if (lane == 0) att_cnt[u] = 0;
                const int b = u / p.Hkv, h = u - b * p.Hkv;
                const int G = p.G;
                const float* pu = p.partials + static_cast<size_t>(u) * S * part_stride;
                if (lane < G) {
                    float M = -INFINITY;
                    for (int s2 = 0; s2 < S; ++s2) M = fmaxf(M, __ldcg(pu + s2 * part_stride + lane));
                    float L = 0.f;
                    for (int s2 = 0; s2 < S; ++s2) {
                        const float ms = __ldcg(pu + s2 * part_stride + lane);
                        const float f = ms == -INFINITY ? 0.f : exp2f(ms - M);
                        sh.pf[s2][lane] = f;
                        L = fmaf(__ldcg(pu + s2 * part_stride + 8 + lane), f, L);
                    }
                    const float inv = L > 0.f ? 1.f / L : 0.f;
                    for (int s2 = 0; s2 < S; ++s2) sh.pf[s2][lane] *= inv;
                    const size_t oi = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * G + lane;
                    if (p.lse) p.lse[oi] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
                }
                __syncwarp();
                float* op = p.out + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * G) * D;
                for (int e4 = lane; e4 < G * D / 4; e4 += 32) {
                    const int g = (4 * e4) / D;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int s2 = 0; s2 < S; ++s2) {
                        const float f = sh.pf[s2][g];
                        const float4 v = __ldcg(reinterpret_cast<const float4*>(pu + s2 * part_stride + 16) + e4);
                        acc.x = fmaf(f, v.x, acc.x);
                        acc.y = fmaf(f, v.y, acc.y);
                        acc.z = fmaf(f, v.z, acc.z);
                        acc.w = fmaf(f, v.w, acc.w);
                    }
                    reinterpret_cast<float4*>(op)[e4] = acc;
                }
                __syncwarp();
            }
        }
    } else {
        // ================= consumers =======================================
        const int w = warp;
        const int gid = lane >> 2, tig = lane & 3;
        const int G = p.G;
        const bool real_head = gid < G;
        uint32_t wf[kR][4];       // score weights of head gid: [min(q,0) | max(q,0)] chunk 4r + tig
        uint32_t qf[D / 32][4];   // attention Q^T B fragments of head gid
        float o[kMTiles][4];
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int i = 0; i < kMTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        int cur_q = -1;
        uint32_t gsync_n = 0;
        auto group_sync = [&]() {  // the 4 consumer warps
            __threadfence_block();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.gbar);
            wait_bar_warp(&sh.gbar, gsync_n & 1);
            ++gsync_n;
        };
        const int ua0 = 8 * (gid >> 1) + (gid & 1);  // attention token row of fragment row gid (see below)

        for (int k = 0;; ++k) {
            const int s = k % kRing;
            if (!wait_bar_warp(&sh.full[w][s], (k / kRing) & 1)) break;
            const int4 d = sh.desc[w][s];
            const uint32_t kind = static_cast<uint32_t>(d.x) & 3u;
            if (kind == kKindEnd) break;
            const int qs = d.x >> 8;
            if (qs != cur_q) {  // the item's query group
                if (!wait_bar_warp(&sh.qfull[qs % kQRing], (qs / kQRing) & 1)) break;
                const uint8_t* qe = qring + size_t(qs % kQRing) * qentry_bytes(D) + gid * (2 * D);
                if (kind == kKindScore) {
#pragma unroll
                    for (int r = 0; r < kR; ++r) {
                        const int c = 4 * r + tig;  // chunk of the [min | max] row
                        const int qc = c % (D / 8);
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (real_head) v = ld_shared_v4(qe + 16 * qc);
                        const bool is_max = c >= D / 8;
                        wf[r][0] = is_max ? bf16x2_max0(v.x) : bf16x2_min0(v.x);
                        wf[r][1] = is_max ? bf16x2_max0(v.y) : bf16x2_min0(v.y);
                        wf[r][2] = is_max ? bf16x2_max0(v.z) : bf16x2_min0(v.z);
                        wf[r][3] = is_max ? bf16x2_max0(v.w) : bf16x2_min0(v.w);
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < D / 32; ++r) {
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (real_head) v = ld_shared_v4(qe + 16 * (4 * r + tig));
                        qf[r][0] = v.x;
                        qf[r][1] = v.y;
                        qf[r][2] = v.z;
                        qf[r][3] = v.w;
                    }
                }
                cur_q = qs;
            }
            const uint8_t* slot = rings + size_t(w * kRing + s) * kSlot;

            if (kind == kKindScore) {
                // ---- 32 pages: two [16 x 2D] x [2D x 8] products ----------
                const int wunit = d.y, pb = d.z, npg = d.w & 255;
                float* srow = p.scores + static_cast<size_t>(wunit) * p.pstride + pb;
                float* orow = p.scores_out ? p.scores_out + static_cast<size_t>(wunit) * p.Pmax + pb : nullptr;
#pragma unroll
                for (int grp = 0; grp < 2; ++grp) {
                    if (16 * grp < npg) {
                        const uint8_t* ra = slot + static_cast<size_t>(16 * grp + gid) * 4 * D;
                        const uint8_t* rb = ra + 8 * 4 * D;
                        float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int r = 0; r < kR; ++r) {
                            const uint4 ka = ld_shared_v4(ra + 16 * (4 * r + tig));
                            const uint4 kb = ld_shared_v4(rb + 16 * (4 * r + tig));
                            mma_bf16_16816(c, ka.x, kb.x, ka.y, kb.y, wf[r][0], wf[r][1]);
                            mma_bf16_16816(c2, ka.z, kb.z, ka.w, kb.w, wf[r][2], wf[r][3]);
                        }
                        // c: [page gid][head 2tig], [gid][2tig+1], [gid+8][2tig], [gid+8][2tig+1]
                        float s_lo, s_hi;
                        if (MODE == 0) {
                            s_lo = (c[0] + c2[0]) + (c[1] + c2[1]);
                            s_hi = (c[2] + c2[2]) + (c[3] + c2[3]);
                            s_lo += __shfl_xor_sync(kFullMask, s_lo, 1);
                            s_hi += __shfl_xor_sync(kFullMask, s_hi, 1);
                            s_lo += __shfl_xor_sync(kFullMask, s_lo, 2);
                            s_hi += __shfl_xor_sync(kFullMask, s_hi, 2);
                        } else {
                            const bool h0 = 2 * tig < G, h1 = 2 * tig + 1 < G;
                            s_lo = fmaxf(h0 ? c[0] + c2[0] : -FLT_MAX, h1 ? c[1] + c2[1] : -FLT_MAX);
                            s_hi = fmaxf(h0 ? c[2] + c2[2] : -FLT_MAX, h1 ? c[3] + c2[3] : -FLT_MAX);
                            s_lo = fmaxf(s_lo, __shfl_xor_sync(kFullMask, s_lo, 1));
                            s_hi = fmaxf(s_hi, __shfl_xor_sync(kFullMask, s_hi, 1));
                            s_lo = fmaxf(s_lo, __shfl_xor_sync(kFullMask, s_lo, 2));
                            s_hi = fmaxf(s_hi, __shfl_xor_sync(kFullMask, s_hi, 2));
                        }
                        if (tig == 0) {
                            const int r0 = 16 * grp + gid;
                            if (r0 < npg) {
                                srow[r0] = s_lo;
                                if (orow) orow[r0] = s_lo;
                            }
                            if (r0 + 8 < npg) {
                                srow[r0 + 8] = s_hi;
                                if (orow) orow[r0 + 8] = s_hi;
                            }
                        }
                    }
                }
                __syncwarp();
                fence_proxy_async_shared();
                if (lane == 0) {
                    mbar_arrive(&sh.empty[w][s]);          // the slot may be refilled
                    mbar_arrive(&sh.qempty[qs % kQRing]);  // and the item's query group freed
                }
                if (d.x & kFlagTicket) {  // the publisher counts this piece of the unit
                    __syncwarp();
                    if (lane == 0) post_notice(wunit + 1);
                }
            } else if (kind == kKindAtt) {
                // ---- one 32-token step (two 16-token sub-tiles) -----------
                const int nv0 = d.z, nv1 = d.w;
                const bool full = (kPPS == 2) ? (nv0 == T && nv1 == T) : (nv0 == T);
                auto valid = [&](int u) { return kPPS == 2 ? ((u >> 4) ? (u & 15) < nv1 : u < nv0) : u < nv0; };
                const uint8_t* ks = slot;
                const uint8_t* vs = slot + kStepTok * D * 2;
                // token u of the step: page u / T (within the step), row u % T.  Sub-tile j,
                // fragment row rho holds token 8*((rho&7)>>1) + 4j + 2*(rho>>3) + (rho&1).
                float x[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint8_t* ra = ks + (ua0 + 4 * j) * (2 * D);
                    const uint8_t* rb = ra + 2 * (2 * D);
                    float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int r = 0; r < D / 32; ++r) {
                        const uint4 ka = ld_shared_v4(ra + 16 * (4 * r + tig));
                        const uint4 kb = ld_shared_v4(rb + 16 * (4 * r + tig));
                        mma_bf16_16816(c, ka.x, kb.x, ka.y, kb.y, qf[r][0], qf[r][1]);
                        mma_bf16_16816(c2, ka.z, kb.z, ka.w, kb.w, qf[r][2], qf[r][3]);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) x[j][i] = (c[i] + c2[i]) * p.scale_log2;
                    if (!full) {
                        if (!valid(ua0 + 4 * j)) x[j][0] = x[j][1] = -INFINITY;
                        if (!valid(ua0 + 4 * j + 2)) x[j][2] = x[j][3] = -INFINITY;
                    }
                }
                float mx0 = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
                float mx1 = fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3]));
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, off));
                }
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
                const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
                const float a0 = fast_exp2(m0 - ref0), a1 = fast_exp2(m1 - ref1);
                float pr[2][4];
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) pr[j][i] = fast_exp2(x[j][i] - ((i & 1) ? ref1 : ref0));
                l0 = fmaf(l0, a0, (pr[0][0] + pr[0][2]) + (pr[1][0] + pr[1][2]));
                l1 = fmaf(l1, a1, (pr[0][1] + pr[0][3]) + (pr[1][1] + pr[1][3]));
                m0 = mn0;
                m1 = mn1;
                if (__any_sync(kFullMask, (a0 != 1.f) || (a1 != 1.f))) {
#pragma unroll
                    for (int i = 0; i < kMTiles; ++i) {
                        o[i][0] *= a0;
                        o[i][1] *= a1;
                        o[i][2] *= a0;
                        o[i][3] *= a1;
                    }
                }
                uint32_t bh[2][2], bl[2][2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t h01 = pack_bf16x2(pr[j][0], pr[j][1]), h23 = pack_bf16x2(pr[j][2], pr[j][3]);
                    const uint32_t r01 = pack_bf16x2(pr[j][0] - bf16_lo(h01), pr[j][1] - bf16_hi(h01));
                    const uint32_t r23 = pack_bf16x2(pr[j][2] - bf16_lo(h23), pr[j][3] - bf16_hi(h23));
                    bh[j][0] = movmatrix_trans(h01);
                    bh[j][1] = movmatrix_trans(h23);
                    bl[j][0] = movmatrix_trans(r01);
                    bl[j][1] = movmatrix_trans(r23);
                }
                // O^T += V^T P^T: lane reads tokens 8tig .. 8tig+7 of dims 16i+gid, 16i+gid+8
                const int u0 = 8 * tig;
                const uint8_t* vrow = vs + (u0 / T) * kPageBytes + (u0 % T) * 2;
                bool vk[8];
                if (!full) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) vk[e] = valid(u0 + e);
                }
#pragma unroll
                for (int i = 0; i < kMTiles; ++i) {
                    uint4 wa = ld_shared_v4(vrow + (16 * i + gid) * (T * 2));
                    uint4 wb = ld_shared_v4(vrow + (16 * i + gid + 8) * (T * 2));
                    if (!full) {
                        wa = make_uint4(keep_halves(wa.x, vk[0], vk[1]), keep_halves(wa.y, vk[2], vk[3]),
                                        keep_halves(wa.z, vk[4], vk[5]), keep_halves(wa.w, vk[6], vk[7]));
                        wb = make_uint4(keep_halves(wb.x, vk[0], vk[1]), keep_halves(wb.y, vk[2], vk[3]),
                                        keep_halves(wb.z, vk[4], vk[5]), keep_halves(wb.w, vk[6], vk[7]));
                    }
                    mma_bf16_16816(o[i], wa.x, wb.x, wa.y, wb.y, bh[0][0], bh[0][1]);
                    mma_bf16_16816(o[i], wa.x, wb.x, wa.y, wb.y, bl[0][0], bl[0][1]);
                    mma_bf16_16816(o[i], wa.z, wb.z, wa.w, wb.w, bh[1][0], bh[1][1]);
                    mma_bf16_16816(o[i], wa.z, wb.z, wa.w, wb.w, bl[1][0], bl[1][1]);
                }
                __syncwarp();
                fence_proxy_async_shared();
                if (lane == 0) mbar_arrive(&sh.empty[w][s]);
            } else {
                // ---- merge marker: the item's four warp partials -> one partial
                if (lane == 0) mbar_arrive(&sh.empty[w][s]);
                const int wunit = d.y, sp = d.z;
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    l0 += __shfl_xor_sync(kFullMask, l0, off);
                    l1 += __shfl_xor_sync(kFullMask, l1, off);
                }
                if (gid == 0) {
                    sh.mm[w][2 * tig] = m0;
                    sh.mm[w][2 * tig + 1] = m1;
                    sh.ml[w][2 * tig] = l0;
                    sh.ml[w][2 * tig + 1] = l1;
                }
                float* mw = mo + size_t(w) * 8 * D;
#pragma unroll
                for (int i = 0; i < kMTiles; ++i) {
                    float* w0 = mw + (2 * tig) * D;
                    float* w1 = w0 + D;
                    w0[16 * i + gid] = o[i][0];
                    w1[16 * i + gid] = o[i][1];
                    w0[16 * i + gid + 8] = o[i][2];
                    w1[16 * i + gid + 8] = o[i][3];
                }
                group_sync();
                const int gt = w * 32 + lane;  // 0 .. 127 over the consumer group
                float* part = p.partials + (static_cast<size_t>(wunit) * S + sp) * part_stride;
                if (gt < G) {
                    float M = -INFINITY;
#pragma unroll
                    for (int ww = 0; ww < kCons; ++ww) M = fmaxf(M, sh.mm[ww][gt]);
                    float L = 0.f;
#pragma unroll
                    for (int ww = 0; ww < kCons; ++ww) {
                        const float mw2 = sh.mm[ww][gt];
                        const float f = mw2 == -INFINITY ? 0.f : exp2f(mw2 - M);
                        sh.f[ww][gt] = f;
                        L = fmaf(sh.ml[ww][gt], f, L);
                    }
                    part[gt] = M;
                    part[8 + gt] = L;
                }
                group_sync();
                for (int e = gt; e < G * D; e += kCons * 32) {
                    const int g = e / D;
                    float O = 0.f;
#pragma unroll
                    for (int ww = 0; ww < kCons; ++ww) O = fmaf(sh.f[ww][g], mo[size_t(ww) * 8 * D + e], O);
                    part[16 + e] = O;
                }
                group_sync();  // the item's partial is written (and the scratch read)
                if (gt == 0) post_notice(-(wunit + 1));  // the publisher counts it
                if (lane == 0) mbar_arrive(&sh.qempty[qs % kQRing]);
#pragma unroll
                for (int i = 0; i < kMTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
                m0 = m1 = -INFINITY;
                l0 = l1 = 0.f;
            }
        }
        if (lane == 0) {
            __threadfence_block();
            atomicAdd(&sh.cons_done, 1);
        }
    }
    // ---- the last CTA out resets the queue counters for the next launch ------
    __syncthreads();
    if (tid == 0) {
        if (aborting()) {
            atomicOr(ctl + kCtlAbort, 1);
            __threadfence();
        }
        sh.last = atomicAdd(ctl + kCtlDone, 1) == static_cast<int>(gridDim.x) - 1;
        if (sh.last) __threadfence();
    }
    __syncthreads();
    if (sh.last) {
        if (__ldcg(ctl + kCtlAbort) != 0) {
            // abandoned work: clear tickets and queue entries
            for (int u = tid; u < 3 * units + n_att; u += kFThreads) score_cnt[u] = 0;
        }
        __syncthreads();
        if (tid == 0) {
            for (int c = 0; c <= kCtlAbort; ++c) ctl[c] = 0;
        }
    }
    if (aborting() && tid == 0) {
        // let any copy still in flight land before the CTA's shared memory is released
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 2000000ull) __nanosleep(1000);
    }
}

template <int D, int T, int MODE>
cudaError_t launch_fused_t(const FusedParams& p, cudaStream_t stream)
{
    static thread_local int dev_cache = -1;
    static thread_local size_t bytes_cache = 0;
    const size_t smem = fused_dyn_smem(D);
    cudaError_t e = allow_smem(fused_decode_kernel<D, T, MODE>, smem, dev_cache, bytes_cache);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148, per_sm = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_decode_kernel<D, T, MODE>, kFThreads, smem);
    if (per_sm < 1) per_sm = 1;
    const long long items = static_cast<long long>(p.B) * p.Hkv * (p.chunks + p.splits);
    const long long slots = static_cast<long long>(sms) * per_sm;
    const long long grid = items < slots ? items : slots;
    return launch_pdl(fused_decode_kernel<D, T, MODE>, dim3(static_cast<unsigned>(grid)), dim3(kFThreads), smem,
                      stream, p);
}

}  // namespace

size_t fused_smem_bytes(int D) { return fused_dyn_smem(D) + sizeof(FusedShared); }

cudaError_t launch_fused_decode(const FusedParams& p, int group_reduce, cudaStream_t stream)
{
    if (p.D == 128) {
        if (p.T == 16) return group_reduce ? launch_fused_t<128, 16, 1>(p, stream) : launch_fused_t<128, 16, 0>(p, stream);
        return group_reduce ? launch_fused_t<128, 32, 1>(p, stream) : launch_fused_t<128, 32, 0>(p, stream);
    }
    if (p.T == 16) return group_reduce ? launch_fused_t<64, 16, 1>(p, stream) : launch_fused_t<64, 16, 0>(p, stream);
    return group_reduce ? launch_fused_t<64, 32, 1>(p, stream) : launch_fused_t<64, 32, 0>(p, stream);
}

}  // namespace kvmm
