// decode_layer.cuh -- one launch per layer: append the new tokens and refresh
// their pages' MinMax, score every page, select the top K, attend over the
// selected pages.  The kernel template also runs its first half or its second
// half alone (PH below): page_score_topk as one launch (score and select) and
// sparse_paged_decode_attn as one launch (attend over kept selections).  Each
// variant is instantiated in a translation unit of its own: decode_layer.cu
// (both phases), decode_score.cu (score and select), decode_attend.cu (attend).
//
// FlexiCache (MLSys'26 blog summary), "Core method, 2. MinMax-metadata page
// scoring" (per-page key bounds, kept up to date as pages fill; the query and
// the bounds give each page's score; the top-K pages of every (layer, KV
// head) are kept) and "Core method, 1. Stability-differentiated placement" /
// "System design, head-level block table" (attention over the selected pages
// only, found through [batch, layer, head, logical_block]).  The results
// equal kv_minmax_update (appending) followed by page_score_topk_attn.
//
// Design (sm_103a).  A thread-block cluster of C CTAs owns NU units (batch,
// KV head): two, or one when two units' score buffers do not fit shared
// memory (long sequences).  C is the most CTAs whose clusters are all resident
// at once.  Every CTA of it streams, in this order, its share of unit 0's
// MinMax rows, its share of unit 1's, its share of unit 0's selected K/V
// pages, its share of unit 1's (all bulk copies with an L2 evict-first
// policy: each byte is read once):
//   - 8 consumer warps each keep their own slots in flight (1-D bulk copies,
//     TMA, one mbarrier per slot).  An attention slot holds one page of K and
//     V: two slots a warp for pages of 16 tokens, one for pages of 32.  The
//     score phase cuts the same bytes into two slots of the [min | max] rows of
//     16 consecutive pages (a score item), whatever the page size.  A score
//     item is scored on the tensor cores (mma.sync m16n8k16)
//     and every score sent to every CTA of the cluster as an asynchronous
//     remote store that completes on the receiver's mbarrier, as does each
//     warp's range of the unit's scores (remote min/max reductions); a page of
//     the item that receives new tokens first has its bounds widened by them.
//     An attention step runs S^T = K Q^T, the online softmax (against a per-
//     head reference raised only when a score exceeds it by 2^8) and
//     O^T += V^T P^T with P as bf16 hi + lo.  At the end of a unit each warp
//     leaves its softmax partial in shared memory and goes on with the next
//     unit's pages, already in flight;
//   - 8 selector warps first take the bounds of the rows a partly filled page
//     already holds (for the consumer that widens it) and append the new
//     tokens (rows, and the MinMax of the pages this CTA owns); then, as soon
//     as all of a unit's scores and their range have arrived, they select the
//     unit's top K exactly (block_topk; for one long unit a cluster, in two
//     levels: each CTA's top K of its share, then the top K of those) and
//     resolve this CTA's share of the pages through the block-table rows
//     (copied to shared memory at the start when they fit) -- unit 0's
//     selection overlaps the streaming of unit 1's rows, unit 1's overlaps
//     unit 0's attention -- and for each unit combine the consumer warps'
//     partials into the CTA's, send every CTA its slice (16-byte remote
//     stores), and combine the slices they receive into out and lse.
// All exchange stays on chip (asynchronous remote shared-memory stores and
// mbarriers), with no fence on the way: a consumer attending over a page that
// receives tokens takes those rows from new_k / new_v rather than waiting for
// the selectors' pool writes, which are for later launches.  Every wait is
// bounded (KVMM_ERR_TIMEOUT, then the kernel runs to its end).
// Launched with programmatic dependent launch: a launch waits for the
// preceding kernel before its first read, or, with early cache reads
// (KVMM_DECODE_EARLY_READS), computes its units' extents, copies their table
// rows and starts streaming their metadata first, and waits before it reads
// the queries, new rows, pools or kept selections, or stores anything but
// error bits (atomic ORs into err).
#pragma once

#include <cfloat>
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "topk_block.cuh"

namespace kvmm {
namespace dl {

constexpr int kDCons = 8;                      // consumer warps
constexpr int kDSel0 = kDCons;                 // first selector warp
constexpr int kDSelWarps = 8;
constexpr int kDSelThreads = kDSelWarps * 32;
constexpr int kDThreads = (kDCons + kDSelWarps) * 32;
constexpr int kDUnits = 2;                     // units per cluster at most (DecodeParams::NU: 1 or 2)
constexpr int kDSelBar = 1;                    // the selector warps' named barrier
constexpr int kDRingMax = 2;

// slots per consumer warp; a slot is one page of K and V (4TD bytes)
__host__ __device__ constexpr int d_ring(int T) { return T == 16 ? 2 : 1; }

using SelGroup = WarpGroup<kDSelBar, kDSel0 * 32, kDSelThreads>;

constexpr uint64_t kDWaitNs = 1000000000ull;   // 1 s: far beyond any legitimate wait
constexpr uint64_t kDAbortNs = 1000000ull;

// one unit of the cluster as this CTA sees it, read from global memory once
struct DUnit {
    size_t ufull;   // its row of the [B][L][Hkv] arrays
    int b, h;
    int seq, P;     // sequence length (clamped to Pmax*T) and its pages
    int lo, hi;     // the pages this CTA scores
    int rescored;
    int tb, te;     // tokens this launch appends (te <= tb: none)
    int pb, pe;     // pages holding appended tokens that this CTA owns (the last CTA also owns those
                    // at or past the unit's page count)
};

struct DecodeShared {
    uint64_t full[kDCons][kDRingMax];  // a consumer warp's slot has landed
    uint64_t qbar;            // the query groups of the cluster's units
    uint64_t btbar;           // the units' block-table rows are in btab (bt_smem)
    uint64_t cbar[kDUnits];   // two-level selection: every CTA's candidates of the unit are here
    uint64_t sbar[kDUnits];   // all of the unit's scores and its range are here (asynchronous remote stores
                              // and reductions, 4 bytes each)
    uint64_t selr[kDUnits];   // this CTA's share of the unit's pages is resolved
    uint64_t rbar[kDUnits];   // every CTA's partial of this CTA's output slice is here (likewise)
    uint64_t pbar;            // prior bounds written (one arrival per selector warp)
    uint64_t pready[kDUnits]; // every consumer warp's partial of the unit is written (kDCons arrivals)
    uint64_t pfree;           // the selector warps have read the consumers' partials of unit 0
    DUnit ud[kDUnits];
    int resn[kDUnits];        // resolved pages of this CTA's share
    int wcount[kDSelWarps];
    float mm[kDCons][8];
    float ml[kDCons][8];
    uint32_t wide[kDUnits][128];   // per unit: key-ordered bounds of all rows below tok_end of the first
                                   // page the new tokens reach, [min | max], two channels a word (D <= 128)
    int wide_ok[kDUnits];          // those bounds are set (the page has a valid table entry)
    uint4 nrow[kDUnits][32];       // per unit, for a one-token append: the token's key row, then its value row
    uint32_t rkey[kDUnits][2];     // per unit: order keys of its smallest and largest score (remote reductions)
    int abort_flag;
};

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

// bf16 pair -> pair of unsigned 16-bit keys ordered like the values
__device__ __forceinline__ uint32_t to_key2(uint32_t w)
{
    const uint32_t neg = (w >> 15) & 0x00010001u;
    return w ^ ((neg * 0xffffu) | 0x80008000u);
}
__device__ __forceinline__ uint32_t from_key2(uint32_t k)
{
    const uint32_t neg = ((~k) >> 15) & 0x00010001u;
    return k ^ ((neg * 0xffffu) | 0x80008000u);
}

__device__ __forceinline__ int ld_volatile(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

// start fetching `bytes` (a multiple of 16, from a 16-byte aligned address) into L2
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// a long wait of an idle warp: poll with short sleeps so that it leaves the issue slots and the
// shared-memory pipe to the warps that stream
__device__ __forceinline__ bool mbar_wait_sleepy(uint64_t* bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        __nanosleep(64);
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Two-level selection: with one unit a cluster, when a unit may have more pages than one CTA's selection holds
// in registers (a launch whose Pmax is above that, with clusters of more than one CTA), each CTA selects the
// top K of the pages it scored, the cluster's candidates (at most C*K) are exchanged, and each CTA selects the
// top K of those.  Every page of the unit's top K is in its own CTA's top K (fewer than K pages of that share
// outrank it), and the candidates are packed in ascending page order, so the result, ties to the lower page
// included, is the one-level selection's -- for every unit of the launch, whatever its own page count.  A CTA
// then keeps only the scores of its own share.  Two units a cluster always select in one level: a compile-time
// fact that keeps that kernel free of the two-level code (measured: the runtime test alone cost it 0.9 us a
// launch at the 8B shape), and at long contexts one unit a cluster was the faster launch anyway.
__host__ __device__ inline bool d_two_level(int NU, int Pmax, int C)
{
    return NU == 1 && C > 1 && Pmax > 8 * kDSelThreads;
}

// Which CTAs of the cluster select a unit (and so receive its scores and range): every one when the launch
// also attends (each resolves its share of the selection) or selects in two levels; in a launch that only
// scores and selects, rank 0 alone, which writes the selection, so that the other CTAs leave after scoring.
__host__ __device__ inline bool d_all_select(int ph, int NU, int Pmax, int C)
{
    return (ph & kPhAttend) != 0 || d_two_level(NU, Pmax, C);
}

// Where a unit's scores and score range go: to every CTA of the cluster (each selects from all of them), to
// rank 0 alone (it alone selects), or to the scoring CTA itself (two levels: each CTA's first level reads
// only the pages it scored and their range, the second only the candidates the CTAs exchange).
enum DScoreDest { kDestAll = 0, kDestRank0 = 1, kDestOwn = 2 };
__host__ __device__ inline int d_score_dest(int ph, int NU, int Pmax, int C)
{
    if (d_two_level(NU, Pmax, C)) return kDestOwn;
    return (ph & kPhAttend) != 0 ? kDestAll : kDestRank0;
}

// the shared-memory plan, identical on host and device
struct DLayout {
    size_t ring, part, qbuf, sbuf, bins, ts, selv, res, recv, btab, cand, total;
    int pstride, slice, recv_stride;
};
__host__ __device__ inline size_t d_align(size_t n) { return (n + 127) & ~static_cast<size_t>(127); }
// bt: the units' block-table rows are copied to shared memory (btab), for the selection's page lookups;
// ph: the phases the launch runs (a buffer only one phase uses takes no room in a launch without it)
__host__ __device__ inline DLayout d_layout(int D, int T, int Pmax, int Kmax, int C, int maxp, int G, bool bt, int NU,
                                            int ph)
{
    const bool sc = (ph & kPhScore) != 0, at = (ph & kPhAttend) != 0;
    const bool two = sc && d_two_level(NU, Pmax, C);
    const int share = (Pmax + C - 1) / C;  // pages a CTA scores at most
    DLayout l{};
    l.pstride = ((two ? share : Pmax) + 3) & ~3;  // per unit: its scores, or this CTA's share of them
    l.slice = ((G * D + C - 1) / C + 3) & ~3;  // outputs a CTA combines: a multiple of 4 (16-byte stores)
    l.recv_stride = 16 * C + l.slice * C;
    l.ring = 0;
    l.part = d_align(l.ring + size_t(kDCons) * d_ring(T) * 4 * T * D);
    l.qbuf = d_align(l.part + (at ? size_t(kDCons) * G * (D + 4) * sizeof(float) : 0));
    l.sbuf = d_align(l.qbuf + size_t(NU) * 8 * D * 2);
    l.bins = d_align(l.sbuf + (sc ? size_t(NU) * l.pstride * sizeof(float) : 0));
    // bins: one per score the general top-K path ranks (a share, or the cluster's candidates, in two levels)
    l.ts = d_align(l.bins + (sc ? size_t(two ? (share > C * Kmax ? share : C * Kmax) : Pmax) * sizeof(int16_t) : 0));
    l.selv = d_align(l.ts + (sc ? sizeof(BlockTopkShared<kDSelThreads>) : 0));
    l.res = d_align(l.selv + (sc ? size_t(Kmax) * sizeof(int32_t) : 0));
    l.recv = d_align(l.res + (at ? size_t(NU) * maxp * 2 * sizeof(int32_t) : 0));
    l.btab = d_align(l.recv + (at ? size_t(NU) * l.recv_stride * sizeof(float) : 0));
    l.cand = d_align(l.btab + (at && bt ? size_t(NU) * Pmax * sizeof(int32_t) : 0));
    l.total = d_align(l.cand + (two ? size_t(NU) * C * Kmax * 8 : 0));
    return l;
}

// ---------------------------------------------------------------------------
template <int D, int T, int MODE, int NU, int PH>
__global__ void __launch_bounds__(kDThreads, 1) decode_layer_kernel(const DecodeParams p,
                                                                     const __grid_constant__ CUtensorMap tmeta)
{
    static_assert(NU >= 1 && NU <= kDUnits, "units per cluster");
    static_assert(PH == kPhScore || PH == kPhAttend || PH == kPhBoth, "phases");
    constexpr bool kScore = (PH & kPhScore) != 0;    // score and select the rescored units
    constexpr bool kAttend = (PH & kPhAttend) != 0;  // attend over the selected pages
    constexpr int kSub = T / 16;                // 16-token sub-tiles of a page
    constexpr int kRing = d_ring(T);            // slots per consumer warp
    constexpr int kRowBytes = 4 * D;            // a page's [min | max] row
    constexpr int kPageBytes = 2 * T * D;       // a page's K (or V) block
    constexpr int kSlot = 2 * kPageBytes;       // an attention slot: one page of K and V
    // the score phase cuts the same bytes into two slots of 16 pages' rows: a T = 32 warp's single
    // attention slot would leave it copying and scoring one after the other
    constexpr int kSRing = 2;                       // score slots per consumer warp
    constexpr int kSSlot = kRing * kSlot / kSRing;  // the [min | max] rows of kSPiece pages
    constexpr int kSPiece = kSSlot / kRowBytes;     // pages per score item
    constexpr int kSGrp = kSPiece / 16;             // 16-page row groups of a score item
    constexpr int kMTiles = D / 16;
    constexpr int kR = (2 * D / 8) / 4;         // 16-byte chunk groups of a [min | max] row
    static_assert(kSGrp == 1 && kSPiece == 16, "a score item is one group of 16 pages");
    // A score item arrives by one tensor copy (TMA) with the 128-byte swizzle: a page's [min | max] row is
    // kLines 128-byte lines, and 16-byte unit u of line l sits at unit u ^ (l & 7) of it, so the fragment loads
    // of rows gid and gid + 1 (512 bytes apart, on the same banks) fall on different banks.
    constexpr int kLines = kRowBytes / 128;
    static_assert(kSSlot == kSPiece * kRowBytes && kSSlot % 1024 == 0, "a score slot is one swizzled box");
    static_assert(kRing <= kDRingMax && kSRing <= kDRingMax, "slot count");
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ DecodeShared sh;

    const int C = p.C;
    const DLayout lay = d_layout(D, T, p.Pmax, p.Kmax, C, p.maxp, p.G, p.bt_smem != 0, NU, PH);
    uint8_t* rings = smem + lay.ring;
    float* part = reinterpret_cast<float*>(smem + lay.part);
    uint8_t* qbuf = smem + lay.qbuf;
    float* sbuf = reinterpret_cast<float*>(smem + lay.sbuf);
    int16_t* bins = reinterpret_cast<int16_t*>(smem + lay.bins);
    auto& ts = *reinterpret_cast<BlockTopkShared<kDSelThreads>*>(smem + lay.ts);
    int32_t* selv = reinterpret_cast<int32_t*>(smem + lay.selv);
    int2* res = reinterpret_cast<int2*>(smem + lay.res);
    float* recv = reinterpret_cast<float*>(smem + lay.recv);
    int32_t* btab = reinterpret_cast<int32_t*>(smem + lay.btab);
    // two-level selection, per unit: C*Kmax candidate scores, then their pages
    float* cand = reinterpret_cast<float*>(smem + lay.cand);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x / C;
    const int U = p.B * p.Hkv;
    const int nunits = min(NU, U - cluster * NU);
    const int G = p.G;
    const int n_out = G * D;

    if (tid == 0) {
        for (int w = 0; w < kDCons; ++w)
            for (int b2 = 0; b2 < kDRingMax; ++b2) mbar_init(&sh.full[w][b2], 1);
        mbar_init(&sh.qbar, 1);
        mbar_init(&sh.btbar, 1);
        for (int j = 0; j < kDUnits; ++j) {
            mbar_init(&sh.cbar[j], 1);
            mbar_init(&sh.sbar[j], 1);
            mbar_init(&sh.selr[j], 1);
            mbar_init(&sh.rbar[j], 1);
            sh.resn[j] = 0;
            sh.rkey[j][0] = 0xffffffffu;
            sh.rkey[j][1] = 0u;
        }
        mbar_init(&sh.pbar, kDSelWarps);
        for (int j = 0; j < kDUnits; ++j) mbar_init(&sh.pready[j], kDCons);
        mbar_init(&sh.pfree, 1);
        sh.abort_flag = 0;
        fence_barrier_init();
    }
    // every CTA's barriers exist before the first remote arrival: the cluster barrier is passed before
    // anything reaches another CTA, and meanwhile the queries and the unit descriptors are fetched
    cluster_arrive();
    // Every input may come from the preceding kernels, and the caller may read what this one writes only
    // after it.  With early cache reads the caller vouches that the preceding kernel writes nothing this
    // launch reads of the cache state (descriptors' inputs, block-table rows, metadata rows): this launch
    // then computes its units' descriptors, copies their table rows and starts streaming their metadata
    // while that kernel drains, and every thread waits for it before it reads the queries or new rows or
    // writes anything (error bits, ORed atomically into err, aside).  Either way a thread lets the next
    // launch be scheduled only after its own wait, so the kernel before the preceding one has finished
    // whenever a launch reads early.
    if (!p.early) pdl_wait_then_release();

    auto aborting = [&]() { return ld_volatile(&sh.abort_flag) != 0; };
    auto set_abort = [&]() {
        *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
        report(p.err, KVMM_ERR_TIMEOUT);
    };
    auto wait_bar_warp = [&](uint64_t* bar, uint32_t parity) {  // every lane of a warp, one outcome
        const bool ok = __all_sync(kFullMask, mbar_wait_bounded(bar, parity, aborting() ? kDAbortNs : kDWaitNs));
        if (!ok && lane == 0) set_abort();
        return ok;
    };

    auto issue_q = [&]() {  // the query groups of the cluster's units (one thread)
        const uint32_t qbytes = static_cast<uint32_t>(G) * D * 2;
        mbar_arrive_expect_tx(&sh.qbar, qbytes * nunits);
        for (int j = 0; j < nunits; ++j) {
            const int wunit = cluster * NU + j;
            const int b = wunit / p.Hkv, h = wunit - (wunit / p.Hkv) * p.Hkv;
            bulk_copy_g2s(qbuf + size_t(j) * 8 * D * 2,
                          p.q + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * G) * D, qbytes, &sh.qbar);
        }
    };
    if (tid == 0 && !p.early) issue_q();
    if (tid < nunits) {  // this CTA's view of unit tid
        DUnit u;
        const int wunit = cluster * NU + tid;
        u.b = wunit / p.Hkv;
        u.h = wunit - u.b * p.Hkv;
        u.ufull = (static_cast<size_t>(u.b) * p.L + p.layer) * p.Hkv + u.h;
        const int cap = p.Pmax * T;
        const bool first_of_batch = rank == 0 && u.h == 0;  // reports a batch's range errors once
        // the four loads are independent: issue them together (an absent array reads seq_len, unused)
        const int* tbp = p.new_k != nullptr ? p.tok_begin + u.b : p.seq_len + u.b;
        const int* tep = p.new_k != nullptr ? p.tok_end + u.b : p.seq_len + u.b;
        const uint8_t* mkp = p.rescore_mask != nullptr ? p.rescore_mask + p.layer * p.Hkv + u.h
                                                       : reinterpret_cast<const uint8_t*>(p.seq_len + u.b);
        int seq = p.seq_len[u.b];
        const int tb_in = *tbp, te_in = *tep;
        const uint8_t mk_in = *mkp;
        if (seq < 0 || seq > cap) {
            if (first_of_batch) report(p.err, KVMM_ERR_OUT_OF_RANGE);
            seq = seq < 0 ? 0 : cap;
        }
        u.seq = seq;
        u.P = (seq + T - 1) / T;
        u.lo = static_cast<int>(static_cast<long long>(u.P) * rank / C);
        u.hi = static_cast<int>(static_cast<long long>(u.P) * (rank + 1) / C);
        u.rescored = kScore && (p.rescore_mask == nullptr || mk_in != 0);  // else the kept selection
        u.tb = u.te = u.pb = u.pe = 0;
        if (p.new_k != nullptr) {
            const int tb = tb_in, te = te_in;
            if (first_of_batch && (tb < 0 || te < tb || tb > cap || te > cap || te - tb > p.n_new))
                report(p.err, KVMM_ERR_OUT_OF_RANGE);
            if (tb >= 0 && te >= tb && tb <= cap) {
                const int te2 = min(min(te, cap), tb + p.n_new);
                if (te2 > tb) {
                    u.tb = tb;
                    u.te = te2;
                    const int own_hi = rank == static_cast<uint32_t>(C - 1) ? p.Pmax : u.hi;
                    u.pb = max(tb / T, u.lo);
                    u.pe = max(u.pb, min((te2 - 1) / T + 1, own_hi));
                }
            }
        }
        sh.ud[tid] = u;
    }
    __syncwarp();  // converged for the aligned barrier
    cluster_wait();
    __syncthreads();  // the descriptors above

    if (warp >= kDSel0) {
        // ================= selectors =======================================
        const int stid = tid - kDSel0 * 32;
        const int swarp = stid >> 5;
        constexpr int kLanesPerRow = D / 8;  // 16 bytes (8 channels) per lane
        constexpr int kRowsPerPass = 32 / kLanesPerRow;
        const int sub = lane % kLanesPerRow;
        if (kAttend && stid == 0 && (p.Pmax & 3) == 0) {
            // the units' block-table rows, read when this CTA's share of the selection is resolved: into
            // shared memory when there is room, else into L2
            const uint32_t row = static_cast<uint32_t>(p.Pmax) * 4u;
            if (p.bt_smem) mbar_arrive_expect_tx(&sh.btbar, row * nunits);
            for (int j = 0; j < nunits; ++j) {
                if (p.bt_smem)
                    bulk_copy_g2s(btab + size_t(j) * p.Pmax, p.block_table + sh.ud[j].ufull * p.Pmax, row, &sh.btbar);
                else
                    prefetch_l2(p.block_table + sh.ud[j].ufull * p.Pmax, row);
            }
        }
        if (stid == 0) {
            // the bytes this CTA receives: every score of a rescored unit (one float a page) and from every
            // consumer warp of every CTA the unit's score range (a min and a max reduction), and from
            // each CTA its (m, l) of every head and its partial of this CTA's slice of the outputs.  A
            // remote store that lands before its barrier is told to expect it leaves the transaction
            // count negative; the pending arrival keeps the phase open until the count is set.
            const int e0 = static_cast<int>(rank) * lay.slice;
            const int own = max(0, min(n_out, e0 + lay.slice) - e0);
            for (int j = 0; j < nunits; ++j) {
                const DUnit& u = sh.ud[j];
                if (!(u.rescored && u.P > p.K && d_two_level(NU, p.Pmax, C))) continue;
                uint32_t n = 0;  // candidates: from every CTA min(K, pages it scored), 8 bytes each
                for (int r = 0; r < C; ++r) {
                    const int pr = static_cast<int>(static_cast<long long>(u.P) * (r + 1) / C) -
                                   static_cast<int>(static_cast<long long>(u.P) * r / C);
                    n += static_cast<uint32_t>(min(p.K, pr));
                }
                mbar_arrive_expect_tx(&sh.cbar[j], n * 8u);
            }
            for (int j = 0; j < nunits; ++j) {
                const DUnit& u = sh.ud[j];
                // every score of the unit and every warp's range, or this CTA's own (two levels), or none
                const int dest = d_score_dest(PH, NU, p.Pmax, C);
                uint32_t bytes = 0u;
                if (u.rescored && dest == kDestOwn)
                    bytes = static_cast<uint32_t>(u.hi - u.lo) * 4u + static_cast<uint32_t>(kDCons * 8);
                else if (u.rescored && (dest == kDestAll || rank == 0))
                    bytes = static_cast<uint32_t>(u.P) * 4u + static_cast<uint32_t>(C * kDCons * 8);
                mbar_arrive_expect_tx(&sh.sbar[j], bytes);
                if (kAttend) mbar_arrive_expect_tx(&sh.rbar[j], static_cast<uint32_t>(C * (2 * G + own)) * 4u);
            }
        }
        if (p.early) {
            pdl_wait_then_release();  // the preceding kernel is done: the queries and new rows are final
            // a launch that only attends has consumer warp 0 copy the queries: the resolution that the first
            // page copies wait for does not stall behind issuing them (attention alone at the 8B shape: 15.52
            // -> 15.45 us)
            if (kScore && stid == 0) issue_q();
        }
        // 0. for the consumer warps, well before they need them: the finished bounds of the first page the
        //    new tokens reach, if this CTA scores it (all its rows below tok_end, old and new), and for a
        //    one-token append the token's key and value rows
        if (swarp < nunits) {
            const int j = swarp;
            const DUnit& u = sh.ud[j];
            if (u.te > u.tb) {
                const size_t src = (static_cast<size_t>(u.b) * p.Hkv + u.h) * p.n_new;  // token tb's row
                if (u.te - u.tb == 1 && lane < D / 8) {
                    sh.nrow[j][lane] = reinterpret_cast<const uint4*>(p.new_k + src * D)[lane];
                    sh.nrow[j][D / 8 + lane] = reinterpret_cast<const uint4*>(p.new_v + src * D)[lane];
                }
                const int pg = u.tb / T, r0 = u.tb - pg * T, r1 = min(u.te - pg * T, T);
                if (u.rescored && u.pb <= pg && pg < min(u.pe, u.hi)) {
                    const int32_t phys = p.block_table[u.ufull * p.Pmax + pg];
                    const bool ok = phys >= 0 && phys < p.n_phys;  // else the page is skipped, and reported below
                    if (ok) {
                        const kvmm_bf16* kpage = p.k_pool + static_cast<size_t>(phys) * T * D;
                        uint32_t lo[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
                        uint32_t hi[4] = {0u, 0u, 0u, 0u};
#pragma unroll 4
                        for (int r = lane / kLanesPerRow; r < r1; r += kRowsPerPass) {
                            const kvmm_bf16* row = r < r0 ? kpage + static_cast<size_t>(r) * D
                                                          : p.new_k + (src + (r - r0)) * D;
                            const uint4 v = reinterpret_cast<const uint4*>(row)[sub];
                            const uint32_t w4[4] = {to_key2(v.x), to_key2(v.y), to_key2(v.z), to_key2(v.w)};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                lo[i] = __vminu2(lo[i], w4[i]);
                                hi[i] = __vmaxu2(hi[i], w4[i]);
                            }
                        }
#pragma unroll
                        for (int off = kLanesPerRow; off < 32; off <<= 1) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                lo[i] = __vminu2(lo[i], __shfl_xor_sync(kFullMask, lo[i], off));
                                hi[i] = __vmaxu2(hi[i], __shfl_xor_sync(kFullMask, hi[i], off));
                            }
                        }
                        if (lane < kLanesPerRow) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                sh.wide[j][4 * sub + i] = lo[i];
                                sh.wide[j][D / 2 + 4 * sub + i] = hi[i];
                            }
                        }
                    }
                    if (lane == 0) sh.wide_ok[j] = ok ? 1 : 0;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.pbar);  // release: the bounds and rows above
        // 1. the appended tokens of the pages this CTA owns: rows, then the pages' MinMax from all
        //    their rows (a consumer scoring such a page widens its own copy of the bounds)
        if (p.new_k != nullptr) {
            for (int j = 0; j < nunits; ++j) {
                const DUnit& u = sh.ud[j];
                const int tb = u.tb, te = u.te;
                for (int page = u.pb + swarp; page < u.pe; page += kDSelWarps) {
                    const int32_t phys = p.block_table[u.ufull * p.Pmax + page];
                    if (phys < 0 || phys >= p.n_phys) {
                        if (lane == 0) report(p.err, phys < 0 ? KVMM_ERR_NULL_BLOCK : KVMM_ERR_OUT_OF_RANGE);
                        continue;
                    }
                    kvmm_bf16* kpage = p.k_pool + static_cast<size_t>(phys) * T * D;
                    kvmm_bf16* vpage = p.v_pool + static_cast<size_t>(phys) * T * D;
                    const int first = page * T;
                    const int r0 = max(tb - first, 0);
                    const int r1 = min(te - first, T);
                    const size_t src_base = (static_cast<size_t>(u.b) * p.Hkv + u.h) * p.n_new;
                    for (int r = r0 + lane / kLanesPerRow; r < r1; r += kRowsPerPass) {
                        const size_t jj = src_base + (first + r - tb);
                        const uint4 kv = reinterpret_cast<const uint4*>(p.new_k + jj * D)[sub];
                        const uint4 vv = reinterpret_cast<const uint4*>(p.new_v + jj * D)[sub];
                        reinterpret_cast<uint4*>(kpage + static_cast<size_t>(r) * D)[sub] = kv;
                        const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                        for (int e = 0; e < 8; ++e)  // values are dimension-major: channel d of token r at [d*T + r]
                            vpage[static_cast<size_t>(8 * sub + e) * T + r] =
                                static_cast<kvmm_bf16>((e & 1) ? (vw[e >> 1] >> 16) : (vw[e >> 1] & 0xffffu));
                    }
                    __syncwarp();  // the rows just written are read back below by other lanes
                    const int n_valid = min(T, te - first);
                    uint32_t lo[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
                    uint32_t hi[4] = {0u, 0u, 0u, 0u};
                    for (int r = lane / kLanesPerRow; r < n_valid; r += kRowsPerPass) {
                        const uint4 v = reinterpret_cast<const uint4*>(kpage + static_cast<size_t>(r) * D)[sub];
                        const uint32_t w4[4] = {to_key2(v.x), to_key2(v.y), to_key2(v.z), to_key2(v.w)};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            lo[i] = __vminu2(lo[i], w4[i]);
                            hi[i] = __vmaxu2(hi[i], w4[i]);
                        }
                    }
#pragma unroll
                    for (int off = kLanesPerRow; off < 32; off <<= 1) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            lo[i] = __vminu2(lo[i], __shfl_xor_sync(kFullMask, lo[i], off));
                            hi[i] = __vmaxu2(hi[i], __shfl_xor_sync(kFullMask, hi[i], off));
                        }
                    }
                    if (lane < kLanesPerRow) {
                        kvmm_bf16* m = p.meta + (u.ufull * p.Pmax + page) * 2 * D;
                        reinterpret_cast<uint4*>(m)[lane] = make_uint4(from_key2(lo[0]), from_key2(lo[1]),
                                                                       from_key2(lo[2]), from_key2(lo[3]));
                        reinterpret_cast<uint4*>(m + D)[lane] = make_uint4(from_key2(hi[0]), from_key2(hi[1]),
                                                                           from_key2(hi[2]), from_key2(hi[3]));
                    }
                }
            }
            // later launches read these rows and bounds; this one never waits for them: the consumer
            // that attends over such a page takes the new rows from new_k / new_v itself
        }

        // 2. each unit's selection, then this CTA's share of its pages through the block table
        for (int j = 0; j < nunits; ++j) {
            const DUnit u = sh.ud[j];
            int cnt;
            const int32_t* src;
            if (kScore && u.rescored) {
                if (rank != 0 && !d_all_select(PH, NU, p.Pmax, C)) continue;  // rank 0 selects this unit alone
                // every score of the unit and its range are here (the histogram is cleared meanwhile)
                block_topk_prepare<kDSelThreads, SelGroup>(ts);
                if (!mbar_wait_sleepy(&sh.sbar[j], 0, aborting() ? kDAbortNs : kDWaitNs)) set_abort();
                float* sj = sbuf + size_t(j) * lay.pstride;  // the unit's scores, or this CTA's share of them
                if (u.P > p.K && d_two_level(NU, p.Pmax, C)) {
                    float* cand_s = cand + size_t(j) * 2 * C * p.Kmax;
                    int32_t* cand_p = reinterpret_cast<int32_t*>(cand_s + size_t(C) * p.Kmax);
                    // this CTA's candidates: the top K of its share, to every CTA, after the earlier CTAs'
                    const int n_l = block_topk<kDSelThreads, SelGroup>(nullptr, u.hi - u.lo, p.K, selv, sj,
                                                                       bins, ts, sh.rkey[j]);
                    int off = 0, n_all = 0;
                    for (int r = 0; r < C; ++r) {
                        const int pr = static_cast<int>(static_cast<long long>(u.P) * (r + 1) / C) -
                                       static_cast<int>(static_cast<long long>(u.P) * r / C);
                        if (r < static_cast<int>(rank)) off += min(p.K, pr);
                        n_all += min(p.K, pr);
                    }
                    for (int i = stid; i < n_l * C; i += kDSelThreads) {
                        const int r = i / n_l, e = i - r * n_l;
                        st_async_f32(cand_s + off + e, &sh.cbar[j], static_cast<uint32_t>(r), sj[selv[e]]);
                        st_async_f32(cand_p + off + e, &sh.cbar[j], static_cast<uint32_t>(r),
                                     __int_as_float(u.lo + selv[e]));
                    }
                    SelGroup::sync();  // selv is read
                    if (!mbar_wait_sleepy(&sh.cbar[j], 0, aborting() ? kDAbortNs : kDWaitNs)) set_abort();
                    cnt = block_topk<kDSelThreads, SelGroup>(nullptr, n_all, p.K, selv, cand_s, bins, ts, nullptr);
                    for (int i = stid; i < cnt; i += kDSelThreads) selv[i] = cand_p[selv[i]];  // positions -> pages
                    SelGroup::sync();
                } else {
                    // two units a cluster: the one call site, inlined (measured 0.17 us a launch at the 8B shape);
                    // one unit a cluster also has the two-level calls, and a second inlined copy slowed it
                    if constexpr (NU == 2)
                        cnt = block_topk_inline<kDSelThreads, SelGroup>(nullptr, u.P, p.K, selv, sj, bins, ts,
                                                                        sh.rkey[j]);
                    else
                        cnt = block_topk<kDSelThreads, SelGroup>(nullptr, u.P, p.K, selv, sj, bins, ts, sh.rkey[j]);
                }
                if (rank == 0) {
                    for (int i = stid; i < cnt; i += kDSelThreads) p.sel_idx[u.ufull * p.Kmax + i] = selv[i];
                    if (stid == 0) p.sel_cnt[u.ufull] = cnt;
                }
                if constexpr (!kAttend) {
                    SelGroup::sync();  // selv is read before the next unit's selection
                    continue;
                }
                src = selv;
            } else {
                if constexpr (!kAttend) continue;  // a unit not rescored keeps its selection
                cnt = p.sel_cnt[u.ufull];
                if (cnt < 0 || cnt > p.Kmax) {
                    if (rank == 0 && stid == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
                    cnt = cnt < 0 ? 0 : p.Kmax;
                }
                src = p.sel_idx + u.ufull * p.Kmax;
            }
            const int beg = static_cast<int>(static_cast<long long>(cnt) * rank / C);
            const int end = static_cast<int>(static_cast<long long>(cnt) * (rank + 1) / C);
            // the rows in shared memory have long landed by now; after a time-out the table is read directly
            const bool bt_here = p.bt_smem && mbar_wait_bounded(&sh.btbar, 0, aborting() ? kDAbortNs : kDWaitNs);
            int2* rl = res + size_t(j) * p.maxp;
            int nres = 0;
            for (int i0 = beg; i0 < end; i0 += kDSelThreads) {
                const int i = i0 + stid;
                int phys = -1;
                int lp = 0;
                if (i < end) {
                    lp = src[i];
                    if (lp < 0 || lp >= u.P) {
                        report(p.err, KVMM_ERR_OUT_OF_RANGE);
                    } else {
                        const int32_t ph = bt_here ? btab[size_t(j) * p.Pmax + lp] : p.block_table[u.ufull * p.Pmax + lp];
                        if (ph < 0) {
                            report(p.err, KVMM_ERR_NULL_BLOCK);
                        } else if (ph >= p.n_phys) {
                            report(p.err, KVMM_ERR_OUT_OF_RANGE);
                        } else if (u.seq > lp * T) {
                            phys = ph;
                        }
                    }
                }
                const bool ok = phys >= 0;
                const unsigned bal = __ballot_sync(kFullMask, ok);
                if (lane == 0) sh.wcount[swarp] = __popc(bal);
                SelGroup::sync();
                int pos = nres, tot = 0;
#pragma unroll
                for (int w = 0; w < kDSelWarps; ++w) {
                    if (w < swarp) pos += sh.wcount[w];
                    tot += sh.wcount[w];
                }
                if (ok) rl[pos + __popc(bal & ((1u << lane) - 1u))] = make_int2(phys, lp);
                nres += tot;
                SelGroup::sync();
            }
            if (stid == 0) {
                sh.resn[j] = nres;
                mbar_arrive(&sh.selr[j]);  // release: the list above, then the consumers
            }
        }

        // 3. each unit's outputs: the consumer warps' partials -> this CTA's, sent to every CTA of the
        //    cluster (each gets its slice); then this CTA's slice from every CTA's partial
        for (int j = 0; kAttend && j < nunits; ++j) {
            const DUnit& u = sh.ud[j];
            if (!mbar_wait_sleepy(&sh.pready[j], 0, aborting() ? kDAbortNs : kDWaitNs)) set_abort();
            float* rj = recv + size_t(j) * lay.recv_stride;  // [C][16] (m, l), then [C][slice] outputs
            // four outputs of one head a thread; each thread weighs the warps' partials of its head itself, and
            // one thread a head sends the head's (m, l) to every CTA
            for (int e4 = 4 * stid; e4 < n_out; e4 += 4 * kDSelThreads) {
                const int g = e4 / D;
                float M = -INFINITY;
#pragma unroll
                for (int ww = 0; ww < kDCons; ++ww) M = fmaxf(M, sh.mm[ww][g]);
                float L = 0.f;
                float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int ww = 0; ww < kDCons; ++ww) {
                    const float mw2 = sh.mm[ww][g];
                    const float f = mw2 == -INFINITY ? 0.f : exp2f(mw2 - M);
                    L = fmaf(sh.ml[ww][g], f, L);
                    const float4 v =
                        *reinterpret_cast<const float4*>(part + size_t(ww) * G * (D + 4) + g * (D + 4) + (e4 - g * D));
                    O.x = fmaf(f, v.x, O.x);
                    O.y = fmaf(f, v.y, O.y);
                    O.z = fmaf(f, v.z, O.z);
                    O.w = fmaf(f, v.w, O.w);
                }
                const int r = e4 / lay.slice;
                st_async_v4_f32(rj + 16 * C + rank * lay.slice + (e4 - r * lay.slice), &sh.rbar[j],
                                static_cast<uint32_t>(r), O.x, O.y, O.z, O.w);
                if (e4 == g * D) {
                    for (int rr = 0; rr < C; ++rr) {
                        st_async_f32(rj + 16 * rank + g, &sh.rbar[j], static_cast<uint32_t>(rr), M);
                        st_async_f32(rj + 16 * rank + 8 + g, &sh.rbar[j], static_cast<uint32_t>(rr), L);
                    }
                }
            }
            SelGroup::sync();  // the consumer warps' partials are read
            if (stid == 0 && j + 1 < nunits) mbar_arrive(&sh.pfree);

            if (!mbar_wait_sleepy(&sh.rbar[j], 0, aborting() ? kDAbortNs : kDWaitNs)) set_abort();
            // this CTA's slice of the outputs from every CTA's partial: each thread weighs the partials of its
            // head itself; rank 0 writes each head's lse
            const int e0 = static_cast<int>(rank) * lay.slice;
            const int e1 = min(n_out, e0 + lay.slice);
            const float* ro = rj + 16 * C;
            float* ob = p.out + (static_cast<size_t>(u.b) * p.Hq + static_cast<size_t>(u.h) * G) * D;
            for (int e = e0 + stid; e < e1; e += kDSelThreads) {
                const int g = e / D;
                float M = -INFINITY;
                for (int c = 0; c < C; ++c) M = fmaxf(M, rj[16 * c + g]);
                float L = 0.f, O = 0.f;
                for (int c = 0; c < C; ++c) {
                    const float mc = rj[16 * c + g];
                    const float f = mc == -INFINITY ? 0.f : exp2f(mc - M);
                    L = fmaf(rj[16 * c + 8 + g], f, L);
                    O = fmaf(f, ro[c * lay.slice + (e - e0)], O);
                }
                ob[e] = O * (L > 0.f ? 1.f / L : 0.f);
            }
            if (rank == 0 && p.lse && stid < G) {
                float M = -INFINITY;
                for (int c = 0; c < C; ++c) M = fmaxf(M, rj[16 * c + stid]);
                float L = 0.f;
                for (int c = 0; c < C; ++c) {
                    const float mc = rj[16 * c + stid];
                    L = fmaf(rj[16 * c + 8 + stid], mc == -INFINITY ? 0.f : exp2f(mc - M), L);
                }
                const size_t oi = static_cast<size_t>(u.b) * p.Hq + static_cast<size_t>(u.h) * G + stid;
                p.lse[oi] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
            }
            SelGroup::sync();
        }
    } else {
        // ================= consumers =======================================
        const int w = warp;
        const int gid = lane >> 2, tig = lane & 3;
        const bool real_head = gid < G;
        uint32_t wf[kR][4];      // score weights of head gid: [min(q,0) | max(q,0)] chunk 4r + tig
        uint32_t qf[D / 32][4];  // attention Q^T B fragments of head gid
        int frag = -1;           // which fragments are loaded: 2*unit + (0 score, 1 attention)
        bool have_q = false;
        uint8_t* my_ring = rings + size_t(w) * kRing * kSlot;
        const uint64_t stream_policy = l2_policy_evict_first();  // metadata and pages: read once
        // the slots: bit b of `held` -- slot b has a copy in flight; bit b of `par` -- the phase its
        // mbarrier completes next; (hj, hs) -- the unit and item it holds
        uint32_t held = 0u, par = 0u;
        int hj0 = 0, hj1 = 0, hs0 = 0, hs1 = 0;
        auto set_slot = [&](int b, int j, int s) {
            held |= 1u << b;
            if (b) {
                hj1 = j;
                hs1 = s;
            } else {
                hj0 = j;
                hs0 = s;
            }
        };
        auto in_flight = [&](int b) { return ((held >> b) & 1u) != 0u; };
        auto land = [&](int b) {
            const bool ok = wait_bar_warp(&sh.full[w][b], (par >> b) & 1u);
            par ^= 1u << b;
            held &= ~(1u << b);
            return ok;
        };
        auto load_frags = [&](int j, bool att) {
            const int want = 2 * j + (att ? 1 : 0);
            if (want == frag) return;
            if (!have_q) {
                wait_bar_warp(&sh.qbar, 0);
                have_q = true;
            }
            const uint8_t* qe = qbuf + size_t(j) * 8 * D * 2 + gid * (2 * D);
            if (!att) {
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
            frag = want;
        };

        // ---- 1. scores: this warp's items (16 pages each) s = w, w + 8, ... of each rescored unit ----
        int nsl[kDUnits] = {0, 0};
        for (int j = 0; j < nunits; ++j) {
            const DUnit& u = sh.ud[j];
            nsl[j] = u.rescored ? (u.hi - u.lo + kSPiece - 1) / kSPiece : 0;
        }
        // advance (j, sl) to this warp's next score item; false when there is none
        auto next_score = [&](int& j, int& sl) {
            sl += kDCons;
            while (j < nunits && sl >= nsl[j]) {
                ++j;
                sl = w;
            }
            return j < nunits;
        };
        auto issue_score = [&](int b2, int j, int sl) {
            const int page0 = sh.ud[j].lo + sl * kSPiece;
            // the 16 rows from page0 in one tensor copy, whole (rows past the unit's pages are read and not
            // used; rows past the array's end arrive as zeros), issued by the slot's own lane: a thread's bulk
            // copies complete one after another
            if (lane == b2) {
                mbar_arrive_expect_tx(&sh.full[w][b2], static_cast<uint32_t>(kSSlot));
                tma_load_3d_hint(my_ring + size_t(b2) * kSSlot, &tmeta, 0, 0,
                                 static_cast<int>(sh.ud[j].ufull * p.Pmax + page0), &sh.full[w][b2], stream_policy);
            }
            set_slot(b2, j, sl);
        };
        // the byte offset in a score slot of 16-byte unit u of page row pr (see kLines)
        auto sw_off = [](int pr, int u) {
            const int line = pr * kLines + (u >> 3);
            return line * 128 + (((u & 7) ^ (line & 7)) << 4);
        };
        // page `pg` of unit j receives tokens in this launch: its bounds in row pr of the score slot (the
        // page's [min | max] row in shared memory, swizzled) become those of all its rows below tok_end.  The selector warps
        // have them ready for the first such page; a later page of a multi-token append holds new rows
        // only.  (The selector warps write the rows and the metadata; a page they skip -- null or
        // out-of-range table entry -- keeps its bounds here too.)
        bool have_prep = false;  // the selector warps' preparations are visible
        auto wait_prep = [&]() {
            if (!have_prep) {
                wait_bar_warp(&sh.pbar, 0);
                have_prep = true;
            }
        };
        auto widen_page = [&](int j, int pg, uint8_t* slot, int pr) {  // pr: the page's row in the slot
            const DUnit& u = sh.ud[j];
            if (pg == u.tb / T) {
                wait_prep();
                if (sh.wide_ok[j] && lane < D / 4) {
                    const uint32_t* wv = sh.wide[j] + 4 * lane;
                    *reinterpret_cast<uint4*>(slot + sw_off(pr, lane)) =
                        make_uint4(from_key2(wv[0]), from_key2(wv[1]), from_key2(wv[2]), from_key2(wv[3]));
                }
                __syncwarp();
                return;
            }
            constexpr int kLanesPerRow = D / 8;  // 16 bytes (8 channels) per lane
            const int first = pg * T;
            const int r1 = min(u.te - first, T);
            const int32_t phys = p.block_table[u.ufull * p.Pmax + pg];
            if (phys < 0 || phys >= p.n_phys || r1 <= 0) return;
            const size_t src_base = (static_cast<size_t>(u.b) * p.Hkv + u.h) * p.n_new;
            const int half = lane / kLanesPerRow;  // 0: min, 1: max
            const int sub = lane % kLanesPerRow;
            if (half < 2) {
                uint32_t acc[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = half == 0 ? 0xffffffffu : 0u;
                for (int r = 0; r < r1; ++r) {
                    const uint4 kv = reinterpret_cast<const uint4*>(p.new_k + (src_base + (first + r - u.tb)) * D)[sub];
                    const uint32_t k4[4] = {to_key2(kv.x), to_key2(kv.y), to_key2(kv.z), to_key2(kv.w)};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        acc[i] = half == 0 ? __vminu2(acc[i], k4[i]) : __vmaxu2(acc[i], k4[i]);
                }
                *reinterpret_cast<uint4*>(slot + sw_off(pr, half * (D / 8) + sub)) =
                    make_uint4(from_key2(acc[0]), from_key2(acc[1]), from_key2(acc[2]), from_key2(acc[3]));
            }
            __syncwarp();
        };
        // the order keys of the smallest and largest score this lane has computed of unit rj; at the end of
        // the unit every CTA of the cluster gets the warp's (for the selection's bins)
        uint32_t kmin = 0xffffffffu, kmax = 0u;
        int rj = 0;
        auto flush_range = [&]() {
            if (sh.ud[rj].rescored) {
                kmin = __reduce_min_sync(kFullMask, kmin);
                kmax = __reduce_max_sync(kFullMask, kmax);
                const int dest = d_score_dest(PH, NU, p.Pmax, C);  // the CTAs that select from the range
                if (dest == kDestAll ? lane < C : lane == 0) {
                    const uint32_t r = dest == kDestAll ? static_cast<uint32_t>(lane) : dest == kDestOwn ? rank : 0u;
                    red_async_minmax_u32<false>(&sh.rkey[rj][0], &sh.sbar[rj], r, kmin);
                    red_async_minmax_u32<true>(&sh.rkey[rj][1], &sh.sbar[rj], r, kmax);
                }
            }
            kmin = 0xffffffffu;
            kmax = 0u;
            ++rj;
        };
        auto score_slot = [&](const uint8_t* slot, int j, int page0, int npg) {
            float* sb = sbuf + size_t(j) * lay.pstride + page0;
            float* orow = p.scores_out ? p.scores_out + static_cast<size_t>(cluster * NU + j) * p.Pmax + page0
                                       : nullptr;
#pragma unroll
            for (int grp = 0; grp < kSGrp; ++grp) {
                if (16 * grp < npg) {
                    // rows gid and gid + 8 share their swizzle (8 rows apart is a multiple of 8 lines)
                    const uint8_t* ra = slot;
                    const uint8_t* rb = slot + 8 * kRowBytes;
                    // four independent accumulation chains (even / odd r, low / high half of the chunk); the scoring
                    // kernels of every path sum them in this same order, so their scores agree bit for bit
                    float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
                    float c3[4] = {0.f, 0.f, 0.f, 0.f}, c4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int r = 0; r < kR; ++r) {
                        const int o = sw_off(16 * grp + gid, 4 * r + tig);
                        const uint4 ka = ld_shared_v4(ra + o);
                        const uint4 kb = ld_shared_v4(rb + o);
                        mma_bf16_16816((r & 1) ? c3 : c, ka.x, kb.x, ka.y, kb.y, wf[r][0], wf[r][1]);
                        mma_bf16_16816((r & 1) ? c4 : c2, ka.z, kb.z, ka.w, kb.w, wf[r][2], wf[r][3]);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) c[i] = (c[i] + c3[i]) + (c2[i] + c4[i]);
                    float s_lo, s_hi;
                    if (MODE == 0) {
                        s_lo = c[0] + c[1];
                        s_hi = c[2] + c[3];
                        s_lo += __shfl_xor_sync(kFullMask, s_lo, 1);
                        s_hi += __shfl_xor_sync(kFullMask, s_hi, 1);
                        s_lo += __shfl_xor_sync(kFullMask, s_lo, 2);
                        s_hi += __shfl_xor_sync(kFullMask, s_hi, 2);
                    } else {
                        const bool h0 = 2 * tig < G, h1 = 2 * tig + 1 < G;
                        s_lo = fmaxf(h0 ? c[0] : -FLT_MAX, h1 ? c[1] : -FLT_MAX);
                        s_hi = fmaxf(h0 ? c[2] : -FLT_MAX, h1 ? c[3] : -FLT_MAX);
                        s_lo = fmaxf(s_lo, __shfl_xor_sync(kFullMask, s_lo, 1));
                        s_hi = fmaxf(s_hi, __shfl_xor_sync(kFullMask, s_hi, 1));
                        s_lo = fmaxf(s_lo, __shfl_xor_sync(kFullMask, s_lo, 2));
                        s_hi = fmaxf(s_hi, __shfl_xor_sync(kFullMask, s_hi, 2));
                    }
                    // lanes tig = 0..3 of a row group send the two scores to CTAs tig, tig + 4, ...
                    const int r0 = 16 * grp + gid;
                    if (r0 < npg) {
                        kmin = min(kmin, topk_order_key(s_lo));
                        kmax = max(kmax, topk_order_key(s_lo));
                    }
                    if (r0 + 8 < npg) {
                        kmin = min(kmin, topk_order_key(s_hi));
                        kmax = max(kmax, topk_order_key(s_hi));
                    }
                    const int dest = d_score_dest(PH, NU, p.Pmax, C);  // the CTAs that select the unit
                    if (dest == kDestAll) {
                        for (int r = tig; r < C; r += 4) {
                            if (r0 < npg) st_async_f32(sb + r0, &sh.sbar[j], static_cast<uint32_t>(r), s_lo);
                            if (r0 + 8 < npg) st_async_f32(sb + r0 + 8, &sh.sbar[j], static_cast<uint32_t>(r), s_hi);
                        }
                    } else if (tig == 0) {
                        // rank 0 keeps the unit's scores by page; a CTA selecting in two levels, its share by
                        // page - lo
                        const uint32_t r = dest == kDestOwn ? rank : 0u;
                        float* so = dest == kDestOwn ? sb - sh.ud[j].lo : sb;
                        if (r0 < npg) st_async_f32(so + r0, &sh.sbar[j], r, s_lo);
                        if (r0 + 8 < npg) st_async_f32(so + r0 + 8, &sh.sbar[j], r, s_hi);
                    }
                    if (orow && tig == 0) {
                        if (r0 < npg) orow[r0] = s_lo;
                        if (r0 + 8 < npg) orow[r0 + 8] = s_hi;
                    }
                }
            }
        };
        if constexpr (!kScore) {
            if (p.early) {
                pdl_wait_then_release();  // before the queries, the kept selections, the pools and any store
                if (w == 0 && lane == 0) issue_q();
            }
        } else {
            int ij = 0, isl = w - kDCons;  // the last issued item
            bool more = next_score(ij, isl);
            for (int b = 0; b < kSRing && more; ++b) {
                issue_score(b, ij, isl);
                more = next_score(ij, isl);
            }
            if (p.early) pdl_wait_then_release();  // before the new rows and any store
            // a slot is refilled as soon as it is consumed, and the slots are consumed in turn: in the
            // order they were filled
            for (int b = 0; in_flight(b); b = (b + 1) % kSRing) {
                const int j = b ? hj1 : hj0;
                const int page0 = sh.ud[j].lo + (b ? hs1 : hs0) * kSPiece;
                const int npg = min(kSPiece, sh.ud[j].hi - page0);
                while (rj < j) flush_range();  // the units before j are done
                land(b);
                load_frags(j, false);
                uint8_t* slot = my_ring + size_t(b) * kSSlot;
                const int pe = min(sh.ud[j].pe, page0 + npg);
                for (int pg = max(sh.ud[j].pb, page0); pg < pe; ++pg)  // pages receiving new tokens
                    widen_page(j, pg, slot, pg - page0);
                score_slot(slot, j, page0, npg);
                __syncwarp();
                fence_proxy_async_shared();  // this slot's reads, then the next copy into it
                if (more) {
                    issue_score(b, ij, isl);
                    more = next_score(ij, isl);
                }
            }
            while (rj < nunits) flush_range();
        }

        // ---- 2. attention: this warp's steps (one page each) s = w, w + 8, ... of each unit, then the
        //         unit's merge; once a unit's steps are all issued, the freed slots fetch the next unit's
        if constexpr (kAttend) {
        float o[kMTiles][4];
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int i = 0; i < kMTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        // token of fragment row rho of sub-tile jj: 4*kSub*((rho&7)>>1) + 4*jj + 2*(rho>>3) + (rho&1), so
        // that lane tig's k-slots of the P^T fragment are tokens 4*kSub*tig .. 4*kSub*tig + 4*kSub - 1
        const int ua0 = 4 * kSub * (gid >> 1) + (gid & 1);
        auto att_step = [&](const uint8_t* slot, int nv) {
            const bool full = nv == T;
            const uint8_t* ks = slot;
            const uint8_t* vs = slot + kPageBytes;
            float x[kSub][4];
#pragma unroll
            for (int jj = 0; jj < kSub; ++jj) {
                const uint8_t* ra = ks + (ua0 + 4 * jj) * (2 * D);
                const uint8_t* rb = ra + 2 * (2 * D);
                // four independent accumulation chains (even / odd r, low / high half of the chunk)
                float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
                float c3[4] = {0.f, 0.f, 0.f, 0.f}, c4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int r = 0; r < D / 32; ++r) {
                    const uint4 ka = ld_shared_v4(ra + 16 * (4 * r + tig));
                    const uint4 kb = ld_shared_v4(rb + 16 * (4 * r + tig));
                    mma_bf16_16816((r & 1) ? c3 : c, ka.x, kb.x, ka.y, kb.y, qf[r][0], qf[r][1]);
                    mma_bf16_16816((r & 1) ? c4 : c2, ka.z, kb.z, ka.w, kb.w, qf[r][2], qf[r][3]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) x[jj][i] = ((c[i] + c3[i]) + (c2[i] + c4[i])) * p.scale_log2;
                if (!full) {
                    if (ua0 + 4 * jj >= nv) x[jj][0] = x[jj][1] = -INFINITY;
                    if (ua0 + 4 * jj + 2 >= nv) x[jj][2] = x[jj][3] = -INFINITY;
                }
            }
            // this lane's largest scores of its two heads
            float mx0 = fmaxf(x[0][0], x[0][2]), mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
            for (int jj = 1; jj < kSub; ++jj) {
                mx0 = fmaxf(mx0, fmaxf(x[jj][0], x[jj][2]));
                mx1 = fmaxf(mx1, fmaxf(x[jj][1], x[jj][3]));
            }
            // The probabilities are taken against a reference per head (m0, m1): kept from the earlier steps
            // while no score of this step exceeds it by more than kSlack (one vote instead of a reduction),
            // else raised to the running maximum, with the sums so far rescaled.  A probability is then at
            // most 2^kSlack, which the fp32 sums and the bf16 hi + lo split carry to the same precision;
            // (m, l, O) stay consistent, which is all the merge and lse use.
            constexpr float kSlack = 8.f;
            if (!__all_sync(kFullMask, mx0 <= m0 + kSlack && mx1 <= m1 + kSlack)) {
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, off));
                }
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float a0 = mn0 == -INFINITY ? 1.f : fast_exp2(m0 - mn0);
                const float a1 = mn1 == -INFINITY ? 1.f : fast_exp2(m1 - mn1);
                l0 *= a0;
                l1 *= a1;
                if (__any_sync(kFullMask, (a0 != 1.f) || (a1 != 1.f))) {
#pragma unroll
                    for (int i = 0; i < kMTiles; ++i) {
                        o[i][0] *= a0;
                        o[i][1] *= a1;
                        o[i][2] *= a0;
                        o[i][3] *= a1;
                    }
                }
                m0 = mn0;
                m1 = mn1;
            }
            const float ref0 = m0 == -INFINITY ? 0.f : m0;
            const float ref1 = m1 == -INFINITY ? 0.f : m1;
            float pr[kSub][4];
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int jj = 0; jj < kSub; ++jj) {
#pragma unroll
                for (int i = 0; i < 4; ++i) pr[jj][i] = fast_exp2(x[jj][i] - ((i & 1) ? ref1 : ref0));
                ps0 += pr[jj][0] + pr[jj][2];
                ps1 += pr[jj][1] + pr[jj][3];
            }
            l0 += ps0;
            l1 += ps1;
            uint32_t bh[kSub][2], bl[kSub][2];
#pragma unroll
            for (int jj = 0; jj < kSub; ++jj) {
                const uint32_t h01 = pack_bf16x2(pr[jj][0], pr[jj][1]), h23 = pack_bf16x2(pr[jj][2], pr[jj][3]);
                const uint32_t r01 = pack_bf16x2(pr[jj][0] - bf16_lo(h01), pr[jj][1] - bf16_hi(h01));
                const uint32_t r23 = pack_bf16x2(pr[jj][2] - bf16_lo(h23), pr[jj][3] - bf16_hi(h23));
                bh[jj][0] = movmatrix_trans(h01);
                bh[jj][1] = movmatrix_trans(h23);
                bl[jj][0] = movmatrix_trans(r01);
                bl[jj][1] = movmatrix_trans(r23);
            }
            // O^T += V^T P^T: lane reads tokens u0 .. u0 + 4*kSub - 1 of dims 16i+gid, 16i+gid+8
            const int u0 = 4 * kSub * tig;
            const uint8_t* vrow = vs + u0 * 2;
            bool vk[4 * kSub];
            if (!full) {
#pragma unroll
                for (int e = 0; e < 4 * kSub; ++e) vk[e] = u0 + e < nv;
            }
#pragma unroll
            for (int i = 0; i < kMTiles; ++i) {
                if constexpr (kSub == 2) {
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
                } else {
                    uint2 wa = ld_shared_v2(vrow + (16 * i + gid) * (T * 2));
                    uint2 wb = ld_shared_v2(vrow + (16 * i + gid + 8) * (T * 2));
                    if (!full) {
                        wa = make_uint2(keep_halves(wa.x, vk[0], vk[1]), keep_halves(wa.y, vk[2], vk[3]));
                        wb = make_uint2(keep_halves(wb.x, vk[0], vk[1]), keep_halves(wb.y, vk[2], vk[3]));
                    }
                    mma_bf16_16816(o[i], wa.x, wb.x, wa.y, wb.y, bh[0][0], bh[0][1]);
                    mma_bf16_16816(o[i], wa.x, wb.x, wa.y, wb.y, bl[0][0], bl[0][1]);
                }
            }
        };
        // a page receiving tokens in this launch may have been copied before or after the selector
        // warps wrote them to the pools: its slot takes those rows from new_k / new_v
        auto patch_page = [&](int j, int lp, uint8_t* slot) {
            constexpr int kDimsPerLane = D / 32;
            const DUnit& u = sh.ud[j];
            const int first = lp * T;
            const int r0 = max(u.tb - first, 0), r1 = min(u.te - first, T);
            const size_t src_base = (static_cast<size_t>(u.b) * p.Hkv + u.h) * p.n_new;
            kvmm_bf16* vt = reinterpret_cast<kvmm_bf16*>(slot + kPageBytes);  // value d of token r at [d*T + r]
            if (u.te - u.tb == 1) {  // the token's rows, staged by the selector warps
                wait_prep();
                if (lane < D / 8)
                    *reinterpret_cast<uint4*>(slot + static_cast<size_t>(r0) * 2 * D + 16 * lane) = sh.nrow[j][lane];
                const kvmm_bf16* vsrc = reinterpret_cast<const kvmm_bf16*>(&sh.nrow[j][D / 8]) + kDimsPerLane * lane;
#pragma unroll
                for (int e = 0; e < kDimsPerLane; ++e) vt[static_cast<size_t>(kDimsPerLane * lane + e) * T + r0] = vsrc[e];
                __syncwarp();
                return;
            }
            for (int r = r0; r < r1; ++r) {
                const size_t jj = src_base + (first + r - u.tb);
                if (lane < D / 8)
                    *reinterpret_cast<uint4*>(slot + static_cast<size_t>(r) * 2 * D + 16 * lane) =
                        reinterpret_cast<const uint4*>(p.new_k + jj * D)[lane];
                const kvmm_bf16* vsrc = p.new_v + jj * D + kDimsPerLane * lane;
#pragma unroll
                for (int e = 0; e < kDimsPerLane; ++e) vt[static_cast<size_t>(kDimsPerLane * lane + e) * T + r] = vsrc[e];
            }
            __syncwarp();
        };
        auto issue_att = [&](int b2, int j, int s) {  // step s of unit j: page s of this CTA's share
            if (lane == 0) mbar_arrive_expect_tx(&sh.full[w][b2], 2u * kPageBytes);
            __syncwarp();
            const int cl = lane - 2 * b2;  // the slot's own copying lanes, as for the scores
            if (cl == 0 || cl == 1) {  // lane cl = 0 copies the page's keys, cl = 1 its values
                uint8_t* dst = my_ring + size_t(b2) * kSlot + cl * kPageBytes;
                const size_t off = static_cast<size_t>(res[size_t(j) * p.maxp + s].x) * T * D;
                bulk_copy_g2s_hint(dst, (cl ? p.v_pool : p.k_pool) + off, kPageBytes, &sh.full[w][b2],
                                   stream_policy);
            }
            set_slot(b2, j, s);
        };
        bool next_known = false;  // the next unit's pages are resolved and its steps may be fetched
        int next_nx = w;          // the next unit's next step to fetch
        int b = 0;                // the slot consumed next: the oldest in flight, if any is
        for (int j = 0; j < nunits; ++j) {
            if (!(j > 0 && next_known)) wait_bar_warp(&sh.selr[j], 0);
            const int n = sh.resn[j];
            int nx = j > 0 && next_known ? next_nx : w;
            next_known = false;
            next_nx = w;
            load_frags(j, true);
            if (kRing == 2 && !in_flight(b) && in_flight(b ^ 1)) b ^= 1;
            for (int t = 0; t < kRing; ++t) {
                const int bb = (b + t) % kRing;
                if (!in_flight(bb) && nx < n) {
                    issue_att(bb, j, nx);
                    nx += kDCons;
                }
            }
            const int jn = j + 1;
            for (; in_flight(b) && (b ? hj1 : hj0) == j; b = (b + 1) % kRing) {
                const int lp = res[size_t(j) * p.maxp + (b ? hs1 : hs0)].y;
                const int nv = min(T, sh.ud[j].seq - lp * T);
                uint8_t* slot = my_ring + size_t(b) * kSlot;
                land(b);
                if (sh.ud[j].te > lp * T && sh.ud[j].tb < (lp + 1) * T) patch_page(j, lp, slot);
                att_step(slot, nv);
                __syncwarp();
                fence_proxy_async_shared();  // this slot's reads, then the next copy into it
                if (nx < n) {
                    issue_att(b, j, nx);
                    nx += kDCons;
                } else if (jn < nunits) {
                    if (!next_known && __all_sync(kFullMask, mbar_try_wait(&sh.selr[jn], 0))) next_known = true;
                    if (next_known && next_nx < sh.resn[jn]) {
                        issue_att(b, jn, next_nx);
                        next_nx += kDCons;
                    }
                }
            }

            // ---- end of the unit: this warp's partial, which the selector warps combine
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0 += __shfl_xor_sync(kFullMask, l0, off);
                l1 += __shfl_xor_sync(kFullMask, l1, off);
            }
            if (j > 0) wait_bar_warp(&sh.pfree, 0);  // the previous unit's partials have been read
            if (gid == 0) {
                sh.mm[w][2 * tig] = m0;
                sh.mm[w][2 * tig + 1] = m1;
                sh.ml[w][2 * tig] = l0;
                sh.ml[w][2 * tig + 1] = l1;
            }
            // [G heads][D + 4]: the padding spreads the four tig lanes over distinct banks
            float* mw = part + size_t(w) * G * (D + 4);
            const bool h0 = 2 * tig < G, h1 = 2 * tig + 1 < G;
#pragma unroll
            for (int i = 0; i < kMTiles; ++i) {
                float* w0 = mw + (2 * tig) * (D + 4);
                float* w1 = w0 + (D + 4);
                if (h0) {
                    w0[16 * i + gid] = o[i][0];
                    w0[16 * i + gid + 8] = o[i][2];
                }
                if (h1) {
                    w1[16 * i + gid] = o[i][1];
                    w1[16 * i + gid + 8] = o[i][3];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.pready[j]);  // release: the partial above
#pragma unroll
            for (int i = 0; i < kMTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }
        }  // kAttend
        // No copy into this CTA's shared memory may still be in flight when it exits.  Only after a time-out
        // can a slot be: it gets the full limit to land, whatever happened before.  The query groups' copy
        // is waited for by the warps that use them, so when no consumer warp had work, warp 0 waits for it.
        for (int bb = 0; bb < kRing; ++bb)
            if (in_flight(bb) && !__all_sync(kFullMask, mbar_wait_bounded(&sh.full[w][bb], (par >> bb) & 1u, kDWaitNs)) &&
                lane == 0)
                set_abort();
        if (w == 0 && !__all_sync(kFullMask, mbar_wait_bounded(&sh.qbar, 0, kDWaitNs)) && lane == 0) set_abort();
    }
    // No final cluster barrier: every access another CTA makes to this one's shared memory is an
    // asynchronous store counted by one of this CTA's mbarriers (scores, partials), and the selector
    // warps have waited for all of them by now -- unless one of those waits timed out (KVMM_ERR_TIMEOUT),
    // after which a peer's late store may still be on its way: the time-outs turn a hang into an error,
    // they do not make the launch's results or its exit safe.
}

}  // namespace dl

// the decode kernel for a shape's (D, T, group reduction, units per cluster), one function per phase set,
// each in its own translation unit
using DecodeKernel = void (*)(DecodeParams, CUtensorMap);
DecodeKernel decode_kernel_both(int D, int T, int mode, int nu);    // decode_layer.cu
DecodeKernel decode_kernel_score(int D, int T, int mode, int nu);   // decode_score.cu
DecodeKernel decode_kernel_attend(int D, int T, int nu);            // decode_attend.cu

}  // namespace kvmm
