// sparse_decode.cu -- GQA decode attention over the selected pages only,
// split across CTAs and merged by log-sum-exp.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 1. Stability-
// differentiated placement": decode attention runs over the top-K pages even
// where the full KV is resident; "System design, head-level block table":
// pages are found through [batch, layer, head, logical_block] and null
// entries are never read.
//
// Design (sm_103a).  The selected pages of one (batch, KV head) are split
// over `splits` CTAs.  A CTA first resolves its pages through the block table
// into a compacted list (null / out-of-range entries dropped and reported),
// then its warps take steps of 32 tokens (two 16-token pages or one 32-token
// page) round robin.  Each warp keeps kSteps steps in flight in a private ring
// (eight warps of one step: 128 KiB per CTA at D = 128):
// every page's K block ([T][D]) and V block ([D][T]) is one contiguous run of
// bytes, moved by a 1-D bulk copy (TMA) into shared memory, the copies of a
// step issued from different lanes and completing on one mbarrier.
//
// Per 16-token sub-tile the GQA group is a small dense contraction on the
// tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate):
//   S^T[16 tok x 8 head] = K[16 x D] * Q^T[D x 8]          (D/16 MMAs)
//   O^T[D x 8 head]     += V^T[D x 16] * P^T[16 x 8]        (2*D/16 MMAs)
// Tokens and head dimensions are visited in fixed permuted orders (the same
// on both sides of each contraction): a lane's K fragment is a 16-byte load
// of two token rows, and, because values are stored dimension-major, a lane's
// V^T fragments for both sub-tiles of a step are one 16-byte load per
// dimension row.  P = exp2(S*scale*log2e - m) is split into bf16 hi + lo parts
// (two MMAs) so the probabilities keep ~16 bits, and is moved from the S^T
// accumulator layout to the B-operand layout with movmatrix.  Softmax
// statistics are online per warp, merged across warps in shared memory and
// across the splits of a unit (one thread-block cluster) by remote
// shared-memory stores and one cluster barrier.  With `select`, rescored
// units first pick their pages from the layer's scores (block_topk, every CTA
// of the cluster computing the same selection).  The kernel is launched with
// programmatic dependent launch and waits for its predecessor before reading
// any input.
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "topk_block.cuh"

#ifndef KVMM_ATTN_WARPS
#define KVMM_ATTN_WARPS 8
#endif
#ifndef KVMM_ATTN_STEPS
#define KVMM_ATTN_STEPS 1
#endif

namespace kvmm {
namespace {

constexpr int kAttnWarps = KVMM_ATTN_WARPS;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kSteps = KVMM_ATTN_STEPS;  // steps in flight per warp
constexpr int kStepTok = 32;             // tokens per step (two 16-token sub-tiles)
static_assert(kSteps >= 1, "at least one step in flight per warp");

__host__ __device__ constexpr int step_bytes(int D) { return 2 * kStepTok * D * 2; }  // K then V
__host__ __device__ constexpr size_t ring_bytes(int D) { return size_t(kAttnWarps) * kSteps * step_bytes(D); }
__host__ __device__ constexpr size_t combine_bytes(int D) { return size_t(kAttnWarps) * 8 * D * sizeof(float); }
__host__ __device__ constexpr size_t ring_region(int D)
{
    return ring_bytes(D) > combine_bytes(D) ? ring_bytes(D) : combine_bytes(D);
}

constexpr int kMaxSplits = kAttnMaxSplits;  // CTAs of one unit = one thread-block cluster

// selection scratch, laid over the ring before streaming starts:
// [BlockTopkShared][scores: Pmax fp32][bins: Pmax int16][selection: Kmax int32]
__host__ __device__ constexpr size_t align16(size_t n) { return (n + 15) & ~static_cast<size_t>(15); }
__host__ __device__ constexpr size_t select_scratch_offset_scores()
{
    return align16(sizeof(BlockTopkShared<kAttnThreads>));
}
__host__ __device__ constexpr size_t select_scratch_offset_sel(int Pmax)
{
    return align16(select_scratch_offset_scores() + size_t(Pmax) * (sizeof(float) + sizeof(int16_t)));
}

struct AttnShared {
    uint64_t bar[kAttnWarps][kSteps];
    uint64_t bt_bar;                  // the unit's block-table row (selecting kernel)
    float m[kAttnWarps][8];
    float l[kAttnWarps][8];
    float fw[kAttnWarps][8];          // weight of each warp's partial in the CTA's
    float fc[kMaxSplits][8];          // weight of each CTA's partial in the unit's
    float inv_l[8];
    float rstat[kMaxSplits][16];      // received: (m, l) per head of every CTA of the cluster
    float ro[8 * 128 + kMaxSplits];   // received: every CTA's partial of this CTA's output slice
    int wcount[kAttnWarps];
};

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// keep the bf16 halves of w whose tokens are valid
__device__ __forceinline__ uint32_t keep_halves(uint32_t w, bool lo, bool hi)
{
    return w & ((lo ? 0x0000ffffu : 0u) | (hi ? 0xffff0000u : 0u));
}

template <int D, int T, bool SELECT>
__global__ void __launch_bounds__(kAttnThreads) sparse_attn_kernel(const AttnParams p)
{
    constexpr int kPPS = kStepTok / T;      // pages per step
    constexpr int kPageBytes = T * D * 2;   // a page's K (or V) block
    constexpr int kMTiles = D / 16;         // m-tiles of O^T
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ AttnShared sh;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int gid = lane >> 2;  // fragment row group
    const int tig = lane & 3;   // thread in group
    const int split = blockIdx.x;
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    const int G = p.G;

    uint8_t* ring = smem;
    // the ring (or, before streaming, the selection scratch) spans p.region0 bytes
    int64_t* pg_row = reinterpret_cast<int64_t*>(smem + p.region0);  // physical page of list entry
    int* pg_nv = reinterpret_cast<int*>(pg_row + p.max_tiles);       // its valid tokens

    const size_t unit = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;

    if (tid < kAttnWarps * kSteps) mbar_init(&sh.bar[tid / kSteps][tid % kSteps], 1);
    if (tid == 0) mbar_init(&sh.bt_bar, 1);
    fence_barrier_init();
    pdl_wait_then_release();  // every input may come from the preceding kernels

    // Q^T as B fragments: lane (gid, tig) holds head gid, 16-byte chunk 4r+tig
    uint32_t qf[D / 32][4];
    {
        const kvmm_bf16* qh = p.q + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * G + gid) * D;
#pragma unroll
        for (int r = 0; r < D / 32; ++r) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (gid < G) v = *reinterpret_cast<const uint4*>(qh + 8 * (4 * r + tig));
            qf[r][0] = v.x;
            qf[r][1] = v.y;
            qf[r][2] = v.z;
            qf[r][3] = v.w;
        }
    }

    int seq = p.seq_len[b];
    const int cap = p.Pmax * T;
    if (seq < 0 || seq > cap) {
        if (split == 0 && tid == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
        seq = seq < 0 ? 0 : cap;
    }
    const int P = (seq + T - 1) / T;
    const int32_t* sel_src = p.sel_idx + unit * p.Kmax;
    const bool selecting = SELECT && (p.rescore_mask == nullptr || p.rescore_mask[p.layer * p.Hkv + h] != 0);
    // the selecting kernel fetches the unit's block-table row while it selects
    const bool bt_prefetch = selecting && p.bt_prefetch && P > 0;
    int32_t* bt_s = reinterpret_cast<int32_t*>(smem + p.bt_offset);
    if (bt_prefetch && tid == 0) {
        const uint32_t bytes = static_cast<uint32_t>((P + 3) / 4) * 16;  // within the 16-byte aligned row
        mbar_arrive_expect_tx(&sh.bt_bar, bytes);
        bulk_copy_g2s(bt_s, p.block_table + unit * p.Pmax, bytes, &sh.bt_bar);
    }
    int cnt;
    if (selecting) {
        // select this unit's pages from its scores (every CTA of the cluster
        // computes the same selection; split 0 also writes it out)
        auto& ts = *reinterpret_cast<BlockTopkShared<kAttnThreads>*>(smem);
        float* sc_s = reinterpret_cast<float*>(smem + select_scratch_offset_scores());
        int16_t* bin_s = reinterpret_cast<int16_t*>(sc_s + p.Pmax);
        int32_t* sel_s = reinterpret_cast<int32_t*>(smem + select_scratch_offset_sel(p.Pmax));
        cnt = block_topk<kAttnThreads>(p.scores + static_cast<size_t>(b * p.Hkv + h) * p.pstride, P, p.K, sel_s,
                                       sc_s, bin_s, ts);
        if (split == 0) {
            for (int i = tid; i < cnt; i += kAttnThreads) p.sel_out[unit * p.Kmax + i] = sel_s[i];
            if (tid == 0) p.cnt_out[unit] = cnt;
        }
        sel_src = sel_s;
    } else {
        cnt = p.sel_cnt[unit];
        if (cnt < 0 || cnt > p.Kmax) {
            if (split == 0 && tid == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
            cnt = cnt < 0 ? 0 : p.Kmax;
        }
    }
    const int beg = static_cast<int>(static_cast<long long>(cnt) * split / p.splits);
    const int end = static_cast<int>(static_cast<long long>(cnt) * (split + 1) / p.splits);

    bool bt_ok = bt_prefetch;
    if (bt_prefetch) bt_ok = __syncthreads_and(mbar_wait_bounded(&sh.bt_bar, 0)) != 0;
    if (bt_prefetch && !bt_ok && tid == 0) report(p.err, KVMM_ERR_TIMEOUT);  // read the table directly instead

    // resolve this CTA's pages and compact the valid ones (in selection order)
    int n_valid = 0;
    for (int i0 = beg; i0 < end; i0 += kAttnThreads) {
        const int i = i0 + tid;
        int64_t row = -1;
        int nv = 0;
        if (i < end) {
            const int lp = sel_src[i];
            if (lp < 0 || lp >= P) {
                report(p.err, KVMM_ERR_OUT_OF_RANGE);
            } else {
                const int32_t phys = bt_ok ? bt_s[lp] : p.block_table[unit * p.Pmax + lp];
                if (phys < 0) {
                    report(p.err, KVMM_ERR_NULL_BLOCK);
                } else if (phys >= p.n_phys) {
                    report(p.err, KVMM_ERR_OUT_OF_RANGE);
                } else {
                    nv = min(T, seq - lp * T);
                    if (nv > 0) row = phys;
                }
            }
        }
        const bool ok = row >= 0;
        const unsigned bal = __ballot_sync(kFullMask, ok);
        if (lane == 0) sh.wcount[warp] = __popc(bal);
        __syncthreads();
        int pos = n_valid, tot = 0;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) {
            if (w < warp) pos += sh.wcount[w];
            tot += sh.wcount[w];
        }
        if (ok) {
            pos += __popc(bal & ((1u << lane) - 1u));
            pg_row[pos] = row;
            pg_nv[pos] = nv;
        }
        n_valid += tot;
        __syncthreads();
    }

    float o[kMTiles][4];
#pragma unroll
    for (int i = 0; i < kMTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    // steps of this CTA: step s covers list entries [s*kPPS, s*kPPS + kPPS); warp w takes s = w, w + warps, ...
    const int n_steps = (n_valid + kPPS - 1) / kPPS;
    const int my_steps = n_steps > warp ? (n_steps - warp + kAttnWarps - 1) / kAttnWarps : 0;
    uint8_t* my_ring = ring + static_cast<size_t>(warp) * kSteps * step_bytes(D);

    auto issue = [&](int k) {  // fetch the warp's k-th step into slot k % kSteps
        const int s = warp + k * kAttnWarps;
        uint8_t* slot = my_ring + static_cast<size_t>(k % kSteps) * step_bytes(D);
        uint64_t* bar = &sh.bar[warp][k % kSteps];
        const int npages = min(kPPS, n_valid - s * kPPS);
        if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(npages) * 2 * kPageBytes);
        __syncwarp();
        if (lane < 2 * npages) {  // lane 2j copies page j's keys, lane 2j+1 its values
            const int j = lane >> 1;
            const size_t off = static_cast<size_t>(pg_row[s * kPPS + j]) * T * D;
            if ((lane & 1) == 0)
                bulk_copy_g2s(slot + j * kPageBytes, p.k_pool + off, kPageBytes, bar);
            else
                bulk_copy_g2s(slot + kStepTok * D * 2 + j * kPageBytes, p.v_pool + off, kPageBytes, bar);
        }
    };
#pragma unroll
    for (int k = 0; k < kSteps; ++k)
        if (k < my_steps) issue(k);

    // token u of a step: page u / T (within the step), row u % T.  Sub-tile j,
    // fragment row rho holds token 8*((rho&7)>>1) + 4j + 2*(rho>>3) + (rho&1).
    const int ua0 = 8 * (gid >> 1) + (gid & 1);  // rows gid (+2 for gid+8), sub-tile 0 (+4 for sub-tile 1)
    bool timed_out = false;
    int k_stop = my_steps;  // first step not consumed
    for (int k = 0; k < my_steps; ++k) {
        const int s = warp + k * kAttnWarps;
        const bool ok = mbar_wait_bounded(&sh.bar[warp][k % kSteps], (k / kSteps) & 1);
        if (__any_sync(kFullMask, !ok)) {  // warp-uniform decision
            timed_out = true;
            k_stop = k;
            break;
        }
        const uint8_t* ks = my_ring + static_cast<size_t>(k % kSteps) * step_bytes(D);
        const uint8_t* vs = ks + kStepTok * D * 2;
        // valid tokens of the step's pages (a missing second page has none)
        const int nv0 = pg_nv[s * kPPS];
        const int nv1 = (kPPS == 2 && s * kPPS + 1 < n_valid) ? pg_nv[s * kPPS + 1] : 0;
        const bool full = (kPPS == 2) ? (nv0 == T && nv1 == T) : (nv0 == T);
        auto valid = [&](int u) { return kPPS == 2 ? ((u >> 4) ? (u & 15) < nv1 : u < nv0) : u < nv0; };

        // ---- S^T = K Q^T for both sub-tiles ------------------------------
        float x[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint8_t* ra = ks + (ua0 + 4 * j) * (2 * D);
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
            for (int i = 0; i < 4; ++i) x[j][i] = ((c[i] + c3[i]) + (c2[i] + c4[i])) * p.scale_log2;
            if (!full) {
                if (!valid(ua0 + 4 * j)) x[j][0] = x[j][1] = -INFINITY;
                if (!valid(ua0 + 4 * j + 2)) x[j][2] = x[j][3] = -INFINITY;
            }
        }
        // x[j]: [row gid][head 2tig], [gid][2tig+1], [gid+8][2tig], [gid+8][2tig+1]
        // this lane's largest scores of its two heads
        float mx0 = fmaxf(fmaxf(x[0][0], x[0][2]), fmaxf(x[1][0], x[1][2]));
        float mx1 = fmaxf(fmaxf(x[0][1], x[0][3]), fmaxf(x[1][1], x[1][3]));
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
        float pr[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) pr[j][i] = fast_exp2(x[j][i] - ((i & 1) ? ref1 : ref0));
        l0 += (pr[0][0] + pr[0][2]) + (pr[1][0] + pr[1][2]);
        l1 += (pr[0][1] + pr[0][3]) + (pr[1][1] + pr[1][3]);

        // ---- P^T as bf16 hi + lo B fragments (k order = the token order above)
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

        // ---- O^T += V^T P^T: lane reads tokens 8tig .. 8tig+7 of dims 16i+gid, 16i+gid+8
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
            // sub-tile 0: tokens u0..u0+3 (words x, y); sub-tile 1: u0+4..u0+7 (z, w)
            mma_bf16_16816(o[i], wa.x, wb.x, wa.y, wb.y, bh[0][0], bh[0][1]);
            mma_bf16_16816(o[i], wa.x, wb.x, wa.y, wb.y, bl[0][0], bl[0][1]);
            mma_bf16_16816(o[i], wa.z, wb.z, wa.w, wb.w, bh[1][0], bh[1][1]);
            mma_bf16_16816(o[i], wa.z, wb.z, wa.w, wb.w, bl[1][0], bl[1][1]);
        }

        // ---- release the slot and refill it ------------------------------
        __syncwarp();
        fence_proxy_async_shared();
        if (k + kSteps < my_steps) issue(k + kSteps);
    }
    if (timed_out) {
        if (lane == 0) report(p.err, KVMM_ERR_TIMEOUT);
        // let copies still in flight land before the CTA leaves (bounded)
        for (int k = k_stop; k < min(my_steps, k_stop + kSteps); ++k)
            mbar_wait_bounded(&sh.bar[warp][k % kSteps], (k / kSteps) & 1, 100000000ull);
    }

    // ---- merge: the CTA's warps, then the cluster's CTAs -------------------
    // Each warp leaves (m, l) per head and its unnormalised O^T in its own
    // ring slot; the CTA combines them into one partial and stores into every
    // CTA of the cluster (the unit's splits) the slice of the outputs that CTA
    // owns (remote shared-memory stores).  After one cluster barrier every CTA
    // combines the partials of its slice locally and writes it out.
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(kFullMask, l0, off);
        l1 += __shfl_xor_sync(kFullMask, l1, off);
    }
    float* my_o = reinterpret_cast<float*>(my_ring);  // [8 heads][D]; this warp's copies are all consumed
    if (gid == 0) {
        sh.m[warp][2 * tig] = m0;
        sh.m[warp][2 * tig + 1] = m1;
        sh.l[warp][2 * tig] = l0;
        sh.l[warp][2 * tig + 1] = l1;
    }
#pragma unroll
    for (int i = 0; i < kMTiles; ++i) {
        float* w0 = my_o + (2 * tig) * D;
        float* w1 = w0 + D;
        w0[16 * i + gid] = o[i][0];
        w1[16 * i + gid] = o[i][1];
        w0[16 * i + gid + 8] = o[i][2];
        w1[16 * i + gid + 8] = o[i][3];
    }
    __syncthreads();

    const int nsp = p.splits;  // CTAs in the cluster
    const uint32_t rank = cluster_ctarank();
    const int n_out = G * D;
    const int slice = (n_out + nsp - 1) / nsp;  // outputs owned by each CTA
    if (tid < G) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, sh.m[w][tid]);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) {
            const float mw = sh.m[w][tid];
            const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
            sh.fw[w][tid] = f;
            L = fmaf(sh.l[w][tid], f, L);
        }
        for (int r = 0; r < nsp; ++r) {
            st_dsmem_f32(&sh.rstat[rank][tid], r, M);
            st_dsmem_f32(&sh.rstat[rank][8 + tid], r, L);
        }
    }
    __syncthreads();
    for (int e = tid; e < n_out; e += kAttnThreads) {
        const int g = e / D;
        float O = 0.f;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w)
            O = fmaf(sh.fw[w][g], reinterpret_cast<const float*>(ring + static_cast<size_t>(w) * kSteps * step_bytes(D))[e], O);
        const int r = e / slice;
        st_dsmem_f32(&sh.ro[rank * slice + (e - r * slice)], r, O);
    }
    cluster_sync();  // every CTA's partial of every slice has arrived

    if (tid < G) {
        float M = -INFINITY;
        for (int c = 0; c < nsp; ++c) M = fmaxf(M, sh.rstat[c][tid]);
        float L = 0.f;
        for (int c = 0; c < nsp; ++c) {
            const float mc = sh.rstat[c][tid];
            const float f = (mc == -INFINITY) ? 0.f : exp2f(mc - M);
            sh.fc[c][tid] = f;
            L = fmaf(sh.rstat[c][8 + tid], f, L);
        }
        sh.inv_l[tid] = L > 0.f ? 1.f / L : 0.f;
        if (rank == 0 && p.lse) {
            const size_t oi = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * G + tid;
            p.lse[oi] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
        }
    }
    __syncthreads();
    const int e0 = static_cast<int>(rank) * slice;
    const int e1 = min(n_out, e0 + slice);
    float* ob = p.out + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * G) * D;
    for (int e = e0 + tid; e < e1; e += kAttnThreads) {
        const int g = e / D;
        float O = 0.f;
        for (int c = 0; c < nsp; ++c) O = fmaf(sh.fc[c][g], sh.ro[c * slice + (e - e0)], O);
        ob[e] = O * sh.inv_l[g];
    }
}

template <int D, int T>
void (*attn_kernel(bool select))(AttnParams)
{
    return select ? sparse_attn_kernel<D, T, true> : sparse_attn_kernel<D, T, false>;
}

void (*attn_kernel_for(int D, int T, bool select))(AttnParams)
{
    if (D == 128) return T == 16 ? attn_kernel<128, 16>(select) : attn_kernel<128, 32>(select);
    return T == 16 ? attn_kernel<64, 16>(select) : attn_kernel<64, 32>(select);
}

// opt-ins of one kernel instantiation, once per device
cudaError_t prepare_attn(void (*kernel)(AttnParams), size_t smem)
{
    struct Prepared {
        void (*kernel)(AttnParams);
        int dev;
        size_t bytes;
    };
    static thread_local Prepared cache[8] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    for (auto& c : cache)
        if (c.kernel == kernel && c.dev == dev && c.bytes >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    for (auto& c : cache)
        if (c.kernel == kernel || c.kernel == nullptr) {
            c = {kernel, dev, smem};
            break;
        }
    return cudaSuccess;
}

size_t region0_bytes(int D, size_t scratch)
{
    const size_t r = ring_region(D) > scratch ? ring_region(D) : scratch;
    return (r + 15) & ~static_cast<size_t>(15);
}

size_t attention_smem_bytes_impl(int D, int max_pages, size_t scratch)
{
    return region0_bytes(D, scratch) + size_t(max_pages) * (sizeof(int64_t) + sizeof(int));
}

// clusters of `c` attention CTAs the device holds at once (0 = not launchable)
int active_clusters(const kvmm_shape& s, int c, bool select)
{
    void (*kernel)(AttnParams) = attn_kernel_for(s.D, s.T, select);
    const size_t smem =
        attention_smem_bytes(s.D, (s.Kmax + c - 1) / c, select ? attention_select_scratch(s.Pmax, s.Kmax) : 0);
    if (prepare_attn(kernel, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c, 1, 1);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

struct SplitCache {
    int dev, D, T, Kmax, Pmax, units, select, splits, max_splits;
};
thread_local SplitCache g_split_cache[8] = {};
thread_local int g_split_next = 0;

SplitCache& split_entry(const kvmm_shape& s, bool select)
{
    int dev = 0;
    cudaGetDevice(&dev);
    const int units = s.B * s.Hkv;
    const int pm = select ? s.Pmax : 0;  // the selecting kernel's scratch depends on Pmax
    for (auto& c : g_split_cache)
        if (c.max_splits > 0 && c.dev == dev && c.D == s.D && c.T == s.T && c.Kmax == s.Kmax && c.Pmax == pm &&
            c.units == units && c.select == int(select))
            return c;
    SplitCache& c = g_split_cache[g_split_next++ % 8];
    c = {dev, s.D, s.T, s.Kmax, pm, units, int(select), 1, 1};
    // largest launchable cluster, and the largest split count whose clusters
    // for every unit fit on the device in one wave
    int best = 1;
    for (int k = 2; k <= kMaxSplits && k <= s.Kmax; ++k) {
        const int n = active_clusters(s, k, select);
        if (n <= 0) break;
        c.max_splits = k;
        if (n >= units) best = k;
    }
    c.splits = best;
    return c;
}

}  // namespace

int attention_max_splits(const kvmm_shape& s, bool select) { return split_entry(s, select).max_splits; }

int attention_slots_per_unit(const kvmm_shape& s, bool select) { return split_entry(s, select).splits; }

size_t attention_smem_bytes(int D, int max_pages, size_t scratch)
{
    return attention_smem_bytes_impl(D, max_pages, scratch);
}

size_t attention_region0(int D, size_t scratch) { return region0_bytes(D, scratch); }

size_t attention_select_scratch(int Pmax, int Kmax)
{
    return select_scratch_offset_sel(Pmax) + size_t(Kmax) * sizeof(int32_t);
}

cudaError_t launch_sparse_attention(const AttnParams& p, cudaStream_t stream)
{
    void (*kernel)(AttnParams) = attn_kernel_for(p.D, p.T, p.select != 0);
    size_t smem = static_cast<size_t>(p.region0) + size_t(p.max_tiles) * (sizeof(int64_t) + sizeof(int));
    if (p.bt_prefetch) smem = static_cast<size_t>(p.bt_offset) + size_t(p.Pmax) * sizeof(int32_t);
    const cudaError_t e = prepare_attn(kernel, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl_cluster(kernel, dim3(p.splits, p.Hkv, p.B), dim3(kAttnThreads), smem, stream,
                              static_cast<unsigned>(p.splits), p);
}

}  // namespace kvmm
