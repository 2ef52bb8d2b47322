// sparse_decode.cu -- GQA decode attention over the selected pages only,
// split across CTAs and merged by log-sum-exp.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 1. Stability-
// differentiated placement": decode attention runs over the top-K pages even
// where the full KV is resident; "System design, head-level block table":
// pages are found through [batch, layer, head, logical_block] and null
// entries are never read.
//
// Design (sm_103a).  The unit of transfer is a 16-token tile of a selected
// page (one tile per page at T = 16, two at T = 32): its K rows and V rows,
// each one contiguous 16*D*2-byte block, moved by two 1-D bulk copies (TMA)
// into shared memory and completing on an mbarrier.  The tiles of one (batch,
// KV head) are split over `splits` CTAs.  Each warp of a CTA walks its own
// tiles through a private ring of kRing slots, refilling a slot as soon as it
// is consumed, and computes two tiles per step (independent MMA chains,
// one softmax update per 32 tokens).
//
// Per tile the GQA group is a small dense contraction and runs on the tensor
// cores with mma.sync m16n8k16 (bf16 in, fp32 accumulate):
//   S^T[16 tok x 8 head]  = K_tile[16 x D] * Q^T[D x 8]            (D/16 MMAs)
//   O^T[D x 8 head]      += V_tile^T[D x 16] * P^T[16 x 8]          (2*D/16 MMAs)
// The K and V fragments are read straight from the bulk-copied row-major
// tile with 16-byte shared loads; the head dimension is visited in a fixed
// permuted order that is the same for Q and K (so S is unchanged) and is
// undone when O is written.  P = exp2(S*scale*log2e - m) is split into
// bf16 hi + lo parts (two MMAs) so the probabilities keep ~16 bits, and is
// moved from the S^T accumulator layout to the B-operand layout with
// movmatrix.  Softmax statistics are online per warp, merged across warps in
// shared memory and across splits by the last CTA of the unit (an atomic
// ticket; nothing spins).  The kernel is launched with programmatic
// dependent launch and waits for its predecessor before reading any input.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

#ifndef KVMM_ATTN_WARPS
#define KVMM_ATTN_WARPS 4
#endif
#ifndef KVMM_ATTN_RING
#define KVMM_ATTN_RING 4
#endif

namespace kvmm {
namespace {

constexpr int kAttnWarps = KVMM_ATTN_WARPS;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kRing = KVMM_ATTN_RING;  // tile slots per warp (>= 2: two tiles per step)
constexpr int kTileTok = 16;           // tokens per tile
static_assert(kRing >= 2, "two tiles per step need two slots");

__host__ __device__ constexpr int tile_bytes(int D) { return kTileTok * D * 2; }

__host__ __device__ constexpr size_t ring_bytes(int D) { return size_t(kAttnWarps) * kRing * 2 * tile_bytes(D); }

__host__ __device__ constexpr size_t combine_bytes(int D) { return size_t(kAttnWarps) * 8 * D * sizeof(float); }

__host__ __device__ constexpr size_t ring_region(int D)
{
    return ring_bytes(D) > combine_bytes(D) ? ring_bytes(D) : combine_bytes(D);
}

struct AttnShared {
    uint64_t bar[kAttnWarps][kRing];
    float m[kAttnWarps][8];
    float l[kAttnWarps][8];
    int last;
};

// S^T of one tile: c = K_tile Q^T over the head dimension, two MMA chains
template <int D>
__device__ __forceinline__ void tile_scores(const uint8_t* ks, const uint32_t (&qf)[D / 32][4], int gid, int tig,
                                            float (&c)[4])
{
    float c2[4] = {0.f, 0.f, 0.f, 0.f};
    c[0] = c[1] = c[2] = c[3] = 0.f;
#pragma unroll
    for (int r = 0; r < D / 32; ++r) {
        const uint4 ka = ld_shared_v4(ks + gid * (2 * D) + 16 * (4 * r + tig));
        const uint4 kb = ld_shared_v4(ks + (gid + 8) * (2 * D) + 16 * (4 * r + tig));
        mma_bf16_16816(c, ka.x, kb.x, ka.y, kb.y, qf[r][0], qf[r][1]);
        mma_bf16_16816(c2, ka.z, kb.z, ka.w, kb.w, qf[r][2], qf[r][3]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] += c2[i];
}

// O^T += V_tile^T P^T with P split into bf16 hi / lo B fragments
template <int D>
__device__ __forceinline__ void tile_accumulate(const uint8_t* vs, int nv, int gid, int tig, uint32_t bh0,
                                                uint32_t bh1, uint32_t bl0, uint32_t bl1, float (&o)[D / 16][4])
{
    constexpr int kDimsPerGroup = D / 8;
    // lane reads tokens 2tig, 2tig+1, 2tig+8, 2tig+9 at dims [gid*D/8, +D/8)
    uint32_t wv[4][kDimsPerGroup / 2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int tok = 2 * tig + (q & 1) + 8 * (q >> 1);
        const uint8_t* rowp = vs + tok * (2 * D) + gid * (2 * kDimsPerGroup);
#pragma unroll
        for (int c16 = 0; c16 < kDimsPerGroup / 8; ++c16) {
            const uint4 v = ld_shared_v4(rowp + 16 * c16);
            wv[q][4 * c16 + 0] = v.x;
            wv[q][4 * c16 + 1] = v.y;
            wv[q][4 * c16 + 2] = v.z;
            wv[q][4 * c16 + 3] = v.w;
        }
        if (nv < kTileTok && tok >= nv) {
#pragma unroll
            for (int i = 0; i < kDimsPerGroup / 2; ++i) wv[q][i] = 0u;
        }
    }
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
        // m-tile i rows: dim gid*D/8 + 2i (row gid) and +1 (row gid+8)
        const uint32_t a0 = prmt(wv[0][i], wv[1][i], 0x5410);
        const uint32_t a1 = prmt(wv[0][i], wv[1][i], 0x7632);
        const uint32_t a2 = prmt(wv[2][i], wv[3][i], 0x5410);
        const uint32_t a3 = prmt(wv[2][i], wv[3][i], 0x7632);
        mma_bf16_16816(o[i], a0, a1, a2, a3, bh0, bh1);
        mma_bf16_16816(o[i], a0, a1, a2, a3, bl0, bl1);
    }
}

// P^T (tokens x heads) of a tile as bf16 hi/lo B fragments for the PV MMA
__device__ __forceinline__ void p_fragments(float p0, float p1, float p2, float p3, uint32_t& bh0, uint32_t& bh1,
                                            uint32_t& bl0, uint32_t& bl1)
{
    const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
    const uint32_t r01 = pack_bf16x2(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
    const uint32_t r23 = pack_bf16x2(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
    bh0 = movmatrix_trans(h01);
    bh1 = movmatrix_trans(h23);
    bl0 = movmatrix_trans(r01);
    bl1 = movmatrix_trans(r23);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads) sparse_attn_kernel(const AttnParams p)
{
    constexpr int kMTiles = D / 16;  // m-tiles of O^T
    constexpr int kDimsPerGroup = D / 8;
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
    const int T = p.T;
    const int tiles_per_page = T / kTileTok;

    uint8_t* ring = smem;
    int64_t* t_row = reinterpret_cast<int64_t*>(smem + ring_region(D));
    int* t_nv = reinterpret_cast<int*>(t_row + p.max_tiles);

    const size_t unit = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
    const int wunit = b * p.Hkv + h;

    if (tid < kAttnWarps * kRing) mbar_init(&sh.bar[tid / kRing][tid % kRing], 1);
    fence_barrier_init();

    pdl_launch_dependents();
    pdl_wait();  // every input may come from the preceding kernels

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
    int cnt = p.sel_cnt[unit];
    if (cnt < 0 || cnt > p.Kmax) {
        if (split == 0 && tid == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
        cnt = cnt < 0 ? 0 : p.Kmax;
    }
    const int tiles = cnt * tiles_per_page;
    const int beg = static_cast<int>(static_cast<long long>(tiles) * split / p.splits);
    const int end = static_cast<int>(static_cast<long long>(tiles) * (split + 1) / p.splits);
    const int ntile = end - beg;

    // resolve this CTA's tiles through the selection and the block table
    for (int i = tid; i < ntile; i += kAttnThreads) {
        const int t = beg + i;
        const int lp = p.sel_idx[unit * p.Kmax + t / tiles_per_page];
        const int first = lp * T + (t % tiles_per_page) * kTileTok;
        int64_t row = -1;
        int nv = 0;
        if (lp < 0 || lp >= P) {
            report(p.err, KVMM_ERR_OUT_OF_RANGE);
        } else {
            const int32_t phys = p.block_table[unit * p.Pmax + lp];
            if (phys < 0) {
                report(p.err, KVMM_ERR_NULL_BLOCK);
            } else if (phys >= p.n_phys) {
                report(p.err, KVMM_ERR_OUT_OF_RANGE);
            } else {
                nv = min(kTileTok, seq - first);
                if (nv > 0) row = static_cast<int64_t>(phys) * T + (t % tiles_per_page) * kTileTok;
            }
        }
        t_row[i] = row;
        t_nv[i] = nv;
    }
    __syncthreads();

    float o[kMTiles][4];
#pragma unroll
    for (int i = 0; i < kMTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    uint8_t* my_ring = ring + static_cast<size_t>(warp) * kRing * 2 * tile_bytes(D);
    auto next_valid = [&](int i) {
        while (i < ntile && t_row[i] < 0) i += kAttnWarps;
        return i;
    };
    auto slot_ptr = [&](int ordinal) { return my_ring + static_cast<size_t>(ordinal % kRing) * 2 * tile_bytes(D); };

    // the warp's valid tiles, numbered 0, 1, ...: tile u lives in slot u % kRing
    int issue_i = next_valid(warp);  // list index of the next tile to fetch
    int issued = 0, consumed = 0;
    auto refill = [&]() {
        while (issued < consumed + kRing && issue_i < ntile) {
            if (lane == 0) {
                uint8_t* ks = slot_ptr(issued);
                uint64_t* bar = &sh.bar[warp][issued % kRing];
                const size_t off = static_cast<size_t>(t_row[issue_i]) * D;
                mbar_arrive_expect_tx(bar, 2 * tile_bytes(D));
                bulk_copy_g2s(ks, p.k_pool + off, tile_bytes(D), bar);
                bulk_copy_g2s(ks + tile_bytes(D), p.v_pool + off, tile_bytes(D), bar);
            }
            ++issued;
            issue_i = next_valid(issue_i + kAttnWarps);
        }
    };
    refill();

    bool timed_out = false;
    int cons_i = warp;
    while (consumed < issued) {
        // up to two tiles this step
        const int i0 = next_valid(cons_i);
        const bool two = consumed + 1 < issued;
        const int i1 = two ? next_valid(i0 + kAttnWarps) : i0;
        bool ok = mbar_wait_bounded(&sh.bar[warp][consumed % kRing], (consumed / kRing) & 1);
        if (two) ok = mbar_wait_bounded(&sh.bar[warp][(consumed + 1) % kRing], ((consumed + 1) / kRing) & 1) && ok;
        if (__any_sync(kFullMask, !ok)) {  // warp-uniform decision
            timed_out = true;
            break;
        }
        const uint8_t* ks0 = slot_ptr(consumed);
        const uint8_t* ks1 = slot_ptr(consumed + 1);
        const int nv0 = t_nv[i0];
        const int nv1 = two ? t_nv[i1] : 0;

        float ca[4], cb[4];
        tile_scores<D>(ks0, qf, gid, tig, ca);
        if (two) {
            tile_scores<D>(ks1, qf, gid, tig, cb);
        } else {
            cb[0] = cb[1] = cb[2] = cb[3] = 0.f;
        }
        // c = S^T[tok gid][head 2tig], [gid][2tig+1], [gid+8][2tig], [gid+8][2tig+1]
        float x[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[i] = ca[i] * p.scale_log2;
            x[4 + i] = cb[i] * p.scale_log2;
        }
        if (nv0 < kTileTok) {
            if (gid >= nv0) x[0] = x[1] = -INFINITY;
            if (gid + 8 >= nv0) x[2] = x[3] = -INFINITY;
        }
        if (nv1 < kTileTok) {  // also masks the absent second tile (nv1 = 0)
            if (gid >= nv1) x[4] = x[5] = -INFINITY;
            if (gid + 8 >= nv1) x[6] = x[7] = -INFINITY;
        }
        float mx0 = fmaxf(fmaxf(x[0], x[2]), fmaxf(x[4], x[6]));
        float mx1 = fmaxf(fmaxf(x[1], x[3]), fmaxf(x[5], x[7]));
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
        const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
        const float a0 = exp2f(m0 - ref0), a1 = exp2f(m1 - ref1);
        float pr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) pr[i] = exp2f(x[i] - ((i & 1) ? ref1 : ref0));
        l0 = fmaf(l0, a0, (pr[0] + pr[2]) + (pr[4] + pr[6]));
        l1 = fmaf(l1, a1, (pr[1] + pr[3]) + (pr[5] + pr[7]));
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

        uint32_t bh0, bh1, bl0, bl1;
        p_fragments(pr[0], pr[1], pr[2], pr[3], bh0, bh1, bl0, bl1);
        tile_accumulate<D>(ks0 + tile_bytes(D), nv0, gid, tig, bh0, bh1, bl0, bl1, o);
        if (two) {
            p_fragments(pr[4], pr[5], pr[6], pr[7], bh0, bh1, bl0, bl1);
            tile_accumulate<D>(ks1 + tile_bytes(D), nv1, gid, tig, bh0, bh1, bl0, bl1, o);
        }

        // ---- release the slots and refill them ---------------------------
        __syncwarp();
        fence_proxy_async_shared();
        consumed += two ? 2 : 1;
        cons_i = (two ? i1 : i0) + kAttnWarps;
        refill();
    }
    if (timed_out) {
        if (lane == 0) report(p.err, KVMM_ERR_TIMEOUT);
        // let copies still in flight land before the CTA leaves (bounded)
        for (int v = consumed; v < issued; ++v)
            mbar_wait_bounded(&sh.bar[warp][v % kRing], (v / kRing) & 1, 100000000ull);
    }

    // ---- merge the warps of this CTA ------------------------------------
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(kFullMask, l0, off);
        l1 += __shfl_xor_sync(kFullMask, l1, off);
    }
    __syncthreads();  // all warps done with the ring: reuse it for O
    float* so = reinterpret_cast<float*>(ring);  // [warps][8 heads][D]
    if (gid == 0) {
        sh.m[warp][2 * tig] = m0;
        sh.m[warp][2 * tig + 1] = m1;
        sh.l[warp][2 * tig] = l0;
        sh.l[warp][2 * tig + 1] = l1;
    }
#pragma unroll
    for (int i = 0; i < kMTiles; ++i) {
        const int d0 = gid * kDimsPerGroup + 2 * i;
        float* w0 = so + (warp * 8 + 2 * tig) * D;
        float* w1 = w0 + D;
        w0[d0] = o[i][0];
        w1[d0] = o[i][1];
        w0[d0 + 1] = o[i][2];
        w1[d0 + 1] = o[i][3];
    }
    __syncthreads();

    const bool single = p.splits == 1;
    float* part_o = p.part_o + (static_cast<size_t>(wunit) * p.splits + split) * G * D;
    float* part_ml = p.part_ml + (static_cast<size_t>(wunit) * p.splits + split) * G * 2;
    for (int e = tid; e < G * D; e += kAttnThreads) {
        const int g = e / D, d = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, sh.m[w][g]);
        float O = 0.f, Lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) {
                const float f = exp2f(sh.m[w][g] - M);
                O = fmaf(so[(w * 8 + g) * D + d], f, O);
                Lsum = fmaf(sh.l[w][g], f, Lsum);
            }
        }
        if (single) {
            const size_t oi = (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * G + g);
            p.out[oi * D + d] = Lsum > 0.f ? O / Lsum : 0.f;
            if (d == 0 && p.lse) p.lse[oi] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.6931471805599453f : -INFINITY;
        } else {
            part_o[e] = O;
            if (d == 0) {
                part_ml[2 * g] = M;
                part_ml[2 * g + 1] = Lsum;
            }
        }
    }
    if (single) return;

    // ---- last CTA of the unit merges the splits -------------------------
    __syncthreads();
    if (tid == 0) {
        __threadfence();  // the CTA's partial (ordered before by the barrier) is visible
        const int ticket = atomicAdd(p.counters + wunit, 1);
        sh.last = (ticket == p.splits - 1);
        if (sh.last) p.counters[wunit] = 0;
        __threadfence();
    }
    __syncthreads();
    if (!sh.last) return;

    const float* uo = p.part_o + static_cast<size_t>(wunit) * p.splits * G * D;
    const float* uml = p.part_ml + static_cast<size_t>(wunit) * p.splits * G * 2;
    for (int e = tid; e < G * D; e += kAttnThreads) {
        const int g = e / D, d = e % D;
        float M = -INFINITY;
        for (int s = 0; s < p.splits; ++s) M = fmaxf(M, __ldcg(uml + (s * G + g) * 2));
        float O = 0.f, Lsum = 0.f;
        if (M != -INFINITY) {
            for (int s = 0; s < p.splits; ++s) {
                const float ms = __ldcg(uml + (s * G + g) * 2);
                if (ms == -INFINITY) continue;
                const float f = exp2f(ms - M);
                O = fmaf(__ldcg(uo + (static_cast<size_t>(s) * G + g) * D + d), f, O);
                Lsum = fmaf(__ldcg(uml + (s * G + g) * 2 + 1), f, Lsum);
            }
        }
        const size_t oi = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * G + g;
        p.out[oi * D + d] = Lsum > 0.f ? O / Lsum : 0.f;
        if (d == 0 && p.lse) p.lse[oi] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.6931471805599453f : -INFINITY;
    }
}

template <int D>
cudaError_t launch_attn(const AttnParams& p, cudaStream_t stream)
{
    static thread_local int dev_cache = -1;
    static thread_local size_t bytes_cache = 0;
    const size_t smem = attention_smem_bytes(D, p.max_tiles);
    cudaError_t e = allow_smem(sparse_attn_kernel<D>, smem, dev_cache, bytes_cache);
    if (e != cudaSuccess) return e;
    return launch_pdl(sparse_attn_kernel<D>, dim3(p.splits, p.Hkv, p.B), dim3(kAttnThreads), smem, stream, p);
}

}  // namespace

size_t attention_smem_bytes(int D, int max_tiles)
{
    return ring_region(D) + size_t(max_tiles) * (sizeof(int64_t) + sizeof(int));
}

int attention_slots_per_unit(const kvmm_shape& s)
{
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int tiles = s.Kmax * (s.T / kTileTok);
    // CTAs resident per SM are bounded by the ring (shared memory) of each CTA
    const size_t per_cta = attention_smem_bytes(s.D, tiles) + sizeof(AttnShared) + 1024;
    int per_sm = static_cast<int>((228u * 1024u) / per_cta);
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 8) per_sm = 8;
    const long long slots = static_cast<long long>(sms) * per_sm;
    const long long units = static_cast<long long>(s.B) * s.Hkv;
    long long splits = slots / units;
    if (splits < 1) splits = 1;
    if (splits > tiles) splits = tiles;
    if (splits > 64) splits = 64;
    return static_cast<int>(splits);
}

cudaError_t launch_sparse_attention(const AttnParams& p, cudaStream_t stream)
{
    return p.D == 128 ? launch_attn<128>(p, stream) : launch_attn<64>(p, stream);
}

}  // namespace kvmm
