// minmax_update.cu -- append token rows and refresh per-page key MinMax.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 2. MinMax-metadata page
// scoring": every KV page keeps the per-channel minimum and maximum of its
// keys, in metadata held apart from the page itself.
//
// One warp owns one (batch, KV head, logical page) touched by the update.
// It writes the new rows of that page through the head-level block table
// (keys as rows of the page's [T][D], values as columns of its [D][T]),
// then re-reads the page's valid rows with 16-byte coalesced loads and
// reduces them.  min/max run on order-preserving 16-bit keys (two channels
// per 32-bit word, SIMD min/max), so -0 sorts below +0 and the result is a
// unique bf16 bit pattern.
#include "common.cuh"
#include "kernels.h"

namespace kvmm {
namespace {

constexpr int kUpdWarps = 8;

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

template <int D>
__global__ void __launch_bounds__(kUpdWarps * 32) minmax_update_kernel(const UpdateParams p)
{
    constexpr int kLanesPerRow = D / 8;            // 16 bytes (8 channels) per lane
    constexpr int kRowsPerPass = 32 / kLanesPerRow;
    const int lane = threadIdx.x & 31;
    const int slot = blockIdx.x * kUpdWarps + (threadIdx.x >> 5);
    const int h = blockIdx.y;
    const int b = blockIdx.z;
    const int T = p.T;
    pdl_wait_then_release();  // the pools, table and metadata may be in use by the previous kernel

    int tb = p.tok_begin[b];
    int te = p.tok_end[b];
    const int cap = p.Pmax * T;
    if (tb < 0 || te < tb || tb > cap) {
        if (slot == 0 && lane == 0 && h == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
        return;
    }
    if (te > cap) {
        if (slot == 0 && lane == 0 && h == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
        te = cap;
    }
    if (p.new_k != nullptr && te - tb > p.n_new) {
        if (slot == 0 && lane == 0 && h == 0) report(p.err, KVMM_ERR_OUT_OF_RANGE);
        te = tb + p.n_new;
    }
    if (te <= tb) return;

    const int page = tb / T + slot;
    if (page * T >= te) return;

    const size_t unit = (static_cast<size_t>(b) * p.L + p.layer) * p.Hkv + h;
    const int32_t phys = p.block_table[unit * p.Pmax + page];
    if (phys < 0 || phys >= p.n_phys) {
        if (lane == 0) report(p.err, phys < 0 ? KVMM_ERR_NULL_BLOCK : KVMM_ERR_OUT_OF_RANGE);
        return;
    }
    kvmm_bf16* kpage = p.k_pool + static_cast<size_t>(phys) * T * D;
    const int sub = lane % kLanesPerRow;  // 16-byte column of the row this lane moves
    const int first = page * T;

    if (p.new_k != nullptr) {
        kvmm_bf16* vpage = p.v_pool + static_cast<size_t>(phys) * T * D;
        const int r0 = max(tb - first, 0);
        const int r1 = min(te - first, T);
        const size_t src_base = (static_cast<size_t>(b) * p.Hkv + h) * p.n_new;
        for (int r = r0 + lane / kLanesPerRow; r < r1; r += kRowsPerPass) {
            const size_t j = src_base + (first + r - tb);
            const uint4 kv = reinterpret_cast<const uint4*>(p.new_k + j * D)[sub];
            const uint4 vv = reinterpret_cast<const uint4*>(p.new_v + j * D)[sub];
            reinterpret_cast<uint4*>(kpage + static_cast<size_t>(r) * D)[sub] = kv;
            // values are stored dimension-major: channel d of token r at vpage[d * T + r]
            const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
            for (int e = 0; e < 8; ++e)
                vpage[static_cast<size_t>(8 * sub + e) * T + r] =
                    static_cast<kvmm_bf16>((e & 1) ? (vw[e >> 1] >> 16) : (vw[e >> 1] & 0xffffu));
        }
        __syncwarp();  // the rows just written are read back below by other lanes
    }

    const int n_valid = min(T, te - first);
    uint32_t lo[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
    uint32_t hi[4] = {0u, 0u, 0u, 0u};
    for (int r = lane / kLanesPerRow; r < n_valid; r += kRowsPerPass) {
        const uint4 v = reinterpret_cast<const uint4*>(kpage + static_cast<size_t>(r) * D)[sub];
        const uint32_t w[4] = {to_key2(v.x), to_key2(v.y), to_key2(v.z), to_key2(v.w)};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = __vminu2(lo[i], w[i]);
            hi[i] = __vmaxu2(hi[i], w[i]);
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
        kvmm_bf16* m = p.meta + (unit * p.Pmax + page) * 2 * D;
        reinterpret_cast<uint4*>(m)[lane] =
            make_uint4(from_key2(lo[0]), from_key2(lo[1]), from_key2(lo[2]), from_key2(lo[3]));
        reinterpret_cast<uint4*>(m + D)[lane] =
            make_uint4(from_key2(hi[0]), from_key2(hi[1]), from_key2(hi[2]), from_key2(hi[3]));
    }
}

}  // namespace

cudaError_t launch_minmax_update(const UpdateParams& p, cudaStream_t stream)
{
    // pages one batch entry can touch: the rows given (append) or the whole table (rebuild)
    const long long span = p.new_k ? (static_cast<long long>(p.n_new) + p.T - 1) / p.T + 1 : p.Pmax;
    const long long pages = span < p.Pmax ? span : p.Pmax;
    const dim3 grid(static_cast<unsigned>((pages + kUpdWarps - 1) / kUpdWarps), p.Hkv, p.B);
    if (p.D == 128) return launch_pdl(minmax_update_kernel<128>, grid, dim3(kUpdWarps * 32), 0, stream, p);
    return launch_pdl(minmax_update_kernel<64>, grid, dim3(kUpdWarps * 32), 0, stream, p);
}

}  // namespace kvmm
