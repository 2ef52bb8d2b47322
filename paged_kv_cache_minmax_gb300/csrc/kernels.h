// kernels.h -- internal launch interface between the C-ABI layer (api.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include "kvmm.h"

namespace kvmm {

// Workspace layout shared by every call that takes a workspace:
//   [control words][scores: B*Hkv rows of Pmax fp32][attention partials]
// The control words (zero before the first use; every launch of the fused
// call leaves them zero again) are the fused call's queue counters, then
// four per-unit arrays: score tickets [U], attention tickets [U], the select
// queue [U] and the ready queue [U * splits].  page_score_topk uses only the
// scores region.
constexpr int kCtrlHead = 16;
inline size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }
// attention items per unit in the fused call: 256 tokens of selected pages each, at most 64
inline int fused_splits(const kvmm_shape& s)
{
    const int item_pages = 256 / s.T;
    int n = (s.Kmax + item_pages - 1) / item_pages;
    return n < 1 ? 1 : (n > 64 ? 64 : n);
}
inline size_t ws_counter_bytes(const kvmm_shape& s)
{
    const size_t units = static_cast<size_t>(s.B) * s.Hkv;
    return round256((kCtrlHead + 3 * units + units * fused_splits(s)) * sizeof(int32_t));
}
// score rows of the fused call start 16-byte aligned: Pmax rounded up to 4
inline int ws_score_stride(const kvmm_shape& s) { return (s.Pmax + 3) & ~3; }
inline size_t ws_scores_bytes(const kvmm_shape& s)
{
    return round256(static_cast<size_t>(s.B) * s.Hkv * ws_score_stride(s) * sizeof(float));
}
// one partial per (unit, attention item): m[8], l[8], O[8][D] (fp32)
inline size_t ws_partials_bytes(const kvmm_shape& s)
{
    return round256(static_cast<size_t>(s.B) * s.Hkv * fused_splits(s) * (16 + 8 * static_cast<size_t>(s.D)) *
                    sizeof(float));
}
inline size_t ws_total_bytes(const kvmm_shape& s)
{
    return ws_counter_bytes(s) + ws_scores_bytes(s) + ws_partials_bytes(s);
}

struct UpdateParams {
    int32_t B, L, Hkv, D, T, Pmax, layer, n_new;
    int64_t n_phys;
    const kvmm_bf16* new_k;
    const kvmm_bf16* new_v;
    const int32_t* tok_begin;
    const int32_t* tok_end;
    kvmm_bf16* k_pool;
    kvmm_bf16* v_pool;
    const int32_t* block_table;
    kvmm_bf16* meta;
    int32_t* err;
};

struct ScoreParams {
    int32_t B, L, Hq, Hkv, G, D, T, Pmax, Kmax, layer, K;
    const kvmm_bf16* q;
    const kvmm_bf16* meta;
    const int32_t* seq_len;
    const uint8_t* rescore_mask;
    int32_t* sel_idx;
    int32_t* sel_cnt;
    float* scores_out;
    int32_t* counters;  // workspace: [B*Hkv]
    float* scores_ws;   // workspace: [B*Hkv][Pmax]
    int32_t* err;
};

struct AttnParams {
    int32_t B, L, Hq, Hkv, G, D, T, Pmax, Kmax, layer;
    int32_t splits;      // CTAs per unit (one cluster)
    int32_t max_tiles;   // upper bound of selected pages handled by one CTA
    int64_t n_phys;
    float scale_log2;    // sm_scale * log2(e)
    const kvmm_bf16* q;
    const kvmm_bf16* k_pool;
    const kvmm_bf16* v_pool;
    const int32_t* block_table;
    const int32_t* seq_len;
    const int32_t* sel_idx;
    const int32_t* sel_cnt;
    float* out;
    float* lse;
    int32_t* err;
};

// page_score_topk_attn runs as one launch for page tables up to this long
constexpr int kFusedMaxPages = 2048;

struct FusedParams {
    int32_t B, L, Hq, Hkv, G, D, T, Pmax, Kmax, layer, K;
    int32_t chunks;  // score items per unit: ceil(Pmax / 128)
    int32_t splits;  // attention items per unit
    int32_t pstride; // floats between the workspace score rows of two units
    int64_t n_phys;
    float scale_log2;  // sm_scale * log2(e)
    const kvmm_bf16* q;
    const kvmm_bf16* meta;
    const kvmm_bf16* k_pool;
    const kvmm_bf16* v_pool;
    const int32_t* block_table;
    const int32_t* seq_len;
    const uint8_t* rescore_mask;
    int32_t* sel_idx;
    int32_t* sel_cnt;
    float* scores_out;
    float* out;
    float* lse;
    int32_t* ctrl;      // workspace: control words
    float* scores;      // workspace: [B*Hkv][pstride]
    float* partials;    // workspace: [B*Hkv][splits][16 + 8*D]
    int32_t* err;
};

struct DiffParams {
    int32_t B, L, Hkv, Kmax, layer, commit;
    const uint8_t* rescore_mask;
    int32_t* prev_idx;
    int32_t* prev_cnt;
    const int32_t* cur_idx;
    const int32_t* cur_cnt;
    int32_t* promoted;
    int32_t* promoted_cnt;
    int32_t* evicted;
    int32_t* evicted_cnt;
    int32_t* total_promoted;
    int32_t* err;
};

// Launch `kernel` on `stream` with programmatic stream serialisation, so it
// may be scheduled while its predecessor drains (it must griddepcontrol.wait
// before using the predecessor's results).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// As launch_pdl, with the grid tiled into thread-block clusters of
// `cluster_x` x 1 x 1 CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               unsigned cluster_x, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raise a kernel's dynamic shared-memory limit to `bytes` (once per device and
// size; the default 48 KiB limit counts static shared memory too).
template <typename Kernel>
cudaError_t allow_smem(Kernel kernel, size_t bytes, int& dev_cache, size_t& bytes_cache)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev_cache == dev && bytes_cache >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    dev_cache = dev;
    bytes_cache = bytes;
    return cudaSuccess;
}

// Launchers return cudaSuccess or the launch error.
cudaError_t launch_minmax_update(const UpdateParams& p, cudaStream_t stream);
cudaError_t launch_score_topk(const ScoreParams& p, int group_reduce, cudaStream_t stream);
cudaError_t launch_sparse_attention(const AttnParams& p, cudaStream_t stream);
cudaError_t launch_promotion_diff(const DiffParams& p, cudaStream_t stream);
cudaError_t launch_fused_decode(const FusedParams& p, int group_reduce, cudaStream_t stream);

// Library-owned scratch of page_score_topk_static_scratch (score_topk.cu):
// counters for up to kStaticScratchCounterBytes/4 units, then the scores.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;
constexpr size_t kStaticScratchCounterBytes = size_t(16) << 10;
// Device address of that scratch on the current device; the first call on a
// device resolves it and zeroes the counters on `stream`.
cudaError_t static_scratch_for_current_device(void** ptr, cudaStream_t stream);

// Attention launch geometry for the current device.
constexpr int kAttnMaxSplits = 16;                   // CTAs of a unit form one cluster
int attention_slots_per_unit(const kvmm_shape& s);  // automatic split count
int attention_max_splits(const kvmm_shape& s);      // largest launchable cluster (<= kAttnMaxSplits)
size_t attention_smem_bytes(int D, int max_pages);

}  // namespace kvmm
