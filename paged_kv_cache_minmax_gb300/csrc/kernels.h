// kernels.h -- internal launch interface between the C-ABI layer (api.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda.h>  // CUtensorMap (the type only; the encoder is reached through the runtime)
#include <cuda_runtime.h>

#include "kvmm.h"

namespace kvmm {

// Workspace layout shared by the calls that take one: the units' page scores,
// B*Hkv rows of Pmax fp32 (every call writes the scores it reads).
inline size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }
inline size_t ws_scores_bytes(const kvmm_shape& s)
{
    return round256(static_cast<size_t>(s.B) * s.Hkv * s.Pmax * sizeof(float));
}
inline size_t ws_total_bytes(const kvmm_shape& s) { return ws_scores_bytes(s); }

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
    float* scores_ws;   // workspace: [B*Hkv][Pmax]
    int32_t* err;
};

struct AttnParams {
    int32_t B, L, Hq, Hkv, G, D, T, Pmax, Kmax, layer;
    int32_t splits;      // CTAs per unit (one cluster)
    int32_t max_tiles;   // upper bound of selected pages handled by one CTA
    int32_t region0;     // shared-memory bytes before the page lists (ring, or selection scratch)
    int32_t select;      // 1: rescored units select their pages from `scores` first
    int32_t K;           // select: pages to keep
    int32_t pstride;     // select: floats between the score rows of two units
    int32_t bt_prefetch; // select: copy each unit's block-table row to shared memory (16-byte aligned rows)
    int32_t bt_offset;   // select: its shared-memory offset
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
    const float* scores;          // select: [B*Hkv][pstride] page scores of the layer
    const uint8_t* rescore_mask;  // select: [L][Hkv] or null (every unit)
    int32_t* sel_out;             // select: where the new selections are written (sel_idx)
    int32_t* cnt_out;             // select: ... and their counts (sel_cnt)
    int32_t* err;
};

// one-launch decode layer (decode_layer.cu): a cluster of C CTAs per NU units (C up to the non-portable
// cluster size 16, NU 1 or 2)
constexpr int kDMaxCluster = 16;
struct DecodeParams {
    int32_t B, L, Hq, Hkv, G, D, T, Pmax, Kmax, layer, K;
    int32_t C;      // CTAs per cluster
    int32_t maxp;   // selected pages one CTA attends over at most: ceil(Kmax / C)
    int32_t bt_smem;  // 1: the units' block-table rows are copied to shared memory
    int32_t NU;       // units per cluster: 1 or 2 (the kernel instantiation takes it too)
    int32_t early;    // 1: the cache state is read before the preceding kernel has finished (KVMM_DECODE_EARLY_READS)
    int32_t n_new;  // appended tokens per batch entry (rows of new_k / new_v)
    int64_t n_phys;
    float scale_log2;  // sm_scale * log2(e)
    const kvmm_bf16* q;
    const kvmm_bf16* new_k;  // null: nothing appended
    const kvmm_bf16* new_v;
    const int32_t* tok_begin;
    const int32_t* tok_end;
    kvmm_bf16* k_pool;
    kvmm_bf16* v_pool;
    const int32_t* block_table;
    kvmm_bf16* meta;
    const int32_t* seq_len;
    const uint8_t* rescore_mask;
    int32_t* sel_idx;
    int32_t* sel_cnt;
    float* scores_out;
    float* out;
    float* lse;
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
// kv_meankey_update
struct MeanParams {
    int B, L, Hkv, T, D, Pmax, layer;
    int64_t n_phys;
    const int32_t* tok_begin;  // or null: 0
    const int32_t* tok_end;
    const kvmm_bf16* k_pool;
    const int32_t* block_table;
    kvmm_bf16* mean;  // [B][L][Hkv][Pmax][D]
    int32_t* err;
};

// block_table_update
struct TableUpdateParams {
    long long n;
    long long entries;  // B * L * Hkv * Pmax
    int64_t n_phys;
    const int64_t* idx;  // device-addressable
    const int32_t* val;
    int32_t* block_table;
    int32_t* err;
};

// promote_pages
struct PromoteParams {
    int B, L, Hkv, T, D, Pmax, Kmax, layer;
    int64_t n_phys;
    const uint8_t* rescore_mask;
    const int32_t* promoted;
    const int32_t* promoted_cnt;
    const int32_t* evicted;
    const int32_t* evicted_cnt;
    const kvmm_bf16* host_k;  // device-addressable host memory
    const kvmm_bf16* host_v;
    kvmm_bf16* k_pool;
    kvmm_bf16* v_pool;
    int32_t* block_table;
    int32_t* moved;
    int32_t* freed;
    int32_t* freed_cnt;
    int32_t* err;
};

// kv_centroid_build / page_score_topk_centroid (centroid.cu)
struct CentroidParams {
    int32_t B, L, Hq, Hkv, G, D, T, Pmax, layer;
    int32_t R;       // pages per initial spatial block
    int32_t Cmax;    // centroids a unit holds at most: ceil(Pmax / R)
    int32_t M, K;    // centroids expanded, pages selected
    int32_t Kmax;    // row length of sel_idx
    const kvmm_bf16* mean;       // [B][L][Hkv][Pmax][D]
    const int32_t* seq_len;      // [B]
    const uint8_t* rescore_mask; // [L][Hkv] or null
    const kvmm_bf16* q;          // [B][Hq][D]
    kvmm_bf16* cent;             // [B][L][Hkv][Cmax][D]
    int32_t* assign;             // [B][L][Hkv][Pmax]
    int32_t* member_off;         // [B][L][Hkv][Cmax + 1]
    int32_t* members;            // [B][L][Hkv][Pmax]
    int32_t* sel_idx;
    int32_t* sel_cnt;
    float* centroid_scores_out;  // [B][Hkv][Cmax] or null
    float* scores_out;           // [B][Hkv][Pmax] or null
    int32_t* err;
};
cudaError_t launch_centroid_build(const CentroidParams& p, int n_iter, cudaStream_t stream);
cudaError_t launch_centroid_select(const CentroidParams& p, int group_reduce, cudaStream_t stream);
size_t centroid_select_smem(int D, int G, int Pmax, int Cmax, int K, int M);  // dynamic shared memory of the selection
size_t centroid_update_smem(int Pmax, int Cmax);                             // ... and of the update

// topk_history_record / topk_stability_rco
struct StabilityParams {
    int B, L, Hkv, T, Pmax, Kmax;
    int W, n, head, lag;  // ring size; steps used, slot of the newest, distance of compared steps
    int layer, slot;      // recording: the layer and the ring slot it goes to
    float unstable_frac;
    const int32_t* sel_idx;
    const int32_t* sel_cnt;
    const int32_t* seq_len;
    int32_t* hist_idx;    // [W][B][L][Hkv][Kmax]
    int32_t* hist_cnt;    // [W][B][L][Hkv]
    int32_t* hist_pages;  // [W][B]
    float* rco_unit;      // [B][L][Hkv]
    float* stability;     // [L][Hkv] or null
    uint8_t* unstable;    // [L][Hkv] or null
    int32_t* err;
};

cudaError_t launch_minmax_update(const UpdateParams& p, cudaStream_t stream);
cudaError_t launch_score_topk(const ScoreParams& p, int group_reduce, cudaStream_t stream);
cudaError_t launch_sparse_attention(const AttnParams& p, cudaStream_t stream);
cudaError_t launch_promotion_diff(const DiffParams& p, cudaStream_t stream);
cudaError_t launch_promote(const PromoteParams& p, int max_ctas, cudaStream_t stream);
cudaError_t launch_table_update(const TableUpdateParams& p, cudaStream_t stream);
cudaError_t launch_meankey(const MeanParams& p, cudaStream_t stream);
cudaError_t launch_history_record(const StabilityParams& p, cudaStream_t stream);
cudaError_t launch_stability_rco(const StabilityParams& p, cudaStream_t stream);
size_t stability_max_heads();  // largest L * Hkv the classification handles
// The phases a launch of the decode kernel runs: decode_layer runs both; page_score_topk runs the first
// alone (score and select), sparse_paged_decode_attn the second (attend over kept selections).
constexpr int kPhScore = 1;   // score every page of the rescored units, select their top K
constexpr int kPhAttend = 2;  // attend over the selected pages and merge the partials
constexpr int kPhBoth = kPhScore | kPhAttend;
cudaError_t launch_decode_layer(DecodeParams p, int group_reduce, int ph, cudaStream_t stream);
constexpr size_t kDSmemLimit = 220 * 1024;  // dynamic shared memory a decode_layer CTA may take
struct DecodeGrid {
    int nu;  // units per cluster (0: the shape's buffers do not fit; the caller takes another path)
    int c;   // CTAs per cluster
};
DecodeGrid decode_layer_grid(const kvmm_shape& s, int ph = kPhBoth);  // the launch shape for a kvmm shape
// the scoring kernel alone (page_score_topk without its selection kernel)
cudaError_t launch_score_only(const ScoreParams& p, int group_reduce, cudaStream_t stream);
cudaError_t launch_score_topk_mean(const ScoreParams& p, int group_reduce, cudaStream_t stream);  // mean-key rows

// Library-owned scratch of page_score_topk_static_scratch (score_topk.cu):
// the scores, laid out as in a caller workspace.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;
// Device address of that scratch on the current device; the first call on a
// device looks it up (cudaGetSymbolAddress) and caches it.
cudaError_t static_scratch_for_current_device(void** ptr);

// Attention launch geometry for the current device.
constexpr int kAttnMaxSplits = 16;                   // CTAs of a unit form one cluster
// `select`: the attention kernel that selects its own pages (page_score_topk_attn)
int attention_slots_per_unit(const kvmm_shape& s, bool select = false);  // automatic split count
int attention_max_splits(const kvmm_shape& s, bool select = false);      // largest launchable cluster
// dynamic shared memory of one attention CTA; `scratch`: the selection scratch (0 without selection)
size_t attention_smem_bytes(int D, int max_pages, size_t scratch = 0);
size_t attention_region0(int D, size_t scratch);
// selection scratch of the selecting attention kernel for a shape
size_t attention_select_scratch(int Pmax, int Kmax);

}  // namespace kvmm
