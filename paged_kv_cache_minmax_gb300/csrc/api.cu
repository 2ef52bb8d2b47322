// api.cu -- the extern "C" entry points declared in include/kvmm.h.
//
// Host side only: synchronous argument checks, workspace carving and kernel
// launches on the caller's stream.  No allocation, no synchronisation.
#include <cmath>

#include "kernels.h"

namespace {

using kvmm::AttnParams;
using kvmm::DiffParams;
using kvmm::ScoreParams;
using kvmm::UpdateParams;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// bf16 arrays and the workspace: present and 16-byte aligned (vector loads, bulk copies)
bool req(const void* p) { return p != nullptr && aligned(p, 16); }
bool opt(const void* p) { return p == nullptr || aligned(p, 16); }
// int32 / float arrays: present (or NULL) and 4-byte aligned
bool req4(const void* p) { return p != nullptr && aligned(p, 4); }
bool opt4(const void* p) { return p == nullptr || aligned(p, 4); }

// The device address of host memory the device can read (the same address under unified addressing),
// or null: pinned or managed memory, or pageable memory where the device reads pageable host memory.
const void* device_view_of_host(const void* h)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeManaged || a.type == cudaMemoryTypeDevice)
        return a.devicePointer != nullptr ? a.devicePointer : h;
    int dev = 0, pageable = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return pageable ? h : nullptr;
}

kvmm_status check_shape(const kvmm_shape* s)
{
    if (s == nullptr) return KVMM_INVALID_ARG;
    if (s->B < 1 || s->L < 1 || s->Hq < 1 || s->Hkv < 1 || s->Pmax < 1 || s->Kmax < 1 || s->n_phys < 1)
        return KVMM_INVALID_ARG;
    if (s->Hq % s->Hkv != 0) return KVMM_INVALID_ARG;
    const int G = s->Hq / s->Hkv;
    if (G > 8) return KVMM_UNSUPPORTED_SHAPE;
    if (s->D != 64 && s->D != 128) return KVMM_UNSUPPORTED_SHAPE;
    if (s->T != 16 && s->T != 32) return KVMM_UNSUPPORTED_SHAPE;
    if (s->Pmax > 32768 || s->Kmax > 32768) return KVMM_UNSUPPORTED_SHAPE;
    if (s->B > 65535 || s->Hkv > 65535) return KVMM_UNSUPPORTED_SHAPE;  // grid y/z limits
    // every element index of the pools, tables and metadata fits in int64 and row ids in int64
    if (s->n_phys > (int64_t(1) << 40)) return KVMM_UNSUPPORTED_SHAPE;
    return KVMM_OK;
}

int resolve_splits(const kvmm_shape& s, int32_t num_splits, bool select = false)
{
    int splits = num_splits > 0 ? num_splits : kvmm::attention_slots_per_unit(s, select);
    if (splits > kvmm::kAttnMaxSplits) splits = kvmm::kAttnMaxSplits;
    if (splits > s.Kmax) splits = s.Kmax;
    if (splits < 1) splits = 1;
    return splits;
}

size_t score_ws_bytes(const kvmm_shape& s) { return kvmm::ws_scores_bytes(s); }

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

kvmm_status launched(cudaError_t e)
{
    if (e == cudaSuccess) return KVMM_OK;
    g_last_cuda_error = e;
    return KVMM_CUDA_ERROR;
}

}  // namespace

extern "C" {

const char* kvmm_status_string(kvmm_status status)
{
    switch (status) {
    case KVMM_OK: return "ok";
    case KVMM_INVALID_ARG: return "invalid argument (null or misaligned pointer, index or flag out of range)";
    case KVMM_UNSUPPORTED_SHAPE: return "unsupported shape (D in {64,128}, T in {16,32}, G <= 8, Pmax and Kmax <= 32768)";
    case KVMM_WORKSPACE_TOO_SMALL: return "workspace too small (see kvmm_workspace_size)";
    case KVMM_CUDA_ERROR: return "CUDA runtime or launch error";
    }
    return "unknown status";
}

const char* kvmm_last_cuda_error(void)
{
    return g_last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(g_last_cuda_error);
}

int32_t kvmm_auto_splits(const kvmm_shape* shape)
{
    if (check_shape(shape) != KVMM_OK) return 0;
    const kvmm::DecodeGrid g = kvmm::decode_layer_grid(*shape, kvmm::kPhAttend);
    return g.nu > 0 ? g.c : resolve_splits(*shape, 0);
}

int32_t kvmm_decode_layer_cluster(const kvmm_shape* shape)
{
    if (check_shape(shape) != KVMM_OK) return 0;
    return kvmm::decode_layer_grid(*shape).c;
}

int32_t kvmm_decode_layer_units(const kvmm_shape* shape)
{
    if (check_shape(shape) != KVMM_OK) return 0;
    return kvmm::decode_layer_grid(*shape).nu;
}

size_t kvmm_workspace_size(const kvmm_shape* shape, int32_t num_splits)
{
    if (check_shape(shape) != KVMM_OK || num_splits < 0) return 0;
    return kvmm::ws_total_bytes(*shape);  // sparse_paged_decode_attn merges on chip and needs none
}

kvmm_status kv_minmax_update(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* new_k,
                             const kvmm_bf16* new_v, int32_t n_new, const int32_t* tok_begin,
                             const int32_t* tok_end, kvmm_bf16* k_pool, kvmm_bf16* v_pool,
                             const int32_t* block_table, kvmm_bf16* meta, int32_t* err,
                             kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < 0 || layer >= s.L) return KVMM_INVALID_ARG;
    if ((new_k == nullptr) != (new_v == nullptr)) return KVMM_INVALID_ARG;
    if (!opt(new_k) || !opt(new_v) || !req4(tok_begin) || !req4(tok_end) || !req(k_pool) ||
        !req4(block_table) || !req(meta) || !opt4(err))
        return KVMM_INVALID_ARG;
    if (new_k != nullptr && (n_new < 1 || !req(v_pool))) return KVMM_INVALID_ARG;
    if (n_new < 0) return KVMM_INVALID_ARG;
    UpdateParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hkv = s.Hkv;
    p.D = s.D;
    p.T = s.T;
    p.Pmax = s.Pmax;
    p.layer = layer;
    p.n_new = n_new;
    p.n_phys = s.n_phys;
    p.new_k = new_k;
    p.new_v = new_v;
    p.tok_begin = tok_begin;
    p.tok_end = tok_end;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.block_table = block_table;
    p.meta = meta;
    p.err = err;
    return launched(kvmm::launch_minmax_update(p, reinterpret_cast<cudaStream_t>(stream)));
}

// the shape part of the clustered decode kernel's parameters; the caller sets the arrays
static kvmm::DecodeParams decode_params(const kvmm_shape& s, int32_t layer, int32_t K, const kvmm::DecodeGrid& g,
                                        float sm_scale)
{
    kvmm::DecodeParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.G = s.Hq / s.Hkv;
    p.D = s.D;
    p.T = s.T;
    p.Pmax = s.Pmax;
    p.Kmax = s.Kmax;
    p.layer = layer;
    p.K = K;
    p.C = g.c;
    p.NU = g.nu;
    p.n_phys = s.n_phys;
    p.scale_log2 = (sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(s.D))) * 1.4426950408889634f;
    return p;
}

// page_score_topk and page_score_topk_mean: the same arguments, MinMax bounds or mean keys as rows
static kvmm_status score_topk_call(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                                   const kvmm_bf16* meta, const int32_t* seq_len, const uint8_t* rescore_mask,
                                   int32_t K, int32_t group_reduce, int32_t* sel_idx, int32_t* sel_cnt,
                                   float* scores_out, void* workspace, size_t workspace_bytes, uint32_t flags,
                                   int32_t* err, kvmm_stream stream, bool mean)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < 0 || layer >= s.L || K < 1 || K > s.Kmax) return KVMM_INVALID_ARG;
    if (group_reduce != 0 && group_reduce != 1) return KVMM_INVALID_ARG;
    if (!req(q) || !req(meta) || !req4(seq_len) || !req4(sel_idx) || !req4(sel_cnt) || !opt4(scores_out) ||
        !req(workspace) || !opt4(err))
        return KVMM_INVALID_ARG;
    if (workspace_bytes < score_ws_bytes(s)) return KVMM_WORKSPACE_TOO_SMALL;
    if ((flags & ~KVMM_EARLY_READS) != 0u) return KVMM_INVALID_ARG;
    if (!mean) {
        // MinMax rows: one launch of the clustered kernel's scoring phase (scores exchanged and selected on
        // chip; the workspace is not touched), when the units' score buffers fit a CTA
        const kvmm::DecodeGrid g = kvmm::decode_layer_grid(s, kvmm::kPhScore);
        if (g.nu > 0) {
            kvmm::DecodeParams dp = decode_params(s, layer, K, g, 0.f);
            dp.early = (flags & KVMM_EARLY_READS) != 0u ? 1 : 0;
            dp.q = q;
            dp.meta = const_cast<kvmm_bf16*>(meta);  // read only: this phase appends nothing
            dp.seq_len = seq_len;
            dp.rescore_mask = rescore_mask;
            dp.sel_idx = sel_idx;
            dp.sel_cnt = sel_cnt;
            dp.scores_out = scores_out;
            dp.err = err;
            return launched(kvmm::launch_decode_layer(dp, group_reduce, kvmm::kPhScore,
                                                      reinterpret_cast<cudaStream_t>(stream)));
        }
    }
    ScoreParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.G = s.Hq / s.Hkv;
    p.D = s.D;
    p.T = s.T;
    p.Pmax = s.Pmax;
    p.Kmax = s.Kmax;
    p.layer = layer;
    p.K = K;
    p.q = q;
    p.meta = meta;
    p.seq_len = seq_len;
    p.rescore_mask = rescore_mask;
    p.sel_idx = sel_idx;
    p.sel_cnt = sel_cnt;
    p.scores_out = scores_out;
    p.scores_ws = static_cast<float*>(workspace);
    p.err = err;
    return launched(mean ? kvmm::launch_score_topk_mean(p, group_reduce, reinterpret_cast<cudaStream_t>(stream))
                         : kvmm::launch_score_topk(p, group_reduce, reinterpret_cast<cudaStream_t>(stream)));
}

kvmm_status page_score_topk(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                            const kvmm_bf16* meta, const int32_t* seq_len,
                            const uint8_t* rescore_mask, int32_t K, int32_t group_reduce,
                            int32_t* sel_idx, int32_t* sel_cnt, float* scores_out,
                            void* workspace, size_t workspace_bytes, uint32_t flags, int32_t* err,
                            kvmm_stream stream)
{
    return score_topk_call(shape, layer, q, meta, seq_len, rescore_mask, K, group_reduce, sel_idx, sel_cnt,
                           scores_out, workspace, workspace_bytes, flags, err, stream, false);
}

kvmm_status page_score_topk_mean(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                                 const kvmm_bf16* mean, const int32_t* seq_len, const uint8_t* rescore_mask,
                                 int32_t K, int32_t group_reduce, int32_t* sel_idx, int32_t* sel_cnt,
                                 float* scores_out, void* workspace, size_t workspace_bytes, int32_t* err,
                                 kvmm_stream stream)
{
    return score_topk_call(shape, layer, q, mean, seq_len, rescore_mask, K, group_reduce, sel_idx, sel_cnt,
                           scores_out, workspace, workspace_bytes, 0u, err, stream, true);
}

kvmm_status kv_meankey_update(const kvmm_shape* shape, int32_t layer, const int32_t* tok_begin,
                              const int32_t* tok_end, const kvmm_bf16* k_pool, const int32_t* block_table,
                              kvmm_bf16* mean, int32_t* err, kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < 0 || layer >= s.L) return KVMM_INVALID_ARG;
    if (!opt4(tok_begin) || !req4(tok_end) || !req(k_pool) || !req4(block_table) || !req(mean) || !opt4(err))
        return KVMM_INVALID_ARG;
    kvmm::MeanParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hkv = s.Hkv;
    p.T = s.T;
    p.D = s.D;
    p.Pmax = s.Pmax;
    p.layer = layer;
    p.n_phys = s.n_phys;
    p.tok_begin = tok_begin;
    p.tok_end = tok_end;
    p.k_pool = k_pool;
    p.block_table = block_table;
    p.mean = mean;
    p.err = err;
    return launched(kvmm::launch_meankey(p, reinterpret_cast<cudaStream_t>(stream)));
}

static kvmm::CentroidParams centroid_params(const kvmm_shape& s, int32_t layer, int32_t R)
{
    kvmm::CentroidParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.G = s.Hq / s.Hkv;
    p.D = s.D;
    p.T = s.T;
    p.Pmax = s.Pmax;
    p.Kmax = s.Kmax;
    p.layer = layer;
    p.R = R;
    p.Cmax = (s.Pmax + R - 1) / R;
    return p;
}

kvmm_status kv_centroid_build(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* mean, const int32_t* seq_len,
                              int32_t R, int32_t n_iter, kvmm_bf16* cent, int32_t* assign, int32_t* member_off,
                              int32_t* members, int32_t* err, kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < 0 || layer >= s.L || R < 1 || R > s.Pmax || n_iter < 0 || n_iter > 64) return KVMM_INVALID_ARG;
    if (!req(mean) || !req4(seq_len) || !req(cent) || !req4(assign) || !req4(member_off) || !req4(members) ||
        !opt4(err))
        return KVMM_INVALID_ARG;
    kvmm::CentroidParams p = centroid_params(s, layer, R);
    if (kvmm::centroid_update_smem(s.Pmax, p.Cmax) > kvmm::kDSmemLimit) return KVMM_UNSUPPORTED_SHAPE;
    p.mean = mean;
    p.seq_len = seq_len;
    p.cent = cent;
    p.assign = assign;
    p.member_off = member_off;
    p.members = members;
    p.err = err;
    return launched(kvmm::launch_centroid_build(p, n_iter, reinterpret_cast<cudaStream_t>(stream)));
}

kvmm_status page_score_topk_centroid(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                                     const kvmm_bf16* mean, const int32_t* seq_len, int32_t R, const kvmm_bf16* cent,
                                     const int32_t* member_off, const int32_t* members, const uint8_t* rescore_mask,
                                     int32_t M, int32_t K, int32_t group_reduce, int32_t* sel_idx, int32_t* sel_cnt,
                                     float* centroid_scores_out, float* scores_out, int32_t* err,
                                     kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < 0 || layer >= s.L || R < 1 || R > s.Pmax || M < 1 || K < 1 || K > s.Kmax) return KVMM_INVALID_ARG;
    if (group_reduce != 0 && group_reduce != 1) return KVMM_INVALID_ARG;
    if (!req(q) || !req(mean) || !req4(seq_len) || !req(cent) || !req4(member_off) || !req4(members) ||
        !req4(sel_idx) || !req4(sel_cnt) || !opt4(centroid_scores_out) || !opt4(scores_out) || !opt4(err))
        return KVMM_INVALID_ARG;
    kvmm::CentroidParams p = centroid_params(s, layer, R);
    p.M = M < p.Cmax ? M : p.Cmax;
    p.K = K;
    if (kvmm::centroid_select_smem(s.D, p.G, s.Pmax, p.Cmax, K, p.M) > kvmm::kDSmemLimit)
        return KVMM_UNSUPPORTED_SHAPE;
    p.q = q;
    p.mean = mean;
    p.seq_len = seq_len;
    p.rescore_mask = rescore_mask;
    p.cent = const_cast<kvmm_bf16*>(cent);  // read only here
    p.member_off = const_cast<int32_t*>(member_off);
    p.members = const_cast<int32_t*>(members);
    p.sel_idx = sel_idx;
    p.sel_cnt = sel_cnt;
    p.centroid_scores_out = centroid_scores_out;
    p.scores_out = scores_out;
    p.err = err;
    return launched(kvmm::launch_centroid_select(p, group_reduce, reinterpret_cast<cudaStream_t>(stream)));
}

kvmm_status page_score_topk_static_scratch(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                                           const kvmm_bf16* meta, const int32_t* seq_len,
                                           const uint8_t* rescore_mask, int32_t K, int32_t group_reduce,
                                           int32_t* sel_idx, int32_t* sel_cnt, float* scores_out,
                                           int32_t* err, kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < 0 || layer >= s.L || K < 1 || K > s.Kmax) return KVMM_INVALID_ARG;
    if (group_reduce != 0 && group_reduce != 1) return KVMM_INVALID_ARG;
    if (!req(q) || !req(meta) || !req4(seq_len) || !req4(sel_idx) || !req4(sel_cnt) || !opt4(scores_out) ||
        !opt4(err))
        return KVMM_INVALID_ARG;
    // the shape must fit the fixed scratch: B*Hkv*Pmax scores
    if (size_t(s.B) * s.Hkv * s.Pmax * sizeof(float) > kvmm::kStaticScratchBytes) return KVMM_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const cudaError_t se = kvmm::static_scratch_for_current_device(&scratch);
    if (se != cudaSuccess) return launched(se);
    ScoreParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.G = s.Hq / s.Hkv;
    p.D = s.D;
    p.T = s.T;
    p.Pmax = s.Pmax;
    p.Kmax = s.Kmax;
    p.layer = layer;
    p.K = K;
    p.q = q;
    p.meta = meta;
    p.seq_len = seq_len;
    p.rescore_mask = rescore_mask;
    p.sel_idx = sel_idx;
    p.sel_cnt = sel_cnt;
    p.scores_out = scores_out;
    p.scores_ws = static_cast<float*>(scratch);
    p.err = err;
    return launched(kvmm::launch_score_topk(p, group_reduce, cs));
}

kvmm_status sparse_paged_decode_attn(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                                     const kvmm_bf16* k_pool, const kvmm_bf16* v_pool,
                                     const int32_t* block_table, const int32_t* seq_len,
                                     const int32_t* sel_idx, const int32_t* sel_cnt,
                                     float sm_scale, int32_t num_splits, float* out, float* lse,
                                     void* workspace, size_t workspace_bytes, uint32_t flags,
                                     int32_t* err, kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < 0 || layer >= s.L || num_splits < 0 || !std::isfinite(sm_scale)) return KVMM_INVALID_ARG;
    if (!req(q) || !req(k_pool) || !req(v_pool) || !req4(block_table) || !req4(seq_len) || !req4(sel_idx) ||
        !req4(sel_cnt) || !req4(out) || !opt4(lse) || !opt4(err))
        return KVMM_INVALID_ARG;
    (void)workspace;
    (void)workspace_bytes;
    if ((flags & ~KVMM_EARLY_READS) != 0u) return KVMM_INVALID_ARG;
    if (num_splits == 0) {
        // automatic: one launch of the clustered kernel's attention phase over the kept selections (units
        // share clusters; a unit's pages follow the previous unit's in the same slots), when it fits
        const kvmm::DecodeGrid g = kvmm::decode_layer_grid(s, kvmm::kPhAttend);
        if (g.nu > 0) {
            kvmm::DecodeParams dp = decode_params(s, layer, s.Kmax, g, sm_scale);
            dp.early = (flags & KVMM_EARLY_READS) != 0u ? 1 : 0;
            dp.q = q;
            dp.k_pool = const_cast<kvmm_bf16*>(k_pool);  // read only: this phase appends nothing
            dp.v_pool = const_cast<kvmm_bf16*>(v_pool);
            dp.block_table = block_table;
            dp.seq_len = seq_len;
            dp.sel_idx = const_cast<int32_t*>(sel_idx);  // read only: the kept selections
            dp.sel_cnt = const_cast<int32_t*>(sel_cnt);
            dp.out = out;
            dp.lse = lse;
            dp.err = err;
            return launched(kvmm::launch_decode_layer(dp, 0, kvmm::kPhAttend, reinterpret_cast<cudaStream_t>(stream)));
        }
    }
    const int splits = resolve_splits(s, num_splits);
    if (num_splits > 0 && splits > kvmm::attention_max_splits(s)) return KVMM_UNSUPPORTED_SHAPE;
    const int max_pages = (s.Kmax + splits - 1) / splits;  // selected pages one CTA may hold
    if (kvmm::attention_smem_bytes(s.D, max_pages) > 200 * 1024) return KVMM_UNSUPPORTED_SHAPE;
    AttnParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.G = s.Hq / s.Hkv;
    p.D = s.D;
    p.T = s.T;
    p.Pmax = s.Pmax;
    p.Kmax = s.Kmax;
    p.layer = layer;
    p.splits = splits;
    p.max_tiles = max_pages;
    p.region0 = static_cast<int32_t>(kvmm::attention_region0(s.D, 0));
    p.n_phys = s.n_phys;
    p.scale_log2 = (sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(s.D))) * 1.4426950408889634f;
    p.q = q;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.block_table = block_table;
    p.seq_len = seq_len;
    p.sel_idx = sel_idx;
    p.sel_cnt = sel_cnt;
    p.out = out;
    p.lse = lse;
    p.err = err;
    return launched(kvmm::launch_sparse_attention(p, reinterpret_cast<cudaStream_t>(stream)));
}

kvmm_status page_score_topk_attn(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                                 const kvmm_bf16* meta, const kvmm_bf16* k_pool, const kvmm_bf16* v_pool,
                                 const int32_t* block_table, const int32_t* seq_len,
                                 const uint8_t* rescore_mask, int32_t K, int32_t group_reduce,
                                 float sm_scale, int32_t* sel_idx, int32_t* sel_cnt, float* scores_out,
                                 float* out, float* lse, void* workspace, size_t workspace_bytes,
                                 int32_t* err, kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < 0 || layer >= s.L || K < 1 || K > s.Kmax || !std::isfinite(sm_scale)) return KVMM_INVALID_ARG;
    if (group_reduce != 0 && group_reduce != 1) return KVMM_INVALID_ARG;
    if (!req(q) || !req(meta) || !req(k_pool) || !req(v_pool) || !req4(block_table) || !req4(seq_len) ||
        !req4(sel_idx) || !req4(sel_cnt) || !opt4(scores_out) || !req4(out) || !opt4(lse) || !req(workspace) ||
        !opt4(err))
        return KVMM_INVALID_ARG;
    if (workspace_bytes < score_ws_bytes(s)) return KVMM_WORKSPACE_TOO_SMALL;
    {
        // one launch of the clustered kernel with both phases and nothing appended: decode_layer without new
        // rows, which leaves what the two calls leave
        const kvmm::DecodeGrid g = kvmm::decode_layer_grid(s, kvmm::kPhBoth);
        if (g.nu > 0) {
            kvmm::DecodeParams dp = decode_params(s, layer, K, g, sm_scale);
            dp.q = q;
            dp.k_pool = const_cast<kvmm_bf16*>(k_pool);  // read only: nothing is appended
            dp.v_pool = const_cast<kvmm_bf16*>(v_pool);
            dp.block_table = block_table;
            dp.meta = const_cast<kvmm_bf16*>(meta);
            dp.seq_len = seq_len;
            dp.rescore_mask = rescore_mask;
            dp.sel_idx = sel_idx;
            dp.sel_cnt = sel_cnt;
            dp.scores_out = scores_out;
            dp.out = out;
            dp.lse = lse;
            dp.err = err;
            return launched(kvmm::launch_decode_layer(dp, group_reduce, kvmm::kPhBoth,
                                                      reinterpret_cast<cudaStream_t>(stream)));
        }
    }
    const size_t scratch = kvmm::attention_select_scratch(s.Pmax, s.Kmax);
    const int splits = resolve_splits(s, 0, true);
    const int max_pages = (s.Kmax + splits - 1) / splits;
    // the unit's block-table row in shared memory too, when its rows are 16-byte aligned and short
    const bool bt_prefetch = s.Pmax % 4 == 0 && s.Pmax <= 4096;
    const size_t base_smem = kvmm::attention_smem_bytes(s.D, max_pages, scratch);
    const size_t bt_offset = (base_smem + 15) & ~static_cast<size_t>(15);
    if (bt_offset + (bt_prefetch ? size_t(s.Pmax) * 4 : 0) > 200 * 1024) {
        // the selection does not fit the attention CTA's shared memory: separate kernels
        st = page_score_topk(shape, layer, q, meta, seq_len, rescore_mask, K, group_reduce, sel_idx, sel_cnt,
                             scores_out, workspace, workspace_bytes, 0u, err, stream);
        if (st != KVMM_OK) return st;
        return sparse_paged_decode_attn(shape, layer, q, k_pool, v_pool, block_table, seq_len, sel_idx, sel_cnt,
                                        sm_scale, 0, out, lse, nullptr, 0, 0u, err, stream);
    }
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    float* scores_ws = static_cast<float*>(workspace);
    ScoreParams sp{};
    sp.B = s.B;
    sp.L = s.L;
    sp.Hq = s.Hq;
    sp.Hkv = s.Hkv;
    sp.G = s.Hq / s.Hkv;
    sp.D = s.D;
    sp.T = s.T;
    sp.Pmax = s.Pmax;
    sp.Kmax = s.Kmax;
    sp.layer = layer;
    sp.K = K;
    sp.q = q;
    sp.meta = meta;
    sp.seq_len = seq_len;
    sp.rescore_mask = rescore_mask;
    sp.sel_idx = sel_idx;
    sp.sel_cnt = sel_cnt;
    sp.scores_out = scores_out;
    sp.scores_ws = scores_ws;
    sp.err = err;
    const cudaError_t e = kvmm::launch_score_only(sp, group_reduce, cs);
    if (e != cudaSuccess) return launched(e);
    AttnParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.G = s.Hq / s.Hkv;
    p.D = s.D;
    p.T = s.T;
    p.Pmax = s.Pmax;
    p.Kmax = s.Kmax;
    p.layer = layer;
    p.splits = splits;
    p.max_tiles = max_pages;
    p.region0 = static_cast<int32_t>(kvmm::attention_region0(s.D, scratch));
    p.select = 1;
    p.K = K;
    p.pstride = s.Pmax;
    p.bt_prefetch = bt_prefetch ? 1 : 0;
    p.bt_offset = static_cast<int32_t>(bt_offset);
    p.n_phys = s.n_phys;
    p.scale_log2 = (sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(s.D))) * 1.4426950408889634f;
    p.q = q;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.block_table = block_table;
    p.seq_len = seq_len;
    p.sel_idx = sel_idx;
    p.sel_cnt = sel_cnt;
    p.out = out;
    p.lse = lse;
    p.scores = scores_ws;
    p.rescore_mask = rescore_mask;
    p.sel_out = sel_idx;
    p.cnt_out = sel_cnt;
    p.err = err;
    return launched(kvmm::launch_sparse_attention(p, cs));
}

kvmm_status decode_layer(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q, const kvmm_bf16* new_k,
                         const kvmm_bf16* new_v, int32_t n_new, const int32_t* tok_begin, const int32_t* tok_end,
                         kvmm_bf16* k_pool, kvmm_bf16* v_pool, const int32_t* block_table, kvmm_bf16* meta,
                         const int32_t* seq_len, const uint8_t* rescore_mask, int32_t K, int32_t group_reduce,
                         float sm_scale, int32_t* sel_idx, int32_t* sel_cnt, float* scores_out, float* out,
                         float* lse, void* workspace, size_t workspace_bytes, uint32_t flags, int32_t* err,
                         kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < 0 || layer >= s.L || K < 1 || K > s.Kmax || !std::isfinite(sm_scale)) return KVMM_INVALID_ARG;
    if ((flags & ~KVMM_DECODE_EARLY_READS) != 0u) return KVMM_INVALID_ARG;
    if (group_reduce != 0 && group_reduce != 1) return KVMM_INVALID_ARG;
    if ((new_k == nullptr) != (new_v == nullptr)) return KVMM_INVALID_ARG;
    if (new_k != nullptr && (n_new < 1 || !req(new_k) || !req(new_v) || !req4(tok_begin) || !req4(tok_end)))
        return KVMM_INVALID_ARG;
    if (!req(q) || !req(meta) || !req(k_pool) || !req(v_pool) || !req4(block_table) || !req4(seq_len) ||
        !req4(sel_idx) || !req4(sel_cnt) || !opt4(scores_out) || !req4(out) || !opt4(lse) || !opt(workspace) ||
        !opt4(err))
        return KVMM_INVALID_ARG;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const kvmm::DecodeGrid grid = kvmm::decode_layer_grid(s);
    if (grid.nu == 0) {
        // the one-launch kernel's buffers do not fit: append, then the two-kernel call
        if (workspace == nullptr || workspace_bytes < score_ws_bytes(s)) return KVMM_WORKSPACE_TOO_SMALL;
        if (new_k != nullptr) {
            st = kv_minmax_update(shape, layer, new_k, new_v, n_new, tok_begin, tok_end, k_pool, v_pool,
                                  block_table, meta, err, stream);
            if (st != KVMM_OK) return st;
        }
        return page_score_topk_attn(shape, layer, q, meta, k_pool, v_pool, block_table, seq_len, rescore_mask, K,
                                    group_reduce, sm_scale, sel_idx, sel_cnt, scores_out, out, lse, workspace,
                                    workspace_bytes, err, stream);
    }
    kvmm::DecodeParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.G = s.Hq / s.Hkv;
    p.D = s.D;
    p.T = s.T;
    p.Pmax = s.Pmax;
    p.Kmax = s.Kmax;
    p.layer = layer;
    p.K = K;
    p.C = grid.c;
    p.NU = grid.nu;
    p.early = (flags & KVMM_DECODE_EARLY_READS) != 0u ? 1 : 0;
    p.n_new = new_k != nullptr ? n_new : 0;
    p.n_phys = s.n_phys;
    p.scale_log2 = (sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(s.D))) * 1.4426950408889634f;
    p.q = q;
    p.new_k = new_k;
    p.new_v = new_v;
    p.tok_begin = tok_begin;
    p.tok_end = tok_end;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.block_table = block_table;
    p.meta = meta;
    p.seq_len = seq_len;
    p.rescore_mask = rescore_mask;
    p.sel_idx = sel_idx;
    p.sel_cnt = sel_cnt;
    p.scores_out = scores_out;
    p.out = out;
    p.lse = lse;
    p.err = err;
    return launched(kvmm::launch_decode_layer(p, group_reduce, kvmm::kPhBoth, cs));
}

kvmm_status topk_promotion_diff(const kvmm_shape* shape, int32_t layer,
                                const uint8_t* rescore_mask, int32_t* prev_idx,
                                int32_t* prev_cnt, const int32_t* cur_idx,
                                const int32_t* cur_cnt, int32_t commit, int32_t* promoted,
                                int32_t* promoted_cnt, int32_t* evicted, int32_t* evicted_cnt,
                                int32_t* total_promoted, int32_t* err, kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < 0 || layer >= s.L) return KVMM_INVALID_ARG;
    if (!req4(prev_idx) || !req4(prev_cnt) || !req4(cur_idx) || !req4(cur_cnt) || !req4(promoted) ||
        !req4(promoted_cnt) || !opt4(evicted) || !opt4(evicted_cnt) || !opt4(total_promoted) || !opt4(err))
        return KVMM_INVALID_ARG;
    DiffParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hkv = s.Hkv;
    p.Kmax = s.Kmax;
    p.layer = layer;
    p.commit = commit != 0;
    p.rescore_mask = rescore_mask;
    p.prev_idx = prev_idx;
    p.prev_cnt = prev_cnt;
    p.cur_idx = cur_idx;
    p.cur_cnt = cur_cnt;
    p.promoted = promoted;
    p.promoted_cnt = promoted_cnt;
    p.evicted = evicted;
    p.evicted_cnt = evicted_cnt;
    p.total_promoted = total_promoted;
    p.err = err;
    return launched(kvmm::launch_promotion_diff(p, reinterpret_cast<cudaStream_t>(stream)));
}

kvmm_status block_table_update(const kvmm_shape* shape, const int64_t* idx, const int32_t* val, int32_t n,
                               int32_t* block_table, int32_t* err, kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (n < 0 || !req4(block_table) || !opt4(err)) return KVMM_INVALID_ARG;
    if (n == 0) return KVMM_OK;
    if (idx == nullptr || val == nullptr || !aligned(idx, 8) || !aligned(val, 4)) return KVMM_INVALID_ARG;
    const void* di = device_view_of_host(idx);
    const void* dv = device_view_of_host(val);
    if (di == nullptr || dv == nullptr) return KVMM_INVALID_ARG;  // memory the device cannot read
    kvmm::TableUpdateParams p{};
    p.n = n;
    p.entries = static_cast<long long>(s.B) * s.L * s.Hkv * s.Pmax;
    p.n_phys = s.n_phys;
    p.idx = static_cast<const int64_t*>(di);
    p.val = static_cast<const int32_t*>(dv);
    p.block_table = block_table;
    p.err = err;
    return launched(kvmm::launch_table_update(p, reinterpret_cast<cudaStream_t>(stream)));
}

kvmm_status promote_pages(const kvmm_shape* shape, int32_t layer, const uint8_t* rescore_mask,
                          const int32_t* promoted, const int32_t* promoted_cnt, const int32_t* evicted,
                          const int32_t* evicted_cnt, const kvmm_bf16* host_k, const kvmm_bf16* host_v,
                          kvmm_bf16* k_pool, kvmm_bf16* v_pool, int32_t* block_table, int32_t* moved,
                          int32_t* freed, int32_t* freed_cnt, int32_t max_ctas, int32_t* err, kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < 0 || layer >= s.L || max_ctas < 0) return KVMM_INVALID_ARG;
    if (!req4(promoted) || !req4(promoted_cnt) || !req4(evicted) || !req4(evicted_cnt) || !req(host_k) ||
        !req(host_v) || !req(k_pool) || !req(v_pool) || !req4(block_table) || !opt4(moved) || !opt4(freed) ||
        !opt4(freed_cnt) || !opt4(err))
        return KVMM_INVALID_ARG;
    const void* hk = device_view_of_host(host_k);
    const void* hv = device_view_of_host(host_v);
    if (hk == nullptr || hv == nullptr) return KVMM_INVALID_ARG;  // host memory the device cannot read
    kvmm::PromoteParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hkv = s.Hkv;
    p.T = s.T;
    p.D = s.D;
    p.Pmax = s.Pmax;
    p.Kmax = s.Kmax;
    p.layer = layer;
    p.n_phys = s.n_phys;
    p.rescore_mask = rescore_mask;
    p.promoted = promoted;
    p.promoted_cnt = promoted_cnt;
    p.evicted = evicted;
    p.evicted_cnt = evicted_cnt;
    p.host_k = static_cast<const kvmm_bf16*>(hk);
    p.host_v = static_cast<const kvmm_bf16*>(hv);
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.block_table = block_table;
    p.moved = moved;
    p.freed = freed;
    p.freed_cnt = freed_cnt;
    p.err = err;
    return launched(kvmm::launch_promote(p, max_ctas, reinterpret_cast<cudaStream_t>(stream)));
}

kvmm_status topk_history_record(const kvmm_shape* shape, int32_t layer, const int32_t* sel_idx,
                                const int32_t* sel_cnt, const int32_t* seq_len, int32_t W, int32_t slot,
                                int32_t* hist_idx, int32_t* hist_cnt, int32_t* hist_pages, int32_t* err,
                                kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (layer < -1 || layer >= s.L || W < 1 || slot < 0 || slot >= W) return KVMM_INVALID_ARG;
    if (!req4(sel_idx) || !req4(sel_cnt) || !req4(seq_len) || !req4(hist_idx) || !req4(hist_cnt) ||
        !req4(hist_pages) || !opt4(err))
        return KVMM_INVALID_ARG;
    kvmm::StabilityParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hkv = s.Hkv;
    p.T = s.T;
    p.Pmax = s.Pmax;
    p.Kmax = s.Kmax;
    p.W = W;
    p.layer = layer;
    p.slot = slot;
    p.sel_idx = sel_idx;
    p.sel_cnt = sel_cnt;
    p.seq_len = seq_len;
    p.hist_idx = hist_idx;
    p.hist_cnt = hist_cnt;
    p.hist_pages = hist_pages;
    p.err = err;
    return launched(kvmm::launch_history_record(p, reinterpret_cast<cudaStream_t>(stream)));
}

kvmm_status topk_stability_rco(const kvmm_shape* shape, const int32_t* hist_idx, const int32_t* hist_cnt,
                               const int32_t* hist_pages, int32_t W, int32_t n, int32_t head, int32_t lag,
                               float unstable_frac, float* rco_unit, float* stability, uint8_t* unstable,
                               int32_t* err, kvmm_stream stream)
{
    kvmm_status st = check_shape(shape);
    if (st != KVMM_OK) return st;
    const kvmm_shape& s = *shape;
    if (W < 1 || n < 1 || n > W || head < 0 || head >= W || lag < 1 || lag >= n) return KVMM_INVALID_ARG;
    if (n > 1024) return KVMM_UNSUPPORTED_SHAPE;  // the window's per-step values live in shared memory
    if (!(unstable_frac >= 0.f && unstable_frac <= 1.f)) return KVMM_INVALID_ARG;
    if (static_cast<size_t>(s.L) * s.Hkv > kvmm::stability_max_heads()) return KVMM_UNSUPPORTED_SHAPE;
    if (!req4(hist_idx) || !req4(hist_cnt) || !req4(hist_pages) || !req4(rco_unit) || !opt4(stability) ||
        !opt4(err))
        return KVMM_INVALID_ARG;
    kvmm::StabilityParams p{};
    p.B = s.B;
    p.L = s.L;
    p.Hkv = s.Hkv;
    p.T = s.T;
    p.Pmax = s.Pmax;
    p.Kmax = s.Kmax;
    p.W = W;
    p.n = n;
    p.head = head;
    p.lag = lag;
    p.unstable_frac = unstable_frac;
    p.hist_idx = const_cast<int32_t*>(hist_idx);
    p.hist_cnt = const_cast<int32_t*>(hist_cnt);
    p.hist_pages = const_cast<int32_t*>(hist_pages);
    p.rco_unit = rco_unit;
    p.stability = stability;
    p.unstable = unstable;
    p.err = err;
    return launched(kvmm::launch_stability_rco(p, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
