// decode_layer.cu -- launch shape and launches of the clustered decode kernel
// (decode_layer.cuh), and its instantiation with both phases: decode_layer,
// one launch per layer that appends, scores, selects and attends.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 2. MinMax-metadata page
// scoring" and "Core method, 1. Stability-differentiated placement" /
// "System design, head-level block table".
#include <cudaTypedefs.h>

#include <mutex>

#include "decode_layer.cuh"

namespace kvmm {

DecodeKernel decode_kernel_both(int D, int T, int mode, int nu)
{
    using namespace dl;
#define KVMM_DL(D_, T_) \
    if (D == D_ && T == T_) \
        return mode ? (nu == 1 ? decode_layer_kernel<D_, T_, 1, 1, kPhBoth> : decode_layer_kernel<D_, T_, 1, 2, kPhBoth>) \
                    : (nu == 1 ? decode_layer_kernel<D_, T_, 0, 1, kPhBoth> : decode_layer_kernel<D_, T_, 0, 2, kPhBoth>);
    KVMM_DL(128, 16)
    KVMM_DL(128, 32)
    KVMM_DL(64, 16)
    KVMM_DL(64, 32)
#undef KVMM_DL
    return nullptr;
}

namespace {

DecodeKernel decode_kernel_for(int D, int T, int mode, int nu, int ph)
{
    if (ph == kPhScore) return decode_kernel_score(D, T, mode, nu);
    if (ph == kPhAttend) return decode_kernel_attend(D, T, nu);
    return decode_kernel_both(D, T, mode, nu);
}

// opt-ins of one instantiation, once per device and size
cudaError_t prepare_decode(DecodeKernel kernel, size_t smem)
{
    struct Prepared {
        DecodeKernel kernel;
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

}  // namespace

// the units' block-table rows go to shared memory when the launch still fits the limit with them
static bool decode_layer_bt(int D, int T, int Pmax, int Kmax, int C, int G, int NU, int ph)
{
    const int maxp = (Kmax + C - 1) / C;
    return (ph & kPhAttend) && Pmax % 4 == 0 &&
           dl::d_layout(D, T, Pmax, Kmax, C, maxp, G, true, NU, ph).total <= kDSmemLimit;
}

static size_t decode_layer_smem(int D, int T, int Pmax, int Kmax, int C, int G, int NU, int ph)
{
    const int maxp = (Kmax + C - 1) / C;
    return dl::d_layout(D, T, Pmax, Kmax, C, maxp, G, decode_layer_bt(D, T, Pmax, Kmax, C, G, NU, ph), NU, ph)
        .total;
}

// Whether `clusters` clusters of c CTAs of `kernel` all fit the GPU at once, with room for an eighth more:
// with programmatic dependent launch the next launch's first clusters take the SMs this one leaves free
// before it ends, and a launch that needs every cluster place the GPU has was measured to run part of its
// grid in a second wave.  Clusters are placed within a GPC, so SMs / c overestimates; the occupancy query
// decides.
static bool one_wave(DecodeKernel kernel, size_t smem, int c, int clusters, int sms)
{
    int n = 0;
    if (c == 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, dl::kDThreads, smem) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        n = per_sm * sms;
    } else {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(clusters * c));
        cfg.blockDim = dim3(dl::kDThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(c);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
    }
    return n >= clusters + (clusters + 7) / 8;
}

// Units per cluster and CTAs per cluster.  For each unit count a cluster (two when there are two units, then
// one), the largest cluster whose buffers fit shared memory and whose clusters fit one wave; of those, the
// one with more CTAs in all, two units a cluster on a tie (one unit's selection then overlaps the other's
// streaming) -- except in a launch that only attends, which takes one unit a cluster on a tie when its
// clusters keep two CTAs or more.  Measured at the 128K shape: clusters of 4 over one unit each (128 CTAs)
// 40.5 us a launch, of 6 over two (96 CTAs) 43.9 us; attention alone at the 8B shape: one unit in clusters of
// 2, 15.6 us, two in clusters of 4, 16.4 us; at the GQA-5 shape single-CTA clusters 27.4 us against two units
// in clusters of 2, 27.3 us.  When no shape fits one wave, two units a cluster if their buffers fit,
// else one; none at all ({0, 0}) sends the caller to the two-kernel path.  Cached per device and shape.
DecodeGrid decode_layer_grid(const kvmm_shape& s, int ph)
{
    struct Choice {
        int dev, D, T, Pmax, Kmax, units, G, ph;
        DecodeGrid g;
    };
    static thread_local Choice cache[8] = {};
    static thread_local int next = 0;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    const int units = s.B * s.Hkv, G = s.Hq / s.Hkv;
    DecodeGrid g{0, 0};
    // a score item's tensor copy addresses its first row by a signed 32-bit coordinate (checked before the
    // cache, which does not key on the layer count)
    if (static_cast<long long>(s.B) * s.L * s.Hkv * s.Pmax > 0x7fffffffLL) return g;
    for (const auto& c : cache)
        if (c.g.nu > 0 && c.dev == dev && c.D == s.D && c.T == s.T && c.Pmax == s.Pmax && c.Kmax == s.Kmax &&
            c.units == units && c.G == G && c.ph == ph)
            return c.g;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long best_ctas = 0;
    bool best_wave = false;
    // two units a cluster only when there are two: one unit in a two-unit layout has half the room
    for (int nu = units < dl::kDUnits ? 1 : dl::kDUnits; nu >= 1; --nu) {
        DecodeKernel kernel = decode_kernel_for(s.D, s.T, 0, nu, ph);  // both reductions: same resources
        const int clusters = (units + nu - 1) / nu;
        int c0 = sms / clusters;
        if (c0 > kDMaxCluster) c0 = kDMaxCluster;
        if (c0 < 1) c0 = 1;
        int found = 0;
        bool wave = false;
        for (int c = c0; c >= 1 && !wave; --c) {
            const size_t smem = decode_layer_smem(s.D, s.T, s.Pmax, s.Kmax, c, G, nu, ph);
            if (smem > kDSmemLimit || prepare_decode(kernel, smem) != cudaSuccess) continue;
            if (one_wave(kernel, smem, c, clusters, sms)) {
                found = c;
                wave = true;
            } else if (found == 0 && c == 1) {
                found = 1;  // more clusters than one wave holds: single CTAs, as many waves as it takes
            }
        }
        if (found == 0) continue;
        const long long ctas = static_cast<long long>(clusters) * found;
        // a launch that only attends has no selection to overlap, and each unit's merge spans the cluster: on a
        // tie it takes one unit a cluster, unless that leaves single-CTA clusters
        const bool tie_to_one = ph == kPhAttend && nu == 1 && found > 1 && ctas == best_ctas;
        if (g.nu == 0 || (wave && !best_wave) || (wave && best_wave && (ctas > best_ctas || tie_to_one))) {
            g = {nu, found};
            best_ctas = ctas;
            best_wave = wave;
        }
    }
    if (g.nu > 0) cache[next++ % 8] = {dev, s.D, s.T, s.Pmax, s.Kmax, units, G, ph, g};
    return g;
}

// The tensor map of the metadata for the score items' tensor copies: a 3-D tensor of 16-bit elements,
// {64 (one 128-byte line), 2D / 64 lines of a [min | max] row, B * L * Hkv * Pmax rows}, read in boxes of
// {64, 2D / 64, 16 rows} with the 128-byte swizzle; rows past the end read as zeros.  The encoder is the
// driver's, reached through the runtime.
static cudaError_t meta_tensor_map(CUtensorMap* m, const DecodeParams& p)
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (encode == nullptr) return cudaErrorNotSupported;
    const cuuint64_t lines = static_cast<cuuint64_t>(2 * p.D / 64);
    const cuuint64_t rows = static_cast<cuuint64_t>(p.B) * p.L * p.Hkv * p.Pmax;
    const cuuint64_t dims[3] = {64, lines, rows};
    const cuuint64_t strides[2] = {128, lines * 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(lines), 16};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, p.meta, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_decode_layer(DecodeParams p, int group_reduce, int ph, cudaStream_t stream)
{
    DecodeKernel kernel = decode_kernel_for(p.D, p.T, group_reduce, p.NU, ph);
    CUtensorMap tmeta{};  // the attention phase alone reads no metadata: left empty
    if (ph & kPhScore) {
        const cudaError_t e = meta_tensor_map(&tmeta, p);
        if (e != cudaSuccess) return e;
    }
    p.maxp = (p.Kmax + p.C - 1) / p.C;
    p.bt_smem = decode_layer_bt(p.D, p.T, p.Pmax, p.Kmax, p.C, p.G, p.NU, ph) ? 1 : 0;
    const size_t smem = decode_layer_smem(p.D, p.T, p.Pmax, p.Kmax, p.C, p.G, p.NU, ph);
    cudaError_t e = prepare_decode(kernel, smem);
    if (e != cudaSuccess) return e;
    const int clusters = (p.B * p.Hkv + p.NU - 1) / p.NU;
    return launch_pdl_cluster(kernel, dim3(static_cast<unsigned>(clusters * p.C)), dim3(dl::kDThreads), smem,
                              stream, static_cast<unsigned>(p.C), p, tmeta);
}

}  // namespace kvmm
