// decode_score.cu -- the clustered decode kernel (decode_layer.cuh) with its
// first phase only: page_score_topk in one launch.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 2. MinMax-metadata page
// scoring": every page of a rescored (layer, KV head) is scored from its key
// bounds and the top-K pages are kept.  The cluster streams the units'
// metadata rows, scores them on the tensor cores, exchanges the scores on chip
// and selects exactly (block_topk); one unit's selection overlaps the next
// unit's stream, and the scores never travel through global memory.
#include "decode_layer.cuh"

namespace kvmm {

DecodeKernel decode_kernel_score(int D, int T, int mode, int nu)
{
    using namespace dl;
#define KVMM_DL(D_, T_) \
    if (D == D_ && T == T_) \
        return mode ? (nu == 1 ? decode_layer_kernel<D_, T_, 1, 1, kPhScore> : decode_layer_kernel<D_, T_, 1, 2, kPhScore>) \
                    : (nu == 1 ? decode_layer_kernel<D_, T_, 0, 1, kPhScore> : decode_layer_kernel<D_, T_, 0, 2, kPhScore>);
    KVMM_DL(128, 16)
    KVMM_DL(128, 32)
    KVMM_DL(64, 16)
    KVMM_DL(64, 32)
#undef KVMM_DL
    return nullptr;
}

}  // namespace kvmm
