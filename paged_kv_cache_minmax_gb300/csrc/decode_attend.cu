// decode_attend.cu -- the clustered decode kernel (decode_layer.cuh) with its
// second phase only: sparse_paged_decode_attn in one launch.
//
// FlexiCache (MLSys'26 blog summary), "Core method, 1. Stability-
// differentiated placement" (decode attention runs over the selected pages
// only) and "System design, head-level block table" (pages are found through
// [batch, layer, head, logical_block]; null entries are never read).  The
// cluster resolves each unit's kept selection through the table, streams the
// selected K/V pages (one unit's pages follow the previous unit's in the same
// slots) and merges the CTAs' softmax partials on chip.  The group reduction
// plays no part here, so one instantiation serves both.
#include "decode_layer.cuh"

namespace kvmm {

DecodeKernel decode_kernel_attend(int D, int T, int nu)
{
    using namespace dl;
#define KVMM_DL(D_, T_) \
    if (D == D_ && T == T_) \
        return nu == 1 ? decode_layer_kernel<D_, T_, 0, 1, kPhAttend> : decode_layer_kernel<D_, T_, 0, 2, kPhAttend>;
    KVMM_DL(128, 16)
    KVMM_DL(128, 32)
    KVMM_DL(64, 16)
    KVMM_DL(64, 32)
#undef KVMM_DL
    return nullptr;
}

}  // namespace kvmm
