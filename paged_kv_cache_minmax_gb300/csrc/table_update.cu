// table_update.cu -- the changed entries of the head-level block table.
//
// FlexiCache (MLSys'26 blog summary), "System design, head-level block
// table": dirty tracking synchronises only the changed regions of the
// [batch, layer, head, logical_block] table instead of the whole table every
// step.  The delta is the list of changed entries; it may sit in pinned host
// memory, read directly through the unified address space, so the table
// itself never crosses the host link.
//
// A grid-stride scatter: each thread reads its updates with independent
// loads (8 in flight) and writes them.  Validation is per update.
#include "common.cuh"
#include "kernels.h"

namespace kvmm {
namespace {

constexpr int kUpdThreads = 256;
constexpr int kUpdBatch = 8;

__global__ void __launch_bounds__(kUpdThreads) table_update_kernel(const TableUpdateParams p)
{
    pdl_wait_then_release();
    const long long stride = static_cast<long long>(gridDim.x) * kUpdThreads;
    for (long long i0 = static_cast<long long>(blockIdx.x) * kUpdThreads + threadIdx.x; i0 < p.n;
         i0 += stride * kUpdBatch) {
        long long idx[kUpdBatch];
        int32_t val[kUpdBatch];
#pragma unroll
        for (int k = 0; k < kUpdBatch; ++k) {
            const long long i = i0 + k * stride;
            idx[k] = -1;
            val[k] = 0;
            if (i < p.n) {
                idx[k] = p.idx[i];
                val[k] = p.val[i];
            }
        }
#pragma unroll
        for (int k = 0; k < kUpdBatch; ++k) {
            if (i0 + k * stride >= p.n) continue;
            if (idx[k] < 0 || idx[k] >= p.entries || val[k] < -1 || val[k] >= p.n_phys)
                report(p.err, KVMM_ERR_OUT_OF_RANGE);
            else
                p.block_table[idx[k]] = val[k];
        }
    }
}

}  // namespace

cudaError_t launch_table_update(const TableUpdateParams& p, cudaStream_t stream)
{
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long per_cta = static_cast<long long>(kUpdThreads) * kUpdBatch;
    const long long need = (p.n + per_cta - 1) / per_cta;
    const int grid = static_cast<int>(need < 2 * sms ? (need > 0 ? need : 1) : 2 * sms);
    return launch_pdl(table_update_kernel, dim3(static_cast<unsigned>(grid)), dim3(kUpdThreads), 0, stream, p);
}

}  // namespace kvmm
