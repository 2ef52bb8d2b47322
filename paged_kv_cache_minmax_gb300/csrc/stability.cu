// stability.cu -- temporal stability of every (layer, KV head), from its
// recorded top-K sets.
//
// FlexiCache (MLSys'26 blog summary), "Core insight: attention heads differ
// in temporal stability": each head's top-K page set is recorded every
// decode step; sets a few steps apart are compared with the Random-Corrected
// Overlap (1 for identical sets, 0 for the overlap random sets would have),
// which is aggregated over a window into a per-head stability score; the
// least stable quarter of the heads is classed unstable.  The formula is
// the reading stated in kvmm.h:
//     RCO(A, B) = (|A n B| - |A||B|/P) / (min(|A|, |B|) - |A||B|/P),
// evaluated as the ratio of the exact integers P|A n B| - |A||B| and
// P min(|A|,|B|) - |A||B| (one correctly rounded division).
//
// Three small kernels (latency-bound, off the decode path):
//  - history_record_kernel: one CTA per (batch, layer, KV head) copies the
//    selections into a ring slot (one layer, or every layer at once);
//  - rco_unit_kernel: one CTA per unit turns the window's n lists into page
//    bitmaps in shared memory (when they fit; else it binary-searches one
//    ascending list in the other in global memory), then each warp takes
//    pairs of steps `lag` apart: the exact overlap is the popcount of the two
//    bitmaps' AND and gives the pair's integer numerator and denominator;
//    the pairs' divisions then run together, one pair per lane (the device's
//    double-precision pipe is narrow, and a warp instruction costs the same
//    with one lane or 32), and one thread averages them in step order;
//  - stability_classify_kernel: one CTA averages the units over the batch
//    and ranks the heads (ties to the lower index) to mark the unstable ones,
//    comparing order-preserving integer keys of the doubles (the device's
//    double-precision rate is low).
#include <climits>
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace kvmm {
namespace {

constexpr int kRcoThreads = 128;
constexpr int kClassifyThreads = 512;

__device__ __forceinline__ bool contains_sorted(const int32_t* list, int n, int32_t x)
{
    int lo = 0, hi = n;  // search [lo, hi)
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const int32_t v = list[mid];
        if (v == x) return true;
        if (v < x)
            lo = mid + 1;
        else
            hi = mid;
    }
    return false;
}

__global__ void __launch_bounds__(kRcoThreads) history_record_kernel(const StabilityParams p)
{
    pdl_wait_then_release();
    const int h = blockIdx.x, b = blockIdx.z;
    const int layer = p.layer >= 0 ? p.layer : static_cast<int>(blockIdx.y);
    const size_t u = (static_cast<size_t>(b) * p.L + layer) * p.Hkv + h;
    const size_t dst = static_cast<size_t>(p.slot) * p.B * p.L * p.Hkv + u;
    for (int i = threadIdx.x; i < p.Kmax; i += kRcoThreads) p.hist_idx[dst * p.Kmax + i] = p.sel_idx[u * p.Kmax + i];
    if (threadIdx.x == 0) {
        p.hist_cnt[dst] = p.sel_cnt[u];
        if (h == 0 && blockIdx.y == 0) {
            const int cap = p.Pmax * p.T;
            int seq = p.seq_len[b];
            if (seq < 0 || seq > cap) {
                report(p.err, KVMM_ERR_OUT_OF_RANGE);
                seq = seq < 0 ? 0 : cap;
            }
            p.hist_pages[static_cast<size_t>(p.slot) * p.B + b] = (seq + p.T - 1) / p.T;
        }
    }
}

// shared memory of rco_unit_kernel: per step of the window its RCO (double), the pair's numerator and
// denominator (int64), its count and page count, then, with bitmaps, one bit per page of every step's list
__host__ __device__ inline int rco_words(int Pmax) { return (Pmax + 31) / 32; }
__host__ __device__ inline size_t rco_smem_bytes(int n, int Pmax, bool bitmaps)
{
    return static_cast<size_t>(n) * (sizeof(double) + 2 * sizeof(long long) + 2 * sizeof(int32_t)) +
           (bitmaps ? static_cast<size_t>(n) * rco_words(Pmax) * sizeof(uint32_t) : 0);
}
constexpr size_t kRcoBitmapMax = 40 * 1024;  // bitmaps when they fit in this many bytes
__host__ __device__ inline bool rco_bitmaps(int n, int Pmax)
{
    return static_cast<size_t>(n) * rco_words(Pmax) * sizeof(uint32_t) <= kRcoBitmapMax;
}

__global__ void __launch_bounds__(kRcoThreads) rco_unit_kernel(const StabilityParams p)
{
    pdl_wait_then_release();
    extern __shared__ __align__(16) uint8_t rsm[];
    const int n = p.n;
    const bool bitmaps = rco_bitmaps(n, p.Pmax);
    const int words = rco_words(p.Pmax);
    double* r = reinterpret_cast<double*>(rsm);                // [n] RCO of pair (t, t + lag)
    long long* num = reinterpret_cast<long long*>(r + n);      // [n] P |A n B| - |A||B|
    long long* den = num + n;                                  // [n] P min(|A|,|B|) - |A||B|
    int32_t* cnt_s = reinterpret_cast<int32_t*>(den + n);      // [n] counts, clamped
    int32_t* pages_s = cnt_s + n;                              // [n] page counts, clamped
    uint32_t* bits = reinterpret_cast<uint32_t*>(pages_s + n);  // [n][words] when bitmaps
    const int h = blockIdx.x, l = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t u = (static_cast<size_t>(b) * p.L + l) * p.Hkv + h;
    const size_t per_slot = static_cast<size_t>(p.B) * p.L * p.Hkv;
    auto slot_of = [&](int t) { return (p.head - t + 2 * p.W) % p.W; };  // t steps before the newest
    for (int t = tid; t < n; t += kRcoThreads) {
        const int sl = slot_of(t);
        int c = p.hist_cnt[static_cast<size_t>(sl) * per_slot + u];
        if (c < 0 || c > p.Kmax) {
            report(p.err, KVMM_ERR_OUT_OF_RANGE);
            c = c < 0 ? 0 : p.Kmax;
        }
        int P = p.hist_pages[static_cast<size_t>(sl) * p.B + b];
        if (P < 0 || P > p.Pmax) {
            report(p.err, KVMM_ERR_OUT_OF_RANGE);
            P = P < 0 ? 0 : p.Pmax;
        }
        cnt_s[t] = c;
        pages_s[t] = P;
    }
    if (bitmaps) {
        for (int e = tid; e < n * words; e += kRcoThreads) bits[e] = 0u;
    }
    __syncthreads();
    if (bitmaps) {
        // element i of every step's list: the loads of 8 steps are issued before their bits are set
        constexpr int kBatch = 8;
        for (int i = tid; i < p.Kmax; i += kRcoThreads) {
            for (int t0 = 0; t0 < n; t0 += kBatch) {
                int32_t pg[kBatch];
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int t = t0 + k;
                    pg[k] = (t < n && i < cnt_s[t])
                                ? p.hist_idx[(static_cast<size_t>(slot_of(t)) * per_slot + u) * p.Kmax + i]
                                : INT_MIN;
                }
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    if (pg[k] == INT_MIN) continue;
                    if (pg[k] >= 0 && pg[k] < p.Pmax)
                        atomicOr(&bits[static_cast<size_t>(t0 + k) * words + (pg[k] >> 5)], 1u << (pg[k] & 31));
                    else
                        report(p.err, KVMM_ERR_OUT_OF_RANGE);
                }
            }
        }
        __syncthreads();
    }
    for (int t = warp; t + p.lag < n; t += kRcoThreads / 32) {
        const int na = cnt_s[t], nb = cnt_s[t + p.lag];
        int c = 0;
        if (bitmaps) {
            const uint32_t* ba = bits + static_cast<size_t>(t) * words;
            const uint32_t* bb = bits + static_cast<size_t>(t + p.lag) * words;
            for (int w = lane; w < words; w += 32) c += __popc(ba[w] & bb[w]);
        } else {
            const int32_t* A = p.hist_idx + (static_cast<size_t>(slot_of(t)) * per_slot + u) * p.Kmax;
            const int32_t* Bl = p.hist_idx + (static_cast<size_t>(slot_of(t + p.lag)) * per_slot + u) * p.Kmax;
            for (int i = lane; i < na; i += 32) {
                const int32_t pg = A[i];
                if (pg >= 0 && pg < p.Pmax) c += contains_sorted(Bl, nb, pg) ? 1 : 0;
                else report(p.err, KVMM_ERR_OUT_OF_RANGE);
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) c += __shfl_xor_sync(kFullMask, c, off);
        if (lane == 0) {
            const long long P = max(pages_s[t], pages_s[t + p.lag]);
            const long long chance_p = static_cast<long long>(na) * nb;
            num[t] = static_cast<long long>(c) * P - chance_p;
            den[t] = P > 0 ? static_cast<long long>(na < nb ? na : nb) * P - chance_p : 0;  // <= 0: RCO = 1
        }
    }
    __syncthreads();
    if (warp == 0) {
        for (int t = lane; t + p.lag < n; t += 32)
            r[t] = den[t] > 0 ? static_cast<double>(num[t]) / static_cast<double>(den[t]) : 1.0;
    }
    __syncthreads();
    if (tid == 0) {
        double sum = 0.0;
        for (int t = 0; t + p.lag < n; ++t) sum += r[t];  // in step order
        p.rco_unit[u] = static_cast<float>(sum / static_cast<double>(n - p.lag));
    }
}

// double -> unsigned 64-bit key with the same order (-0 taken as +0)
__device__ __forceinline__ unsigned long long order_key(double x)
{
    if (x == 0.0) x = 0.0;
    const unsigned long long bitsv = static_cast<unsigned long long>(__double_as_longlong(x));
    return (bitsv >> 63) ? ~bitsv : (bitsv | 0x8000000000000000ull);
}

__global__ void __launch_bounds__(kClassifyThreads) stability_classify_kernel(const StabilityParams p)
{
    pdl_wait_then_release();
    extern __shared__ unsigned long long skey[];  // [L * Hkv] order keys of the stabilities
    const int n = p.L * p.Hkv;
    for (int i = threadIdx.x; i < n; i += kClassifyThreads) {
        double s = 0.0;
        for (int b = 0; b < p.B; ++b) s += static_cast<double>(p.rco_unit[static_cast<size_t>(b) * n + i]);
        s /= static_cast<double>(p.B);
        skey[i] = order_key(s);
        if (p.stability) p.stability[i] = static_cast<float>(s);
    }
    __syncthreads();
    if (p.unstable == nullptr) return;
    const int k = static_cast<int>(floor(static_cast<double>(p.unstable_frac) * n + 0.5));
    for (int i = threadIdx.x; i < n; i += kClassifyThreads) {
        const unsigned long long ki = skey[i];
        int rank = 0;  // heads ranked before head i: less stable, or as stable and of lower index
        for (int j = 0; j < n; ++j) {
            const unsigned long long kj = skey[j];
            rank += (kj < ki || (kj == ki && j < i)) ? 1 : 0;
        }
        p.unstable[i] = rank < k ? 1 : 0;
    }
}

}  // namespace

cudaError_t launch_history_record(const StabilityParams& p, cudaStream_t stream)
{
    const unsigned layers = p.layer >= 0 ? 1u : static_cast<unsigned>(p.L);
    return launch_pdl(history_record_kernel, dim3(static_cast<unsigned>(p.Hkv), layers, static_cast<unsigned>(p.B)),
                      dim3(kRcoThreads), 0, stream, p);
}

cudaError_t launch_stability_rco(const StabilityParams& p, cudaStream_t stream)
{
    cudaError_t e = launch_pdl(rco_unit_kernel,
                               dim3(static_cast<unsigned>(p.Hkv), static_cast<unsigned>(p.L), static_cast<unsigned>(p.B)),
                               dim3(kRcoThreads), rco_smem_bytes(p.n, p.Pmax, rco_bitmaps(p.n, p.Pmax)), stream, p);
    if (e != cudaSuccess || (p.stability == nullptr && p.unstable == nullptr)) return e;
    const size_t smem = static_cast<size_t>(p.L) * p.Hkv * sizeof(unsigned long long);
    return launch_pdl(stability_classify_kernel, dim3(1), dim3(kClassifyThreads), smem, stream, p);
}

size_t stability_max_heads() { return 4096; }  // [L * Hkv] doubles fit the default shared-memory limit

}  // namespace kvmm
