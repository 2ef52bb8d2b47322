// common.cuh -- device helpers shared by the kvmm kernels (sm_103a).
//
// Inline PTX for the Blackwell data-movement path used by the kernels:
// 1-D bulk copies (cp.async.bulk, the TMA unit) completing on shared-memory
// mbarriers, bounded mbarrier waits, bf16 unpacking, and the warp-level
// mma.sync / movmatrix forms used by the attention tile.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "kvmm.h"

namespace kvmm {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// error word
__device__ __forceinline__ void report(int32_t* err, int32_t bit)
{
    if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarriers and bulk copies
__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// make initialised barriers visible to the async (bulk-copy) proxy
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// order earlier generic-proxy shared-memory accesses before later bulk copies
__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the barrier phase with the given parity, giving up after about
// `limit_ns` nanoseconds.  Returns false on time-out (the caller reports
// KVMM_ERR_TIMEOUT); a completed copy never takes anywhere near that long.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 1000000000ull)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 255u) == 255u && global_timer_ns() - t0 > limit_ns) return false;
    }
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// An L2 policy for data read once: its lines are the first to go, so a stream
// larger than L2 does not push out the code, tables and small per-launch state.
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_copy_g2s with an L2 cache policy for the source lines
__device__ __forceinline__ void bulk_copy_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                   uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 3-D tensor copy (TMA) global -> shared of the box at coordinates (c0, c1, c2) of the tensor map at `tmap`
// (the generic address of a __grid_constant__ kernel parameter), completing the box's bytes of transaction
// on `bar`, with an L2 cache policy for the source lines.  c0 times the element size must be a multiple of
// 16 bytes; the destination is aligned as the map's swizzle requires (1024 bytes for the 128-byte swizzle).
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const void* tmap, int c0, int c1, int c2, uint64_t* bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, "
        "%4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// thread-block clusters and distributed shared memory
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// every thread of every CTA of the cluster arrives and waits; release/acquire
// make each CTA's earlier shared-memory writes visible to the others
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// the two halves of cluster_sync, for work that needs neither in between
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// store a float into the shared memory of CTA `rank` of the cluster, at the
// address that `local` has in this CTA's shared memory (visible to that CTA
// after the next cluster barrier)
__device__ __forceinline__ void st_dsmem_f32(void* local, uint32_t rank, float v)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// asynchronous store of v to the float at `local`'s address in CTA `rank` of
// the cluster, completing 4 bytes of transaction on the mbarrier at
// `local_bar`'s address in that CTA.  A thread that sees the barrier's phase
// complete sees the value; the sender needs no fence.
__device__ __forceinline__ void st_async_f32(void* local, uint64_t* local_bar, uint32_t rank, float v)
{
    uint32_t ra, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_addr(local_bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(ra),
                 "r"(__float_as_uint(v)), "r"(rb)
                 : "memory");
}

// st_async_f32 of four consecutive floats (16 bytes of transaction); `local` 16-byte aligned
__device__ __forceinline__ void st_async_v4_f32(void* local, uint64_t* local_bar, uint32_t rank, float a, float b,
                                                float c, float d)
{
    uint32_t ra, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_addr(local_bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(ra),
                 "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)), "r"(__float_as_uint(d)),
                 "r"(rb)
                 : "memory");
}

// asynchronous atomic min (MAX = false) or max (MAX = true) of v into the
// unsigned word at `local`'s address in CTA `rank` of the cluster, completing
// 4 bytes of transaction on the mbarrier at `local_bar`'s address in that
// CTA, like st_async_f32
template <bool MAX>
__device__ __forceinline__ void red_async_minmax_u32(uint32_t* local, uint64_t* local_bar, uint32_t rank, uint32_t v)
{
    uint32_t ra, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_addr(local_bar)), "r"(rank));
    if (MAX)
        asm volatile("red.async.relaxed.cluster.shared::cluster.mbarrier::complete_tx::bytes.max.u32 [%0], %1, [%2];" ::"r"(ra),
                     "r"(v), "r"(rb)
                     : "memory");
    else
        asm volatile("red.async.relaxed.cluster.shared::cluster.mbarrier::complete_tx::bytes.min.u32 [%0], %1, [%2];" ::"r"(ra),
                     "r"(v), "r"(rb)
                     : "memory");
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: the next kernel in the stream may be
// scheduled once every CTA of this one has called launch_dependents; a kernel
// must call wait before touching memory its predecessor writes (or reads).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Every kvmm kernel lets its dependents be scheduled only after its own wait
// has returned: in a chain A -> B -> C of these launches, C's CTAs then start
// only once A has finished, so a launch that reads part of its inputs before
// its wait (decode_layer with KVMM_DECODE_EARLY_READS) overlaps the kernel
// launched just before it and no earlier one.
__device__ __forceinline__ void pdl_wait_then_release()
{
    pdl_wait();
    pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// loads
__device__ __forceinline__ uint4 ld_shared_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

__device__ __forceinline__ uint2 ld_shared_v2(const void* p)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_addr(p)));
    return v;
}

// streaming read-only global load that does not allocate in L1
__device__ __forceinline__ uint4 ld_stream_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// bf16 helpers (a 32-bit word holds two bf16: element 0 in the low half)
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// round two floats to bf16 (nearest-even) and pack: lo in bits 0..15
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// ---------------------------------------------------------------------------
// warp-level tensor-core tile ops
//
// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col).  Fragment
// layout, lane = 4*g + t: A regs {(g, 2t..2t+1), (g+8, 2t..), (g, 2t+8..),
// (g+8, 2t+8..)}; B regs {(k 2t..2t+1, n g), (k 2t+8.., n g)}; C regs
// {(g, 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)}.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// transpose an 8x8 matrix of 16-bit elements held in the standard fragment
// layout (lane 4*g + t holds row g, columns 2t and 2t+1)
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a)
{
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

}  // namespace kvmm
