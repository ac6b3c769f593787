// pkm_device.cuh -- sm_103a building blocks written as inline PTX: mbarriers with bounded
// waits, TMA (cp.async.bulk.tensor) loads/stores, cp.async, tcgen05 (TMEM alloc, MMA,
// commit, loads) and the shared-memory / instruction descriptors the MMAs take.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "paged_kv_mla.h"

namespace pkm {

// ------------------------------------------------------------------------------------
// generic helpers
// ------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void report(int32_t* status, int code) {
    if (status != nullptr) atomicMax(status, code);
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Register reallocation between warpgroups (four consecutive warps, every thread of the
// warpgroup executes the same instruction).  The pool is what the CTA was launched with:
// the warpgroups' new counts must add up to no more than that.
template <int N>
__device__ __forceinline__ void warpgroup_reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void warpgroup_reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------------------------
// programmatic dependent launch: a prepass lets the kernel that consumes its output start
// its prologue early; the consumer waits for the prepass's writes before reading them
// ------------------------------------------------------------------------------------

__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Blocks until every prerequisite grid has completed and its memory operations are visible
// (returns at once when the kernel was not launched as a dependent).
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Shared control block of a CTA's pipeline: the abort flag every wait polls, the caller's
// status word and the wait limit.
struct WaitCtl {
    volatile int* abort_flag;
    int32_t* status;
    uint64_t timeout_ns;
};

// Slow path of mbar_wait: spins until the phase completes, the abort flag rises or the wait
// outlives timeout_ns.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, const WaitCtl& w,
                                               bool obey_abort) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31) == 0) {
            if (obey_abort && *w.abort_flag) return false;
            if (globaltimer_ns() - t0 > w.timeout_ns) {
                report(w.status, PKM_ERR_TIMEOUT);
                *w.abort_flag = 1;
                return false;
            }
        }
    }
}

// The same, as a function of its own: the wait sites stay small.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity,
                                                   const WaitCtl& w, bool obey_abort) {
    return mbar_wait_spin(bar, parity, w, obey_abort);
}

// Waits until the phase with the given parity of `bar` has completed (acquire, CTA scope).
// Returns false when another role raised the abort flag (if `obey_abort`) or when the wait
// outlived timeout_ns; in the latter case it records PKM_ERR_TIMEOUT and raises the abort
// flag so that every role of the CTA winds down.
//
// CTA scope is enough for every barrier whose phase is completed by the asynchronous proxy
// (TMA complete_tx, tcgen05.commit) or by arrivals that only hand over tensor-memory
// accumulators ordered with tcgen05 fences, including arrivals from the other CTA of a pair.
// A satisfied wait then costs a few tens of cycles, against several hundred for the
// cluster-scope acquire of mbar_wait_cluster.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w,
                                          bool obey_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, w, obey_abort);
}

// mbar_wait with the slow path inlined, for kernels whose warpgroups change their register
// counts (setmaxnreg): such a region cannot call a separately compiled function.
__device__ __forceinline__ bool mbar_wait_inl(uint64_t* bar, uint32_t parity, const WaitCtl& w,
                                              bool obey_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_spin(bar, parity, w, obey_abort);
}

// ------------------------------------------------------------------------------------
// clusters and CTA pairs (two CTAs whose %cluster_ctarank differ in bit 0)
// ------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared::cluster address of the object at shared::cta address `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive (release, cluster scope) on an mbarrier given by its shared::cluster address,
// possibly in another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// Adds `bytes` to the transaction count of an mbarrier of either CTA of the cluster, without
// arriving: the thread that will later arrive announces the bytes of a TMA load it issues.
__device__ __forceinline__ void mbar_expect_tx_cluster(uint32_t cluster_addr, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cluster.shared::cluster.b64 [%0], %1;" ::"r"(
                     cluster_addr),
                 "r"(bytes)
                 : "memory");
}

// Arrive on an mbarrier of either CTA of the cluster (shared::cluster address) with the
// default release-at-CTA semantics.  Used for hand-offs whose data is ordered by tcgen05
// fences (a TMEM accumulator drained by the epilogue), where a cluster-scope release would
// only add latency.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// mbar_wait with acquire at cluster scope, for a barrier whose completion publishes ordinary
// (generic-proxy) shared-memory writes made by threads of the other CTA of the pair.  Same
// limits and abort behaviour as mbar_wait.
static __device__ __noinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                      const WaitCtl& w, bool obey_abort = true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 31) == 0) {
            if (obey_abort && *w.abort_flag) return false;
            if (globaltimer_ns() - t0 > w.timeout_ns) {
                report(w.status, PKM_ERR_TIMEOUT);
                *w.abort_flag = 1;
                return false;
            }
        }
    }
}

// All threads of every CTA in the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Spins for about `ns` nanoseconds.
__device__ __forceinline__ void spin_ns(uint64_t ns) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < ns) {
    }
}

// ------------------------------------------------------------------------------------
// TMA (tensor maps are __grid_constant__ kernel parameters)
// ------------------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Adds `bytes` to the transaction count of a CTA-local mbarrier without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// 4-byte asynchronous copy global -> shared (both 4-byte aligned).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Makes `bar` wait, in its current phase, for every cp.async this thread has issued so far
// (one extra pending arrival, performed when they complete).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Untiled bulk copy of `bytes` contiguous bytes (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`'s transaction count.
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
        "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map,
                                                 uint64_t* bar, int32_t c0, int32_t c1,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1),
        "l"(policy)
        : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on an mbarrier of
// either CTA of the pair (`bar_cluster` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2.L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// 4-D variant without an L2 policy (rows gathered from a paged cache, all k-blocks at once).
__device__ __forceinline__ void tma_load_4d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1,
                                                 int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2 [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3)
        : "memory");
}

// 3-D variant (e.g. several k-blocks of a matrix in one operation).
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1,
                                                 int32_t c2, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2.L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2),
        "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src,
                                             int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::
            "l"(reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(c0), "r"(c1)
        : "memory");
}

// 3-D tiled store from this CTA's shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::
            "l"(reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// accesses (TMA stores, tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// L2 eviction-priority policies for cache hints.
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------------------------
// cp.async (16-byte, L2 only; src_bytes = 0 writes zeros)
// ------------------------------------------------------------------------------------

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// cp.async.wait_group takes an immediate; this dispatches a runtime count (0..7).
__device__ __forceinline__ void cp_async_wait_dyn(int pending) {
    switch (pending) {
        case 0: cp_async_wait<0>(); break;
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        case 5: cp_async_wait<5>(); break;
        case 6: cp_async_wait<6>(); break;
        default: cp_async_wait<7>(); break;
    }
}

// ------------------------------------------------------------------------------------
// plain vector memory ops
// ------------------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// d0 = a * b0 + d0 and d1 = a * b1 + d1, each rounded to nearest once (one packed
// fma.rn.f32x2 instruction instead of two).
__device__ __forceinline__ void fma2(float& d0, float& d1, float a, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %2};\n\t"
        "mov.b64 rb, {%3, %4};\n\t"
        "mov.b64 rc, {%0, %1};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a), "f"(b0), "f"(b1));
}

// Walks the tile ids [t_begin, t_end) of a persistent CTA (pair) as (m, n), n = t mod
// n_tiles, with one division at the start instead of one per tile: the loops of the
// MMA-issuing warp and of the warps sharing its scheduler stay short.
struct TileWalk {
    int64_t t, end, m;
    int n, n_tiles;
    __device__ __forceinline__ TileWalk(int64_t t_begin, int64_t t_end, int tiles)
        : t(t_begin), end(t_end), m(t_begin / tiles),
          n(static_cast<int>(t_begin % tiles)), n_tiles(tiles) {}
    __device__ __forceinline__ bool valid() const { return t < end; }
    __device__ __forceinline__ void next() {
        ++t;
        if (++n == n_tiles) {
            n = 0;
            ++m;
        }
    }
};

// Slot and phase parity of a ring of `stages` slots, advanced one slot at a time.
struct RingPos {
    uint32_t stage = 0, phase = 0;
    __device__ __forceinline__ void next(uint32_t stages) {
        if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

// Stores a warp's 32-row x 64-column bf16 box to global memory in whole 128-byte row
// segments.  On entry lane r holds row r as 32 packed bf16 pairs in `p`; the rows pass
// through `stage` (4 KB of shared memory owned by the warp, 16-byte chunk j of row r kept
// at chunk j ^ (r & 7), so both passes are free of bank conflicts) and come back out eight
// lanes per row, so each store instruction writes four complete rows.  Row r goes to
// row0 + r * pitch (elements) when bit r of `valid` is set.  This costs the warp a few
// dozen instructions, where issuing a TMA store costs its thread several hundred cycles.
__device__ __forceinline__ void warp_store_rows_32x64(uint32_t stage, const uint32_t (&p)[32],
                                                      uint16_t* row0, int64_t pitch,
                                                      uint32_t valid, int lane) {
    const uint32_t rowaddr = stage + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        st_shared_v4(rowaddr + ((j ^ (lane & 7)) << 4), p[4 * j], p[4 * j + 1], p[4 * j + 2],
                     p[4 * j + 3]);
    __syncwarp();
    const int chunk = lane & 7;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int r = it * 4 + (lane >> 3);
        const uint4 v = ld_shared_v4(stage + r * 128 + ((chunk ^ (r & 7)) << 4));
        if ((valid >> r) & 1u) st_v4(row0 + r * pitch + chunk * 8, v);
    }
    __syncwarp();  // the box may be overwritten once every lane has read its part
}

// Maximum of v over the 32 lanes of a warp, in one instruction (every lane must execute it).
// For non-negative floats the bit patterns order like the values, so this also takes the
// maximum of magnitudes.
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
    uint32_t r;
    asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
    return r;
}

// The two bf16 halves of a packed word as fp32 values (exact): each half plus -0.0 by the
// mixed-precision add (bf16 operand, fp32 result), which keeps the sign of a zero and
// leaves the integer/logic pipe to other work.
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, 0f80000000;\n\t"
        "add.rn.f32.bf16 %1, h, 0f80000000;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
}

// max(|a|, |b|, |c|) in one instruction.
__device__ __forceinline__ float fmax3_abs(float a, float b, float c) {
    float r;
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Two fp32 values to e4m3 (round to nearest even, saturating to +-448); lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// (d0, d1) += (a0, a1) * (b0, b1), one packed fp32x2 FMA (each lane rounded as fmaf).
__device__ __forceinline__ void fma2v(float& d0, float& d1, float a0, float a1, float b0,
                                      float b1) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%0, %1};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// (d0, d1) = (a0, a1) * (b0, b1), one packed fp32x2 multiply (each lane rounded as a * b).
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0,
                                     float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
    return *reinterpret_cast<uint32_t*>(&h);
}

// (d0, d1) = (a0, a1) * (b0, b1) + (c0, c1), one packed fp32x2 FMA (each lane as fmaf).
__device__ __forceinline__ void fma2x(float& d0, float& d1, float a0, float a1, float b0,
                                      float b1, float c0, float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ float rcp_approx(float s) {
    float y;
    asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(s));
    return y;
}

// x / s for a block scale s > 0 with an approximate reciprocal y ~ 1 / s (within an ulp or
// so) that the caller computes once per block: the remainder correction of Markstein (IBM
// J. Res. Develop. 34(1), 1990).  q0 = RN(x * y) is within a few ulps of x / s, the
// remainder r = x - q0 * s is exact in one FMA, and RN(q0 + r * y) is RN(x / s) or its
// neighbour.  The sign of a zero quotient is the sign of x.
__device__ __forceinline__ float div_by_scale(float x, float s, float y) {
    const float q0 = __fmul_rn(x, y);
    const float r = __fmaf_rn(-q0, s, x);
    return copysignf(__fmaf_rn(r, y, q0), x);
}

// RN(amax / 448) for amax >= 2^-100 (a normal quotient): the same correction with the
// correctly rounded constant c = RN(1 / 448), q0 = RN(amax * c), r = amax - 448 * q0
// (exact), RN(q0 + r * c).  Checked equal to the correctly rounded quotient for every
// bf16 amax in that range.
__device__ __forceinline__ float scale_of_amax(float amax) {
    const float c = 0x1.24924ap-9f;  // RN(1 / 448)
    const float q0 = __fmul_rn(amax, c);
    return __fmaf_rn(__fmaf_rn(-q0, 448.0f, amax), c, q0);
}

// One 128-value block quantised to e4m3: s = RN(amax / 448) (1 for an all-zero block) and
// codes e4m3_rne_satfinite(RN(x / s)) for |x| <= amax, x and amax bf16 values.  For
// amax >= 2^-100 the quotients are div_by_scale's with the hardware's approximate
// reciprocal, taken in pairs by packed fp32x2 operations: they can miss RN(x / s) by an
// ulp, but never where that changes the e4m3 code (checked exhaustively over every bf16 x
// and amax; code differences appear only for amax < 2^-104).  Smaller blocks divide
// correctly rounded.  The scale is always the correctly rounded quotient (amax * RN(1 /
// 448) alone differs from it for about half the bf16 values of amax).
struct E4m3Block {
    float s, yn;  // the scale and minus its approximate reciprocal
    bool fast;
    E4m3Block() = default;
    __device__ __forceinline__ explicit E4m3Block(float amax) {
        fast = amax >= 0x1p-100f;
        if (fast) s = scale_of_amax(amax);
        else s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        yn = -rcp_approx(s);
    }
    // Codes of four values, the first in the low byte, when `fast` holds.  The quotient is
    // carried negated: n = x * (-y) = -q0, r = fma(n, s, x) = x - q0 * s, fma(r, -y, n) =
    // -RN(q0 + r * y); with that arrangement a zero quotient comes out with the sign
    // opposite to x's, so flipping the sign bit of each code (e4m3 is sign-magnitude and
    // its rounding symmetric) gives the codes of the quotients themselves, signed zeros
    // included.
    __device__ __forceinline__ uint32_t codes4_fast(float a, float b, float c, float d) const {
        float n0, n1, n2, n3, r0, r1, r2, r3;
        mul2(n0, n1, a, b, yn, yn);
        mul2(n2, n3, c, d, yn, yn);
        fma2x(r0, r1, n0, n1, s, s, a, b);
        fma2x(r2, r3, n2, n3, s, s, c, d);
        fma2x(n0, n1, r0, r1, yn, yn, n0, n1);
        fma2x(n2, n3, r2, r3, yn, yn, n2, n3);
        return (e4m3x2(n0, n1) | (e4m3x2(n2, n3) << 16)) ^ 0x80808080u;
    }
    // Codes of four values in every case.
    __device__ __forceinline__ uint32_t codes4(float a, float b, float c, float d) const {
        if (fast) return codes4_fast(a, b, c, d);
        return e4m3x2(__fdiv_rn(a, s), __fdiv_rn(b, s)) |
               (e4m3x2(__fdiv_rn(c, s), __fdiv_rn(d, s)) << 16);
    }
};

// ------------------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads
// ------------------------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// CTA-pair TMEM management: one warp in EACH CTA of the pair issues these together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, e4m3 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Pair MMA (issued by one thread of the even CTA): M = 256 split as 128 rows of A per CTA,
// B split along N between the two CTAs, D = each CTA's 128 rows x N in its own TMEM.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on the mbarrier at `bar`'s offset in every CTA of `cta_mask` when all pair
// MMAs this thread issued so far complete.
// Pair MMA, e4m3 x e4m3 -> fp32 (M = 256 over the two CTAs).
__device__ __forceinline__ void mma_e4m3_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued so far completes.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 TMEM lanes x 32 consecutive 32-bit columns: thread i of the warp receives lane
// (base lane + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// 32 TMEM lanes x 16 consecutive 32-bit columns (tmem_ld_x32's layout, half the columns).
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle (the layout TMA
// writes with CU_TENSOR_MAP_SWIZZLE_128B): start address, leading / stride byte offsets,
// descriptor version 1 (bits 46-47), layout type 2 = SWIZZLE_128B (bits 61-63).
//   K-major operand: rows of 128 bytes, 8-row core groups SBO = 1024 bytes apart, LBO
//   unused.  MN-major operand: LBO = distance between 64-element MN chunks, SBO =
//   distance between 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// The descriptor's start-address field counts 16-byte units: adding bytes / 16 to a
// descriptor moves its start by that many bytes (shared addresses stay below 256 KB).
__device__ __forceinline__ uint64_t desc_add_bytes(uint64_t d, uint32_t bytes) {
    return d + (bytes >> 4);
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9,
// 10-12 = 1), A / B major-ness (bits 15 / 16: 0 = K-major, 1 = MN-major), N >> 3 at bit
// 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((static_cast<uint32_t>(n) >> 3) << 17) |
           ((static_cast<uint32_t>(m) >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with A and B e4m3 (format 0), D fp32, K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int m, int n) {
    return (1u << 4) | ((static_cast<uint32_t>(n) >> 3) << 17) |
           ((static_cast<uint32_t>(m) >> 4) << 24);
}

}  // namespace pkm
