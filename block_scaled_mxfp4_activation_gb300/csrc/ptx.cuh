// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// (tensor and 1-D bulk copies), tcgen05 (tensor-memory allocation, block-scaled
// MMA, shared->tensor-memory copies, tensor-memory loads) and cluster
// shared-memory access.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace mxfp4 {

// Bits of the device-side failure word (read by mxfp4_device_error()): which
// wait gave up.
enum DeviceError : uint32_t {
  kErrWaitTma = 1u << 0,     // MMA issuer waiting for a TMA stage
  kErrWaitA = 1u << 1,       // MMA issuer waiting for the activation stage
  kErrWaitEmpty = 1u << 2,   // a producer waiting for a free stage
  kErrWaitAccum = 1u << 3,   // epilogue waiting for the accumulator
  kErrWaitDrain = 1u << 4,   // teardown waiting for copies in flight
  kErrDiag = 1u << 5,        // the diagnostic kernel's wait (expected to give up)
  kErrBadPlan = 1u << 6,     // launch geometry disagrees with the kernel
  kErrWaitFlag = 1u << 7,    // a wait on another CTA's completion counter (multi-layer kernel)
  kErrBounds = 1u << 8,      // checked build: an index outside its buffer (the access was skipped)
  kErrWaitReduce = 1u << 9,  // split-K owner waiting for its peers' partial sums
};

__device__ __forceinline__ void report_error(uint32_t* word, uint32_t bits) {
  if (word != nullptr) atomicOr(word, bits);
}

// Guard of a computed-index memory access.  In the library's checked build
// (-DMXFP4_CHECKED) it tests the index against its buffer, and on failure
// reports kErrBounds and returns false so the access is skipped; in the normal
// build it is `true` and costs nothing.
#ifdef MXFP4_CHECKED
__device__ __forceinline__ bool in_bounds(bool ok, uint32_t* err) {
  if (!ok) report_error(err, kErrBounds);
  return ok;
}
#define MXFP4_IN_BOUNDS(cond, err) ::mxfp4::in_bounds((cond), (err))
#else
#define MXFP4_IN_BOUNDS(cond, err) true
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One lane of the (fully converged) warp gets true: the lowest-numbered lane.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits until the phase with the given parity has completed, for at most
// timeout_ns of global time.  Returns false if it gave up.  A phase that has
// already completed is seen by the non-blocking test, without the potentially
// suspending try_wait.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_test(bar, parity) || mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0 && global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// ----------------------------------------------------------------------------- proxies / fences
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tcgen05.mma / tcgen05.cp operands).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ----------------------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
}

// 2-D tiled tensor load into this CTA's shared memory, completing on `bar`.
// x (innermost, in elements of the map) must keep x * element size a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int32_t x, int32_t y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// 2-D tiled tensor store from this CTA's shared memory (bulk-group
// completion); elements outside the tensor are not written.  x as for loads.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, int32_t x, int32_t y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tm), "r"(x),
               "r"(y), "r"(src)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until every committed bulk store of this thread has finished reading
// shared memory (the global writes complete with the grid).
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// 1-D bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Prefetch of a 2-D tensor box / a byte range into L2 (no shared-memory write,
// no completion tracking).  L2 is the GPU's point of coherence, so prefetching
// data that an earlier grid is still writing cannot make a later read stale.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* tm, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(tm), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ----------------------------------------------------------------------------- grid dependencies
// Programmatic dependent launch: let the next grid in the stream start its
// prologue now / wait until the previous grid has completed and its memory
// operations are visible (a no-op when launched without the attribute).
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Loads of data that an earlier grid on the stream may have written, for use
// after grid_dependency_wait().  Inline asm keeps them after the wait (a load
// through __ldg or a const __restrict__ pointer counts as invariant for the
// kernel's lifetime and may be hoisted above it, reading the input before the
// previous grid has written it), and .cg reads at L2, the point of coherence.
__device__ __forceinline__ uint4 ld_after_wait_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ uint2 ld_after_wait_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.cg.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_after_wait_u8(const void* p) {
  uint32_t v;
  asm volatile("ld.global.cg.u8 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ----------------------------------------------------------------------------- counters between CTAs
// Completion counters in global memory that one CTA releases and others wait
// for (the multi-layer kernel's layer-to-layer hand-off).  The producer's
// threads store their results, then each makes them visible at GPU scope
// (fence_proxy_async_global for later TMA readers, then __threadfence), the
// CTA synchronises, and one thread adds to the counter with release
// semantics.  A consumer thread polls, orders its later accesses after the
// observed value with an acquire fence, and its own later TMA reads after
// that with fence_proxy_async_global.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Orders this thread's generic-proxy global accesses with its async-proxy
// (TMA, bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Waits until the counter equals `target` exactly, for at most timeout_ns of
// global time; false if it gave up.  Polls with relaxed loads; once the value
// is there, one acquire load of it orders the caller's later accesses.
// Equality, not >=: each counter receives exactly its expected number of
// increments per launch, so a value past the target means the counters did
// not start at zero (an uncleared workspace), which then ends in a reported
// timeout instead of a wrong result.
__device__ __forceinline__ bool wait_count_eq(const uint32_t* p, uint32_t target, uint64_t timeout_ns) {
  bool done = ld_relaxed_gpu(p) == target;
  if (!done) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
      if (ld_relaxed_gpu(p) == target) {
        done = true;
        break;
      }
      if ((it & 15u) == 0 && global_timer_ns() - t0 > timeout_ns) break;
    }
  }
  if (done) done = ld_acquire_gpu(p) == target;
  return done;
}

__device__ __forceinline__ float ld_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

// ----------------------------------------------------------------------------- tcgen05
// Allocates `ncols` tensor-memory columns (a power of two >= 32); the whole
// warp executes it and the address lands in shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
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

// Shared-memory matrix descriptor (tcgen05 form): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1 at bit 46, swizzle mode
// at bits 61-63 (0 none, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle_mode) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(swizzle_mode & 7u) << 61);
}

// D[tmem] (+)= A[smem, M=128 x K=64 E2M1] * B[smem, N x 64 E2M1]^T with one
// UE8M0 scale per 32 K elements of every row of A and B, read from tensor memory.
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
      "}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Copies a 32-row x 16-byte block of shared memory to tensor memory, once into
// each of the four 32-lane sub-partitions (lane 32q + i <- row i), 4 columns.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t src_desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc)
               : "memory");
}

// Arrives once on `bar` when every tcgen05 async operation this thread issued
// before it has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Each lane reads 16 consecutive 32-bit columns of its own tensor-memory lane.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ----------------------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// The two halves of cluster_sync_all, for a barrier whose arrival and wait are
// far apart (every thread of the CTA executes each, warp-uniformly).
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// This CTA's coordinates inside its thread-block cluster.
__device__ __forceinline__ uint32_t cluster_ctaid_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctaid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_ctaid_y() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctaid.y;" : "=r"(r));
  return r;
}

// Asynchronous stores into a cluster CTA's shared memory (shared::cluster
// addresses, from map_to_rank) that count their bytes on that CTA's mbarrier
// `cbar` (complete_tx): the receiver waits on its own barrier, armed with the
// number of bytes it expects, and needs no other synchronisation.
__device__ __forceinline__ void st_async_v2(uint32_t caddr, uint32_t a, uint32_t b, uint32_t cbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(caddr),
               "r"(a), "r"(b), "r"(cbar)
               : "memory");
}

__device__ __forceinline__ void st_async_b32(uint32_t caddr, uint32_t a, uint32_t cbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(caddr), "r"(a),
               "r"(cbar)
               : "memory");
}

// Address of the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t caddr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(caddr), "f"(v) : "memory");
}

// Barrier over a subset of the CTA's warps (id 1..15; `threads` a multiple of 32).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t saddr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(saddr)
               : "memory");
  return v;
}

}  // namespace mxfp4
