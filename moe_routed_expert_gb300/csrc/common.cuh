// Shared device helpers: status word, bf16 packing, and inline-PTX wrappers for
// mbarrier, TMA (cp.async.bulk.tensor) and tcgen05 (TMEM + 5th-gen tensor cores).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"
#include "moe_gmm.h"

namespace moe {

// ----------------------------------------------------------------- status word
// The first 4 bytes of every workspace; the first error sticks.
__device__ __forceinline__ void set_status(uint32_t* status, uint32_t code) {
  if (status) atomicCAS(status, 0u, code);
}

// Bounds-checking build (MOE_BOUNDS_CHECK=1, the library
// libmoe_gb300_bounds.so): true when 0 <= i < n; otherwise the status word
// takes MOE_ERR_BOUNDS and the caller skips the access it guards.  The
// checks sit where a kernel derives an index from its own arithmetic (a row
// from group offsets and tile numbers, a permuted row from a rank) rather
// than reading one that it validates anyway.  Release build: always true, no
// code.
#ifndef MOE_BOUNDS_CHECK
#define MOE_BOUNDS_CHECK 0
#endif
__device__ __forceinline__ bool in_bounds(int64_t i, int64_t n, uint32_t* status) {
#if MOE_BOUNDS_CHECK
  if (i >= 0 && i < n) return true;
  set_status(status, MOE_ERR_BOUNDS);
  return false;
#else
  (void)i;
  (void)n;
  (void)status;
  return true;
#endif
}

// ----------------------------------------------------------------- bf16 helpers
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Round two floats to bf16 (nearest even) and pack (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// acc[i] += w * (bf16 element i of v), one fused multiply-add each: the
// combine's per-slot step (the standalone kernel and the fused down GMM share
// it, so both give the same bits).
__device__ __forceinline__ void add8(float (&acc)[8], uint4 v, float w) {
  acc[0] = fmaf(w, bf16_lo(v.x), acc[0]);
  acc[1] = fmaf(w, bf16_hi(v.x), acc[1]);
  acc[2] = fmaf(w, bf16_lo(v.y), acc[2]);
  acc[3] = fmaf(w, bf16_hi(v.y), acc[3]);
  acc[4] = fmaf(w, bf16_lo(v.z), acc[4]);
  acc[5] = fmaf(w, bf16_hi(v.z), acc[5]);
  acc[6] = fmaf(w, bf16_lo(v.w), acc[6]);
  acc[7] = fmaf(w, bf16_hi(v.w), acc[7]);
}

// Eight floats rounded to bf16 (nearest even) and packed.
__device__ __forceinline__ uint4 pack8(const float (&a)[8]) {
  uint4 q;
  q.x = pack_bf16x2(a[0], a[1]);
  q.y = pack_bf16x2(a[2], a[3]);
  q.z = pack_bf16x2(a[4], a[5]);
  q.w = pack_bf16x2(a[6], a[7]);
  return q;
}

// sigma(z) = 1 / (1 + e^-z) with the hardware exponential and an approximate
// reciprocal (2 ulp): every use rounds its result to bf16 (8 significant bits).
__device__ __forceinline__ float sigmoid_fast(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// tanh from its exponential form, 1 - 2 / (1 + e^{2z}); exact at the limits
// (e^{2z} overflows to +inf for large z, underflows to 0 for very negative z).
__device__ __forceinline__ float tanh_fast(float z) { return 1.0f - __fdividef(2.0f, 1.0f + __expf(2.0f * z)); }

// The gated activations of "MegaMoE" (激活函数公式) for one element: g, u are
// the bf16-valued gate / up pre-activations (see Act in internal.h).
__device__ __forceinline__ float act_forward(float g, float u, const Act& a) {
  const float uc = fminf(fmaxf(u, -a.c), a.c);
  switch (a.kind) {
    case MOE_ACT_SWIGLUSTEP: return fminf(g * sigmoid_fast(g), a.c) * uc;
    case MOE_ACT_SWIGLUOAI: {
      const float gc = fminf(g, a.c);
      return gc * sigmoid_fast(a.alpha * gc) * (uc + a.beta);
    }
    case MOE_ACT_SITUGLU: {
      const float lu = a.lbeta > 0.0f ? a.lbeta * tanh_fast(u / a.lbeta) : u;
      return a.beta * tanh_fast(g / a.beta) * sigmoid_fast(g) * lu;
    }
    default: {
      const float gc = fminf(g, a.c);
      return gc * sigmoid_fast(gc) * uc;
    }
  }
}

// Its gradient: dG, dU from d = dA (already bf16-valued).  The pages give no
// gradients; these are the formulas' derivatives, every min / clip kink
// passing the gradient (d/dG = 1 where G <= c, d/dU = 1 where -c <= U <= c,
// swiglustep's min(SiLU(G), c) where SiLU(G) <= c).  SiLU'(z) = s (1 + z (1 - s)).
// One definition, shared by the standalone kernel and the dX epilogues.
__device__ __forceinline__ void act_grad(float g, float u, float d, const Act& a, float& dg, float& du) {
  const bool u_in = (u >= -a.c && u <= a.c);
  const float uc = fminf(fmaxf(u, -a.c), a.c);
  switch (a.kind) {
    case MOE_ACT_SWIGLUSTEP: {
      const float s = sigmoid_fast(g);
      const float silu = g * s;
      dg = (silu <= a.c) ? d * uc * s * (1.0f + g * (1.0f - s)) : 0.0f;
      du = u_in ? d * fminf(silu, a.c) : 0.0f;
      return;
    }
    case MOE_ACT_SWIGLUOAI: {
      const float gc = fminf(g, a.c);
      const float s = sigmoid_fast(a.alpha * gc);
      dg = (g <= a.c) ? d * (uc + a.beta) * (s + a.alpha * gc * s * (1.0f - s)) : 0.0f;
      du = u_in ? d * gc * s : 0.0f;
      return;
    }
    case MOE_ACT_SITUGLU: {
      const float t = tanh_fast(g / a.beta);
      const float s = sigmoid_fast(g);
      float lu = u, dlu = 1.0f;
      if (a.lbeta > 0.0f) {
        const float tl = tanh_fast(u / a.lbeta);
        lu = a.lbeta * tl;
        dlu = 1.0f - tl * tl;
      }
      dg = d * lu * ((1.0f - t * t) * s + a.beta * t * s * (1.0f - s));
      du = d * a.beta * t * s * dlu;
      return;
    }
    default: {
      const float gc = fminf(g, a.c);
      const float s = sigmoid_fast(gc);
      dg = (g <= a.c) ? d * uc * s * (1.0f + gc * (1.0f - s)) : 0.0f;
      du = u_in ? d * gc * s : 0.0f;
      return;
    }
  }
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------- programmatic dependent launch
// Every kernel of the library is launched with programmatic stream
// serialisation: it may start while the previous kernel on the stream drains.
// pdl_wait() blocks until that kernel has finished and its writes are visible;
// no kernel reads or writes global memory before it (an L2 prefetch of an
// input, which returns nothing and changes nothing, is the one exception).
// pdl_trigger() lets the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ----------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

// `count` arrivals at once.
__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait for the phase with parity `parity` of barrier `bar`.
// Gives up (returns false) when *abort becomes non-zero or after timeout_ns,
// in which case it raises *abort itself so the other roles stop too.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile uint32_t* abort, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) {
      *abort = 1u;
      return false;
    }
  }
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Shared -> global tile store (bulk async-group completion).  The source
// must be visible to the async proxy (fence_proxy_async_smem by the writers).
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];"
               :: "l"(reinterpret_cast<uint64_t>(tmap)), "r"(src), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The issuing thread's committed stores have read their shared memory source.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Four rows of a 2D tensor whose map has a one-row box (64 bf16 columns), rows
// r0..r3 at column c0, written to consecutive 128-byte rows at dst (with the
// map's swizzle, which follows the shared-memory address like a tile copy's).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0, int32_t r0,
                                            int32_t r1, int32_t r2, int32_t r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}

// An L2 policy under which lines are the first to be evicted (for data read
// once, such as streamed weights, so it does not push out data read again).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// An L2 policy under which lines are the last to be evicted (data read again
// soon, while streamed data passes through L2).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0,
                                                 int32_t c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

// 16-byte global store under an L2 cache policy.
__device__ __forceinline__ void st_v4_hint(void* p, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy) : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void* tmap, uint32_t bar, int32_t c0,
                                                 int32_t c1, int32_t c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

// 16-byte global -> shared copy that does not block the thread (cp.async),
// cached in L2 only; completion is signalled with cp_async_arrive_noinc.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}
// The same under an L2 cache policy (createpolicy).
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "l"(pol)
               : "memory");
}

// Atomic add with release (this thread's earlier writes are visible GPU-wide
// first) and acquire (writes released before the values it read are visible
// to this thread's later reads) semantics, GPU scope; returns the old value.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Add with release semantics at GPU scope (no value returned).
__device__ __forceinline__ void red_add_release_gpu(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Load with acquire semantics at GPU scope.
__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Orders this thread's earlier generic-proxy accesses to global memory (and
// the writes of other threads they made visible) before its later async-proxy
// (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bring the 128-byte line holding p into L2 (no value returned).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

// Bring [p, p + bytes) into L2 through the bulk-copy unit (no value returned).
// p 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// 16-byte load cached in L2 only (data another SM wrote during this kernel).
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
  return r;
}

// Drop a 128-byte line from L2 without writing it back: for scratch that is
// dead once read (its memory then holds undefined values).
__device__ __forceinline__ void discard_l2_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" :: "l"(p) : "memory");
}

// ----------------------------------------------------------------- TMA descriptors edited on the device
// Field edits of a 128-byte tensor map held in shared memory.
__device__ __forceinline__ void tmap_set_address(uint32_t smem_map, uint64_t addr) {
  asm volatile("tensormap.replace.tile.global_address.shared::cta.b1024.b64 [%0], %1;" :: "r"(smem_map), "l"(addr)
               : "memory");
}
__device__ __forceinline__ void tmap_set_rows(uint32_t smem_map, uint32_t rows) {  // extent of dimension 1
  asm volatile("tensormap.replace.tile.global_dim.shared::cta.b1024.b32 [%0], 1, %1;" :: "r"(smem_map), "r"(rows)
               : "memory");
}
// Copy an edited map to global memory for the TMA unit (whole warp), then make
// it visible to this thread's later copies.
__device__ __forceinline__ void tmap_publish(void* gmem_map, uint32_t smem_map) {
  asm volatile("tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.cta.sync.aligned [%0], [%1], 128;"
               :: "l"(gmem_map), "r"(smem_map) : "memory");
}
__device__ __forceinline__ void tmap_acquire(const void* gmem_map) {
  asm volatile("fence.proxy.tensormap::generic.acquire.cta [%0], 128;" :: "l"(gmem_map) : "memory");
}

// ----------------------------------------------------------------- clusters (CTA pairs)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// arrive on an mbarrier given by its shared::cluster address (this CTA or a peer)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(caddr) : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, uint32_t bar_caddr, int32_t c0,
                                                 int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_caddr), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* tmap, uint32_t bar_caddr, int32_t c0,
                                                 int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_caddr), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane (base+i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// CTA-pair forms: allocation, MMA and commit for cta_group::2.  Both CTAs of
// the pair allocate and free together; one thread of the even CTA issues the MMA.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive once on the mbarrier at offset `bar` in every CTA of `mask` when the
// tcgen05 ops issued so far by this thread complete.
__device__ __forceinline__ void tc_commit_pair_multicast(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               :: "r"(bar), "h"(mask) : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format, version 1), 128-byte swizzle.
//   lbo / sbo in bytes: for K-major operands sbo = stride between 8-row groups
//   (lbo unused); for MN-major operands lbo = stride between 64-element MN
//   chunks and sbo = stride between 8-row K groups.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for tcgen05
  d |= 2ull << 61;  // SWIZZLE_128B
  return d;
}

// Shared-memory matrix descriptor without swizzle (tcgen05 format, version 1):
// 8-row x 16-byte core matrices, `sbo` bytes between 8-row groups and `lbo`
// between 16-byte column groups.
__device__ __forceinline__ uint64_t smem_desc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version for tcgen05; layout bits 61-63 = 0: no swizzle
  return d;
}

// Shared memory (32 rows x 16 bytes, described by `sdesc`) -> TMEM lanes 0-31,
// four 32-bit columns from `taddr`, replicated into all four lane quarters.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(sdesc) : "memory");
}

// D[tmem] (+)= (A * scale_A) (B * scale_B), fp8 / fp6 / fp4 operands with one
// E8M0 scale per 32 elements of K (kind::mxf8f6f4, scale_vec::1X); the scales
// are read from TMEM at sfa / sfb, the byte chosen by the descriptor's ids.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor, kind::mxf8f6f4 with block scaling: A / B element
// formats (0 E4M3, 1 E5M2), K-major A and B, fp32 D, E8M0 scales; the scale
// byte ids (bits 4-5 for B, 29-30 for A) are or-ed in per K step.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int a_fmt, int b_fmt) {
  return (static_cast<uint32_t>(a_fmt) << 7)        // A format
         | (static_cast<uint32_t>(b_fmt) << 10)     // B format
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (1u << 23)                               // scale format: E8M0
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}
__host__ __device__ constexpr uint32_t idesc_sf_ids(uint32_t a_id, uint32_t b_id) { return (b_id << 4) | (a_id << 29); }

// 4-byte global -> shared copy that does not block the thread (cp.async);
// src_bytes = 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// One arrival on `bar` (counted in its expected arrivals) once every cp.async
// this thread has issued so far has landed; the thread does not wait.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, dense.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | ((a_mn_major ? 1u : 0u) << 15)            // A major: 0 = K, 1 = MN
         | ((b_mn_major ? 1u : 0u) << 16)            // B major
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

}  // namespace moe
