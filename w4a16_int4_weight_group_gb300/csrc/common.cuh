// Device-side helpers shared by the kernels of libw4a16.so: dtype tags, inline-PTX wrappers for
// byte permutes, packed 16-bit arithmetic with explicit rounding, warp-level MMA, cp.async,
// thread-block-cluster barriers and distributed shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace w4a16 {

// ---------------------------------------------------------------------------------------------
// dtype tags
// ---------------------------------------------------------------------------------------------
struct F16 {
  using T = __half;
  static constexpr bool kBF16 = false;
  __device__ static __forceinline__ float to_float(T x) { return __half2float(x); }
  __device__ static __forceinline__ T from_float_rn(float x) { return __float2half_rn(x); }
};
struct BF16 {
  using T = __nv_bfloat16;
  static constexpr bool kBF16 = true;
  __device__ static __forceinline__ float to_float(T x) { return __bfloat162float(x); }
  __device__ static __forceinline__ T from_float_rn(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ float bits_to_float(uint16_t b, bool is_bf16) {
  return is_bf16 ? __uint_as_float(uint32_t(b) << 16) : __half2float(__ushort_as_half(b));
}

// ---------------------------------------------------------------------------------------------
// integer bit manipulation
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// (a & mask) | bits, one LOP3 (truth table 0xEA for (A & B) | C)
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t bits) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));
  return d;
}

// ---------------------------------------------------------------------------------------------
// packed 16-bit arithmetic, round-to-nearest-even made explicit (no contraction into FMA)
// ---------------------------------------------------------------------------------------------
template <bool BF>
__device__ __forceinline__ uint32_t sub2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (BF) asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
template <bool BF>
__device__ __forceinline__ uint32_t mul2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (BF) asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ---------------------------------------------------------------------------------------------
// warp-level MMA m16n8k16, fp32 accumulate: D = A(16x16, row) * B(16x8, col) + D
// ---------------------------------------------------------------------------------------------
template <bool BF>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  if constexpr (BF) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}
// d = a . b (accumulator starts from zero)
template <bool BF>
__device__ __forceinline__ void mma_16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                            uint32_t b1) {
  const float z = 0.f;
  if constexpr (BF) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
  }
}

// ---------------------------------------------------------------------------------------------
// shared memory addressing, cp.async (16-byte, L2-only caching, optional zero fill)
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Copies 16 bytes global -> shared. When `valid` is false nothing is read and 16 zero bytes are
// written (src-size 0); `src` must still be a valid address.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void lds64(uint32_t addr, uint32_t &x, uint32_t &y) {
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(x), "=r"(y) : "r"(addr));
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t x;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(x) : "r"(addr));
  return x;
}
__device__ __forceinline__ void lds128(uint32_t addr, uint32_t &x, uint32_t &y, uint32_t &z,
                                       uint32_t &w) {
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(x), "=r"(y), "=r"(z), "=r"(w)
               : "r"(addr));
}

// ---------------------------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched with programmatic stream serialization may
// start while the previous kernel of the stream is still running; griddep_wait() blocks until that
// kernel has completed and its memory is visible (call it before the first global access), and
// griddep_launch_dependents() lets the next kernel start launching. Both are no-ops otherwise.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------------------------
// thread-block clusters: hardware barrier and distributed shared memory reads
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Cluster barrier without memory ordering (used only to keep shared memory alive for peers).
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}
// Split phases of the cluster barrier: arrive (no memory ordering) now, wait later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
// Asynchronous 4-byte store into the shared memory of a CTA of the cluster (shared::cluster address),
// completion counted in bytes on that CTA's mbarrier (shared::cluster address).
__device__ __forceinline__ void st_async_f32(uint32_t cluster_addr, float v, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(cluster_addr),
               "r"(__float_as_uint(v)), "r"(cluster_bar)
               : "memory");
}
// Asynchronous 16-byte store (16-byte aligned) into the shared memory of a CTA of the cluster, completion
// counted in bytes on that CTA's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, float a, float b, float c, float d,
                                            uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(cluster_addr),
               "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)), "r"(__float_as_uint(d)),
               "r"(cluster_bar)
               : "memory");
}
// Maps a shared::cta address of this CTA to the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// 16-byte load from another CTA's shared memory (a shared::cluster address, 16-byte aligned).
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t cluster_addr) {
  float4 v;
  asm("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(cluster_addr));
  return v;
}
// Plain (non-volatile) load so that the compiler may issue several remote loads back to back; the
// ordering against the writers comes from the cluster barrier that precedes the reads.
__device__ __forceinline__ float ld_dsmem_f32(uint32_t cluster_addr) {
  float v;
  asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr));
  return v;
}


// ---------------------------------------------------------------------------------------------
// mbarrier, TMA (cp.async.bulk.tensor) and bounded waits
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Returns true once the phase with the given parity has completed (the instruction itself waits
// for a short, hardware-defined time before reporting that it has not).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// A shared-memory flag read and written through the shared window (not a generic pointer).
__device__ __forceinline__ uint32_t ld_flag(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_flag(uint32_t addr, uint32_t v) {
  asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Fetches a TMA descriptor (a __grid_constant__ kernel parameter) ahead of its first use.
__device__ __forceinline__ void prefetch_tensormap(const void *tensor_map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tensor_map)) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// 2-D tiled TMA load into shared memory, completion counted on an mbarrier (bytes).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tensor_map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tensor_map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// Asks the memory system to bring a 2-D tile of a tensor into L2 (no shared-memory destination, no
// completion to wait for): a hint that lets a kernel start HBM reads before it may consume them.
__device__ __forceinline__ void tma_prefetch_l2_2d(const void *tensor_map, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(tensor_map)),
               "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Orders this thread's earlier generic-proxy view of global memory (e.g. after an acquire of data
// other CTAs wrote) before its later async-proxy (bulk copy) reads of it.
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// Bulk copy of `bytes` contiguous bytes (16-byte aligned, a multiple of 16) from global into shared
// memory, completion counted on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Bounded wait on an mbarrier phase. On expiry it sets the CTA's abort flag (a shared-memory word
// at `abort_flag`) and ORs 1 into the kernel's device error word; it also returns false early once
// another thread has set the flag.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, uint32_t abort_flag,
                                           uint64_t limit_ns, unsigned int *error_word) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (ld_flag(abort_flag)) return false;
    if (globaltimer() - t0 > limit_ns) {
      st_flag(abort_flag, 1u);
      atomicOr(error_word, 1u);
      return false;
    }
  }
}
// Wait used after an abort to let this CTA's own copies or MMAs land: ignores the abort flag and
// has its own fixed bound.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity, unsigned int *error_word,
                                            uint64_t limit_ns = 1000000000ull) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) {
      atomicOr(error_word, 2u);
      return;
    }
  }
}

// ---------------------------------------------------------------------------------------------
// ldmatrix: four 8x8 matrices of 16-bit elements; lanes 8i..8i+7 give the row addresses of matrix i.
// Without .trans lane t receives (row t/4, columns 2(t%4), 2(t%4)+1); with .trans it receives
// (rows 2(t%4), 2(t%4)+1 of column t/4).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

}  // namespace w4a16
