// common.cuh -- sm_103a building blocks shared by the verification kernels:
// mbarrier + bulk-copy (TMA) pipeline, bounded waits, thread-block-cluster
// barriers and distributed shared memory, warp/block reductions and scans.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Row-status bits: bit c set <=> code c applies (the reported code is the
// lowest set bit).  Values mirror SPEC_ROW_* in include/specverify.h.
enum : uint32_t {
  F_NONFINITE = 1u << 1,
  F_BAD_TOKEN = 1u << 2,
  F_BAD_UNIFORM = 1u << 3,
  F_BAD_PARENT = 1u << 4,
  F_EMPTY = 1u << 5,
  F_TIMEOUT = 1u << 6,
  F_BAD_TEMPERATURE = 1u << 7,
};

__host__ __device__ inline int lowest_code(uint32_t flags) {
  for (int c = 1; c < 32; ++c)
    if (flags & (1u << c)) return c;
  return 0;
}

// ------------------------------------------------------------- bounds checks
// A measurement and test aid: built with -DSV_BOUNDS, the kernels check every
// computed global or shared-memory index (SV_INB: 0 <= i < n; SV_INR: the
// range [i, i + len) inside [0, n)) before the access.  A bad index is
// counted, the first one's source line kept, and the access skipped: nothing
// traps, and the row comes out wrong or flagged instead.  Each translation
// unit keeps its own record (g_sv_oob: {count, first line}); the library's
// spec_debug_bounds reads and clears them all.  In the default build both
// macros are the constant true.
#ifdef SV_BOUNDS
static __device__ unsigned int g_sv_oob[2];
__device__ __forceinline__ bool sv_in_bounds(long long i, long long len, long long n, int line) {
  if (i >= 0 && len >= 0 && i + len <= n) return true;
  if (atomicAdd(&g_sv_oob[0], 1u) == 0u) g_sv_oob[1] = static_cast<unsigned>(line);
  return false;
}
#define SV_INB(i, n) ::sv::sv_in_bounds(static_cast<long long>(i), 1LL, static_cast<long long>(n), __LINE__)
#define SV_INR(i, len, n)                                                                     \
  ::sv::sv_in_bounds(static_cast<long long>(i), static_cast<long long>(len), static_cast<long long>(n), \
                     __LINE__)
// host side: this unit's record, then cleared
#define SV_OOB_READER(fn)                                                       \
  cudaError_t fn(unsigned *count, unsigned *line) {                             \
    unsigned h[2] = {0u, 0u};                                                   \
    cudaError_t e = cudaMemcpyFromSymbol(h, g_sv_oob, sizeof(h));               \
    if (e != cudaSuccess) return e;                                             \
    *count += h[0];                                                             \
    if (!*line) *line = h[1];                                                   \
    const unsigned z[2] = {0u, 0u};                                             \
    return cudaMemcpyToSymbol(g_sv_oob, z, sizeof(z));                          \
  }
#else
#define SV_INB(i, n) true
#define SV_INR(i, len, n) true
#endif

// ------------------------------------------------------------ shared memory
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes mbarrier initialisation visible to the async (bulk copy) proxy and to
// the other CTAs of the cluster.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One bounded probe of phase `parity`: the thread may sleep (not spin) until
// the phase completes or about `sleep_ns` passes.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity,
                                              uint32_t sleep_ns = 20000) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(sleep_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch.  grid_dependency_wait returns once every grid
// this one was launched as a programmatic dependent of has completed and its
// memory operations are visible (at once for a plain launch); the kernels it
// waits for are bounded themselves.  allow_dependents lets the grid launched
// after this one as a programmatic dependent be scheduled once every CTA of
// this grid has issued it or exited.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait for phase `parity` of `bar` to complete; give up after limit_ns.
// Returns false on timeout.  Never spins without a bound.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------- bulk copy (TMA)
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Non-multicast bulk copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) from global memory into this CTA's shared memory; completion is
// signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Asynchronous 16-byte copy from global to this CTA's shared memory (both
// addresses 16-byte aligned), through L2 only; cp_async_wait_all waits for
// every copy this thread issued.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Bulk prefetch of `bytes` (multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Full cluster barrier: every thread of every CTA of the cluster arrives;
// release/acquire orders shared-memory writes before it with reads after it,
// including reads of other CTAs' shared memory.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Relaxed 64-bit accesses at GPU scope: single-copy atomic, never served from
// a stale L1 line.
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// ------------------------------------------------------------------ math
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed fp32 pairs (Blackwell f32x2): two IEEE round-to-nearest operations
// per instruction, bit-identical to the scalar ones.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// max that propagates NaN (IEEE maxNum would drop it)
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 16-byte loads
__device__ __forceinline__ uint4 ld_shared_u4(const void *p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// Streaming 16-byte global load of read-once data: not kept in L1, and
// marked in L2 with `policy` (l2_policy_evict_first for data read once).
__device__ __forceinline__ uint4 ld_stream_u4(const void *p, uint64_t policy) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

// ------------------------------------------------------- warp primitives
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  return v;
}
// inclusive prefix sum over the lanes of a warp (Hillis-Steele)
__device__ __forceinline__ float warp_inclusive_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float n = __shfl_up_sync(FULL_MASK, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

}  // namespace sv
