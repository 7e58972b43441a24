// Device helpers shared by the libreplayssm kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "replayssm.h"

namespace rssm {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kThreads = 256;  // threads per CTA of the per-head kernels
constexpr int kWarps = kThreads / 32;
constexpr int kMaxL = 32;  // ring capacity limit (one warp lane per entry)
constexpr int kMaxT = 8;   // verify window limit

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------------------
// typed loads/stores: 4 consecutive elements as a float4, scalars as float
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

__device__ __forceinline__ float4 load4(const bf16 *p) {
  // bf16 -> f32 is exact: the bf16 bits are the high half of the f32 bits.
  const uint2 u = *reinterpret_cast<const uint2 *>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

__device__ __forceinline__ float load1(const float *p) { return *p; }
__device__ __forceinline__ float load1(const bf16 *p) {
  return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(p)) << 16);
}

__device__ __forceinline__ float2 load2(const float *p) { return *reinterpret_cast<const float2 *>(p); }
__device__ __forceinline__ float2 load2(const bf16 *p) {
  const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

__device__ __forceinline__ void store1(float *p, float v) { *p = v; }
__device__ __forceinline__ void store1(bf16 *p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

// Copy one element without changing its representation.
template <typename T>
__device__ __forceinline__ void copy1(T *dst, const T *src) {
  *dst = *src;
}

// Streaming 16-byte load of checkpoint/state data that is read once per launch.
__device__ __forceinline__ float4 ldg_stream4(const float *p) {
  return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void stg_stream4(float *p, float4 v) { __stcs(reinterpret_cast<float4 *>(p), v); }

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// Sum over an aligned group of LG lanes (LG a power of two <= 32). Every lane
// of the warp must execute the call.
template <int LG>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = LG / 2; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Sum of V values over an aligned group of LG lanes with V-1 + log2(LG/V)
// shuffles instead of V*log2(LG) (recursive halving).  V and LG are powers of
// two with V <= LG.  On return x[0] of lane l holds the group total of value
// index (l % LG) / (LG / V).
template <int LG, int V>
__device__ __forceinline__ void group_sum_multi(float (&x)[V], int lane) {
  static_assert(V <= LG, "V must not exceed the group size");
  int cnt = V;
#pragma unroll
  for (int off = LG / 2; off >= LG / V && off > 0; off >>= 1) {
    const bool upper = (lane & off) != 0;
    const int half = cnt / 2;
#pragma unroll
    for (int m = 0; m < V / 2; ++m) {
      if (m < half) {
        const float send = upper ? x[m] : x[m + half];
        const float keep = upper ? x[m + half] : x[m];
        x[m] = keep + __shfl_xor_sync(kFull, send, off);
      }
    }
    cnt = half;
  }
#pragma unroll
  for (int off = LG / (2 * V); off > 0; off >>= 1) x[0] += __shfl_xor_sync(kFull, x[0], off);
}

__device__ __forceinline__ void set_err(int32_t *err, int bit) {
  if (err) atomicOr(err, bit);
}

// Bounds-checked build (compiled with -DRSSM_CHECKED; a stand-in for a memory
// sanitizer, which this library's tests cannot run): every ring slot a kernel
// writes and every pointer value it decodes from a workspace record is checked
// against its extent.  A failed check ORs RSSM_EBIT_BOUNDS into the error
// word; an item-level check (rssm_check) then skips the item, a slot check
// (checked_slot) redirects the access to slot 0 of the same ring so that no
// access leaves the caller's arrays.  Neither traps.  In the ordinary build
// both compile to nothing.
#ifdef RSSM_CHECKED
__device__ __forceinline__ bool rssm_check(bool ok, int32_t *err) {
  if (!ok) set_err(err, RSSM_EBIT_BOUNDS);
  return ok;
}
__device__ __forceinline__ int checked_slot(int s, int L, int32_t *err) {
  if (static_cast<unsigned>(s) >= static_cast<unsigned>(L)) {
    set_err(err, RSSM_EBIT_BOUNDS);
    return 0;
  }
  return s;
}
#else
__device__ __forceinline__ bool rssm_check(bool, int32_t *) { return true; }
__device__ __forceinline__ int checked_slot(int s, int, int32_t *) { return s; }
#endif

// Arrival counter of a sequence's thread blocks.  Every block of sequence b
// calls this once, after it has read start/count/flag of b; it returns true
// in exactly one block, the last to arrive, which may then rewrite the
// pointers (no other block of this launch reads them afterwards).  The
// counter is left at zero.
__device__ __forceinline__ bool last_arrival(int32_t *sync, int b, int blocks_per_seq) {
  __threadfence();
  const int old = atomicAdd(sync + b, 1);
  if (old == blocks_per_seq - 1) {
    __threadfence();
    sync[b] = 0;
    return true;
  }
  return false;
}

// Suffix sums of per-entry log decays over the first p entries, one entry per
// lane of a warp (p <= 32).  For lane j < p returns the exclusive suffix
// sum_{m > j, m < p} la_m; `total` receives sum_{m < p} la_m.  Lanes >= p must
// pass la = 0.
__device__ __forceinline__ float excl_suffix_sum(float la, int lane, float &total) {
  float incl = la;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_down_sync(kFull, incl, o);
    if (lane + o < 32) incl += t;
  }
  total = __shfl_sync(kFull, incl, 0);
  float ex = __shfl_down_sync(kFull, incl, 1);
  if (lane == 31) ex = 0.f;
  return ex;
}

}  // namespace rssm

// ---------------------------------------------------------------------------
// mbarrier / bulk-copy (TMA) helpers, inline PTX for sm_90+ / sm_100+
// ---------------------------------------------------------------------------
namespace rssm {

// Time limit of every wait inside a kernel (mbarrier phases, the fold-unit
// lock): about one second of GPU global time.  A wait that runs out sets
// RSSM_EBIT_TIMEOUT in the error word and the kernel winds down instead of
// hanging the GPU.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Warp-level 16x8x16 bf16 product with fp32 accumulation, for the small dot
// tables of the precompute kernels (a few MMAs per block, where the CUDA-core
// form spends its time in shuffles).  Fragments: row g = lane / 4 and column
// pair 2 (lane % 4) of each 8x8 quarter, as ldmatrix delivers them.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void mma_16816_bf16(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// Raise the transaction count of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of the given parity; false if the time limit
// ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

// Bounded wait with a limit chosen at launch.  A limit of 0 counts the wait
// as run out without polling: the host sets it only to exercise the recovery
// path of the caller (which must still drain its copies with mbar_wait).
__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}

// Bulk (non-tensor) asynchronous copy global -> shared; completion is counted
// in bytes on `bar`.  dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Volatile shared/global int access (a flag other threads poll).
__device__ __forceinline__ int ld_volatile(const int *p) { return *reinterpret_cast<const volatile int *>(p); }
__device__ __forceinline__ void st_volatile(int *p, int v) { *reinterpret_cast<volatile int *>(p) = v; }

// Barrier over a subset of warps (ids 1..15; id 0 is __syncthreads).
__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads, so
// that a decision (e.g. a wait that ran out) is the same in all of them.
__device__ __forceinline__ bool named_bar_or(int id, int threads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %3, 0;\n\t"
      "bar.red.or.pred q, %1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(out)
      : "r"(id), "r"(threads), "r"(pred ? 1u : 0u)
      : "memory");
  return out != 0;
}

// Whether the precompute kernel left a valid record for every group of one
// sequence.  The records of the sequence's heads are `stride` floats apart
// from `first`; a group's precompute block writes the records of its `hpg`
// heads, so the first head of each group speaks for the block; its int info
// word sits at float `info_off` and carries `valid_bit` when the block
// finished.  A block that gave up (a wait that ran out, pointers out of range)
// clears it, and every streaming block of that sequence then skips the
// sequence.  group_records_load issues this lane's loads (call it early: the
// answer is needed only before the first write), group_records_valid combines
// them over the warp (call with the whole warp; the same answer in every lane).
__device__ __forceinline__ bool group_records_load(const float *first, int groups, int hpg, int stride, int info_off,
                                                   int valid_bit) {
  const int lane = threadIdx.x & 31;
  int all = valid_bit;
  for (int g = lane; g < groups; g += 32)
    all &= reinterpret_cast<const int *>(first + static_cast<size_t>(g) * hpg * stride)[info_off];
  return all != 0;
}
__device__ __forceinline__ bool group_records_valid(bool lane_ok) { return __all_sync(kFull, lane_ok); }
// Both at once, for a block about to change the sequence's state.  Not
// inlined, and called where little else is live: the streaming kernels sit at
// their register caps, and inlined its loads made them spill.
static __device__ __noinline__ bool sequence_records_valid(const float *first, int groups, int hpg, int stride,
                                                       int info_off, int valid_bit) {
  return group_records_valid(group_records_load(first, groups, hpg, stride, info_off, valid_bit));
}

}  // namespace rssm

namespace rssm {

// Per-thread 16-byte asynchronous copy global -> shared (L1 bypassed); the
// thread waits for its own copies with cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

}  // namespace rssm

namespace rssm {

// Programmatic dependent launch (sm_90+).  A grid launched with the
// programmatic stream-serialization attribute may start once every block of
// the preceding grid has called pdl_launch_dependents (or exited);
// pdl_wait blocks until that preceding grid has completed and its memory
// writes are visible.  Without the attribute pdl_wait returns at once.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace rssm
