// 5th-generation tensor core (tcgen05) helpers for sm_100a/sm_103a, inline PTX.
//
// Only what the flush contraction needs: tensor-memory (TMEM) allocation, a
// single-CTA bf16 x bf16 -> fp32 MMA with both operands in shared memory in
// the no-swizzle K-major layout, the commit to an mbarrier, and 32x32b loads
// of the accumulator back to registers.
#pragma once

#include "common.cuh"

namespace rssm {
namespace tc05 {

// Shared-memory matrix descriptor, no swizzle, K-major.  The operand is a grid
// of 8-row x 16-byte "core matrices" (128 contiguous bytes, row stride 16 B);
// lbo is the byte distance between core matrices adjacent along K, sbo along
// M/N.  Bits: [0,14) start address >> 4, [16,30) lbo >> 4, [32,46) sbo >> 4,
// [46,48) descriptor version (1 on sm_100 and later), [61,64) swizzle mode (0).
__device__ __forceinline__ uint64_t smem_desc(const void *base, uint32_t lbo, uint32_t sbo) {
  const uint64_t addr = smem_addr(base);
  return ((addr >> 4) & 0x3FFFull) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulator,
// both operands K-major, dense.  Bits: [4,6) D format (1 = f32), [7,10) A
// format (1 = bf16), [10,13) B format (1 = bf16), 15/16 A/B major (0 = K),
// [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Byte offset of element (row, k) in a no-swizzle K-major operand of `rows`
// rows and 16 K-elements (bf16) per MMA step, with k-step s stored after the
// previous one: core matrix (row/8, k/8) at (row/8)*256 + (k/8)*128, element
// at (row%8)*16 + (k%8)*2 inside it.  lbo = 128, sbo = 256.
__host__ __device__ constexpr uint32_t kmajor_offset(int rows, int row, int k) {
  return static_cast<uint32_t>((k >> 4) * rows * 32 + (row >> 3) * 256 + ((k & 15) >> 3) * 128 + (row & 7) * 16 +
                               (k & 7) * 2);
}
constexpr uint32_t kLBO = 128, kSBO = 256;

// Allocate `ncols` TMEM columns (a power of two >= 32) for this CTA; one full
// warp executes it; the TMEM address is written to *dst (shared memory).
__device__ __forceinline__ void alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// Arrive on an mbarrier once all previously issued MMAs of this thread finish.
__device__ __forceinline__ void commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Make generic-proxy writes to shared memory visible to the async proxy
// (the tensor core reads its operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Load 32 consecutive fp32 columns of this warp's 32 TMEM lanes (lane i of the
// warp gets TMEM lane 32*(warp%4) + i).  taddr: lane in bits [16,32), column
// in [0,16).
__device__ __forceinline__ void ld_32x32b_x32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Split x into three bf16 terms with hi + mid + lo = x to about 2^-25
// relative (each term carries the next 8 significant bits of the remainder):
// the split-precision operand of a bf16 tensor-core product whose other
// factor is exact in bf16, accurate to fp32 level.
__device__ __forceinline__ void split3_bf16(float x, bf16 &hi, bf16 &mid, bf16 &lo) {
  hi = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(hi);
  mid = __float2bfloat16_rn(r1);
  lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
}

}  // namespace tc05
}  // namespace rssm
