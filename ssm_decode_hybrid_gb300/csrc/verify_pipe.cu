// Speculative verify, the S_0 stream as a persistent, warp-specialised
// TMA + tcgen05 pipeline (sm_103a), for both families.
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- "Algorithm -- speculative
// decoding" and the appendix "GDN: speculative decoding": per item the
// checkpoint meets the window's vectors once, Z = S_0 X, and every output row
// follows from its row of Z and the terms the precompute kernel left in the
// workspace.
//   GDN:     an item is a (sequence, value head): 128 rows (d_v) x 128
//            columns (d_k); X = [k_1 .. k_T, q_1 .. q_T] of its key head; each
//            row follows from the chunked T x T solve whose terms
//            gdn_split.cu's precompute left in the record.
//   Mamba-2: an item is two heads of one group of a sequence: 2 x 64 rows
//            (d) x 128 columns (n); X = [q_1 .. q_T] of the group; row r of
//            head i gives y_s[r] = abar_s Z[r][s] + buf_s[r] (decode_split.cu's
//            records).
//
// One CTA per SM walks the items of the grid.  Each item's 128 x 128 fp32
// block is four 128-row x 32-column chunks.  Roles:
//   warp 0     TMA producer: each chunk lands in a stage of an eight-stage
//              ring (one cp.async.bulk.tensor box of 16 KB, 128-byte
//              swizzle);
//   warps 2-5  convert: thread r (TMEM lane r) reads row r of each landed
//              chunk (eight conflict-free 16-byte loads), frees the stage, and
//              writes hi = tf32(S) and lo = S - hi of the row into one of four
//              A-operand slots in tensor memory (tcgen05.st; the tensor core
//              reads fp32 as tf32 by dropping the low 13 mantissa bits, and
//              hi + lo carries S to about 2^-21); it also stages the item's
//              window vectors (bf16, exact in tf32) into one of two B-operand
//              slots in shared memory;
//   warp 1     MMA issuer: per chunk four tf32 MMAs on hi and four on lo
//              (M = 128 rows, N = 16 vectors, K = 8; A from tensor memory, B
//              from shared memory) into one of four TMEM accumulators; a
//              commit frees the A slot once they have read it;
//   warps 6-21 epilogue, four groups of four warps taking every fourth item,
//              each with its own TMEM accumulator: once an item's accumulator
//              is complete, thread r of its group reads row r (tcgen05.ld) and
//              finishes it (four groups, so that the loads of the rows' inputs
//              of several items are in flight at once).
// So the S_0 loads of later items are always in flight while earlier items
// are converted, multiplied and solved.  Shared memory carries each chunk
// twice (the copy in, one read); the tensor cores read S_0 from tensor memory.
// Every wait is bounded (RSSM_EBIT_TIMEOUT); after one runs out each role
// stops at its next wait, in-flight copies are drained and TMEM is released.
#include <cudaTypedefs.h>

#include <cuda.h>

#include <type_traits>

#include "kernels.cuh"
#include "tc05.cuh"

namespace rssm {

namespace {

constexpr int kPvStages = 8;
constexpr int kPvTSlots = 4;                        // A-operand slots in tensor memory (hi and lo of one chunk)
constexpr int kPvRows = 128;                        // rows of an item: MMA M, TMEM lanes
constexpr int kPvK = 128;                           // columns of S_0 (d_k, n)
constexpr int kPvM2Rows = 64;                       // Mamba-2 head dimension d (two heads per item)
constexpr int kPvChunks = 4;                        // 32-column chunks of a row
constexpr uint32_t kPvChunkBytes = kPvRows * 128;   // 16 KB: one TMA box
constexpr uint32_t kPvStageBytes = kPvChunkBytes;
constexpr int kPvN = 16;                            // GDN: 8 key, 8 query columns; Mamba-2: 8 query columns, 8 zero
constexpr uint32_t kPvXChunkBytes = kPvN * 128;     // 2 KB
constexpr uint32_t kPvXBytes = kPvChunks * kPvXChunkBytes;  // 8 KB per slot
constexpr uint32_t kPvStagesOff = 0;
constexpr uint32_t kPvXOff = kPvStagesOff + kPvStages * kPvStageBytes;
constexpr uint32_t kPvHdrOff = kPvXOff + 2 * kPvXBytes;
constexpr int kPvGroups = 4;                        // epilogue groups of 128 threads
constexpr uint32_t kPvSmem = kPvHdrOff + kPvGroups * kGdnWorkHeader * 4 + 1024;  // + alignment slack
static_assert(kM2VerifyHeader <= kGdnWorkHeader, "record header staging");
constexpr int kPvThreads = 64 + 128 + kPvGroups * 128;
constexpr uint32_t kPvAccCols = kPvGroups * 16;     // one accumulator of 16 columns per group
constexpr uint32_t kPvTSlotCols = 64;               // hi: 32 columns (K = 32 fp32), lo: 32
constexpr uint32_t kPvTmemCols = 512;               // >= kPvAccCols + kPvTSlots * kPvTSlotCols, a power of two
static_assert(kPvAccCols + kPvTSlots * kPvTSlotCols <= kPvTmemCols, "tensor memory budget");
constexpr int kInfoValid = 1 << 16;

// kind::tf32, fp32 accumulator, A and B tf32, both K-major, M = 128, N = 16.
constexpr uint32_t kPvIdesc = (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(kPvN >> 3) << 17) |
                              (static_cast<uint32_t>(kPvRows >> 4) << 24);

// Shared-memory descriptor of a K-major operand in the 128-byte swizzle layout
// (8-row x 128-byte atoms stacked at 1024 B; bits [61,64) = 2).
__device__ __forceinline__ uint64_t pv_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// D (TMEM) += A (TMEM: lane = row, one column per K element) x B (shared memory).
__device__ __forceinline__ void pv_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(kPvIdesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// 16 columns of this warp's 32 TMEM lanes from registers (thread = lane).
__device__ __forceinline__ void pv_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// 2-D tiled bulk tensor copy global -> shared, completion counted in bytes on bar.
__device__ __forceinline__ void pv_tma_load(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void pv_lds4(uint32_t a, float4 &v) {
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
}
__device__ __forceinline__ void pv_sts4(uint32_t a, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}
__device__ __forceinline__ float pv_trunc(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

__device__ __forceinline__ void pv_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Bounded wait that also gives up as soon as another role has given up.
__device__ __forceinline__ bool pv_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

struct PvBars {
  uint64_t full[kPvStages];   // TMA landed (tx bytes)
  uint64_t empty[kPvStages];  // the stage is read (the 128 convert threads)
  uint64_t tfull[kPvTSlots];  // hi and lo of a chunk in tensor memory (the 128 convert threads)
  uint64_t tempty[kPvTSlots]; // MMAs have read the A slot (commit)
  uint64_t xfull[2];          // window vectors written (the 128 convert threads)
  uint64_t xempty[2];         // MMAs of the slot's item done (commit)
  uint64_t afull[kPvGroups];  // accumulator complete (commit)
  uint64_t aempty[kPvGroups]; // accumulator read (the group's 128 threads)
  uint64_t drain;             // every MMA issued has completed (commit)
};

// Items of each family, and where vector v (row v of X) of item `it` comes
// from (nullptr: a zero row).
__device__ __forceinline__ int pv_items(const GdnLaunch &a) { return a.B * a.Hv; }
__device__ __forceinline__ int pv_items(const M2Launch &a) { return a.B * (a.H / 2); }
template <typename TI>
__device__ __forceinline__ const TI *pv_vector(const GdnLaunch &a, int it, int v) {
  const int b = it / a.Hv, kh = (it - b * a.Hv) / (a.Hv / a.Hk), m = v & 7;
  if (m >= a.T) return nullptr;
  return static_cast<const TI *>(v < 8 ? a.k : a.q) + ((static_cast<size_t>(b) * a.T + m) * a.Hk + kh) * kPvK;
}
template <typename TI>
__device__ __forceinline__ const TI *pv_vector(const M2Launch &a, int it, int v) {
  const int hp = a.H / 2, b = it / hp, g = 2 * (it - b * hp) / (a.H / a.G);
  if (v >= a.T) return nullptr;
  return static_cast<const TI *>(a.q) + ((static_cast<size_t>(b) * a.T + v) * a.G + g) * kPvK;
}

template <typename LaunchT, typename TI, typename TU, typename TO>
__global__ void __launch_bounds__(kPvThreads, 1)
    verify_pipe_kernel(const __grid_constant__ CUtensorMap s0map, LaunchT a, int stride, int P) {
  constexpr bool kM2 = std::is_same<LaunchT, M2Launch>::value;
  extern __shared__ unsigned char pv_raw[];
  __shared__ PvBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = (smem_addr(pv_raw) + 1023u) & ~1023u;
  const int T = a.T, L = a.L;
  const int items = pv_items(a);
  volatile int *abort = &s_abort;

  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < kPvStages; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 128);
    }
    for (int t = 0; t < kPvTSlots; ++t) {
      mbar_init(&bars.tfull[t], 128);
      mbar_init(&bars.tempty[t], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.xfull[x], 128);
      mbar_init(&bars.xempty[x], 1);
    }
    for (int g = 0; g < kPvGroups; ++g) {
      mbar_init(&bars.afull[g], 1);
      mbar_init(&bars.aempty[g], 128);
    }
    mbar_init(&bars.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc05::alloc(&s_tmem, kPvTmemCols);
    tc05::relinquish();
  }
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ---- TMA producer -------------------------------------------------------
    if (lane == 0) {
      int q = 0;
      for (int it = blockIdx.x; it < items && !*abort; it += gridDim.x) {
        for (int c = 0; c < kPvChunks; ++c, ++q) {
          const int s = q % kPvStages;
          if (!pv_wait(&bars.empty[s], ((q / kPvStages) & 1) ^ 1, abort)) break;
          mbar_arrive_expect_tx(&bars.full[s], kPvChunkBytes);
          pv_tma_load(base + kPvStagesOff + s * kPvStageBytes, &s0map, c * 32, it * kPvRows, &bars.full[s]);
        }
      }
      // drain: the last copy issued to each stage must land before the CTA ends
      for (int k = 1; k <= kPvStages && q - k >= 0; ++k) {
        const int qq = q - k;
        mbar_wait(&bars.full[qq % kPvStages], (qq / kPvStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer -----------------------------------------------------------
    if (lane == 0) {
      int q = 0, k = 0;
      for (int it = blockIdx.x; it < items && !*abort; it += gridDim.x, ++k) {
        const int sl = k & 1, ag = k % kPvGroups;
        if (!pv_wait(&bars.aempty[ag], ((k / kPvGroups) & 1) ^ 1, abort)) break;
        if (!pv_wait(&bars.xfull[sl], (k >> 1) & 1, abort)) break;
        tc05::fence_after_sync();
        const uint32_t d = tmem + static_cast<uint32_t>(ag * kPvN);
        const uint32_t xb = base + kPvXOff + sl * kPvXBytes;
        bool ok = true;
        for (int c = 0; c < kPvChunks; ++c, ++q) {
          const int t = q % kPvTSlots;
          if (!pv_wait(&bars.tfull[t], (q / kPvTSlots) & 1, abort)) {
            ok = false;
            break;
          }
          tc05::fence_after_sync();
          const uint32_t hi = tmem + kPvAccCols + static_cast<uint32_t>(t) * kPvTSlotCols, lo = hi + 32;
#pragma unroll
          for (int s2 = 0; s2 < 4; ++s2)
            pv_mma_ts(d, hi + 8 * s2, pv_desc(xb + c * kPvXChunkBytes + s2 * 32), c > 0 || s2 > 0);
#pragma unroll
          for (int s2 = 0; s2 < 4; ++s2) pv_mma_ts(d, lo + 8 * s2, pv_desc(xb + c * kPvXChunkBytes + s2 * 32), true);
          tc05::commit(&bars.tempty[t]);
        }
        if (!ok) break;
        tc05::commit(&bars.afull[ag]);
        tc05::commit(&bars.xempty[sl]);
      }
      // every MMA issued must be complete before TMEM is released
      tc05::commit(&bars.drain);
      mbar_wait(&bars.drain, 0);
    }
  } else if (warp < 6) {
    // ---- convert: hi and lo of each landed chunk into tensor memory, and the
    // window vectors.  The next item's vectors are loaded into registers
    // while the current item's chunks are converted, so that this role never
    // waits on global memory.
    const int ct = tid - 64;                       // 0..127
    const int r = 32 * (warp & 3) + lane;          // the TMEM lane (row) this thread writes
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    constexpr int kXUnits = kPvN * (kPvK / 4) / 128;  // 16-byte units of the vectors per thread
    uint2 xr[kXUnits];
    auto load_x = [&](int it) {
#pragma unroll
      for (int j = 0; j < kXUnits; ++j) {
        const int idx = ct + 128 * j, v = idx / (kPvK / 4), u = idx % (kPvK / 4);
        const TI *src = pv_vector<TI>(a, it, v);
        xr[j] = src != nullptr ? *reinterpret_cast<const uint2 *>(src + 4 * u) : make_uint2(0u, 0u);
      }
    };
    static_assert(sizeof(TI) == 2, "bf16 window vectors");
    if (blockIdx.x < items) load_x(blockIdx.x);
    int q = 0, k = 0;
    for (int it = blockIdx.x; it < items && !*abort; it += gridDim.x, ++k) {
      const int sl = k & 1;
      if (!pv_wait(&bars.xempty[sl], ((k >> 1) & 1) ^ 1, abort)) break;
      // vector v (pv_vector); 16-byte unit u of chunk u / 8 at atom v / 8,
      // row v % 8, unit (u % 8) ^ (v % 8); bf16 to fp32 is exact
      const uint32_t xb = base + kPvXOff + sl * kPvXBytes;
#pragma unroll
      for (int j = 0; j < kXUnits; ++j) {
        const int idx = ct + 128 * j, v = idx / (kPvK / 4), u = idx % (kPvK / 4);
        const int cc = u >> 3, lu = u & 7;
        const float4 x = make_float4(__uint_as_float(xr[j].x << 16), __uint_as_float(xr[j].x & 0xffff0000u),
                                     __uint_as_float(xr[j].y << 16), __uint_as_float(xr[j].y & 0xffff0000u));
        pv_sts4(xb + cc * kPvXChunkBytes + (v >> 3) * 1024 + (v & 7) * 128 + ((lu ^ (v & 7)) << 4), x);
      }
      tc05::fence_proxy_async_smem();
      mbar_arrive(&bars.xfull[sl]);
      if (it + static_cast<int>(gridDim.x) < items) load_x(it + gridDim.x);  // in flight during the conversions
      bool ok = true;
      for (int c = 0; c < kPvChunks; ++c, ++q) {
        const int s = q % kPvStages, t = q % kPvTSlots;
        if (!pv_wait(&bars.full[s], (q / kPvStages) & 1, abort) ||
            !pv_wait(&bars.tempty[t], ((q / kPvTSlots) & 1) ^ 1, abort)) {
          ok = false;
          break;
        }
        // row r of the chunk: 16-byte unit u at r * 128 + ((u ^ (r % 8)) << 4) in the swizzled box
        const uint32_t row = base + kPvStagesOff + s * kPvStageBytes + r * 128;
        const uint32_t ta = tmem + lane_base + kPvAccCols + static_cast<uint32_t>(t) * kPvTSlotCols;
        tc05::fence_after_sync();  // after the wait on tempty: the MMAs that read this slot are complete
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float4 x;
            pv_lds4(row + (((4 * half + u) ^ (r & 7)) << 4), x);
            const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float h = pv_trunc(xs[e]);
              hi[4 * u + e] = __float_as_uint(h);
              lo[4 * u + e] = __float_as_uint(xs[e] - h);
            }
          }
          pv_st16(ta + 16 * half, hi);
          pv_st16(ta + 32 + 16 * half, lo);
        }
        mbar_arrive(&bars.empty[s]);  // the stage is read: the producer may refill it
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc05::fence_before_sync();
        mbar_arrive(&bars.tfull[t]);
      }
      if (!ok) break;
    }
  } else {
    // ---- epilogue: group g finishes items k = g, g + 4, ...; thread r row r ----
    const int g = (warp - 6) / 4;     // group
    const int ew = warp % 4;          // this warp reads TMEM lanes 32 ew .. 32 ew + 31
    const int r = 32 * ew + lane;     // TMEM lane, row of the item
    pdl_wait();  // the precompute grid has finished: workspace, drafts' entries, pointers
    // the group's 128 threads take every decision to stop together (named
    // barriers with an OR), since a named barrier has no time limit
    int k = g;
    for (int it = blockIdx.x + g * gridDim.x; it < items; it += kPvGroups * gridDim.x, k += kPvGroups) {
      if constexpr (kM2) {
        const int hp = a.H / 2, b = it / hp, i = 2 * (it - b * hp) + (r >> 6), row = r & (kPvM2Rows - 1);
        const float *wk = a.work + (static_cast<size_t>(b) * a.H + i) * stride;
        if (named_bar_or(1 + 2 * g, 128, *abort != 0)) break;
        // this row's terms: abar_s, buf_s[row] and the record's info, loaded
        // while the MMAs run
        float ab[kMaxT], buf[kMaxT];
#pragma unroll
        for (int s2 = 0; s2 < kMaxT; ++s2) {
          ab[s2] = buf[s2] = 0.f;
          if (s2 < T) {
            ab[s2] = wk[s2];
            buf[s2] = wk[kM2VerifyHeader + s2 * kPvM2Rows + row];
          }
        }
        const int info = reinterpret_cast<const int *>(wk)[kMaxT];
        const bool failed = !pv_wait(&bars.afull[g], (k / kPvGroups) & 1, abort);
        if (named_bar_or(2 + 2 * g, 128, failed)) break;  // the accumulator is complete
        tc05::fence_after_sync();
        float z[16];
        pv_ld16(tmem + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(g * kPvN), z);
        tc05::fence_before_sync();
        mbar_arrive(&bars.aempty[g]);
        if (info & kInfoValid) {
          TO *y = static_cast<TO *>(a.y);
#pragma unroll
          for (int s2 = 0; s2 < kMaxT; ++s2)
            if (s2 < T)
              store1(y + ((static_cast<size_t>(b) * T + s2) * a.H + i) * kPvM2Rows + row, fmaf(ab[s2], z[s2], buf[s2]));
        }
        // the flag, once every group's precompute block of the sequence finished
        if (i == 0 && ew == 0) {
          const float *first = a.work + static_cast<size_t>(b) * a.H * stride;
          if ((info & kInfoValid) && sequence_records_valid(first, a.G, a.H / a.G, stride, kMaxT, kInfoValid) &&
              lane == 0)
            a.flag[b] = ((info & 0xff) + 2 * T > L) ? 1 : 0;  // early flush, one window ahead
        }
      } else {
        const int b = it / a.Hv, i = it - b * a.Hv;
        const size_t bh = static_cast<size_t>(b) * a.Hv + i;
        const float *wk = a.work + bh * stride;
        float *shdr = reinterpret_cast<float *>(pv_raw + (base - smem_addr(pv_raw)) + kPvHdrOff) + g * kGdnWorkHeader;
        if (named_bar_or(1 + 2 * g, 128, *abort != 0)) break;  // the previous item's header is no longer read
        for (int c = r; c < kGdnWorkHeader; c += 128) shdr[c] = wk[c];
        float pk[kMaxT], pq[kMaxT], pv[kMaxT];
#pragma unroll
        for (int m = 0; m < kMaxT; ++m) {
          pk[m] = pq[m] = pv[m] = 0.f;
          if (m < T) {
            pk[m] = wk[kGwBuf + m * kPvRows + r];
            pq[m] = wk[kGwBuf + (P + m) * kPvRows + r];  // the record holds P key vectors, then the queries
            pv[m] = load1(static_cast<const TI *>(a.v) + ((static_cast<size_t>(b) * T + m) * a.Hv + i) * kPvRows + r);
          }
        }
        const bool failed = !pv_wait(&bars.afull[g], (k / kPvGroups) & 1, abort);
        if (named_bar_or(2 + 2 * g, 128, failed)) break;  // the header is in place; the accumulator is complete
        tc05::fence_after_sync();
        float z[16];
        pv_ld16(tmem + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(g * kPvN), z);
        tc05::fence_before_sync();
        mbar_arrive(&bars.aempty[g]);
        const int info = __float_as_int(shdr[kGwInfo]);
        if ((info & kInfoValid) && rssm_check(((info >> 8) & 0xff) < L && (info & 0xff) + T <= L, a.err)) {
          const int h = info & 0xff, st = (info >> 8) & 0xff;
          const float abar = shdr[kGwAbar];
          TO *y = static_cast<TO *>(a.y);
          TU *ru = static_cast<TU *>(a.ring_u) + bh * L * kPvRows;
          float u[kMaxT];
#pragma unroll
          for (int m = 0; m < kMaxT; ++m) {
            u[m] = 0.f;
            if (m < T) {
              const size_t tvm = (static_cast<size_t>(b) * T + m) * a.Hv + i;
              const float Shk = fmaf(abar, z[m], pk[m]);
              const float Shq = fmaf(abar, z[8 + m], pq[m]);
              const float eG = shdr[kGwEG + m];
              float um = shdr[kGwBeta + m] * (pv[m] - eG * Shk);
#pragma unroll
              for (int mp = 0; mp < m; ++mp) um = fmaf(-shdr[kGwA + m * kMaxT + mp], u[mp], um);
              u[m] = um;
              float ym = eG * Shq;
#pragma unroll
              for (int mp = 0; mp <= m; ++mp) ym = fmaf(shdr[kGwY + m * kMaxT + mp], u[mp], ym);
              store1(y + tvm * kPvRows + r, ym);
              store1(ru + static_cast<size_t>(checked_slot((st + h + m) % L, L, a.err)) * kPvRows + r, um);
            }
          }
          // the flag, once every group's precompute block of the sequence finished
          if (i == 0 && ew == 0 &&
              sequence_records_valid(a.work + static_cast<size_t>(b) * a.Hv * stride, a.Hk, a.Hv / a.Hk, stride,
                                     kGwInfo, kInfoValid) &&
              lane == 0)
            a.flag[b] = (h + 2 * T > L) ? 1 : 0;  // early flush, one window ahead
        }
      }
    }
  }
  if (tid == 0 && *abort) set_err(a.err, RSSM_EBIT_TIMEOUT);
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc05::dealloc(tmem, kPvTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// S_0 as a 2-D fp32 tensor: 128 columns, `rows` rows; boxes of 128 rows x 32
// columns (128 bytes) in the 128-byte swizzle.
bool pv_map(CUtensorMap *map, float *S, long long rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kPvK), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kPvK) * 4};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kPvRows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, S, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <typename LaunchT, typename TU, typename TO>
cudaError_t launch_pv(const LaunchT &a, const CUtensorMap &map, int items, int stride, int P, cudaStream_t stream) {
  auto kern = verify_pipe_kernel<LaunchT, bf16, TU, TO>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kPvSmem))) !=
      cudaSuccess)
    return e;
  const int grid = items < sm_count() ? items : sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kPvThreads);
  cfg.dynamicSmemBytes = kPvSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, map, a, stride, P);
}

}  // namespace

bool gdn_verify_pipe_eligible(const GdnLaunch &a) {
  return a.dk == kPvK && a.dv == kPvRows && a.in_dtype == RSSM_BF16 && a.T >= 2 && a.T <= kMaxT &&
         static_cast<long long>(a.B) * a.Hv * kPvRows < (1ll << 31) && (reinterpret_cast<uintptr_t>(a.S) & 15u) == 0 &&
         encode_fn() != nullptr;
}

cudaError_t launch_gdn_verify_pipe(const GdnLaunch &a, int stride, int P, cudaStream_t stream) {
  CUtensorMap map;
  if (!pv_map(&map, a.S, static_cast<long long>(a.B) * a.Hv * kPvRows)) return cudaErrorInvalidValue;
  const int items = a.B * a.Hv;
  const bool ub = a.u_dtype == RSSM_BF16, yb = a.y_dtype == RSSM_BF16;
  if (ub && yb) return launch_pv<GdnLaunch, bf16, bf16>(a, map, items, stride, P, stream);
  if (ub) return launch_pv<GdnLaunch, bf16, float>(a, map, items, stride, P, stream);
  if (yb) return launch_pv<GdnLaunch, float, bf16>(a, map, items, stride, P, stream);
  return launch_pv<GdnLaunch, float, float>(a, map, items, stride, P, stream);
}

bool m2_verify_pipe_eligible(const M2Launch &a) {
  // two heads of one group per item; up to four queries the CUDA-core stream
  // is faster (it reads S_0 at a higher fraction of the bandwidth)
  return a.n == kPvK && a.d == kPvM2Rows && a.in_dtype == RSSM_BF16 && a.H % 2 == 0 && (a.H / a.G) % 2 == 0 &&
         a.T >= 5 && a.T <= kMaxT && static_cast<long long>(a.B) * a.H * kPvM2Rows < (1ll << 31) &&
         (reinterpret_cast<uintptr_t>(a.S) & 15u) == 0 && encode_fn() != nullptr;
}

cudaError_t launch_m2_verify_pipe(const M2Launch &a, int stride, cudaStream_t stream) {
  CUtensorMap map;
  if (!pv_map(&map, a.S, static_cast<long long>(a.B) * a.H * kPvM2Rows)) return cudaErrorInvalidValue;
  const int items = a.B * (a.H / 2);
  if (a.y_dtype == RSSM_BF16) return launch_pv<M2Launch, float, bf16>(a, map, items, stride, 0, stream);
  return launch_pv<M2Launch, float, float>(a, map, items, stride, 0, stream);
}

}  // namespace rssm
