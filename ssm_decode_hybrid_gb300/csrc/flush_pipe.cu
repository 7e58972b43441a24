// Flush as a persistent, warp-specialised TMA + tcgen05 pipeline (sm_103a).
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- "Algorithm: Mamba-2 standard
// decode" (flush: S_0 <- abar S_0 + sum_j s_j v_j k_j^T over the committed
// entries, then clear the buffer) and the GDN appendix (the same history form
// with the cached corrections u_j and the gates g_j).
//
// Items are 64-row halves of the (sequence, head) tiles of flagged sequences
// (a head of d = 64 rows is one item, one of d = 128 two), numbered in
// sequence order over the flagged sequences only and dealt round-robin to the
// persistent CTAs, so that every CTA gets the same share however the flags
// fall.  Roles:
//   warp 0     TMA producer: an item's 64 x 128 fp32 rows land in its group's
//              stage as four 64-row x 32-column boxes in the 128-byte swizzle,
//              issued as soon as the group has released the stage;
//   warps 2-17 four worker groups of four warps, taking every fourth item.
//              While the tile is on its way a group forms the decay weights
//              (one warp scan), builds the two operands of D^T = K (W V)^T in
//              shared memory (keys, exact in bf16, K-major, one copy; each
//              w_j v_j[r] split into three bf16 terms, so the product keeps
//              fp32 accuracy) and issues three MMAs (M = 128 state columns =
//              TMEM lanes, N = 64 rows, K = 16 each, one per term) into its
//              own 64 TMEM columns; it then loads the keys, vectors and decays
//              of its next item, and thread c (state column c) reads
//              D^T[c][0..64) and writes S_0[r][c] = abar S_0[r][c] + D^T[c][r]
//              from the landed tile, a warp writing 128 contiguous bytes of a
//              row.
// A second, one-thread-per-sequence launch resets the pointers of every
// flagged sequence and clears its flag once all items are folded (no
// arrival counting inside the pipeline).  Every wait is bounded (RSSM_EBIT_TIMEOUT); a group decides
// to stop together (named barriers with an OR), the producer drains its last
// copies and the groups their MMAs before TMEM is released.
#include <cudaTypedefs.h>

#include <cuda.h>

#include "kernels.cuh"
#include "tc05.cuh"

namespace rssm {

namespace {

constexpr int kFpGroups = 4;
constexpr int kFpRows = 64;                              // rows of an item: MMA N
constexpr int kFpN = 128;                                // state columns: MMA M, TMEM lanes
constexpr int kFpKE = 16;                                // entries, zero-padded (L <= 16)
constexpr int kFpKT = 3 * kFpKE;                         // split-precision K extent
constexpr uint32_t kFpBoxBytes = kFpRows * 128;          // 64 rows x 32 fp32: 8 KB
constexpr uint32_t kFpTileBytes = 4 * kFpBoxBytes;       // 32 KB
constexpr uint32_t kFpABytes = kFpN * kFpKE * 2;         // keys operand (one copy serves the three MMAs): 4 KB
constexpr uint32_t kFpBBytes = kFpRows * kFpKT * 2;      // weighted-vector operand: 6 KB
constexpr uint32_t kFpTilesOff = 0;
constexpr uint32_t kFpOpsOff = kFpTilesOff + kFpGroups * kFpTileBytes;
constexpr int kFpListMax = 1024;                        // items one CTA may hold (its gids, in order)
constexpr uint32_t kFpListOff = kFpOpsOff + kFpGroups * (kFpABytes + kFpBBytes);
constexpr uint32_t kFpSmem = kFpListOff + 3 * kFpListMax * 4 + 1024;  // + alignment slack: gid, count, start
constexpr int kFpThreads = 64 + kFpGroups * 128;
constexpr uint32_t kFpTmemCols = kFpGroups * kFpRows;  // 256

__device__ __forceinline__ void fp_tma_load(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t bf16_pair(bf16 lo, bf16 hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) | (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

__device__ __forceinline__ float fp_lds(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}

// Bounded wait that also gives up as soon as another role has given up.
__device__ __forceinline__ bool fp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
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

template <typename TV>
__global__ void __launch_bounds__(kFpThreads, 1)
    flush_pipe_kernel(const __grid_constant__ CUtensorMap s0map, FlushLaunch a, int halves) {
  extern __shared__ unsigned char fp_raw[];
  __shared__ uint64_t full[kFpGroups], empty[kFpGroups], mma_bar[kFpGroups];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_w[kFpGroups][kMaxL];
  __shared__ float s_abar[kFpGroups];
  __shared__ int s_wcount[kFpThreads / 32 + 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = (smem_addr(fp_raw) + 1023u) & ~1023u;
  const int H = a.H, L = a.L, HpG = a.H / a.G;
  const int per_seq = H * halves;                    // items of one sequence
  const long total = static_cast<long>(a.B) * per_seq;
  volatile int *abort = &s_abort;

  if (tid == 0) {
    s_abort = 0;
    for (int g = 0; g < kFpGroups; ++g) {
      mbar_init(&full[g], 1);
      mbar_init(&empty[g], 128);
      mbar_init(&mma_bar[g], 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tc05::alloc(&s_tmem, kFpTmemCols);
    tc05::relinquish();
  }
  // launched with programmatic serialisation: the flags, pointers, rings and
  // S_0 are read only once the previous grid has completed; the pointer reset
  // that follows may be scheduled at once (it waits for this grid)
  pdl_wait();
  pdl_launch_dependents();
  // this CTA's items: the flagged sequences' items numbered t = 0, 1, ... in
  // sequence order, and this CTA takes t = blockIdx.x + j gridDim.x, so every
  // CTA gets the same share whichever sequences are flagged.  One pass over the
  // flags (the pointers read with them) writes the gids and pointers of those
  // items into shared memory in order.
  int *items = reinterpret_cast<int *>(fp_raw + (base - smem_addr(fp_raw)) + kFpListOff);
  int *item_cnt = items + kFpListMax, *item_st = item_cnt + kFpListMax;
  int n_items = 0, n_seq = 0;  // items listed so far, flagged sequences seen so far
  const int grid = static_cast<int>(gridDim.x), bid = static_cast<int>(blockIdx.x);
  for (int b0 = 0; b0 < a.B; b0 += kFpThreads) {
    const int b = b0 + tid;
    const bool inb = b < a.B;
    const bool f = inb && a.flag[b] != 0;
    const int cb = inb ? a.count[b] : 0, sb = inb ? a.start[b] : 0;
    const unsigned m = __ballot_sync(kFull, f);
    if (lane == 0) s_wcount[warp] = __popc(m);
    __syncthreads();
    if (tid == 0) {
      int acc = 0;
      for (int w = 0; w < kFpThreads / 32; ++w) {
        const int cw = s_wcount[w];
        s_wcount[w] = acc;
        acc += cw;
      }
      s_wcount[kFpThreads / 32] = acc;
    }
    __syncthreads();
    // sequence number p among the flagged ones; its items t = p per_seq + r
    const long p = n_seq + s_wcount[warp] + __popc(m & ((1u << lane) - 1u));
    const int r0 = f ? static_cast<int>(((bid - p * per_seq) % grid + grid) % grid) : per_seq;
    const int mine = r0 < per_seq ? (per_seq - 1 - r0) / grid + 1 : 0;
    // exclusive prefix of `mine` over the block, in thread (= sequence) order
    int inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += v;
    }
    __syncthreads();  // the flag counts are read
    if (lane == 31) s_wcount[warp] = inc;
    __syncthreads();
    if (tid == 0) {
      int acc = 0;
      for (int w = 0; w < kFpThreads / 32; ++w) {
        const int cw = s_wcount[w];
        s_wcount[w] = acc;
        acc += cw;
      }
      s_wcount[kFpThreads / 32] = acc;
    }
    __syncthreads();
    int pos = n_items + s_wcount[warp] + inc - mine;
    for (int q = 0; q < mine; ++q, ++pos) {
      if (pos < kFpListMax) {
        items[pos] = b * per_seq + r0 + q * grid;
        item_cnt[pos] = cb;
        item_st[pos] = sb;
      }
    }
    n_items += s_wcount[kFpThreads / 32];
    n_seq += __syncthreads_count(f);
  }
  n_items = min(n_items, kFpListMax);  // no effect: flush_pipe_eligible bounds a CTA's share by kFpListMax

  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ---- TMA producer: item k into stage k % 4 --------------------------------
    if (lane == 0) {
      int k = 0;
      for (; k < n_items && !*abort;) {
        const int gid = items[k];
        const int b = gid / per_seq;
        const int s = k % kFpGroups;
        if (!fp_wait(&empty[s], ((k / kFpGroups) & 1) ^ 1, abort)) break;
        const int rest = gid - b * per_seq;
        const int i = rest / halves, hf = rest - i * halves;
        const int row = (b * H + i) * a.d + hf * kFpRows;
        mbar_arrive_expect_tx(&full[s], kFpTileBytes);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          fp_tma_load(base + kFpTilesOff + s * kFpTileBytes + c4 * kFpBoxBytes, &s0map, c4 * 32, row, &full[s]);
        ++k;
      }
      // drain: the last copy issued to each stage must land before the CTA ends
      for (int j = 1; j <= kFpGroups && k - j >= 0; ++j) {
        const int kk = k - j;
        mbar_wait(&full[kk % kFpGroups], (kk / kFpGroups) & 1);
      }
    }
  } else if (warp >= 2) {
    // ---- worker group g: items k = g, g + 4, ... ------------------------------
    const int g = (warp - 2) / 4;
    const int gt = tid - 64 - g * 128;         // 0..127 within the group: the A row (state column) it writes
    const int c = 32 * (warp % 4) + lane;      // state column = TMEM lane this thread reads
    const int gw = gt >> 5;                    // warp within the group
    const int vr = gt & (kFpRows - 1), vh = gt >> 6;  // B operand: row vr, entries 8 vh .. 8 vh + 7
    const uint32_t tile = base + kFpTilesOff + g * kFpTileBytes;
    const uint32_t opA = base + kFpOpsOff + g * (kFpABytes + kFpBBytes), opB = opA + kFpABytes;
    unsigned char *pA = fp_raw + (opA - smem_addr(fp_raw));
    unsigned char *pB = fp_raw + (opB - smem_addr(fp_raw));
    const uint32_t d_tmem = tmem + static_cast<uint32_t>(g * kFpRows);
    const uint32_t idesc = tc05::idesc_bf16_f32(kFpN, kFpRows);
    // an item's loads, issued one item ahead: the keys of state column gt
    // (bf16 pairs), v_e[vr] for this thread's eight entries, and the log decay
    // of entry `lane` (the group's first warp)
    uint32_t kp[kFpKE / 2];
    float vv[8];
    float ld = 0.f;
    auto fetch = [&](int k) {
      const int gid = items[k], cnt = item_cnt[k], st = item_st[k];
      const int b = gid / per_seq, rest = gid - b * per_seq;
      const int i = rest / halves, hf = rest - i * halves;
      const size_t bh = static_cast<size_t>(b) * H + i;
      const size_t bg = static_cast<size_t>(b) * a.G + i / HpG;
      const bool valid = cnt >= 0 && cnt <= L && st >= 0 && st < L;
      ld = 0.f;
#pragma unroll
      for (int e = 0; e < kFpKE / 2; ++e) kp[e] = 0u;
#pragma unroll
      for (int q = 0; q < 8; ++q) vv[q] = 0.f;
      if (!valid) return;
      const unsigned short *key = static_cast<const unsigned short *>(a.ring_key) + bg * L * kFpN + gt;
      int sl = st;
#pragma unroll
      for (int e = 0; e < kFpKE; e += 2) {
        const uint32_t k0 = e < cnt ? key[static_cast<size_t>(sl) * kFpN] : 0u;
        sl = sl + 1 == L ? 0 : sl + 1;
        const uint32_t k1 = e + 1 < cnt ? key[static_cast<size_t>(sl) * kFpN] : 0u;
        sl = sl + 1 == L ? 0 : sl + 1;
        kp[e / 2] = k0 | (k1 << 16);
      }
      const TV *vec = static_cast<const TV *>(a.ring_vec) + bh * L * a.d + hf * kFpRows + vr;
      int sv = (st + 8 * vh) % L;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        vv[q] = 8 * vh + q < cnt ? load1(vec + static_cast<size_t>(sv) * a.d) : 0.f;
        sv = sv + 1 == L ? 0 : sv + 1;
      }
      if (gw == 0 && lane < cnt) ld = a.ring_ld[bh * L + (st + lane) % L];
    };
    int j = 0, mj = 0;  // j: this group's items so far, mj: its MMA commits so far
    if (g < n_items) fetch(g);
    for (int k = g; k < n_items; k += kFpGroups) {
      const int gid = items[k], cnt = item_cnt[k], st = item_st[k];
      const int b = gid / per_seq, rest = gid - b * per_seq;
      const int i = rest / halves, hf = rest - i * halves;
      const size_t bh = static_cast<size_t>(b) * H + i;
      const bool valid = cnt >= 0 && cnt <= L && st >= 0 && st < L;
      if (valid) {
        if (gw == 0) {
          // decay weights over the committed entries, one per lane
          const float la = a.mamba2 ? a.A[i] * ld : ld;
          float tot;
          const float ex = excl_suffix_sum(lane < cnt ? la : 0.f, lane, tot);
          s_w[g][lane] = (lane < cnt) ? (a.mamba2 ? ld : 1.f) * expf(ex) : 0.f;
          if (lane == 0) s_abar[g] = expf(tot);
        }
        // A operand: row gt = the keys' column gt over the 16 entries (two
        // 16-byte units); the three MMAs share it
        *reinterpret_cast<uint4 *>(pA + tc05::kmajor_offset(kFpN, gt, 0)) = make_uint4(kp[0], kp[1], kp[2], kp[3]);
        *reinterpret_cast<uint4 *>(pA + tc05::kmajor_offset(kFpN, gt, 8)) = make_uint4(kp[4], kp[5], kp[6], kp[7]);
      }
      // s_w ready; every thread is past the previous item's TMEM reads
      if (named_bar_or(1 + g, 128, *abort != 0)) break;
      if (valid) {
        // B operand: row vr of the item, K = entries: hi(w_e v_e[r]), then mid, then lo
        uint32_t t0[4], t1[4], t2[4];
#pragma unroll
        for (int q = 0; q < 8; q += 2) {
          bf16 h0, m0, l0, h1, m1, l1;
          tc05::split3_bf16(s_w[g][8 * vh + q] * vv[q], h0, m0, l0);
          tc05::split3_bf16(s_w[g][8 * vh + q + 1] * vv[q + 1], h1, m1, l1);
          t0[q / 2] = bf16_pair(h0, h1);
          t1[q / 2] = bf16_pair(m0, m1);
          t2[q / 2] = bf16_pair(l0, l1);
        }
        *reinterpret_cast<uint4 *>(pB + tc05::kmajor_offset(kFpRows, vr, 8 * vh)) = make_uint4(t0[0], t0[1], t0[2], t0[3]);
        *reinterpret_cast<uint4 *>(pB + tc05::kmajor_offset(kFpRows, vr, kFpKE + 8 * vh)) =
            make_uint4(t1[0], t1[1], t1[2], t1[3]);
        *reinterpret_cast<uint4 *>(pB + tc05::kmajor_offset(kFpRows, vr, 2 * kFpKE + 8 * vh)) =
            make_uint4(t2[0], t2[1], t2[2], t2[3]);
        tc05::fence_proxy_async_smem();
      }
      tc05::fence_before_sync();
      if (named_bar_or(1 + g, 128, false)) break;  // operands in place
      if (valid && gt == 0) {
        tc05::fence_after_sync();
        const uint64_t adesc = tc05::smem_desc(pA, tc05::kLBO, tc05::kSBO);
        for (int s = 0; s < kFpKT / 16; ++s)
          tc05::mma_bf16(d_tmem, adesc, tc05::smem_desc(pB + static_cast<size_t>(s) * kFpRows * 32, tc05::kLBO, tc05::kSBO),
                         idesc, s > 0);
        tc05::commit(&mma_bar[g]);
      }
      // the group's next item: its loads overlap this one's MMA and write-back
      if (k + kFpGroups < n_items) fetch(k + kFpGroups);
      bool failed = valid && !fp_wait(&mma_bar[g], mj & 1, abort);
      if (valid) ++mj;
      failed = failed || !fp_wait(&full[g], j & 1, abort);  // the tile has landed (the stage is this group's)
      const float abar = s_abar[g];  // read before the barrier: the next item's warp 0 may overwrite it after
      if (named_bar_or(1 + g, 128, failed)) break;
      if (valid) {
        tc05::fence_after_sync();
        float *S0 = a.S0 + (bh * a.d + hf * kFpRows) * kFpN + c;
        // column c in the tile: box c / 32, 16-byte unit (c % 32) / 4 swizzled by the row
        const uint32_t col_base = tile + (c >> 5) * kFpBoxBytes + (c & 3) * 4;
        const uint32_t unit = (c & 31) >> 2;
#pragma unroll
        for (int r0 = 0; r0 < kFpRows; r0 += 32) {
          float dv[32];
          tc05::ld_32x32b_x32(d_tmem + (static_cast<uint32_t>(32 * (warp % 4)) << 16) + static_cast<uint32_t>(r0), dv);
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int r = r0 + u;
            const float s = fp_lds(col_base + r * 128 + ((unit ^ (r & 7)) << 4));
            __stcs(S0 + static_cast<size_t>(r) * kFpN, fmaf(abar, s, dv[u]));
          }
        }
      } else if (gt == 0) {
        set_err(a.err, RSSM_EBIT_COUNT_RANGE);
      }
      tc05::fence_before_sync();
      mbar_arrive(&empty[g]);  // the stage may be refilled
      ++j;
    }
    // every MMA this group issued must be complete before TMEM is released
    if (gt == 0 && mj > 0) {
      tc05::commit(&mma_bar[g]);
      mbar_wait(&mma_bar[g], mj & 1);
    }
  }
  if (tid == 0 && *abort) set_err(a.err, RSSM_EBIT_TIMEOUT);
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc05::dealloc(tmem, kFpTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 fp_encode_fn() {
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

// After the fold of every flagged sequence: start <- (start + count) mod L,
// count <- 0, flag <- 0 (a sequence whose pointers were out of range was not
// folded and keeps them; the fold set RSSM_EBIT_COUNT_RANGE).
__global__ void fp_reset_kernel(int B, int L, int32_t *start, int32_t *count, int32_t *flag) {
  pdl_wait();  // every item of the flush is folded
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B || flag[b] == 0) return;
  const int c = count[b], st = start[b];
  if (c >= 0 && c <= L && st >= 0 && st < L) {
    start[b] = (st + c) % L;
    count[b] = 0;
  }
  flag[b] = 0;
}

template <typename TV>
cudaError_t launch_fp(const FlushLaunch &a, cudaStream_t stream) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = fp_encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  // S_0 as a 2-D fp32 tensor: 128 columns, B H d rows; boxes of 64 rows x 32
  // columns (128 bytes) in the 128-byte swizzle
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kFpN), static_cast<cuuint64_t>(a.B) * a.H * a.d};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kFpN) * 4};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kFpRows)};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.S0, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  auto kern = flush_pipe_kernel<TV>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kFpSmem))) !=
      cudaSuccess)
    return e;
  const int halves = a.d / kFpRows;
  const long items = static_cast<long>(a.B) * a.H * halves;
  const int sms = a.num_sms > 0 ? a.num_sms : sm_count();
  const int grid = items < sms ? static_cast<int>(items) : sms;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kFpThreads);
  cfg.dynamicSmemBytes = kFpSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, kern, map, a, halves)) != cudaSuccess) return e;
  cudaLaunchConfig_t rcfg = {};
  rcfg.gridDim = dim3(static_cast<unsigned>((a.B + 255) / 256));
  rcfg.blockDim = dim3(256);
  rcfg.stream = stream;
  rcfg.attrs = attr;
  rcfg.numAttrs = 1;
  return cudaLaunchKernelEx(&rcfg, fp_reset_kernel, a.B, a.L, a.start, a.count, a.flag);
}

}  // namespace

bool flush_pipe_eligible(const FlushLaunch &a) {
  const long long items = static_cast<long long>(a.B) * a.H * (a.d / kFpRows);
  const int sms = a.num_sms > 0 ? a.num_sms : sm_count();
  return a.n == kFpN && a.key_dtype == RSSM_BF16 && (a.d == 64 || a.d == 128) && a.L <= kFpKE &&
         (reinterpret_cast<uintptr_t>(a.S0) & 15u) == 0 && static_cast<long long>(a.B) * a.H * a.d < (1ll << 31) &&
         (items + sms - 1) / sms <= kFpListMax && fp_encode_fn() != nullptr;
}

cudaError_t launch_flush_pipe(const FlushLaunch &a, cudaStream_t stream) {
  return a.vec_dtype == RSSM_BF16 ? launch_fp<bf16>(a, stream) : launch_fp<float>(a, stream);
}

}  // namespace rssm
