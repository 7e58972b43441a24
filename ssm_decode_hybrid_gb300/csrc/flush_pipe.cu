// Flush as a persistent, warp-specialised TMA + tcgen05 pipeline (sm_103a).
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- "Algorithm: Mamba-2 standard
// decode" (flush: S_0 <- abar S_0 + sum_j s_j v_j k_j^T over the committed
// entries, then clear the buffer) and the GDN appendix (the same history form
// with the cached corrections u_j and the gates g_j).
//
// Items are 64-row halves of the (sequence, head) tiles of flagged sequences
// (a head of d = 64 rows is one item, one of d = 128 two), spread over the
// persistent CTAs by their index so that every CTA gets its share.  Roles:
//   warp 0     TMA producer: an item's 64 x 128 fp32 rows land in its group's
//              stage as four 64-row x 32-column boxes in the 128-byte swizzle,
//              issued as soon as the group has released the stage;
//   warps 2-17 four worker groups of four warps, taking every fourth item.
//              While the tile is on its way a group reads the pointers, forms
//              the decay weights (one warp scan), builds the two operands of
//              D^T = K (W V)^T in shared memory (keys, exact in bf16, K-major;
//              each w_j v_j[r] split into three bf16 terms, so the product
//              keeps fp32 accuracy) and issues the three MMAs (M = 128 state
//              columns = TMEM lanes, N = 64 rows, K = 48) into its own 64 TMEM
//              columns; then thread c (state column c) reads D^T[c][0..64)
//              and writes S_0[r][c] = abar S_0[r][c] + D^T[c][r] from the
//              landed tile, a warp writing 128 contiguous bytes of a row.
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
constexpr uint32_t kFpABytes = kFpN * kFpKT * 2;         // keys operand: 12 KB
constexpr uint32_t kFpBBytes = kFpRows * kFpKT * 2;      // weighted-vector operand: 6 KB
constexpr uint32_t kFpTilesOff = 0;
constexpr uint32_t kFpOpsOff = kFpTilesOff + kFpGroups * kFpTileBytes;
constexpr int kFpListMax = 1024;                        // items one CTA may hold (its gids, compacted)
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
  // this CTA's items (gid = blockIdx.x + j gridDim.x of flagged sequences),
  // compacted in order into shared memory once, so that no role walks the
  // flags with a dependent load per candidate
  int *items = reinterpret_cast<int *>(fp_raw + (base - smem_addr(fp_raw)) + kFpListOff);
  int *item_cnt = items + kFpListMax, *item_st = item_cnt + kFpListMax;
  const int per_cta = static_cast<int>((total - blockIdx.x + gridDim.x - 1) / gridDim.x);
  int n_items = 0;
  for (int j0 = 0; j0 < per_cta; j0 += kFpThreads) {
    const int jj = j0 + tid;
    const long gid = blockIdx.x + static_cast<long>(jj) * gridDim.x;
    const bool f = jj < per_cta && a.flag[gid / per_seq] != 0;
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
    if (f) items[n_items + s_wcount[warp] + __popc(m & ((1u << lane) - 1u))] = static_cast<int>(gid);
    n_items += s_wcount[kFpThreads / 32];
    __syncthreads();
  }
  // and their pointers, all read before any item is folded (every item of a
  // sequence reads them before the last one resets them)
  for (int kk = tid; kk < n_items; kk += kFpThreads) {
    const int b = items[kk] / per_seq;
    item_cnt[kk] = a.count[b];
    item_st[kk] = a.start[b];
  }

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
    const int gt = tid - 64 - g * 128;        // 0..127 within the group
    const int c = 32 * (warp % 4) + lane;     // state column = TMEM lane this thread reads
    const int gw = gt >> 5;                   // warp within the group
    const uint32_t tile = base + kFpTilesOff + g * kFpTileBytes;
    const uint32_t opA = base + kFpOpsOff + g * (kFpABytes + kFpBBytes), opB = opA + kFpABytes;
    unsigned char *pA = fp_raw + (opA - smem_addr(fp_raw));
    unsigned char *pB = fp_raw + (opB - smem_addr(fp_raw));
    const uint32_t d_tmem = tmem + static_cast<uint32_t>(g * kFpRows);
    const uint32_t idesc = tc05::idesc_bf16_f32(kFpN, kFpRows);
    int j = 0, mj = 0;  // j: this group's items so far, mj: its MMA commits so far
    for (int k = g; k < n_items; k += kFpGroups) {
      const int gid = items[k];
      const int b = gid / per_seq;
      const int rest = gid - b * per_seq;
      const int i = rest / halves, hf = rest - i * halves;
      const size_t bh = static_cast<size_t>(b) * H + i;
      const size_t bg = static_cast<size_t>(b) * a.G + i / HpG;
      const int cnt = item_cnt[k], st = item_st[k];
      const bool valid = cnt >= 0 && cnt <= L && st >= 0 && st < L;
      // every load of the item at once: keys (this thread's state column), the
      // vectors of its rows, the log decays (warp 0)
      constexpr int kVPer = kFpRows * kFpKE / 128;  // vector values per thread
      bf16 kv[kFpKE];
      float vv[kVPer];
      float ld = 0.f;
      if (valid) {
        const bf16 *key = static_cast<const bf16 *>(a.ring_key) + bg * L * kFpN;
#pragma unroll
        for (int e = 0; e < kFpKE; ++e)
          kv[e] = (e < cnt) ? key[static_cast<size_t>((st + e) % L) * kFpN + gt] : __float2bfloat16_rn(0.f);
        const TV *vec = static_cast<const TV *>(a.ring_vec) + bh * L * a.d + hf * kFpRows;
#pragma unroll
        for (int u = 0; u < kVPer; ++u) {
          const int idx = gt + 128 * u, e = idx / kFpRows, r = idx - e * kFpRows;
          vv[u] = (e < cnt) ? load1(vec + static_cast<size_t>((st + e) % L) * a.d + r) : 0.f;
        }
        if (gw == 0 && lane < cnt) ld = a.ring_ld[bh * L + (st + lane) % L];
      }
      if (valid) {
        if (gw == 0) {
          // decay weights over the committed entries, one per lane
          const float la = a.mamba2 ? a.A[i] * ld : ld;
          float tot;
          const float ex = excl_suffix_sum(lane < cnt ? la : 0.f, lane, tot);
          s_w[g][lane] = (lane < cnt) ? (a.mamba2 ? ld : 1.f) * expf(ex) : 0.f;
          if (lane == 0) s_abar[g] = expf(tot);
        }
        // A operand: row = state column gt, K = entries (the keys, three times)
#pragma unroll
        for (int e = 0; e < kFpKE; e += 2) {
          __nv_bfloat162 pr;
          pr.x = kv[e];
          pr.y = kv[e + 1];
#pragma unroll
          for (int t = 0; t < 3; ++t)
            *reinterpret_cast<__nv_bfloat162 *>(pA + tc05::kmajor_offset(kFpN, gt, t * kFpKE + e)) = pr;
        }
      }
      // s_w ready; every thread is past the previous item's TMEM reads
      if (named_bar_or(1 + g, 128, *abort != 0)) break;
      if (valid) {
        // B operand: row r of the item, K = entries: hi(w_e v_e[r]), then mid, then lo
#pragma unroll
        for (int u = 0; u < kVPer; ++u) {
          const int idx = gt + 128 * u, e = idx / kFpRows, r = idx - e * kFpRows;
          bf16 t0, t1, t2;
          tc05::split3_bf16(s_w[g][e] * vv[u], t0, t1, t2);
          *reinterpret_cast<bf16 *>(pB + tc05::kmajor_offset(kFpRows, r, e)) = t0;
          *reinterpret_cast<bf16 *>(pB + tc05::kmajor_offset(kFpRows, r, kFpKE + e)) = t1;
          *reinterpret_cast<bf16 *>(pB + tc05::kmajor_offset(kFpRows, r, 2 * kFpKE + e)) = t2;
        }
        tc05::fence_proxy_async_smem();
      }
      tc05::fence_before_sync();
      if (named_bar_or(1 + g, 128, false)) break;  // operands in place
      if (valid && gt == 0) {
        tc05::fence_after_sync();
        for (int s = 0; s < kFpKT / 16; ++s)
          tc05::mma_bf16(d_tmem, tc05::smem_desc(pA + static_cast<size_t>(s) * kFpN * 32, tc05::kLBO, tc05::kSBO),
                         tc05::smem_desc(pB + static_cast<size_t>(s) * kFpRows * 32, tc05::kLBO, tc05::kSBO), idesc,
                         s > 0);
        tc05::commit(&mma_bar[g]);
      }
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
  kern<<<grid, kFpThreads, kFpSmem, stream>>>(map, a, halves);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fp_reset_kernel<<<(a.B + 255) / 256, 256, 0, stream>>>(a.B, a.L, a.start, a.count, a.flag);
  return cudaGetLastError();
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
