// Flush: fold the committed ring entries of flagged sequences into S_0.
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- "Algorithm: Mamba-2 standard
// decode" (flush: S_0 <- abar S_0 + sum_j s_j v_j k_j^T, then clear the
// buffer) and the GDN appendix (same history form with the cached
// corrections u_j and the gates g_j).
//
// Two launches.  The first is a persistent grid: every CTA compacts the
// flagged sequences (in sequence order, so all CTAs build the same list) and
// takes every grid-th (sequence, head) item of that list.  For an item, the
// c committed entries (c x d vectors, c x n keys) are staged in shared memory;
// each thread owns one 16-byte column slice of up to 8 rows of S_0, loads it,
// and accumulates abar * S_0 + sum_j (w_j v_j[r]) k_j[col..col+3] with the
// key slice read once per entry.  The last of a sequence's items to arrive
// resets start and count.  The flags themselves are cleared by the second,
// one-thread-per-sequence launch, because every CTA of the first reads them.
#include "kernels.cuh"
#include "tc05.cuh"

namespace rssm {

namespace {

constexpr int kPass = 8;

template <int N, typename TV, typename TK>
__global__ void __launch_bounds__(kThreads) flush_kernel(FlushLaunch a) {
  constexpr int LPR = N / 4, RPW = 32 / LPR, RPP = kWarps * RPW;
  extern __shared__ float smem[];  // [L][d] vectors, then [L][N] keys (f32)
  __shared__ int s_list[kThreads];
  __shared__ int s_wsum[kWarps + 1];
  __shared__ float s_wt[kMaxL];
  __shared__ float s_abar;
  __shared__ int s_ptr[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = a.B, H = a.H, d = a.d, L = a.L;
  const int HpG = H / a.G;
  const int grid = gridDim.x;
  float *s_vec = smem;
  float *s_key = smem + static_cast<size_t>(L) * d;
  const int col = (lane % LPR) * 4;
  const int row0 = warp * RPW + lane / LPR;

  int done = 0;  // flagged sequences in earlier chunks
  for (int base = 0; base < B; base += kThreads) {
    // ordered compaction of the flagged sequences of this chunk
    const int bq = base + tid;
    const bool f = bq < B && a.flag[bq] != 0;
    const unsigned m = __ballot_sync(kFull, f);
    if (lane == 0) s_wsum[warp] = __popc(m);
    __syncthreads();
    if (tid == 0) {
      int acc = 0;
      for (int w = 0; w < kWarps; ++w) {
        const int c = s_wsum[w];
        s_wsum[w] = acc;
        acc += c;
      }
      s_wsum[kWarps] = acc;
    }
    __syncthreads();
    if (f) s_list[s_wsum[warp] + __popc(m & ((1u << lane) - 1u))] = bq;
    __syncthreads();
    const int nf = s_wsum[kWarps];
    const long first = static_cast<long>(done) * H;  // global index of this chunk's first item
    int k = static_cast<int>(((static_cast<long>(blockIdx.x) - first) % grid + grid) % grid);
    for (; k < nf * H; k += grid) {
      const int b = s_list[k / H], i = k % H;
      if (tid == 0) {
        s_ptr[0] = a.count[b];
        s_ptr[1] = a.start[b];
      }
      __syncthreads();
      const int c = s_ptr[0], st = s_ptr[1];
      __syncthreads();
      if (c < 0 || c > L || st < 0 || st >= L) {
        if (tid == 0) set_err(a.err, RSSM_EBIT_COUNT_RANGE);
        continue;
      }
      if (tid == 0 && last_arrival(a.sync, b, H)) {
        a.start[b] = (st + c) % L;
        a.count[b] = 0;
      }
      const size_t bh = static_cast<size_t>(b) * H + i;
      const size_t bg = static_cast<size_t>(b) * a.G + i / HpG;
      float *S0 = a.S0 + bh * d * N;
      const TV *vec = static_cast<const TV *>(a.ring_vec) + bh * L * d;
      const TK *key = static_cast<const TK *>(a.ring_key) + bg * L * N;
      if (warp == 0) {
        float ld = 0.f;
        if (lane < c) ld = a.ring_ld[bh * L + (st + lane) % L];
        const float la = a.mamba2 ? a.A[i] * ld : ld;
        float total;
        const float ex = excl_suffix_sum(lane < c ? la : 0.f, lane, total);
        if (lane < c) s_wt[lane] = (a.mamba2 ? ld : 1.f) * expf(ex);
        if (lane == 0) s_abar = expf(total);
      }
      for (int idx = tid; idx < c * d; idx += kThreads) {
        const int j = idx / d, r = idx - j * d;
        s_vec[idx] = load1(vec + static_cast<size_t>((st + j) % L) * d + r);
      }
      for (int idx = tid; idx < c * (N / 4); idx += kThreads) {
        const int j = idx / (N / 4), c4 = (idx - j * (N / 4)) * 4;
        store4(s_key + j * N + c4, load4(key + static_cast<size_t>((st + j) % L) * N + c4));
      }
      for (int rb = 0; rb < d; rb += kPass * RPP) {
        float4 acc[kPass];
#pragma unroll
        for (int p = 0; p < kPass; ++p) {
          const int r = rb + row0 + p * RPP;
          acc[p] = (r < d) ? ldg_stream4(S0 + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();  // s_vec, s_key, s_wt, s_abar ready (first pass); loads in flight
        const float abar = s_abar;
#pragma unroll
        for (int p = 0; p < kPass; ++p) {
          acc[p].x *= abar;
          acc[p].y *= abar;
          acc[p].z *= abar;
          acc[p].w *= abar;
        }
        for (int j = 0; j < c; ++j) {
          const float4 kv = *reinterpret_cast<const float4 *>(s_key + j * N + col);
          const float w = s_wt[j];
#pragma unroll
          for (int p = 0; p < kPass; ++p) {
            const int r = rb + row0 + p * RPP;
            const float wv = (r < d) ? w * s_vec[j * d + r] : 0.f;
            acc[p].x = fmaf(wv, kv.x, acc[p].x);
            acc[p].y = fmaf(wv, kv.y, acc[p].y);
            acc[p].z = fmaf(wv, kv.z, acc[p].z);
            acc[p].w = fmaf(wv, kv.w, acc[p].w);
          }
        }
#pragma unroll
        for (int p = 0; p < kPass; ++p) {
          const int r = rb + row0 + p * RPP;
          if (r < d) stg_stream4(S0 + static_cast<size_t>(r) * N + col, acc[p]);
        }
      }
      __syncthreads();  // shared staging is reused by the next item
    }
    done += nf;
    __syncthreads();  // s_list / s_wsum are rebuilt for the next chunk
  }
}

// ---------------------------------------------------------------------------
// Tensor-core flush (n = 128, bf16 keys).  The fold of one (sequence, head)
// is the d x c by c x n contraction D = sum_j (w_j v_j) k_j^T.  It runs on the
// 5th-generation tensor core in transposed form, D^T = K (w V)^T: M = n = 128
// rows (TMEM lanes, one per state column), N = d columns, K = the ring
// entries.  Keys are exact in bf16; each weighted vector w_j v_j[r] is split
// into three bf16 terms (hi + mid + lo, about 2^-25 relative), so the K
// extent is 3 * KE (KE = L rounded up to 16) and the fp32 accumulator sees
// the product to fp32 accuracy.  Operands are built in shared memory in the no-swizzle K-major
// layout, one thread issues the MMAs and commits them to an mbarrier, and
// each thread then owns one state column c: it loads D^T[c][0..d) from TMEM
// and writes S_0[r][c] = abar S_0[r][c] + D^T[c][r] with warp-coalesced
// accesses along the row.
// ---------------------------------------------------------------------------
constexpr int kTcThreads = 128;

template <typename TV>
__global__ void __launch_bounds__(kTcThreads) flush_tc_kernel(FlushLaunch a, int ke, uint32_t ncols) {
  constexpr int N = 128;
  extern __shared__ __align__(1024) unsigned char tc_smem[];
  __shared__ uint64_t mma_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_list[kTcThreads];
  __shared__ int s_wsum[kTcThreads / 32 + 1];
  __shared__ float s_wt[kMaxL];
  __shared__ float s_abar;
  __shared__ int s_ptr[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = a.B, H = a.H, d = a.d, L = a.L;
  const int HpG = H / a.G;
  const int grid = gridDim.x;
  const int KT = 3 * ke;
  bf16 *opA = reinterpret_cast<bf16 *>(tc_smem);                                   // [KT/16][128 rows][16]
  bf16 *opB = reinterpret_cast<bf16 *>(tc_smem + static_cast<size_t>(N) * KT * 2);  // [KT/16][d rows][16]
  const uint32_t idesc = tc05::idesc_bf16_f32(N, d);

  if (warp == 0) {
    tc05::alloc(&s_tmem, ncols);
    tc05::relinquish();
  }
  if (tid == 0) {
    mbar_init(&mma_bar, 1);
    fence_mbar_init();
  }
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tmem = s_tmem;
  uint32_t phase = 0;
  bool alive = true;

  int done = 0;
  for (int base = 0; base < B && alive; base += kTcThreads) {
    const int bq = base + tid;
    const bool f = bq < B && a.flag[bq] != 0;
    const unsigned m = __ballot_sync(kFull, f);
    if (lane == 0) s_wsum[warp] = __popc(m);
    __syncthreads();
    if (tid == 0) {
      int acc = 0;
      for (int w = 0; w < kTcThreads / 32; ++w) {
        const int c = s_wsum[w];
        s_wsum[w] = acc;
        acc += c;
      }
      s_wsum[kTcThreads / 32] = acc;
    }
    __syncthreads();
    if (f) s_list[s_wsum[warp] + __popc(m & ((1u << lane) - 1u))] = bq;
    __syncthreads();
    const int nf = s_wsum[kTcThreads / 32];
    const long first = static_cast<long>(done) * H;
    int k = static_cast<int>(((static_cast<long>(blockIdx.x) - first) % grid + grid) % grid);
    for (; k < nf * H && alive; k += grid) {
      const int b = s_list[k / H], i = k % H;
      if (tid == 0) {
        s_ptr[0] = a.count[b];
        s_ptr[1] = a.start[b];
      }
      __syncthreads();
      const int c = s_ptr[0], st = s_ptr[1];
      __syncthreads();
      if (c < 0 || c > L || st < 0 || st >= L) {
        if (tid == 0) set_err(a.err, RSSM_EBIT_COUNT_RANGE);
        continue;
      }
      const size_t bh = static_cast<size_t>(b) * H + i;
      const size_t bg = static_cast<size_t>(b) * a.G + i / HpG;
      // this thread's state column for the first kPre rows, loaded now so that
      // the loads overlap the operand staging and the MMA
      constexpr int kPre = 64;
      float *S0 = a.S0 + bh * d * N;
      float spre[kPre];
#pragma unroll
      for (int u = 0; u < kPre; ++u) spre[u] = (u < d) ? __ldcs(S0 + static_cast<size_t>(u) * N + tid) : 0.f;
      if (warp == 0) {
        float ld = 0.f;
        if (lane < c) ld = a.ring_ld[bh * L + (st + lane) % L];
        const float la = a.mamba2 ? a.A[i] * ld : ld;
        float total;
        const float ex = excl_suffix_sum(lane < c ? la : 0.f, lane, total);
        s_wt[lane] = (lane < c) ? (a.mamba2 ? ld : 1.f) * expf(ex) : 0.f;
        if (lane == 0) s_abar = expf(total);
      }
      // A operand: row = state column (this thread), K = entries (keys, twice)
      const bf16 *key = static_cast<const bf16 *>(a.ring_key) + bg * L * N;
      for (int j = 0; j < ke; j += 2) {
        bf16 k0 = __float2bfloat16_rn(0.f), k1 = k0;
        if (j < c) k0 = key[static_cast<size_t>((st + j) % L) * N + tid];
        if (j + 1 < c) k1 = key[static_cast<size_t>((st + j + 1) % L) * N + tid];
        __nv_bfloat162 pr;
        pr.x = k0;
        pr.y = k1;
#pragma unroll
        for (int t = 0; t < 3; ++t)
          *reinterpret_cast<__nv_bfloat162 *>(reinterpret_cast<unsigned char *>(opA) +
                                              tc05::kmajor_offset(N, tid, t * ke + j)) = pr;
      }
      __syncthreads();  // s_wt ready
      // B operand: row r of S_0, K = entries: hi(w_j v_j[r]), then mid, then lo
      const TV *vec = static_cast<const TV *>(a.ring_vec) + bh * L * d;
      const int half = ke / 2;
      for (int idx = tid; idx < d * half; idx += kTcThreads) {
        const int jp = idx / d, r = idx - jp * d, j = 2 * jp;
        const float w0 = (j < c) ? s_wt[j] * load1(vec + static_cast<size_t>((st + j) % L) * d + r) : 0.f;
        const float w1 = (j + 1 < c) ? s_wt[j + 1] * load1(vec + static_cast<size_t>((st + j + 1) % L) * d + r) : 0.f;
        __nv_bfloat162 t3[3];
        tc05::split3_bf16(w0, t3[0].x, t3[1].x, t3[2].x);
        tc05::split3_bf16(w1, t3[0].y, t3[1].y, t3[2].y);
#pragma unroll
        for (int t = 0; t < 3; ++t)
          *reinterpret_cast<__nv_bfloat162 *>(reinterpret_cast<unsigned char *>(opB) +
                                              tc05::kmajor_offset(d, r, t * ke + j)) = t3[t];
      }
      tc05::fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc05::fence_after_sync();
        for (int s = 0; s < KT / 16; ++s)
          tc05::mma_bf16(tmem, tc05::smem_desc(opA + static_cast<size_t>(s) * N * 16, tc05::kLBO, tc05::kSBO),
                         tc05::smem_desc(opB + static_cast<size_t>(s) * d * 16, tc05::kLBO, tc05::kSBO), idesc, s > 0);
        tc05::commit(&mma_bar);
      }
      const bool timed_out = !mbar_wait(&mma_bar, phase);
      if (__syncthreads_or(timed_out)) {  // the same decision in every thread
        if (tid == 0) set_err(a.err, RSSM_EBIT_TIMEOUT);
        alive = false;
        break;
      }
      phase ^= 1u;
      tc05::fence_after_sync();
      // epilogue: this thread owns state column tid (TMEM lane tid)
      const float abar = s_abar;
#pragma unroll
      for (int r0 = 0; r0 < kPre; r0 += 32) {
        if (r0 < d) {
          float dv[32];
          tc05::ld_32x32b_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(r0), dv);
#pragma unroll
          for (int u = 0; u < 32; ++u)
            __stcs(S0 + static_cast<size_t>(r0 + u) * N + tid, fmaf(abar, spre[r0 + u], dv[u]));
        }
      }
      for (int r0 = kPre; r0 < d; r0 += 32) {
        float dv[32], sv[32];
        tc05::ld_32x32b_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(r0), dv);
#pragma unroll
        for (int u = 0; u < 32; ++u) sv[u] = __ldcs(S0 + static_cast<size_t>(r0 + u) * N + tid);
#pragma unroll
        for (int u = 0; u < 32; ++u) __stcs(S0 + static_cast<size_t>(r0 + u) * N + tid, fmaf(abar, sv[u], dv[u]));
      }
      // the pointers of b are reset once every item of b has read them
      if (tid == 0 && last_arrival(a.sync, b, H)) {
        a.start[b] = (st + c) % L;
        a.count[b] = 0;
      }
      tc05::fence_before_sync();
      __syncthreads();  // TMEM and the operand buffers are reused by the next item
    }
    done += nf;
    __syncthreads();
  }
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc05::dealloc(tmem, ncols);
}

__global__ void clear_flags_kernel(int B, int32_t *flag) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) flag[b] = 0;
}

template <int N, typename TV, typename TK>
cudaError_t launch_flush_n(const FlushLaunch &a, cudaStream_t stream) {
  const size_t sm = static_cast<size_t>(a.L) * (a.d + N) * sizeof(float);
  auto kern = flush_kernel<N, TV, TK>;
  if (sm > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm));
    if (e != cudaSuccess) return e;
  }
  const long items = static_cast<long>(a.B) * a.H;
  const long cap = static_cast<long>(a.num_sms > 0 ? a.num_sms : 148) * 4;
  const unsigned grid = static_cast<unsigned>(items < cap ? items : cap);
  kern<<<grid, kThreads, sm, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  clear_flags_kernel<<<(a.B + 255) / 256, 256, 0, stream>>>(a.B, a.flag);
  return cudaGetLastError();
}

template <typename TV, typename TK>
cudaError_t launch_flush_t(const FlushLaunch &a, cudaStream_t stream) {
  switch (a.n) {
    case 16: return launch_flush_n<16, TV, TK>(a, stream);
    case 32: return launch_flush_n<32, TV, TK>(a, stream);
    case 64: return launch_flush_n<64, TV, TK>(a, stream);
    case 128: return launch_flush_n<128, TV, TK>(a, stream);
  }
  return cudaErrorInvalidValue;
}

template <typename TV>
cudaError_t launch_flush_tc(const FlushLaunch &a, cudaStream_t stream) {
  int dev = 0, sms = 0, smem_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
  const int ke = a.L <= 16 ? 16 : 32;
  uint32_t ncols = 32;
  while (ncols < static_cast<uint32_t>(a.d)) ncols <<= 1;
  // at most 512 / ncols CTAs may hold TMEM on one SM: request enough shared
  // memory that no more than that many are resident at once
  const int per_sm = static_cast<int>(512u / ncols) < 4 ? static_cast<int>(512u / ncols) : 4;
  const size_t need = static_cast<size_t>(128 + a.d) * 3 * ke * 2;
  size_t smem = static_cast<size_t>(smem_sm) / (per_sm + 1) + 1024;
  if (smem < need) smem = need;
  auto kern = flush_tc_kernel<TV>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) !=
      cudaSuccess)
    return e;
  const long items = static_cast<long>(a.B) * a.H;
  const long cap = static_cast<long>(sms) * per_sm;
  const unsigned grid = static_cast<unsigned>(items < cap ? items : cap);
  kern<<<grid, kTcThreads, smem, stream>>>(a, ke, ncols);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  clear_flags_kernel<<<(a.B + 255) / 256, 256, 0, stream>>>(a.B, a.flag);
  return cudaGetLastError();
}

}  // namespace

bool flush_tc_eligible(const FlushLaunch &a) {
  return a.n == 128 && a.key_dtype == RSSM_BF16 && a.d % 32 == 0 && a.d <= 256 && a.L <= kMaxL;
}

cudaError_t launch_flush(const FlushLaunch &a, cudaStream_t stream) {
  if (flush_pipe_eligible(a)) return launch_flush_pipe(a, stream);
  if (flush_tc_eligible(a))
    return a.vec_dtype == RSSM_BF16 ? launch_flush_tc<bf16>(a, stream) : launch_flush_tc<float>(a, stream);
  const bool vb = a.vec_dtype == RSSM_BF16, kb = a.key_dtype == RSSM_BF16;
  if (vb && kb) return launch_flush_t<bf16, bf16>(a, stream);
  if (!vb && kb) return launch_flush_t<float, bf16>(a, stream);
  if (vb && !kb) return launch_flush_t<bf16, float>(a, stream);
  return launch_flush_t<float, float>(a, stream);
}

}  // namespace rssm
