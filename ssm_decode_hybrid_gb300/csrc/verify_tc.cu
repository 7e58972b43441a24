// GDN chunked speculative verify, the S_0 contraction on the 5th-generation
// tensor cores (sm_103a).
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- appendix "GDN: speculative
// decoding": the T corrections come from one T x T lower-triangular solve, so
// the verify step becomes GEMM-shaped.  Per (sequence, value head) the
// checkpoint meets the window's 2T vectors once:
//   Z = S_0 [k_1 .. k_T, q_1 .. q_T]    (dv x dk times dk x 2T)
// and every output row r follows from row r of Z and the precomputed terms:
//   u_m[r] = beta_m (v_m[r] - e^{G_m} (abar Z[r][m] + bk_m[r])) - sum_{m'<m} A[m][m'] u_m'[r]
//   y_m[r] = e^{G_m} (abar Z[r][T'+m] + bq_m[r]) + sum_{m'<=m} Y[m][m'] u_m'[r]
// (the precompute kernel of gdn_split.cu forms abar, e^{G_m}, beta_m, A, Y
// and the buffer vectors bk, bq in the caller's workspace).
//
// One CTA per (sequence, value head), 256 threads.  The head's 128 x 128 fp32
// S_0 block is loaded with every 16-byte load in flight at once (each warp
// reads whole 512-byte rows) and stored into shared memory in the 128-byte
// swizzled K-major layout of the MMA operand.  The tensor core reads fp32
// operands as tf32 by dropping the low 13 mantissa bits, so the MMAs on the
// raw block multiply hi = S_0 truncated; lo = S_0 - hi (exact in fp32, its
// own tf32 rounding is 2^-11 of lo) is then written in place from the
// registers that still hold S_0, once those MMAs have read the block, and
// multiplied in as well: S_0 x to about 2^-21 relative, fp32 level.  The
// window vectors are bf16, exact in tf32.  The accumulator (TMEM lanes =
// state rows, 16 fp32 columns: keys in 0..7, queries in 8..15) is read back
// with tcgen05.ld by warps 0-3 and thread r solves row r.
#include "kernels.cuh"
#include "tc05.cuh"

namespace rssm {

namespace {

constexpr int kVtRows = 128;                         // state rows per item: MMA M, TMEM lanes
constexpr int kVtK = 128;                            // state columns (dk)
constexpr int kVtChunks = 4;                         // 32-column (128-byte) chunks of a row
constexpr int kVtN = 16;                             // MMA N: 8 key columns, then 8 query columns
constexpr uint32_t kVtChunkBytes = kVtRows * 128;    // one chunk of A: 16 KB
constexpr uint32_t kVtXChunkBytes = kVtN * 128;      // one chunk of the vectors: 2 KB
constexpr uint32_t kVtA = 0;                                     // [4][16 KB] S_0, swizzled
constexpr uint32_t kVtX = kVtA + kVtChunks * kVtChunkBytes;      // [4][2 KB] window vectors, swizzled
constexpr uint32_t kVtHdr = kVtX + kVtChunks * kVtXChunkBytes;   // [kGdnWorkHeader] floats
constexpr uint32_t kVtSmem = kVtHdr + kGdnWorkHeader * 4 + 1024;  // + alignment slack
constexpr uint32_t kVtTmemCols = 32;
constexpr int kVtThreads = 256;                      // 8 warps stage S_0; warps 0-3 own TMEM lanes 0-127
constexpr int kVtWarps = kVtThreads / 32;
constexpr int kVtRowsPerThread = kVtRows / kVtWarps;  // 16 rows per warp, one 16-byte unit of each per lane

constexpr int kInfoValid = 1 << 16;

// Shared-memory descriptor of a K-major operand in the 128-byte swizzle
// layout: 8-row x 128-byte atoms stacked along M/N (sbo = 1024 B); lbo is
// unused for this layout (encoded as 1).  Bits [61,64) = 2: 128-byte swizzle.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// kind::tf32, fp32 accumulator, A and B tf32, both K-major, M = 128, N = 16.
constexpr uint32_t kVtIdesc = (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(kVtN >> 3) << 17) |
                              (static_cast<uint32_t>(kVtRows >> 4) << 24);

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(kVtIdesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

__device__ __forceinline__ void ld_32x32b_x16(uint32_t taddr, float (&v)[16]) {
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

__device__ __forceinline__ float4 lds4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts4(uint32_t a, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}
// The part of x the tensor core keeps when it reads an fp32 operand as tf32:
// the low 13 mantissa bits are dropped (truncation; a split that assumes
// rounding instead misses the parity tolerance by orders of magnitude).
__device__ __forceinline__ float tf32_part(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

// Shared parts of the two verify kernels.  A CTA contracts one 128 x 128
// fp32 block (128 consecutive state rows) with 16 window vectors.
struct TcBlock {
  uint32_t base;   // 1024-byte aligned shared-memory base
  uint32_t tmem;   // accumulator: TMEM lanes = rows, 16 columns
  uint32_t aoff;   // this thread's unit offset within a row of A
  float4 sv[kVtRowsPerThread];
};

// Issue the loads of the block (warp w takes rows w, w + 8, ...; lane l the
// row's 16-byte unit l: one coalesced 512-byte row per load, all in flight).
__device__ __forceinline__ void tc_load(TcBlock &t, const float *S, int warp, int lane) {
#pragma unroll
  for (int j = 0; j < kVtRowsPerThread; ++j)
    t.sv[j] = ldg_stream4(S + static_cast<size_t>(warp + kVtWarps * j) * kVtK + 4 * lane);
}

// Window vector v (16-byte unit u) into the swizzled K-major B operand: unit u
// of chunk u / 8 at atom v / 8, row v % 8, unit (u % 8) ^ (v % 8).
__device__ __forceinline__ void tc_put_x(const TcBlock &t, int v, int u, float4 x) {
  const int c = u >> 3, lu = u & 7;
  sts4(t.base + kVtX + c * kVtXChunkBytes + (v >> 3) * 1024 + (v & 7) * 128 + ((lu ^ (v & 7)) << 4), x);
}

// Set-up: barriers, TMEM.  Every thread calls it; ends with a block barrier
// after the caller has written the window vectors (tc_put_x) before it.
__device__ __forceinline__ void tc_setup(TcBlock &t, unsigned char *raw, uint64_t *hi_bar, uint64_t *mma_bar,
                                         uint32_t *s_tmem, int tid, int warp, int lane) {
  t.base = (smem_addr(raw) + 1023u) & ~1023u;  // the swizzle pattern repeats every 1024 bytes
  t.aoff = t.base + kVtA + (lane >> 3) * kVtChunkBytes + (((lane & 7) ^ (warp & 7)) << 4);
  if (tid == 0) {
    mbar_init(hi_bar, 1);
    mbar_init(mma_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tc05::alloc(s_tmem, kVtTmemCols);
    tc05::relinquish();
  }
}

__device__ __forceinline__ void tc_mma_all(const TcBlock &t, bool accumulate_first) {
#pragma unroll
  for (int c = 0; c < kVtChunks; ++c)
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2)
      mma_tf32(t.tmem, desc_sw128(t.base + kVtA + c * kVtChunkBytes + s2 * 32),
               desc_sw128(t.base + kVtX + c * kVtXChunkBytes + s2 * 32), accumulate_first || c > 0 || s2 > 0);
}

// Store the raw block, then (one thread) the MMAs on it: the tensor core
// reads the fp32 values as tf32 by dropping the low 13 mantissa bits, so this
// multiplies hi = S truncated.
__device__ __forceinline__ void tc_hi(TcBlock &t, uint32_t *s_tmem, uint64_t *hi_bar, int tid, int warp) {
#pragma unroll
  for (int j = 0; j < kVtRowsPerThread; ++j) {
    const int row = warp + kVtWarps * j;
    sts4(t.aoff + (row >> 3) * 1024 + (row & 7) * 128, t.sv[j]);
  }
  tc05::fence_proxy_async_smem();
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  t.tmem = *s_tmem;
  if (tid == 0) {
    tc_mma_all(t, false);
    tc05::commit(hi_bar);
  }
}

// Once the MMAs on hi have read the block: lo = S - hi (exact in fp32) in
// place, from the registers that still hold S, and the MMAs on it.  False
// if a bounded wait ran out.
__device__ __forceinline__ bool tc_lo(TcBlock &t, uint64_t *hi_bar, uint64_t *mma_bar, int tid, int warp) {
  if (__syncthreads_or(!mbar_wait(hi_bar, 0))) return false;
  tc05::fence_after_sync();
#pragma unroll
  for (int j = 0; j < kVtRowsPerThread; ++j) {
    const int row = warp + kVtWarps * j;
    const float4 x = t.sv[j];
    sts4(t.aoff + (row >> 3) * 1024 + (row & 7) * 128,
         make_float4(x.x - tf32_part(x.x), x.y - tf32_part(x.y), x.z - tf32_part(x.z), x.w - tf32_part(x.w)));
  }
  tc05::fence_proxy_async_smem();
  tc05::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    tc05::fence_after_sync();
    tc_mma_all(t, true);
    tc05::commit(mma_bar);
  }
  return true;
}

// Row `lane + 32 warp` of the accumulator, columns 0..15 (warps 0-3).
__device__ __forceinline__ void tc_read(const TcBlock &t, int warp, float (&z)[16]) {
  tc05::fence_after_sync();
  ld_32x32b_x16(t.tmem + (static_cast<uint32_t>(warp * 32) << 16), z);
}

__device__ __forceinline__ void tc_release(const TcBlock &t, int warp) {
  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc05::dealloc(t.tmem, kVtTmemCols);
}

template <typename TI, typename TU, typename TO>
__global__ void __launch_bounds__(kVtThreads, 3) gdn_verify_tc_kernel(GdnLaunch a, int stride, int P) {
  extern __shared__ unsigned char vt_raw[];
  __shared__ __align__(8) uint64_t hi_bar;
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.x, b = blockIdx.y;
  const int kh = i / (a.Hv / a.Hk);
  const int L = a.L, T = a.T;
  constexpr int dv = kVtRows, N = kVtK;
  const size_t bh = static_cast<size_t>(b) * a.Hv + i;
  TcBlock t;
  tc_load(t, a.S + bh * dv * N, warp, lane);
  tc_setup(t, vt_raw, &hi_bar, &mma_bar, &s_tmem, tid, warp, lane);
  float *shdr = reinterpret_cast<float *>(vt_raw + (t.base - smem_addr(vt_raw)) + kVtHdr);
  // window vectors: key m in row m, query m in row 8 + m, zero past T
  for (int idx = tid; idx < kVtN * (N / 4); idx += kVtThreads) {
    const int v = idx / (N / 4), u = idx % (N / 4);
    const int m = v & 7;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m < T)
      x = load4(static_cast<const TI *>(v < 8 ? a.k : a.q) + ((static_cast<size_t>(b) * T + m) * a.Hk + kh) * N + 4 * u);
    tc_put_x(t, v, u, x);
  }
  const float *wk = a.work + bh * stride;
  tc_hi(t, &s_tmem, &hi_bar, tid, warp);
  pdl_wait();  // the precompute grid has finished: workspace, drafts' k and g, pointers
  for (int c = tid; c < kGdnWorkHeader; c += kVtThreads) shdr[c] = wk[c];
  bool ok = tc_lo(t, &hi_bar, &mma_bar, tid, warp);
  // the solve's per-row inputs, loaded while the MMAs run
  const int r = tid;
  const bool rowt = r < dv;  // threads 0..127 own the rows (TMEM lanes)
  float pk[kMaxT], pq[kMaxT], pv[kMaxT];
#pragma unroll
  for (int m = 0; m < kMaxT; ++m) {
    pk[m] = pq[m] = pv[m] = 0.f;
    if (m < T && rowt) {
      pk[m] = wk[kGwBuf + m * dv + r];
      pq[m] = wk[kGwBuf + (P + m) * dv + r];  // the record holds P key vectors, then the queries
      pv[m] = load1(static_cast<const TI *>(a.v) + ((static_cast<size_t>(b) * T + m) * a.Hv + i) * dv + r);
    }
  }
  if (ok) ok = !__syncthreads_or(!mbar_wait(&mma_bar, 0));
  const int info = __float_as_int(shdr[kGwInfo]);
  const bool valid = (info & kInfoValid) && rssm_check(((info >> 8) & 0xff) < L && (info & 0xff) + T <= L, a.err);
  if (!ok) {
    if (tid == 0) set_err(a.err, RSSM_EBIT_TIMEOUT);
  } else if (valid) {
    if (rowt) {
      float z[16];
      tc_read(t, warp, z);
      const int h = info & 0xff, st = (info >> 8) & 0xff;
      const float abar = shdr[kGwAbar];
      TO *y = static_cast<TO *>(a.y);
      TU *ru = static_cast<TU *>(a.ring_u) + bh * L * dv;
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
          store1(y + tvm * dv + r, ym);
          store1(ru + static_cast<size_t>(checked_slot((st + h + m) % L, L, a.err)) * dv + r, um);
        }
      }
    }
  }
  if (ok && i == 0 && warp == 0) {
    // the flag, once every group's precompute block of the sequence finished
    // (the header is read again: nothing of the solve stays live up to here)
    const int inf = __float_as_int(shdr[kGwInfo]);
    if ((inf & kInfoValid) &&
        sequence_records_valid(a.work + static_cast<size_t>(b) * a.Hv * stride, a.Hk, a.Hv / a.Hk, stride, kGwInfo,
                               kInfoValid) &&
        lane == 0)
      a.flag[b] = ((inf & 0xff) + 2 * T > L) ? 1 : 0;  // early flush, one window ahead
  }
  tc_release(t, warp);
}

// Mamba-2 verify ("Algorithm -- speculative decoding"): the checkpoint term
// H_{:,s} = abar_s (S_0 q_s) for all T drafts at once.  Heads of one group
// share their queries, so one CTA takes two consecutive heads of a group
// (2 x d = 128 rows, d = 64) against the group's T queries; thread r writes
// Y_s[r] = abar_s(head) Z[r][s] + buf_s(head)[r] from the workspace record of
// the Mamba-2 precompute kernel: [abar_1..abar_8, info, pad, buf_s[0..d)].
constexpr int kM2Rows = 64;

template <typename TI, typename TO>
__global__ void __launch_bounds__(kVtThreads, 3) m2_verify_tc_kernel(M2Launch a, int stride) {
  extern __shared__ unsigned char vt_raw[];
  __shared__ __align__(8) uint64_t hi_bar;
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i0 = 2 * blockIdx.x, b = blockIdx.y;
  const int g = i0 / (a.H / a.G);
  const int L = a.L, T = a.T;
  constexpr int d = kM2Rows, N = kVtK;
  const size_t bh0 = static_cast<size_t>(b) * a.H + i0;
  TcBlock t;
  tc_load(t, a.S + bh0 * d * N, warp, lane);
  tc_setup(t, vt_raw, &hi_bar, &mma_bar, &s_tmem, tid, warp, lane);
  // window vectors: query s in row s, zero past T
  for (int idx = tid; idx < kVtN * (N / 4); idx += kVtThreads) {
    const int v = idx / (N / 4), u = idx % (N / 4);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (v < T) x = load4(static_cast<const TI *>(a.q) + ((static_cast<size_t>(b) * T + v) * a.G + g) * N + 4 * u);
    tc_put_x(t, v, u, x);
  }
  tc_hi(t, &s_tmem, &hi_bar, tid, warp);
  pdl_wait();  // the precompute grid has finished: workspace, drafts' entries, pointers
  bool ok = tc_lo(t, &hi_bar, &mma_bar, tid, warp);
  const int r = tid;
  const bool rowt = r < 2 * d;
  const int head = i0 + (r >= d ? 1 : 0), row = r & (d - 1);
  const float *wk = a.work + (static_cast<size_t>(b) * a.H + head) * stride;
  float ab[kMaxT], buf[kMaxT];
#pragma unroll
  for (int s2 = 0; s2 < kMaxT; ++s2) {
    ab[s2] = buf[s2] = 0.f;
    if (s2 < T && rowt) {
      ab[s2] = wk[s2];
      buf[s2] = wk[kM2VerifyHeader + s2 * d + row];
    }
  }
  const int info = rowt ? reinterpret_cast<const int *>(wk)[kMaxT] : 0;
  if (ok) ok = !__syncthreads_or(!mbar_wait(&mma_bar, 0));
  if (!ok) {
    if (tid == 0) set_err(a.err, RSSM_EBIT_TIMEOUT);
  } else if (rowt) {
    float z[16];
    tc_read(t, warp, z);
    if (info & kInfoValid) {
      TO *y = static_cast<TO *>(a.y);
#pragma unroll
      for (int s2 = 0; s2 < kMaxT; ++s2)
        if (s2 < T) store1(y + ((static_cast<size_t>(b) * T + s2) * a.H + head) * d + row, fmaf(ab[s2], z[s2], buf[s2]));
    }
  }
  if (ok && i0 == 0 && warp == 0) {
    // the flag, once every group's precompute block of the sequence finished
    // (the record is read again: nothing of the epilogue stays live up to here)
    const float *first = a.work + static_cast<size_t>(b) * a.H * stride;
    const int inf = reinterpret_cast<const int *>(first)[kMaxT];
    if ((inf & kInfoValid) && sequence_records_valid(first, a.G, a.H / a.G, stride, kMaxT, kInfoValid) && lane == 0)
      a.flag[b] = ((inf & 0xff) + 2 * T > L) ? 1 : 0;  // early flush, one window ahead
  }
  tc_release(t, warp);
}

template <typename TU, typename TO>
cudaError_t launch_vt(const GdnLaunch &a, int stride, int P, cudaStream_t stream) {
  auto kern = gdn_verify_tc_kernel<bf16, TU, TO>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kVtSmem))) !=
      cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.Hv), static_cast<unsigned>(a.B));
  cfg.blockDim = dim3(kVtThreads);
  cfg.dynamicSmemBytes = kVtSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, stride, P);
}

template <typename TO>
cudaError_t launch_m2vt(const M2Launch &a, int stride, cudaStream_t stream) {
  auto kern = m2_verify_tc_kernel<bf16, TO>;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kVtSmem))) !=
      cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.H / 2), static_cast<unsigned>(a.B));
  cfg.blockDim = dim3(kVtThreads);
  cfg.dynamicSmemBytes = kVtSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, stride);
}

}  // namespace

bool gdn_verify_tc_eligible(const GdnLaunch &a) {
  // T = 1 (two window vectors) stays on the CUDA cores, where it is cheaper
  return a.dk == kVtK && a.dv == kVtRows && a.in_dtype == RSSM_BF16 && a.T >= 2 && a.T <= kMaxT &&
         a.B <= 65535 && (reinterpret_cast<uintptr_t>(a.S) & 15u) == 0;
}

cudaError_t launch_gdn_verify_tc(const GdnLaunch &a, int stride, int P, cudaStream_t stream) {
  const bool ub = a.u_dtype == RSSM_BF16, yb = a.y_dtype == RSSM_BF16;
  if (ub && yb) return launch_vt<bf16, bf16>(a, stride, P, stream);
  if (ub) return launch_vt<bf16, float>(a, stride, P, stream);
  if (yb) return launch_vt<float, bf16>(a, stride, P, stream);
  return launch_vt<float, float>(a, stride, P, stream);
}

}  // namespace rssm

namespace rssm {

bool m2_verify_tc_eligible(const M2Launch &a) {
  // two heads of one group per 128-row block; up to four queries the CUDA
  // cores keep up with the S_0 stream and stay faster
  return a.n == kVtK && a.d == kM2Rows && a.in_dtype == RSSM_BF16 && a.H % 2 == 0 && (a.H / a.G) % 2 == 0 &&
         a.T >= 5 && a.T <= kMaxT && a.B <= 65535 && (reinterpret_cast<uintptr_t>(a.S) & 15u) == 0;
}

cudaError_t launch_m2_verify_tc(const M2Launch &a, int stride, cudaStream_t stream) {
  return a.y_dtype == RSSM_BF16 ? launch_m2vt<bf16>(a, stride, stream) : launch_m2vt<float>(a, stride, stream);
}

}  // namespace rssm
