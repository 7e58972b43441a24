// Gated DeltaNet decode step and chunked speculative verify as two launches
// (sm_103a): a small precompute kernel per (sequence, key head) and a kernel
// streaming S_0 per (sequence, value head, row block).
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- appendix "GDN: standard decode"
// (cache u; S_h from the decayed checkpoint plus the buffer), "GDN:
// speculative decoding" (u_s = R_s - sum_{s'<s} A_{s,s'} u_{s'}), and "Kernel
// design details" (a small precompute kernel for the buffer-dependent terms,
// the main kernel streaming the checkpoint).
//
// With the window's vectors x_v (the T drafts' keys, then their queries),
//   S_h x_v = abar (S_0 x_v) + sum_{j<h} w_j (k_j . x_v) u_j,
// and both the solve and the outputs act row by row:
//   u_m[r] = beta_m (v_m[r] - e^{G_m} (S_h k_m)[r]) - sum_{m'<m} A[m][m'] u_{m'}[r],
//   y_m[r] = e^{G_m} (S_h q_m)[r] + sum_{m'<=m} Y[m][m'] u_{m'}[r],
// A[m][m'] = beta_m e^{G_m - G_m'} (k_m . k_m'), Y[m][m'] = e^{G_m - G_m'} (k_m' . q_m).
// The precompute kernel forms every scalar (abar, e^{G_m}, beta_m, A, Y) and
// the buffer vectors sum_j w_j (k_j . x_v) u_j per value head, appends the
// drafts' k and g, and leaves them in the workspace.  The streaming kernel
// brings its block of S_0 rows into shared memory with one bulk copy, forms
// S_0 x_v for all window vectors, solves its rows, writes y and the drafts'
// u, and -- for a fused decode step whose buffer fills -- folds all L entries
// into its rows of S_0.  Decode is the
// T = 1 window with the pointers advanced.
#include "kernels.cuh"

namespace rssm {

namespace {

constexpr int kInfoValid = 1 << 16;

constexpr int kInfoFold = 1 << 17;

__device__ __forceinline__ int wrapL(int s, int L) { return s >= L ? s - L : s; }

template <typename T>
__device__ __forceinline__ float round_as(float x);
template <>
__device__ __forceinline__ float round_as<float>(float x) { return x; }
template <>
__device__ __forceinline__ float round_as<bf16>(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// ---------------------------------------------------------------------------
// precompute: one CTA per (sequence, key head), one warp per value head
// ---------------------------------------------------------------------------
// Window widths up to this read the committed u entries from global memory
// in the precompute (several in flight per lane) instead of staging the u
// rings in shared memory: more precompute blocks fit on an SM.  Width 8
// stages them (its 16 accumulators per row leave no registers to spare).
constexpr int kUGlobalMaxP = 4;

// Byte offsets in shared memory.  The first five parts are filled by bulk
// copies (each 16-byte sized and aligned); the rest is scratch.
struct GPrepSmem {
  uint32_t k_ring, u_ring, g_ring, k_in, q_in, copied_end, dots, kk, coef, total;
  __host__ __device__ GPrepSmem(int L, int N, int dv, int HpK, int P, int es, int eu) {
    k_ring = 0;
    u_ring = k_ring + L * N * es;
    g_ring = u_ring + (P > kUGlobalMaxP ? HpK * L * dv * eu : 0);  // narrow windows read u from global memory
    k_in = g_ring + HpK * L * 4;
    q_in = k_in + P * N * es;
    copied_end = q_in + P * N * es;
    dots = copied_end;               // float [2P][kMaxL]: k_j . x_v, committed j
    kk = dots + 2 * P * kMaxL * 4;   // float [P][2P]: k_m . x_v, drafts m
    coef = kk + P * 2 * P * 4;       // float [HpK][2P][kMaxL]: w_j (k_j . x_v)
    total = coef + HpK * 2 * P * kMaxL * 4;
  }
};

template <int N, int NT, bool kDecode, bool kFuse, typename TI, typename TU>
__global__ void __launch_bounds__(1024) gdn_prep_kernel(GdnLaunch a, int stride) {
  constexpr int LPR = N / 4;
  constexpr int NV = 2 * NT;
  constexpr int es = sizeof(TI), eu = sizeof(TU);
  extern __shared__ __align__(128) unsigned char psm[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_ptr[2];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int HpK = a.Hv / a.Hk;
  const int b = blockIdx.x / a.Hk, kh = blockIdx.x - b * a.Hk;
  const int i = kh * HpK + w;  // this warp's value head
  const int dv = a.dv, L = a.L;
  const int T = kDecode ? 1 : a.T;
  const size_t bk = static_cast<size_t>(b) * a.Hk + kh;
  const size_t h0 = static_cast<size_t>(b) * a.Hv + kh * HpK;  // first value head of the group
  const size_t bh = h0 + w;
  const GPrepSmem lay(L, N, dv, HpK, NT, es, eu);

  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    // the g rings first; then this step's k, q and, once the pointers are in,
    // only the committed slots of the k and u rings (they sit at their own
    // slot positions in shared memory)
    mbar_expect_tx(&bar, (lay.k_in - lay.g_ring) + 2u * T * N * es);
    bulk_g2s(psm + lay.g_ring, a.ring_g + h0 * L, lay.k_in - lay.g_ring, &bar);
  }
  // This grid may start while the previous call's streaming grid finishes (it
  // is launched with programmatic serialisation, and a streaming grid lets it
  // start once all its blocks are past their own wait on their precompute):
  // the g rings are final by then (only precompute grids write them), but the
  // pointers, the u ring and the workspace records are not, nor need the
  // inputs be (the caller may pass that grid's output), so everything below
  // waits for that grid.
  pdl_wait();
  // the streaming kernel may start its S_0 loads now; it waits for this grid
  // before it reads the workspace
  pdl_launch_dependents();
  if (tid == 0) {
    for (int m = 0; m < T; ++m) {
      const size_t off = ((static_cast<size_t>(b) * T + m) * a.Hk + kh) * N * es;
      bulk_g2s(psm + lay.k_in + m * N * es, static_cast<const unsigned char *>(a.k) + off, N * es, &bar);
      bulk_g2s(psm + lay.q_in + m * N * es, static_cast<const unsigned char *>(a.q) + off, N * es, &bar);
    }
    const int hc = a.count[b], sc = a.start[b];
    s_ptr[0] = hc;
    s_ptr[1] = sc;
    if (hc >= 1 && hc <= L && sc >= 0 && sc < L) {
      const int n1 = min(hc, L - sc), n2 = hc - n1;
      mbar_expect_tx(&bar, static_cast<uint32_t>(hc) * (N * es + (NT > kUGlobalMaxP ? HpK * dv * eu : 0)));
      const unsigned char *gk = static_cast<const unsigned char *>(a.ring_k) + bk * L * N * es;
      bulk_g2s(psm + lay.k_ring + sc * N * es, gk + static_cast<size_t>(sc) * N * es, n1 * N * es, &bar);
      if (n2 > 0) bulk_g2s(psm + lay.k_ring, gk, n2 * N * es, &bar);
      if (NT > kUGlobalMaxP)  // wider windows stage the u rings; narrow ones read them from global memory
      for (int hw = 0; hw < HpK; ++hw) {
        const unsigned char *gu = static_cast<const unsigned char *>(a.ring_u) + (h0 + hw) * L * dv * eu;
        unsigned char *su = psm + lay.u_ring + static_cast<size_t>(hw) * L * dv * eu;
        bulk_g2s(su + static_cast<size_t>(sc) * dv * eu, gu + static_cast<size_t>(sc) * dv * eu, n1 * dv * eu, &bar);
        if (n2 > 0) bulk_g2s(su, gu, n2 * dv * eu, &bar);
      }
    }
    mbar_arrive(&bar);
  }
  const size_t tv = (static_cast<size_t>(b) * T + (lane < T ? lane : 0)) * a.Hv + i;  // draft `lane` of this head
  const float g_m = (lane < T) ? a.g[tv] : 0.f;
  const float beta_m = (lane < T) ? a.beta[tv] : 0.f;
  float *wk = a.work + bh * stride;
  __syncthreads();  // barrier initialised, pointers read
  // one warp waits for the copies; the block barrier passes them on to the rest
  bool arrived = true;
  if (w == 0) arrived = mbar_wait_limit(&bar, 0, a.wait_ns);
  if (__syncthreads_or(!arrived)) {
    // give the sequence up: no valid record, so every streaming block of it
    // skips it and its pointers, S_0, ring and y stay as they were
    if (lane == 0) reinterpret_cast<int *>(wk)[kGwInfo] = 0;
    if (tid == 0) {
      set_err(a.err, RSSM_EBIT_TIMEOUT);
      mbar_wait(&bar, 0);  // bounded: the copies must land before shared memory is released
    }
    return;
  }

  const int h = s_ptr[0], st = s_ptr[1];
  const bool ok = kDecode ? (h >= 0 && h < L && st >= 0 && st < L) : (h >= 0 && st >= 0 && st < L && h + T <= L);
  if (!ok) {
    if (lane == 0) reinterpret_cast<int *>(wk)[kGwInfo] = 0;
    if (tid == 0) set_err(a.err, kDecode ? RSSM_EBIT_COUNT_RANGE : RSSM_EBIT_WINDOW);
    return;
  }
  const TI *kring = reinterpret_cast<const TI *>(psm + lay.k_ring);
  const TU *uring = reinterpret_cast<const TU *>(psm + lay.u_ring) + static_cast<size_t>(w) * L * dv;
  const float *gring = reinterpret_cast<const float *>(psm + lay.g_ring) + w * L;
  const TI *kin = reinterpret_cast<const TI *>(psm + lay.k_in);
  const TI *qin = reinterpret_cast<const TI *>(psm + lay.q_in);
  float *sD = reinterpret_cast<float *>(psm + lay.dots);
  float *sK = reinterpret_cast<float *>(psm + lay.kk);
  float *scoef = reinterpret_cast<float *>(psm + lay.coef) + w * NV * kMaxL;

  // dots of every key (committed j < h, then drafts m) with every window vector
  // x_v (v < NT: k_v, v >= NT: q_{v-NT}), zero for v past the drafts
  if constexpr (sizeof(TI) == 2) {
    // bf16: D[e][v] on the tensor cores (m16n8k16, fp32 out), one warp per
    // tile of 16 keys x 8 vectors.  Rows past the last key and vectors past
    // the last draft read key 0 and vector 0 and store zero or nothing.
    const int nw = blockDim.x / 32;
    const int ne = h + T, mt_n = (ne + 15) / 16, nt_n = (NV + 7) / 8;
    for (int t = w; t < mt_n * nt_n; t += nw) {
      const int mt = t / nt_n, nt = t - mt * nt_n;
      const int e = mt * 16 + (lane & 15), ec = e < ne ? e : 0;
      const TI *key = ec < h ? kring + static_cast<size_t>(wrapL(st + ec, L)) * N : kin + (ec - h) * N;
      const int v = nt * 8 + (lane & 7), mv = v < NT ? v : v - NT;
      const TI *xv = (v < NV && mv < T) ? (v < NT ? kin : qin) + mv * N : kin;
      const uint32_t aaddr = smem_addr(key + (lane >> 4) * 8);
      const uint32_t baddr = smem_addr(xv + ((lane >> 3) & 1) * 8);
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < N / 16; ++kk) {
        uint32_t af[4], bfr[2];
        ldsm_x4(af, aaddr + kk * 32);
        ldsm_x2(bfr, baddr + kk * 32);
        mma_16816_bf16(c, af, bfr);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int er = mt * 16 + (lane >> 2) + (j >> 1) * 8, vc = nt * 8 + 2 * (lane & 3) + (j & 1);
        const int mvc = vc < NT ? vc : vc - NT;
        if (er < ne && vc < NV) {
          const float x = mvc < T ? c[j] : 0.f;
          if (er < h)
            sD[vc * kMaxL + er] = x;
          else
            sK[(er - h) * NV + vc] = x;
        }
      }
    }
  } else {
    // pairs spread over the lane groups, V of them reduced together
    constexpr int V = LPR >= 4 ? 4 : LPR;
    constexpr int RPW = 32 / LPR;
    const int col = (lane % LPR) * 4;
    const int nw = blockDim.x / 32, grp = lane / LPR;
    const int npair = (h + T) * NV;
    for (int base = w * RPW * V; base < npair; base += nw * RPW * V) {
      float x[V];
#pragma unroll
      for (int m = 0; m < V; ++m) {
        const int pi = base + grp * V + m;
        x[m] = 0.f;
        if (pi < npair) {
          const int e = pi / NV, v = pi - e * NV;
          const int mv = v < NT ? v : v - NT;
          if (mv < T) {
            const TI *key = e < h ? kring + static_cast<size_t>(wrapL(st + e, L)) * N : kin + (e - h) * N;
            x[m] = dot4(load4(key + col), load4((v < NT ? kin : qin) + mv * N + col));
          }
        }
      }
      group_sum_multi<LPR, V>(x, lane);
      const int pi = base + grp * V + (lane % LPR) / (LPR / V);
      if ((lane % (LPR / V)) == 0 && pi < npair) {
        const int e = pi / NV, v = pi - e * NV;
        if (e < h)
          sD[v * kMaxL + e] = x[0];
        else
          sK[(e - h) * NV + v] = x[0];
      }
    }
  }

  // decay of this value head: committed weights w_j = exp(sum_{j<m<h} g_m),
  // abar = exp(sum_{m<h} g_m); drafts' prefix sums G_m
  float wj, abar;
  {
    const float gj = (lane < h) ? gring[wrapL(st + lane, L)] : 0.f;
    float tot;
    const float ex = excl_suffix_sum(gj, lane, tot);
    wj = (lane < h) ? expf(ex) : 0.f;
    abar = expf(tot);
  }
  float G = g_m;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(kFull, G, o);
    if (lane >= o) G += t;
  }
  __syncthreads();  // sD, sK complete

#pragma unroll
  for (int v = 0; v < NV; ++v) scoef[v * kMaxL + lane] = (lane < h) ? wj * sD[v * kMaxL + lane] : 0.f;
  // the window's triangular coefficients
  for (int base = 0; base < NT * NT; base += 32) {
    const int idx = base + lane;
    const int m = idx / NT, mp = idx - m * NT;
    const float Gm = __shfl_sync(kFull, G, m & 31);
    const float Gmp = __shfl_sync(kFull, G, mp & 31);
    const float bm = __shfl_sync(kFull, beta_m, m & 31);
    if (idx < NT * NT) {
      const float Av = (m < T && mp < m) ? bm * expf(Gm - Gmp) * sK[m * NV + mp] : 0.f;
      const float Yv = (m < T && mp <= m) ? expf(Gm - Gmp) * sK[mp * NV + NT + m] : 0.f;
      wk[kGwA + m * kMaxT + mp] = Av;
      wk[kGwY + m * kMaxT + mp] = Yv;
    }
  }
  if (lane < NT) {
    wk[kGwEG + lane] = (lane < T) ? expf(G) : 0.f;
    wk[kGwBeta + lane] = beta_m;
  }
  const float eg0 = expf(__shfl_sync(kFull, G, 0));  // e^{g_t} of a decode step
  const bool fold = kDecode && kFuse && (h + 1 == L);
  if (kDecode && kFuse) wk[kGwW + lane] = (lane < h) ? wj * eg0 : (lane == h ? 1.f : 0.f);
  if (lane == 0) {
    wk[kGwAbar] = abar;
    wk[kGwAbarFold] = abar * eg0;
    reinterpret_cast<int *>(wk)[kGwInfo] = h | (st << 8) | kInfoValid | (fold ? kInfoFold : 0);
  }
  __syncwarp();

  // buffer vectors of this value head: sum_{j<h} w_j (k_j . x_v) u_j[r]
  if constexpr (NT <= kUGlobalMaxP) {
    // u read from global memory, eight entries of four (two for width 4)
    // rows per lane in flight at once
    const TU *gu = static_cast<const TU *>(a.ring_u) + bh * L * dv;
    constexpr int RPL = NT == 1 ? 4 : 2;
    for (int r0 = lane; r0 < dv; r0 += 32 * RPL) {
      float acc[RPL][NV];
#pragma unroll
      for (int m = 0; m < RPL; ++m)
#pragma unroll
        for (int v = 0; v < NV; ++v) acc[m][v] = 0.f;
      for (int j0 = 0; j0 < h; j0 += 8) {
        float uu[8][RPL];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          const int sl = wrapL(st + (j < h ? j : 0), L);
#pragma unroll
          for (int m = 0; m < RPL; ++m) {
            const int r = r0 + 32 * m;
            uu[jj][m] = (j < h && r < dv) ? load1(gu + static_cast<size_t>(sl) * dv + r) : 0.f;
          }
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          if (j < h) {
#pragma unroll
            for (int m = 0; m < RPL; ++m)
#pragma unroll
              for (int v = 0; v < NV; ++v) acc[m][v] = fmaf(scoef[v * kMaxL + j], uu[jj][m], acc[m][v]);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < RPL; ++m) {
        const int r = r0 + 32 * m;
        if (r < dv)
#pragma unroll
          for (int v = 0; v < NV; ++v) wk[kGwBuf + v * dv + r] = acc[m][v];
      }
    }
  } else
  for (int r = lane; r < dv; r += 32) {
    float acc[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[v] = 0.f;
    int sl = st;
    for (int j = 0; j < h; ++j) {
      const float u = load1(uring + static_cast<size_t>(sl) * dv + r);
#pragma unroll
      for (int v = 0; v < NV; ++v) acc[v] = fmaf(scoef[v * kMaxL + j], u, acc[v]);
      if (++sl == L) sl = 0;
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) wk[kGwBuf + v * dv + r] = acc[v];
  }

  // tentative / appended entries: the drafts' k (per key head) and g (per value
  // head)
  if (lane < T) a.ring_g[bh * L + checked_slot(wrapL(st + h + lane, L) % L, L, a.err)] = g_m;
  if (w == 0) {
    for (int m = 0; m < T; ++m) {
      uint32_t *dst =
          reinterpret_cast<uint32_t *>(static_cast<TI *>(a.ring_k) + (bk * L + checked_slot((st + h + m) % L, L, a.err)) * N);
      const uint32_t *src = reinterpret_cast<const uint32_t *>(kin + m * N);
      for (int c = lane; c < N * es / 4; c += 32) dst[c] = src[c];
    }
  }
}

// ---------------------------------------------------------------------------
// stream: one CTA per (sequence, value head, block of CHUNK = 2 HALF rows).
// The first HALF rows come in through registers (streaming 16-byte loads), the
// second HALF through one bulk copy into shared memory, both issued at once,
// so that a block keeps 2 x HALF rows of S_0 in flight and works on the
// register half while the copy lands.
// ---------------------------------------------------------------------------
template <int N>
struct GRows {
  static constexpr int LPR = N / 4;  // lanes per row, four columns each
  static constexpr int RPW = 32 / LPR;
  static constexpr int RPP = kWarps * RPW;
  static constexpr int kPass = 8;
  static constexpr int HALF = kPass * RPP;
  static constexpr int CHUNK = 2 * HALF;
};

// Shared-memory layout of the streaming kernel (floats).
template <int N, int NT>
struct GStreamSmem {
  static constexpr int CHUNK = GRows<N>::CHUNK, HALF = GRows<N>::HALF;
  static constexpr int kSxStride = CHUNK + 4;  // padded: a reduction's lanes store to different banks
  static constexpr size_t tile = 0;                                 // [HALF][N] second half of the rows
  static constexpr size_t sx = tile + size_t(HALF) * N;             // [2NT][kSxStride] S_0 x_v
  static constexpr size_t su = sx + size_t(2 * NT) * kSxStride;     // [CHUNK] this step's u (fold)
  static constexpr size_t hdr = su + CHUNK;                         // [kGwBuf] workspace header
  static constexpr size_t fold = hdr + kGwBuf;                      // [L][CHUNK] u (TU), [L][N] keys (TI)
  static size_t bytes(bool fused, int L, int eu, int es) {
    return 4 * fold + (fused ? size_t(L) * (size_t(CHUNK) * eu + size_t(N) * es) : 0);
  }
  static_assert((sx * 4) % 16 == 0 && (hdr * 4) % 16 == 0 && (fold * 4) % 16 == 0, "16-byte aligned parts");
};

// Partial dots of kPass rows (row0 + p RPP of `rows`, taken from s[]) with the
// window vectors, reduced over each row's lane group; results to sx[v][off + row].
template <int N, int NT>
__device__ __forceinline__ void gdn_row_dots(const float4 (&s)[GRows<N>::kPass], const float4 (&xv)[2 * NT],
                                             float *sx, int off, int row0, int lane) {
  using RM = GRows<N>;
  constexpr int LPR = RM::LPR, RPP = RM::RPP, kPass = RM::kPass;
  constexpr int NV = 2 * NT;
  constexpr int kSxStride = GStreamSmem<N, NT>::kSxStride;
  static_assert(NV <= LPR, "window vectors per lane group");
  constexpr int PB = (kPass * NV <= LPR) ? kPass : LPR / NV;
#pragma unroll
  for (int p0 = 0; p0 < kPass; p0 += PB) {
    float x[PB * NV];
#pragma unroll
    for (int pp = 0; pp < PB; ++pp)
#pragma unroll
      for (int v = 0; v < NV; ++v) x[pp * NV + v] = dot4(s[p0 + pp], xv[v]);
    group_sum_multi<LPR, PB * NV>(x, lane);
    constexpr int SPAN = LPR / (PB * NV);
    const int idx = (lane % LPR) / SPAN;
    const int pp = idx / NV, v = idx - pp * NV;
    if ((lane % SPAN) == 0) sx[v * kSxStride + off + row0 + (p0 + pp) * RPP] = x[0];
  }
}

template <int N, int NT, bool kDecode, bool kFuse, typename TI, typename TU, typename TO>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 4 : (NT == 8 ? 1 : 2)) gdn_stream_kernel(GdnLaunch a, int stride) {
  using RM = GRows<N>;
  using SM = GStreamSmem<N, NT>;
  constexpr int LPR = RM::LPR, RPP = RM::RPP, HALF = RM::HALF, CHUNK = RM::CHUNK, kPass = RM::kPass;
  constexpr int NV = 2 * NT;
  constexpr int kSxStride = SM::kSxStride;
  extern __shared__ __align__(128) float ssm[];
  __shared__ __align__(8) uint64_t bar;
  float *tile = ssm + SM::tile;
  float *sx = ssm + SM::sx;
  float *su = ssm + SM::su;
  float *shdr = ssm + SM::hdr;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rb = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
  const int HpK = a.Hv / a.Hk;
  const int kh = i / HpK;
  const int dv = a.dv, L = a.L;
  const int T = kDecode ? 1 : a.T;
  const int r_base = rb * CHUNK;
  const int rows1 = min(HALF, dv - r_base);
  const int rows2 = max(0, min(HALF, dv - r_base - HALF));
  const size_t bh = static_cast<size_t>(b) * a.Hv + i;
  const size_t bk = static_cast<size_t>(b) * a.Hk + kh;
  const float *wk = a.work + bh * stride;
  const int col = (lane % LPR) * 4;
  const int row0 = warp * RM::RPW + lane / LPR;
  const float *S0 = a.S + (bh * dv + r_base) * N;

  if (tid == 0 && rows2 > 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(rows2) * N * 4);
    bulk_g2s(tile, S0 + static_cast<size_t>(HALF) * N, static_cast<uint32_t>(rows2) * N * 4, &bar);
  }
  float4 s[kPass];
#pragma unroll
  for (int p = 0; p < kPass; ++p) {
    const int rl = row0 + p * RPP;
    s[p] = (rl < rows1) ? ldg_stream4(S0 + static_cast<size_t>(rl) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float4 xv[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int mv = v < NT ? v : v - NT;
    xv[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mv < T)
      xv[v] = load4(static_cast<const TI *>(v < NT ? a.k : a.q) +
                    ((static_cast<size_t>(b) * T + mv) * a.Hk + kh) * N + col);
  }
  pdl_wait();  // the precompute grid has finished: workspace, drafts' k and g, pointers
  // the next call's precompute may start its first copies once every block is
  // past this wait (it waits for this grid before it reads anything this grid
  // writes)
  pdl_launch_dependents();
  // this thread's row of the solve, and the header, fetched before they are needed
  float pk[NT], pq[NT], pv[NT];
  const int rs = r_base + tid;
#pragma unroll
  for (int m = 0; m < NT; ++m) {
    pk[m] = pq[m] = pv[m] = 0.f;
    if (m < T && tid < rows1 + rows2) {
      pk[m] = wk[kGwBuf + m * dv + rs];
      pq[m] = wk[kGwBuf + (NT + m) * dv + rs];
      pv[m] = load1(static_cast<const TI *>(a.v) + ((static_cast<size_t>(b) * T + m) * a.Hv + i) * dv + rs);
    }
  }
  if (tid < kGwBuf) shdr[tid] = wk[tid];
  gdn_row_dots<N, NT>(s, xv, sx, 0, row0, lane);  // the register half
  __syncthreads();  // barrier initialised, header staged
  // one warp waits for the copy; the block barrier passes it on to the rest
  bool arrived = true;
  if (warp == 0 && rows2 > 0) arrived = mbar_wait(&bar, 0);
  if (__syncthreads_or(!arrived)) {
    if (tid == 0) {
      set_err(a.err, RSSM_EBIT_TIMEOUT);
      mbar_wait(&bar, 0);  // bounded: the copy must land before shared memory is released
    }
    return;
  }
  const int info = __float_as_int(shdr[kGwInfo]);
  if (!(info & kInfoValid)) return;
  const int h = info & 0xff, st = (info >> 8) & 0xff;
  if (!rssm_check(st < L && h + T <= L, a.err)) return;
  // outputs and the entries past the committed window are written whatever the
  // other groups' precompute blocks did; a block that changes the sequence's
  // state (S_0 by a fold, the pointers) first makes sure that every group's
  // precompute block finished, so that a sequence given up keeps its state whole
  const float *first = a.work + static_cast<size_t>(b) * a.Hv * stride;
  bool checked = false;
  if (rows2 > 0) {  // the shared-memory half
    float4 t2[kPass];
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int rl = row0 + p * RPP;
      t2[p] = (rl < rows2) ? *reinterpret_cast<const float4 *>(tile + rl * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    gdn_row_dots<N, NT>(t2, xv, sx, HALF, row0, lane);
  }
  __syncthreads();

  // per row: the window's solve, outputs and the drafts' u
  const float abar = shdr[kGwAbar];
  if (tid < CHUNK) {
    float u[NT];
    float u_last = 0.f;
    if (tid < rows1 + rows2) {
      TO *y = static_cast<TO *>(a.y);
      TU *ru = static_cast<TU *>(a.ring_u) + bh * L * dv;
#pragma unroll
      for (int m = 0; m < NT; ++m) {
        u[m] = 0.f;
        if (m < T) {
          const size_t tvm = (static_cast<size_t>(b) * T + m) * a.Hv + i;
          const float Shk = fmaf(abar, sx[m * kSxStride + tid], pk[m]);
          const float Shq = fmaf(abar, sx[(NT + m) * kSxStride + tid], pq[m]);
          const float eG = shdr[kGwEG + m];
          float um = shdr[kGwBeta + m] * (pv[m] - eG * Shk);
#pragma unroll
          for (int mp = 0; mp < m; ++mp) um = fmaf(-shdr[kGwA + m * kMaxT + mp], u[mp], um);
          u[m] = um;
          float ym = eG * Shq;
#pragma unroll
          for (int mp = 0; mp <= m; ++mp) ym = fmaf(shdr[kGwY + m * kMaxT + mp], u[mp], ym);
          store1(y + tvm * dv + rs, ym);
          store1(ru + static_cast<size_t>(checked_slot((st + h + m) % L, L, a.err)) * dv + rs, um);
          u_last = round_as<TU>(um);
        }
      }
    }
    if (kDecode && kFuse) su[tid] = u_last;
  }

  if constexpr (kDecode && kFuse) {
    if ((info & kInfoFold) && sequence_records_valid(first, a.Hk, HpK, stride, kGwInfo, kInfoValid)) {
      checked = true;
      // every slot holds an entry: the L - 1 committed ones and this step's.
      // The block's rows of the u ring and the group's keys are staged raw, in
      // window order j, with copies issued together; this step's u (slot j = h)
      // is taken from su.  The register half of S_0 is read again with all of
      // its loads in flight at once (its registers were released).
      constexpr int es = sizeof(TI), eu = sizeof(TU);
      const int rows = rows1 + rows2;
      unsigned char *ustage = reinterpret_cast<unsigned char *>(ssm + SM::fold);  // [L][CHUNK] TU
      unsigned char *kstage = ustage + static_cast<size_t>(L) * CHUNK * eu;       // [L][N] TI
      const unsigned char *gu =
          reinterpret_cast<const unsigned char *>(static_cast<const TU *>(a.ring_u) + bh * L * dv + r_base);
      const unsigned char *gk = reinterpret_cast<const unsigned char *>(static_cast<const TI *>(a.ring_k) + bk * L * N);
      const int uc = rows * eu / 16, kc = N * es / 16;  // 16-byte chunks per slot
      __syncthreads();  // su complete; every u of this step stored
      for (int idx = tid; idx < L * (uc + kc); idx += kThreads) {
        const int j = idx / (uc + kc), c = idx - j * (uc + kc);
        const int sl = wrapL(st + j, L);
        if (c < uc)
          cp_async16(ustage + (static_cast<size_t>(j) * CHUNK * eu) + c * 16,
                     gu + static_cast<size_t>(sl) * dv * eu + c * 16);
        else
          cp_async16(kstage + static_cast<size_t>(j) * N * es + (c - uc) * 16, gk + static_cast<size_t>(sl) * N * es + (c - uc) * 16);
      }
      cp_async_commit();
      const float af = shdr[kGwAbarFold];
      float4 o[kPass];
#pragma unroll
      for (int p = 0; p < kPass; ++p) {
        const int rl = row0 + p * RPP;
        o[p] = (rl < rows1) ? ldg_stream4(S0 + static_cast<size_t>(rl) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      cp_async_wait_all();
      __syncthreads();
      const TU *us = reinterpret_cast<const TU *>(ustage);
      const TI *ks = reinterpret_cast<const TI *>(kstage);
      float *S0w = a.S + (bh * dv + r_base) * N;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const int off = half * HALF;
        const int lim = half ? rows2 : rows1;
        if (half) {
#pragma unroll
          for (int p = 0; p < kPass; ++p) {
            const int rl = row0 + p * RPP;
            o[p] = (rl < rows2) ? *reinterpret_cast<const float4 *>(tile + rl * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int p = 0; p < kPass; ++p) {
          o[p].x *= af;
          o[p].y *= af;
          o[p].z *= af;
          o[p].w *= af;
        }
#pragma unroll 2
        for (int j = 0; j < L; ++j) {
          const float wj = shdr[kGwW + j];
          const float4 kv = load4(ks + static_cast<size_t>(j) * N + col);
#pragma unroll
          for (int p = 0; p < kPass; ++p) {
            const int rb2 = off + row0 + p * RPP;
            const float uv = (j == h) ? su[rb2] : load1(us + static_cast<size_t>(j) * CHUNK + rb2);
            const float w = wj * uv;
            o[p].x = fmaf(w, kv.x, o[p].x);
            o[p].y = fmaf(w, kv.y, o[p].y);
            o[p].z = fmaf(w, kv.z, o[p].z);
            o[p].w = fmaf(w, kv.w, o[p].w);
          }
        }
#pragma unroll
        for (int p = 0; p < kPass; ++p) {
          const int rl = row0 + p * RPP;
          if (rl < lim) stg_stream4(S0w + static_cast<size_t>(off + rl) * N + col, o[p]);
        }
      }
    }
  }
  if (i == 0 && rb == 0 && warp == 0 &&
      (checked || sequence_records_valid(first, a.Hk, HpK, stride, kGwInfo, kInfoValid)) && lane == 0) {
    // every precompute block has read this sequence's pointers: advance them
    if (kDecode) {
      const int p = h + 1;
      a.count[b] = (kFuse && p == L) ? 0 : p;  // fused: a filled buffer is folded above
      a.flag[b] = (!kFuse && p == L) ? 1 : 0;
    } else {
      a.flag[b] = (h + 2 * T > L) ? 1 : 0;  // early flush, one window ahead
    }
  }
}

template <int N, int NT, bool kDecode, bool kFuse, typename TU, typename TO>
cudaError_t launch_gs(const GdnLaunch &a, cudaStream_t stream) {
  using TI = bf16;
  constexpr int es = sizeof(TI), eu = sizeof(TU);
  constexpr int CHUNK = GRows<N>::CHUNK;
  const int HpK = a.Hv / a.Hk;
  const int stride = gdn_work_stride_floats(a.dv, NT);
  const size_t psm = GPrepSmem(a.L, N, a.dv, HpK, NT, es, eu).total;
  auto prep = gdn_prep_kernel<N, NT, kDecode, kFuse, TI, TU>;
  cudaError_t e;
  if (psm > 48 * 1024 &&
      (e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(psm))) !=
          cudaSuccess)
    return e;
  // programmatic dependent launches: the precompute's first copies overlap the
  // previous streaming grid's tail, and the S_0 stream the precompute's tail
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t pcfg = {};
  pcfg.gridDim = dim3(static_cast<unsigned>(a.B) * a.Hk);
  pcfg.blockDim = dim3(32 * HpK);
  pcfg.dynamicSmemBytes = psm;
  pcfg.stream = stream;
  pcfg.attrs = attr;
  pcfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&pcfg, prep, a, stride)) != cudaSuccess) return e;
  if (!kDecode && gdn_verify_pipe_eligible(a)) return launch_gdn_verify_pipe(a, stride, NT, stream);
  const int nrb = (a.dv + CHUNK - 1) / CHUNK;
  const size_t ssm = GStreamSmem<N, NT>::bytes(kDecode && kFuse, a.L, eu, es);
  auto strm = gdn_stream_kernel<N, NT, kDecode, kFuse, TI, TU, TO>;
  if (ssm > 48 * 1024 &&
      (e = cudaFuncSetAttribute(strm, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ssm))) !=
          cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nrb), static_cast<unsigned>(a.Hv), static_cast<unsigned>(a.B));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = ssm;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, strm, a, stride);
}

template <int N, typename TU, typename TO>
cudaError_t launch_gs_kind(GdnKind kind, const GdnLaunch &a, cudaStream_t stream) {
  if (kind == GdnKind::Decode) return launch_gs<N, 1, true, false, TU, TO>(a, stream);
  if (kind == GdnKind::DecodeFused) return launch_gs<N, 1, true, true, TU, TO>(a, stream);
  switch (gdn_window_width(a.T)) {
    case 1: return launch_gs<N, 1, false, false, TU, TO>(a, stream);
    case 4: return launch_gs<N, 4, false, false, TU, TO>(a, stream);
    default: return launch_gs<N, 8, false, false, TU, TO>(a, stream);
  }
}

template <typename TU, typename TO>
cudaError_t launch_gs_n(GdnKind kind, const GdnLaunch &a, cudaStream_t stream) {
  if (a.dk == 64) return launch_gs_kind<64, TU, TO>(kind, a, stream);
  return launch_gs_kind<128, TU, TO>(kind, a, stream);
}

}  // namespace

bool gdn_split_eligible(GdnKind kind, const GdnLaunch &a) {
  if (kind != GdnKind::Decode && kind != GdnKind::DecodeFused && kind != GdnKind::Verify) return false;
  if (a.in_dtype != RSSM_BF16 || (a.dk != 64 && a.dk != 128)) return false;
  const int T = kind == GdnKind::Verify ? a.T : 1;
  if (T < 1 || T > kMaxT) return false;
  const int P = gdn_window_width(T);
  const int eu = a.u_dtype == RSSM_BF16 ? 2 : 4;
  const int HpK = a.Hv / a.Hk;
  if (HpK > 32 || a.L % 4 != 0 || a.L > kMaxL || (a.dv * eu) % 16 != 0) return false;
  if (a.B > 65535 || a.Hv > 65535) return false;  // grid dimensions of the streaming kernel
  const int64_t need = static_cast<int64_t>(a.B) * a.Hv * gdn_work_stride_floats(a.dv, P) * 4;
  auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (a.work == nullptr || a.work_bytes < need || !a16(a.work)) return false;
  if (GPrepSmem(a.L, a.dk, a.dv, HpK, P, 2, eu).total > 160u * 1024u) return false;
  return a16(a.S) && a16(a.ring_u) && a16(a.ring_k) && a16(a.ring_g) && a16(a.k) && a16(a.q);
}

cudaError_t launch_gdn_split(GdnKind kind, const GdnLaunch &a, cudaStream_t stream) {
  const bool ub = a.u_dtype == RSSM_BF16, yb = a.y_dtype == RSSM_BF16;
  if (ub && yb) return launch_gs_n<bf16, bf16>(kind, a, stream);
  if (ub) return launch_gs_n<bf16, float>(kind, a, stream);
  if (yb) return launch_gs_n<float, bf16>(kind, a, stream);
  return launch_gs_n<float, float>(kind, a, stream);
}

}  // namespace rssm
