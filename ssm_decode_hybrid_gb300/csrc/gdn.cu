// Gated DeltaNet decode kernels: baseline state update, ReplaySSM decode and
// chunked speculative verify, and the per-draft snapshot baseline.
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- appendix "GDN: standard decode"
// (cache the correction u; S_h from the decayed checkpoint plus the buffer)
// and "GDN: speculative decoding" (the window unrolls into
// u_s = R_s - sum_{s'<s} A_{s,s'} u_{s'}, a T x T lower-triangular solve).
//
// One CTA of 256 threads per (sequence, value head).  The replay kernels never
// build S_h: S_h x = abar (S_0 x) + sum_j w_j u_j (k_j . x) for x in the
// window's keys and queries, the output-only association, which is exact in
// real arithmetic and reads S_0 once for all 2T vectors.  The decode step is
// the T = 1 case with the pointers advanced by one.
#include "kernels.cuh"

namespace rssm {

namespace {

constexpr int kPass = 8;

template <int N>
struct RowMap {
  static constexpr int LPR = N / 4;
  static constexpr int RPW = 32 / LPR;
  static constexpr int RPP = kWarps * RPW;
  static constexpr int CHUNK = kPass * RPP;
};

// ---------------------------------------------------------------------------
// Baseline: alpha = e^g; u = beta (v - alpha S k); S <- alpha S + u k^T; y = S q
// ---------------------------------------------------------------------------
template <int N, typename TI, typename TO>
__global__ void __launch_bounds__(kThreads) gdn_baseline_kernel(GdnLaunch a) {
  using M = RowMap<N>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.Hv, i = blockIdx.x - b * a.Hv;
  const int kh = i / (a.Hv / a.Hk);
  const int dv = a.dv;
  float *S = a.S + static_cast<size_t>(blockIdx.x) * dv * N;
  const int col = (lane % M::LPR) * 4;
  const int row0 = warp * M::RPW + lane / M::LPR;
  const size_t bh = static_cast<size_t>(b) * a.Hv + i;
  const size_t bk = static_cast<size_t>(b) * a.Hk + kh;
  const float alpha = expf(a.g[bh]);
  const float beta = a.beta[bh];
  const float4 k4 = load4(static_cast<const TI *>(a.k) + bk * N + col);
  const float4 q4 = load4(static_cast<const TI *>(a.q) + bk * N + col);
  const float kq = group_sum<M::LPR>(dot4(k4, q4));  // k . q, in every lane
  const TI *v = static_cast<const TI *>(a.v) + bh * dv;
  TO *y = static_cast<TO *>(a.y) + bh * dv;

  for (int base = 0; base < dv; base += M::CHUNK) {
    float4 s[kPass];
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int r = base + row0 + p * M::RPP;
      s[p] = (r < dv) ? ldg_stream4(S + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int r = base + row0 + p * M::RPP;
      const float sk = group_sum<M::LPR>(dot4(s[p], k4));
      const float sq = group_sum<M::LPR>(dot4(s[p], q4));
      const float vr = (r < dv) ? load1(v + r) : 0.f;
      const float u = beta * (vr - alpha * sk);
      float4 o;
      o.x = fmaf(alpha, s[p].x, u * k4.x);
      o.y = fmaf(alpha, s[p].y, u * k4.y);
      o.z = fmaf(alpha, s[p].z, u * k4.z);
      o.w = fmaf(alpha, s[p].w, u * k4.w);
      if (r < dv) {
        stg_stream4(S + static_cast<size_t>(r) * N + col, o);
        if ((lane % M::LPR) == 0) store1(y + r, fmaf(alpha, sq, u * kq));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Replay decode (NT = 1, kDecode) and chunked verify (NT = 4 or 8).
// ---------------------------------------------------------------------------
template <int N, int NT, bool kDecode, typename TI, typename TU, typename TO>
__global__ void __launch_bounds__(kThreads) gdn_replay_kernel(GdnLaunch a) {
  using M = RowMap<N>;
  constexpr int LPR = M::LPR;
  constexpr int NV = 2 * NT;  // vectors dotted with S_0 rows: k_1..k_T, q_1..q_T
  // dynamic smem: [L][dv] buffered u (f32), then [NV][dv] S_h x results
  extern __shared__ float smem[];
  __shared__ float s_c[NV][kMaxL];   // w_j (k_j . x_v) for committed j
  __shared__ float s_w[kMaxL];       // w_j
  __shared__ float s_kx[NT][NV];     // k_s . x_v among the window's own vectors
  __shared__ float s_abar;
  __shared__ float s_G[NT];          // inclusive prefix sums of the drafts' g
  __shared__ int s_ptr[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.Hv, i = blockIdx.x - b * a.Hv;
  const int HpK = a.Hv / a.Hk;
  const int kh = i / HpK;
  const int dv = a.dv, L = a.L;
  const int T = kDecode ? 1 : a.T;
  const float *S0 = a.S + static_cast<size_t>(blockIdx.x) * dv * N;
  const int col = (lane % LPR) * 4;
  const int row0 = warp * M::RPW + lane / LPR;
  const size_t bh = static_cast<size_t>(b) * a.Hv + i;
  const size_t bk = static_cast<size_t>(b) * a.Hk + kh;

  if (tid == 0) {
    s_ptr[0] = a.count[b];
    s_ptr[1] = a.start[b];
  }
  float4 s[kPass];
#pragma unroll
  for (int p = 0; p < kPass; ++p) {
    const int r = row0 + p * M::RPP;
    s[p] = (r < dv) ? ldg_stream4(S0 + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  const int h = s_ptr[0], st = s_ptr[1];
  if (kDecode) {
    if (h < 0 || h >= L || st < 0 || st >= L) {
      if (tid == 0) set_err(a.err, RSSM_EBIT_COUNT_RANGE);
      return;
    }
    if (tid == 0 && last_arrival(a.sync, b, a.Hv)) {
      a.count[b] = h + 1;
      a.flag[b] = (h + 1 == L) ? 1 : 0;
    }
  } else {
    if (h < 0 || st < 0 || st >= L || h + T > L) {
      if (tid == 0) set_err(a.err, RSSM_EBIT_WINDOW);
      return;
    }
    if (tid == 0 && i == 0) a.flag[b] = (h + 2 * T > L) ? 1 : 0;
  }

  // inputs: token m of this round at [b][m] (decode: m = 0, T = 1)
  const TI *qin = static_cast<const TI *>(a.q);
  const TI *kin = static_cast<const TI *>(a.k);
  const TI *vin = static_cast<const TI *>(a.v);
  const size_t tk0 = static_cast<size_t>(b) * T * a.Hk + kh;  // + m*Hk
  const size_t tv0 = static_cast<size_t>(b) * T * a.Hv + i;   // + m*Hv
  const TU *ring_u = static_cast<const TU *>(a.ring_u) + bh * L * dv;
  const TI *ring_k = static_cast<const TI *>(a.ring_k) + bk * L * N;
  const float *ring_g = a.ring_g + bh * L;

  // window vectors x_v: v < T -> k_{v+1}, v >= T -> q_{v-T+1}
  float4 xv[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const int m = v < NT ? v : v - NT;
    xv[v] = (m < T) ? load4((v < NT ? kin : qin) + (tk0 + static_cast<size_t>(m) * a.Hk) * N + col)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // committed u entries -> smem
  for (int idx = tid; idx < h * dv; idx += kThreads) {
    const int j = idx / dv, r = idx - j * dv;
    smem[idx] = load1(ring_u + static_cast<size_t>((st + j) % L) * dv + r);
  }
  // committed decay weights: w_j = exp(sum_{j<m<h} g_m), abar = exp(sum_{m<h} g_m)
  if (warp == 0) {
    const float gj = (lane < h) ? ring_g[(st + lane) % L] : 0.f;
    float total;
    const float ex = excl_suffix_sum(gj, lane, total);
    s_w[lane] = (lane < h) ? expf(ex) : 0.f;
    if (lane == 0) s_abar = expf(total);
  } else if (warp == 1) {
    // prefix sums of the drafts' g (T <= 8 lanes)
    float gm = (lane < T) ? a.g[tv0 + static_cast<size_t>(lane) * a.Hv] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(kFull, gm, o);
      if (lane >= o) gm += t;
    }
    if (lane < NT) s_G[lane] = gm;
  }
  // dots of committed keys with the window vectors: one lane group per entry
  for (int jb = warp * M::RPW; jb < h; jb += M::RPP) {
    const int j = jb + lane / LPR;
    float4 kj = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < h) kj = load4(ring_k + static_cast<size_t>((st + j) % L) * N + col);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const float cv = group_sum<LPR>(dot4(kj, xv[v]));
      if (j < h && (lane % LPR) == 0) s_c[v][j] = cv;
    }
  }
  // dots among the window's own vectors: k_s . x_v (warp s handles k_s)
  for (int m = warp; m < T; m += kWarps) {
    const TI *km = kin + (tk0 + static_cast<size_t>(m) * a.Hk) * N;
    // lanes stride the key in 4-element slices
    float part[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) part[v] = 0.f;
    for (int c4 = lane * 4; c4 < N; c4 += 128) {
      const float4 kk = load4(km + c4);
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const int mm = v < NT ? v : v - NT;
        if (mm < T) {
          const float4 xx = load4((v < NT ? kin : qin) + (tk0 + static_cast<size_t>(mm) * a.Hk) * N + c4);
          part[v] += dot4(kk, xx);
        }
      }
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const float t = group_sum<32>(part[v]);
      if (lane == 0) s_kx[m][v] = t;
    }
  }
  __syncthreads();
  // fold the weights into the dots
  for (int idx = tid; idx < NV * kMaxL; idx += kThreads) {
    const int v = idx / kMaxL, j = idx - v * kMaxL;
    s_c[v][j] = (j < h) ? s_c[v][j] * s_w[j] : 0.f;
  }
  __syncthreads();

  // buffer part of S_h x_v: bufx[v][r] = sum_{j<h} c_{j,v} u_j[r]
  float *s_x = smem + static_cast<size_t>(L) * dv;  // [NV][dv]
  for (int idx = tid; idx < NV * dv; idx += kThreads) {
    const int v = idx / dv, r = idx - v * dv;
    const int m = v < NT ? v : v - NT;
    float acc = 0.f;
    if (m < T)
      for (int j = 0; j < h; ++j) acc = fmaf(s_c[v][j], smem[j * dv + r], acc);
    s_x[idx] = acc;
  }
  __syncthreads();

  // checkpoint part: s_x[v][r] += abar (S_0 x_v)[r]
  const float abar = s_abar;
  constexpr bool kMulti = NV <= LPR;
  for (int base = 0; base < dv; base += M::CHUNK) {
    if (base > 0) {
#pragma unroll
      for (int p = 0; p < kPass; ++p) {
        const int r = base + row0 + p * M::RPP;
        s[p] = (r < dv) ? ldg_stream4(S0 + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int r = base + row0 + p * M::RPP;
      if constexpr (kMulti) {
        float x[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) x[v] = dot4(s[p], xv[v]);
        group_sum_multi<LPR, NV>(x, lane);
        constexpr int SPAN = LPR / NV;
        const int v = (lane % LPR) / SPAN;
        const int m = v < NT ? v : v - NT;
        if (r < dv && (lane % SPAN) == 0 && m < T) s_x[v * dv + r] += abar * x[0];
      } else {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          const float t = group_sum<LPR>(dot4(s[p], xv[v]));
          const int m = v < NT ? v : v - NT;
          if (r < dv && (lane % LPR) == 0 && m < T) s_x[v * dv + r] += abar * t;
        }
      }
    }
  }
  __syncthreads();

  // per row: chunked solve over the window, outputs, tentative ring entries
  TO *y = static_cast<TO *>(a.y);
  TU *ru = static_cast<TU *>(a.ring_u) + bh * L * dv;
  for (int r = tid; r < dv; r += kThreads) {
    float u[NT];
#pragma unroll
    for (int m = 0; m < NT; ++m) {
      if (m < T) {
        const float Gm = s_G[m];
        const float bm = a.beta[tv0 + static_cast<size_t>(m) * a.Hv];
        const float vr = load1(vin + (tv0 + static_cast<size_t>(m) * a.Hv) * dv + r);
        // R_m = beta_m (v_m - e^{G_m} S_h k_m)
        float um = bm * (vr - expf(Gm) * s_x[m * dv + r]);
        // u_m = R_m - sum_{m'<m} A_{m,m'} u_{m'},  A_{m,m'} = beta_m e^{G_m - G_m'} (k_m . k_m')
#pragma unroll
        for (int mp = 0; mp < NT; ++mp)
          if (mp < m) um -= bm * expf(Gm - s_G[mp]) * s_kx[m][mp] * u[mp];
        u[m] = um;
        // y_m = e^{G_m} S_h q_m + sum_{m'<=m} e^{G_m - G_m'} (k_m' . q_m) u_m'
        float ym = expf(Gm) * s_x[(NT + m) * dv + r];
#pragma unroll
        for (int mp = 0; mp < NT; ++mp)
          if (mp <= m) ym = fmaf(expf(Gm - s_G[mp]) * s_kx[mp][NT + m], u[mp], ym);
        store1(y + (tv0 + static_cast<size_t>(m) * a.Hv) * dv + r, ym);
        store1(ru + static_cast<size_t>(checked_slot((st + h + m) % L, L, a.err)) * dv + r, um);
      } else {
        u[m] = 0.f;
      }
    }
  }
  if (tid < T) a.ring_g[bh * L + checked_slot((st + h + tid) % L, L, a.err)] = a.g[tv0 + static_cast<size_t>(tid) * a.Hv];
  if (i % HpK == 0) {
    TI *rk = static_cast<TI *>(a.ring_k) + bk * L * N;
    for (int idx = tid; idx < T * N; idx += kThreads) {
      const int m = idx / N, c = idx - m * N;
      copy1(rk + static_cast<size_t>(checked_slot((st + h + m) % L, L, a.err)) * N + c, kin + (tk0 + static_cast<size_t>(m) * a.Hk) * N + c);
    }
  }
}

// ---------------------------------------------------------------------------
// Baseline speculative verify with per-draft snapshots
// ---------------------------------------------------------------------------
template <int N, typename TI, typename TO>
__global__ void __launch_bounds__(kThreads) gdn_snapshot_verify_kernel(GdnLaunch a) {
  using M = RowMap<N>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.Hv, i = blockIdx.x - b * a.Hv;
  const int kh = i / (a.Hv / a.Hk);
  const int dv = a.dv, T = a.T;
  const int cur = a.cur[b];
  if (cur < 0 || cur > T) {
    if (tid == 0) set_err(a.err, RSSM_EBIT_CUR);
    return;
  }
  const size_t slot_elems = static_cast<size_t>(a.Hv) * dv * N;
  float *slots = a.S + static_cast<size_t>(b) * (T + 1) * slot_elems + static_cast<size_t>(i) * dv * N;
  const int col = (lane % M::LPR) * 4;
  const int row0 = warp * M::RPW + lane / M::LPR;
  const TI *qin = static_cast<const TI *>(a.q);
  const TI *kin = static_cast<const TI *>(a.k);
  const TI *vin = static_cast<const TI *>(a.v);
  TO *y = static_cast<TO *>(a.y);

  for (int base = 0; base < dv; base += M::CHUNK) {
    float4 s[kPass];
    const float *src = slots + static_cast<size_t>(cur) * slot_elems;
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int r = base + row0 + p * M::RPP;
      s[p] = (r < dv) ? ldg_stream4(src + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int m = 0; m < T; ++m) {
      const size_t tvh = (static_cast<size_t>(b) * T + m) * a.Hv + i;
      const size_t tkh = (static_cast<size_t>(b) * T + m) * a.Hk + kh;
      const float alpha = expf(a.g[tvh]);
      const float beta = a.beta[tvh];
      const float4 k4 = load4(kin + tkh * N + col);
      const float4 q4 = load4(qin + tkh * N + col);
      const float kq = group_sum<M::LPR>(dot4(k4, q4));
      float *dst = slots + static_cast<size_t>((cur + m + 1) % (T + 1)) * slot_elems;
#pragma unroll
      for (int p = 0; p < kPass; ++p) {
        const int r = base + row0 + p * M::RPP;
        const float sk = group_sum<M::LPR>(dot4(s[p], k4));
        const float sq = group_sum<M::LPR>(dot4(s[p], q4));
        const float vr = (r < dv) ? load1(vin + tvh * dv + r) : 0.f;
        const float u = beta * (vr - alpha * sk);
        s[p].x = fmaf(alpha, s[p].x, u * k4.x);
        s[p].y = fmaf(alpha, s[p].y, u * k4.y);
        s[p].z = fmaf(alpha, s[p].z, u * k4.z);
        s[p].w = fmaf(alpha, s[p].w, u * k4.w);
        if (r < dv) {
          stg_stream4(dst + static_cast<size_t>(r) * N + col, s[p]);
          if ((lane % M::LPR) == 0) store1(y + tvh * dv + r, fmaf(alpha, sq, u * kq));
        }
      }
    }
  }
}

template <int N, typename TI, typename TU, typename TO>
cudaError_t launch_gdn_n(GdnKind kind, const GdnLaunch &a, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(a.B) * a.Hv);
  switch (kind) {
    case GdnKind::Baseline:
      gdn_baseline_kernel<N, TI, TO><<<grid, kThreads, 0, stream>>>(a);
      break;
    case GdnKind::Decode: {
      const size_t sm = static_cast<size_t>(a.L + 2) * a.dv * sizeof(float);
      gdn_replay_kernel<N, 1, true, TI, TU, TO><<<grid, kThreads, sm, stream>>>(a);
      break;
    }
    case GdnKind::Verify: {
      if (a.T <= 4) {
        const size_t sm = static_cast<size_t>(a.L + 8) * a.dv * sizeof(float);
        auto kern = gdn_replay_kernel<N, 4, false, TI, TU, TO>;
        if (sm > 48 * 1024) {
          cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm));
          if (e != cudaSuccess) return e;
        }
        kern<<<grid, kThreads, sm, stream>>>(a);
      } else {
        const size_t sm = static_cast<size_t>(a.L + 16) * a.dv * sizeof(float);
        auto kern = gdn_replay_kernel<N, 8, false, TI, TU, TO>;
        if (sm > 48 * 1024) {
          cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm));
          if (e != cudaSuccess) return e;
        }
        kern<<<grid, kThreads, sm, stream>>>(a);
      }
      break;
    }
    case GdnKind::SnapshotVerify:
      gdn_snapshot_verify_kernel<N, TI, TO><<<grid, kThreads, 0, stream>>>(a);
      break;
    case GdnKind::DecodeFused:
      return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

template <typename TI, typename TU, typename TO>
cudaError_t launch_gdn_t(GdnKind kind, const GdnLaunch &a, cudaStream_t stream) {
  switch (a.dk) {
    case 16: return launch_gdn_n<16, TI, TU, TO>(kind, a, stream);
    case 32: return launch_gdn_n<32, TI, TU, TO>(kind, a, stream);
    case 64: return launch_gdn_n<64, TI, TU, TO>(kind, a, stream);
    case 128: return launch_gdn_n<128, TI, TU, TO>(kind, a, stream);
  }
  return cudaErrorInvalidValue;
}

template <typename TI, typename TO>
cudaError_t launch_gdn_u(GdnKind kind, const GdnLaunch &a, cudaStream_t stream) {
  if (a.u_dtype == RSSM_BF16) return launch_gdn_t<TI, bf16, TO>(kind, a, stream);
  return launch_gdn_t<TI, float, TO>(kind, a, stream);
}

}  // namespace

cudaError_t launch_gdn(GdnKind kind, const GdnLaunch &a, cudaStream_t stream) {
  if ((kind == GdnKind::Decode || kind == GdnKind::Verify) && gdn_split_eligible(kind, a))
    return launch_gdn_split(kind, a, stream);
  if (kind == GdnKind::DecodeFused) return cudaErrorNotSupported;  // caller: decode, then flush
  if (a.in_dtype == RSSM_F32 && a.y_dtype == RSSM_F32) return launch_gdn_u<float, float>(kind, a, stream);
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_F32) return launch_gdn_u<bf16, float>(kind, a, stream);
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_BF16) return launch_gdn_u<bf16, bf16>(kind, a, stream);
  if (a.in_dtype == RSSM_F32 && a.y_dtype == RSSM_BF16) return launch_gdn_u<float, bf16>(kind, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace rssm
