// Mamba-2 decode kernels: baseline state update, ReplaySSM output-only decode,
// speculative verify, commit, and the per-draft snapshot baseline.
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- "Algorithm: Mamba-2 standard
// decode" and "speculative decoding"; ring buffer indexing from "Kernel design
// details".
//
// Work decomposition (all per-head kernels): one CTA of 256 threads per
// (sequence, head).  The head's d x n fp32 block of S_0 (or S) is read with
// coalesced 16-byte loads: a row of n floats is covered by n/4 lanes, so a
// warp covers 128/n rows per load and the CTA 8 * 128/n rows.  Each thread
// issues up to 8 such loads before consuming any of them, so a CTA keeps
// 32 KB of the checkpoint in flight while it fetches the (small) ring entries.
// Dot products along n (S_0 q, k_j^T q) are reduced with warp shuffles.
#include "kernels.cuh"

namespace rssm {

namespace {

constexpr int kPass = 8;  // 16-byte checkpoint loads in flight per thread

template <int N>
struct RowMap {
  static constexpr int LPR = N / 4;        // lanes per row
  static constexpr int RPW = 32 / LPR;     // rows per warp per pass
  static constexpr int RPP = kWarps * RPW;  // rows per CTA per pass
  static constexpr int CHUNK = kPass * RPP;  // rows per chunk of kPass passes
};

// ---------------------------------------------------------------------------
// Baseline: S <- a S + dt v k^T ; y = S q   (one CTA per (b, head))
// ---------------------------------------------------------------------------
template <int N, typename TI, typename TO>
__global__ void __launch_bounds__(kThreads) m2_baseline_kernel(M2Launch a) {
  using M = RowMap<N>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.H, i = blockIdx.x - b * a.H;
  const int g = i / (a.H / a.G);
  const int d = a.d;
  float *S = a.S + static_cast<size_t>(blockIdx.x) * d * N;
  const int col = (lane % M::LPR) * 4;
  const int row0 = warp * M::RPW + lane / M::LPR;
  const size_t bh = static_cast<size_t>(b) * a.H + i;
  const size_t bg = static_cast<size_t>(b) * a.G + g;

  const float dt = a.dt[bh];
  const float decay = expf(a.A[i] * dt);
  const float4 k4 = load4(static_cast<const TI *>(a.k) + bg * N + col);
  const float4 q4 = load4(static_cast<const TI *>(a.q) + bg * N + col);
  const TI *v = static_cast<const TI *>(a.v) + bh * d;
  TO *y = static_cast<TO *>(a.y) + bh * d;

  for (int base = 0; base < d; base += M::CHUNK) {
    float4 s[kPass];
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int r = base + row0 + p * M::RPP;
      s[p] = (r < d) ? ldg_stream4(S + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int r = base + row0 + p * M::RPP;
      const float dv = (r < d) ? dt * load1(v + r) : 0.f;
      float4 o;
      o.x = fmaf(decay, s[p].x, dv * k4.x);
      o.y = fmaf(decay, s[p].y, dv * k4.y);
      o.z = fmaf(decay, s[p].z, dv * k4.z);
      o.w = fmaf(decay, s[p].w, dv * k4.w);
      if (r < d) stg_stream4(S + static_cast<size_t>(r) * N + col, o);
      const float yr = group_sum<M::LPR>(dot4(o, q4));
      if (r < d && (lane % M::LPR) == 0) store1(y + r, yr);
    }
  }
}

// ---------------------------------------------------------------------------
// ReplaySSM decode step / speculative verify (one CTA per (b, head)).
//
// NT = 0: decode step (one query, the current token is entry h+1, pointers
//         advance by one).
// NT > 0: verify of T <= NT drafts (entries h+1..h+T, pointers unchanged,
//         flag <- h + 2T > L).
// ---------------------------------------------------------------------------
template <int N, int NT, typename TI, typename TO>
__global__ void __launch_bounds__(kThreads) m2_replay_kernel(M2Launch a) {
  using M = RowMap<N>;
  constexpr bool kVerify = NT > 0;
  constexpr int Q = kVerify ? NT : 1;  // queries per head
  extern __shared__ float smem[];      // [L][d] buffered v entries as f32, then [Q][d] outputs
  __shared__ float s_coef[Q][kMaxL];   // w_{j,s} (k_j^T q_s), zero for j > p_s
  __shared__ float s_wt[Q][kMaxL];     // w_{j,s}
  __shared__ float s_M[Q][kMaxL];      // k_j^T q_s
  __shared__ float s_abar[Q];
  __shared__ int s_ptr[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.H, i = blockIdx.x - b * a.H;
  const int HpG = a.H / a.G;
  const int g = i / HpG;
  const int d = a.d, L = a.L;
  const int T = kVerify ? a.T : 1;
  const float *S0 = a.S + static_cast<size_t>(blockIdx.x) * d * N;
  const int col = (lane % M::LPR) * 4;
  const int row0 = warp * M::RPW + lane / M::LPR;
  const size_t bh = static_cast<size_t>(b) * a.H + i;
  const size_t bg = static_cast<size_t>(b) * a.G + g;

  // 1. pointers, then the first chunk of checkpoint loads (independent of them)
  if (tid == 0) {
    s_ptr[0] = a.count[b];
    s_ptr[1] = a.start[b];
  }
  float4 s[kPass];
#pragma unroll
  for (int p = 0; p < kPass; ++p) {
    const int r = row0 + p * M::RPP;
    s[p] = (r < d) ? ldg_stream4(S0 + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  const int h = s_ptr[0], st = s_ptr[1];
  if (kVerify) {
    if (h < 0 || st < 0 || st >= L || h + T > L) {
      if (tid == 0) set_err(a.err, RSSM_EBIT_WINDOW);
      return;
    }
    if (tid == 0 && i == 0) a.flag[b] = (h + 2 * T > L) ? 1 : 0;
  } else {
    if (h < 0 || h >= L || st < 0 || st >= L) {
      if (tid == 0) set_err(a.err, RSSM_EBIT_COUNT_RANGE);
      return;
    }
    if (tid == 0 && last_arrival(a.sync, b, a.H)) {
      a.count[b] = h + 1;
      a.flag[b] = (h + 1 == L) ? 1 : 0;
    }
  }
  const int P = h + T;  // entries touched: committed h plus T new ones

  // token m (0-based) of this step's inputs for this head/group
  const TI *vin = static_cast<const TI *>(a.v);
  const TI *kin = static_cast<const TI *>(a.k);
  const TI *qin = static_cast<const TI *>(a.q);
  const size_t in_h = kVerify ? (static_cast<size_t>(b) * T) * a.H + i : bh;  // + m*H
  const size_t in_g = kVerify ? (static_cast<size_t>(b) * T) * a.G + g : bg;  // + m*G
  const TI *ring_v = static_cast<const TI *>(a.ring_v) + bh * L * d;
  const TI *ring_k = static_cast<const TI *>(a.ring_k) + bg * L * N;
  const float *ring_dt = a.ring_dt + bh * L;

  // 2. buffered + new v entries -> smem (f32), coalesced over (j, r)
  for (int idx = tid; idx < P * d; idx += kThreads) {
    const int j = idx / d, r = idx - j * d;
    const TI *src = (j < h) ? ring_v + static_cast<size_t>((st + j) % L) * d + r
                            : vin + (in_h + static_cast<size_t>(j - h) * a.H) * d + r;
    smem[idx] = load1(src);
  }

  // 3. decay weights: warp s handles query s; lane j < p_s is entry j+1
  for (int qs = warp; qs < T; qs += kWarps) {
    const int p = h + (kVerify ? qs + 1 : 1);
    float dtj = 0.f;
    if (lane < p) dtj = (lane < h) ? ring_dt[(st + lane) % L] : a.dt[in_h + static_cast<size_t>(lane - h) * a.H];
    const float la = a.A[i] * dtj;
    float total;
    const float ex = excl_suffix_sum(la, lane, total);
    s_wt[qs][lane] = (lane < p) ? dtj * expf(ex) : 0.f;
    if (lane == 0) s_abar[qs] = expf(total);
  }

  // 4. k_j^T q_s: one lane group of n/4 lanes per entry j
  float4 qv[Q];
#pragma unroll
  for (int qs = 0; qs < Q; ++qs)
    qv[qs] = (qs < T) ? load4(qin + (in_g + static_cast<size_t>(qs) * a.G) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int jb = warp * M::RPW; jb < P; jb += M::RPP) {
    const int j = jb + lane / M::LPR;
    float4 kv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < P) {
      const TI *src = (j < h) ? ring_k + static_cast<size_t>((st + j) % L) * N + col
                              : kin + (in_g + static_cast<size_t>(j - h) * a.G) * N + col;
      kv = load4(src);
    }
#pragma unroll
    for (int qs = 0; qs < Q; ++qs) {
      const float m = group_sum<M::LPR>(dot4(kv, qv[qs]));
      if (j < P && (lane % M::LPR) == 0) s_M[qs][j] = m;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < T * kMaxL; idx += kThreads) {
    const int qs = idx / kMaxL, j = idx - qs * kMaxL;
    const int p = h + (kVerify ? qs + 1 : 1);
    s_coef[qs][j] = (j < p) ? s_wt[qs][j] * s_M[qs][j] : 0.f;
  }
  __syncthreads();

  // 5. buffer term per (query, row): buf[s][r] = sum_{j <= p_s} coef_{j,s} v_j[r]
  float *s_buf = smem + static_cast<size_t>(L) * d;  // [Q][d]
  for (int idx = tid; idx < T * d; idx += kThreads) {
    const int qs = idx / d, r = idx - qs * d;
    const int p_s = h + (kVerify ? qs + 1 : 1);
    float acc = 0.f;
    for (int j = 0; j < p_s; ++j) acc = fmaf(s_coef[qs][j], smem[j * d + r], acc);
    s_buf[idx] = acc;
  }
  __syncthreads();

  // 6. consume the checkpoint: out_s[r] = abar_s (S_0 q_s)[r] + buf[s][r]
  constexpr int LPR = M::LPR;
  constexpr bool kMulti = Q <= LPR;
  for (int base = 0; base < d; base += M::CHUNK) {
    if (base > 0) {
#pragma unroll
      for (int p = 0; p < kPass; ++p) {
        const int r = base + row0 + p * M::RPP;
        s[p] = (r < d) ? ldg_stream4(S0 + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int r = base + row0 + p * M::RPP;
      if constexpr (kMulti) {
        float x[Q];
#pragma unroll
        for (int qs = 0; qs < Q; ++qs) x[qs] = dot4(s[p], qv[qs]);
        group_sum_multi<LPR, Q>(x, lane);
        constexpr int SPAN = LPR / Q;  // lanes holding the same query's total
        const int qs = (lane % LPR) / SPAN;
        if (r < d && (lane % SPAN) == 0 && qs < T) s_buf[qs * d + r] += s_abar[qs] * x[0];
      } else {
#pragma unroll
        for (int qs = 0; qs < Q; ++qs) {
          const float sq = group_sum<LPR>(dot4(s[p], qv[qs]));
          if (r < d && (lane % LPR) == 0 && qs < T) s_buf[qs * d + r] += s_abar[qs] * sq;
        }
      }
    }
  }
  __syncthreads();
  TO *y = static_cast<TO *>(a.y);
  for (int idx = tid; idx < T * d; idx += kThreads) {
    const int qs = idx / d, r = idx - qs * d;
    const size_t yo = kVerify ? ((static_cast<size_t>(b) * T + qs) * a.H + i) * d + r : bh * d + r;
    store1(y + yo, s_buf[idx]);
  }

  // 7. append the new entries to the ring (slots past the committed window)
  TI *rv = static_cast<TI *>(a.ring_v) + bh * L * d;
  for (int idx = tid; idx < T * d; idx += kThreads) {
    const int m = idx / d, r = idx - m * d;
    copy1(rv + static_cast<size_t>(checked_slot((st + h + m) % L, L, a.err)) * d + r, vin + (in_h + static_cast<size_t>(m) * a.H) * d + r);
  }
  if (tid < T) a.ring_dt[bh * L + checked_slot((st + h + tid) % L, L, a.err)] = a.dt[in_h + static_cast<size_t>(tid) * a.H];
  if (i % HpG == 0) {
    TI *rk = static_cast<TI *>(a.ring_k) + bg * L * N;
    for (int idx = tid; idx < T * N; idx += kThreads) {
      const int m = idx / N, c = idx - m * N;
      copy1(rk + static_cast<size_t>(checked_slot((st + h + m) % L, L, a.err)) * N + c, kin + (in_g + static_cast<size_t>(m) * a.G) * N + c);
    }
  }
}

// ---------------------------------------------------------------------------
// Baseline speculative verify with per-draft snapshots (one CTA per (b, head))
// ---------------------------------------------------------------------------
template <int N, typename TI, typename TO>
__global__ void __launch_bounds__(kThreads) m2_snapshot_verify_kernel(M2Launch a) {
  using M = RowMap<N>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.H, i = blockIdx.x - b * a.H;
  const int g = i / (a.H / a.G);
  const int d = a.d, T = a.T;
  const int cur = a.cur[b];
  if (cur < 0 || cur > T) {
    if (tid == 0) set_err(a.err, RSSM_EBIT_CUR);
    return;
  }
  const size_t slot_elems = static_cast<size_t>(a.H) * d * N;
  float *slots = a.S + static_cast<size_t>(b) * (T + 1) * slot_elems + static_cast<size_t>(i) * d * N;
  const int col = (lane % M::LPR) * 4;
  const int row0 = warp * M::RPW + lane / M::LPR;
  const TI *vin = static_cast<const TI *>(a.v);
  const TI *kin = static_cast<const TI *>(a.k);
  const TI *qin = static_cast<const TI *>(a.q);
  TO *y = static_cast<TO *>(a.y);

  for (int base = 0; base < d; base += M::CHUNK) {
    float4 s[kPass];
    const float *src = slots + static_cast<size_t>(cur) * slot_elems;
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int r = base + row0 + p * M::RPP;
      s[p] = (r < d) ? ldg_stream4(src + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int m = 0; m < T; ++m) {
      const size_t th = (static_cast<size_t>(b) * T + m) * a.H + i;
      const size_t tg = (static_cast<size_t>(b) * T + m) * a.G + g;
      const float dt = a.dt[th];
      const float decay = expf(a.A[i] * dt);
      const float4 k4 = load4(kin + tg * N + col);
      const float4 q4 = load4(qin + tg * N + col);
      float *dst = slots + static_cast<size_t>((cur + m + 1) % (T + 1)) * slot_elems;
#pragma unroll
      for (int p = 0; p < kPass; ++p) {
        const int r = base + row0 + p * M::RPP;
        const float dv = (r < d) ? dt * load1(vin + th * d + r) : 0.f;
        s[p].x = fmaf(decay, s[p].x, dv * k4.x);
        s[p].y = fmaf(decay, s[p].y, dv * k4.y);
        s[p].z = fmaf(decay, s[p].z, dv * k4.z);
        s[p].w = fmaf(decay, s[p].w, dv * k4.w);
        if (r < d) stg_stream4(dst + static_cast<size_t>(r) * N + col, s[p]);
        const float yr = group_sum<M::LPR>(dot4(s[p], q4));
        if (r < d && (lane % M::LPR) == 0) store1(y + th * d + r, yr);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Commit kernels (one thread per sequence)
// ---------------------------------------------------------------------------
__global__ void replay_commit_kernel(int B, int T, int L, const int32_t *accepted, int32_t *count, int32_t *err) {
  // launched with programmatic serialisation: scheduled while the previous
  // grid finishes, it reads nothing before that grid has completed
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int acc = accepted[b], c = count[b];
  if (acc < 0 || acc > T || c < 0 || c + acc > L) {
    set_err(err, RSSM_EBIT_ACCEPTED);
    return;
  }
  count[b] = c + acc;
}

__global__ void snapshot_commit_kernel(int B, int T, const int32_t *accepted, int32_t *cur, int32_t *err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int acc = accepted[b], c = cur[b];
  if (acc < 0 || acc > T || c < 0 || c > T) {
    set_err(err, acc < 0 || acc > T ? RSSM_EBIT_ACCEPTED : RSSM_EBIT_CUR);
    return;
  }
  cur[b] = (c + acc) % (T + 1);
}

template <int N, typename TI, typename TO>
cudaError_t launch_m2_n(M2Kind kind, const M2Launch &a, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(a.B) * a.H);
  switch (kind) {
    case M2Kind::Baseline:
      m2_baseline_kernel<N, TI, TO><<<grid, kThreads, 0, stream>>>(a);
      break;
    case M2Kind::Decode: {
      const size_t sm = static_cast<size_t>(a.L + 1) * a.d * sizeof(float);
      m2_replay_kernel<N, 0, TI, TO><<<grid, kThreads, sm, stream>>>(a);
      break;
    }
    case M2Kind::Verify: {
      if (a.T <= 4) {
        const size_t sm = static_cast<size_t>(a.L + 4) * a.d * sizeof(float);
        m2_replay_kernel<N, 4, TI, TO><<<grid, kThreads, sm, stream>>>(a);
      } else {
        const size_t sm = static_cast<size_t>(a.L + 8) * a.d * sizeof(float);
        m2_replay_kernel<N, 8, TI, TO><<<grid, kThreads, sm, stream>>>(a);
      }
      break;
    }
    case M2Kind::SnapshotVerify:
      m2_snapshot_verify_kernel<N, TI, TO><<<grid, kThreads, 0, stream>>>(a);
      break;
  }
  return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_m2_t(M2Kind kind, const M2Launch &a, cudaStream_t stream) {
  switch (a.n) {
    case 16: return launch_m2_n<16, TI, TO>(kind, a, stream);
    case 32: return launch_m2_n<32, TI, TO>(kind, a, stream);
    case 64: return launch_m2_n<64, TI, TO>(kind, a, stream);
    case 128: return launch_m2_n<128, TI, TO>(kind, a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_m2(M2Kind kind, const M2Launch &a, cudaStream_t stream) {
  if (kind == M2Kind::Verify && m2_verify_split_eligible(a)) return launch_m2_verify_split(a, stream);
  if ((kind == M2Kind::Decode || kind == M2Kind::DecodeFused) && m2_decode_split_eligible(a))
    return launch_m2_decode_split(a, kind == M2Kind::DecodeFused, stream);
  if ((kind == M2Kind::Decode || kind == M2Kind::DecodeFused) && m2_decode_flat_eligible(a))
    return launch_m2_decode_flat(a, kind == M2Kind::DecodeFused, stream);
  if (kind == M2Kind::DecodeFused) return cudaErrorNotSupported;  // caller: decode, then flush
  if (a.in_dtype == RSSM_F32 && a.y_dtype == RSSM_F32) return launch_m2_t<float, float>(kind, a, stream);
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_F32) return launch_m2_t<bf16, float>(kind, a, stream);
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_BF16) return launch_m2_t<bf16, bf16>(kind, a, stream);
  if (a.in_dtype == RSSM_F32 && a.y_dtype == RSSM_BF16) return launch_m2_t<float, bf16>(kind, a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_replay_commit(int B, int T, int L, const int32_t *accepted, int32_t *count, int32_t *err,
                                 cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((B + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, replay_commit_kernel, B, T, L, accepted, count, err);
}

cudaError_t launch_snapshot_commit(int B, int T, const int32_t *accepted, int32_t *cur, int32_t *err,
                                   cudaStream_t stream) {
  snapshot_commit_kernel<<<(B + 255) / 256, 256, 0, stream>>>(B, T, accepted, cur, err);
  return cudaGetLastError();
}

}  // namespace rssm
