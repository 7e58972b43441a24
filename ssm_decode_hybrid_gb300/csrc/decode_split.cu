// ReplaySSM decode step for Mamba-2 as two launches (sm_103a): a small
// precompute kernel per (sequence, group) and a streaming kernel per
// (sequence, head).
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- "Kernel design details": the
// inner products k_j^T q are shared by the heads of a group and computed once
// per group by a small precompute kernel; the main kernel reads them from a
// staging buffer.  "Algorithm: Mamba-2 standard decode": output-only decode,
// and "if the buffer is full, flush".
//
// Precompute (grid B x G, one warp per head of the group) works on data that
// sits in L2 (the ring entries, this step's inputs): it reads the pointers,
// computes k_j^T q for the group, per head the decay weights w_j and abar
// and the buffer term buf[r] = sum_j w_j (k_j^T q) v_j[r], appends this step's
// entry to the ring, advances the pointers, and leaves per head in the
// caller's workspace: abar, (h, start, flags), w_1..w_L, buf[0..d).
//
// Stream (grid B x H, 256 threads) is then as lean as the baseline kernel:
// each thread loads its eight 16-byte slices of the head's S_0 block, forms
// S_0 q with shuffle reductions and writes y = abar (S_0 q) + buf.  Its CTAs
// live little longer than their loads, so the S_0 stream runs near the HBM
// roofline.  With the flush fused, a head whose buffer filled also reads its
// ring (all L slots, the new entry included) and writes back
// S_0 <- abar S_0 + sum_j w_j v_j k_j^T from the registers.
#include "kernels.cuh"

namespace rssm {

namespace {

constexpr int kInfoValid = 1 << 16;
constexpr int kInfoFold = 1 << 17;

__device__ __forceinline__ int wrapL(int s, int L) { return s >= L ? s - L : s; }

// ---------------------------------------------------------------------------
// precompute: one CTA per (sequence, group), one warp per head of the group
// ---------------------------------------------------------------------------
template <int N, bool kFuse, typename TI>
__global__ void __launch_bounds__(1024) m2_prep_kernel(M2Launch a, int stride) {
  constexpr int LPR = N / 4;
  constexpr int es = sizeof(TI);
  extern __shared__ __align__(16) unsigned char psm[];
  __shared__ float s_M[kMaxL];
  __shared__ int s_ptr[2];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int nthreads = blockDim.x;
  const int HpG = a.H / a.G;
  const int b = blockIdx.x / a.G, g = blockIdx.x - b * a.G;
  const int i = g * HpG + w;  // this warp's head
  const int d = a.d, L = a.L;
  const size_t bg = static_cast<size_t>(b) * a.G + g;
  const size_t bh = static_cast<size_t>(b) * a.H + i;
  const int vc = d * es / 16, kc = N * es / 16;

  // shared: [L][N] group k ring | k | q | per head: [L][d] v ring, v, [L] Delta ring, [32] weights
  unsigned char *sk = psm;
  unsigned char *skin = sk + static_cast<size_t>(L) * N * es;
  unsigned char *sqin = skin + static_cast<size_t>(N) * es;
  unsigned char *shead = sqin + static_cast<size_t>(N) * es;
  const size_t head_bytes = static_cast<size_t>(L) * d * es + static_cast<size_t>(d) * es + L * 4 + kMaxL * 4;
  unsigned char *sv = shead + w * head_bytes;
  unsigned char *svin = sv + static_cast<size_t>(L) * d * es;
  float *sdt = reinterpret_cast<float *>(svin + static_cast<size_t>(d) * es);
  float *swt = sdt + L;

  if (tid == 0) {
    s_ptr[0] = a.count[b];
    s_ptr[1] = a.start[b];
  }
  // all ring slots and this step's inputs, 16 bytes per copy
  {
    const unsigned char *gk = static_cast<const unsigned char *>(a.ring_k) + bg * L * N * es;
    const int ng = L * kc + 2 * kc;
    for (int idx = tid; idx < ng; idx += nthreads) {
      if (idx < L * kc)
        cp_async16(sk + idx * 16, gk + idx * 16);
      else if (idx < L * kc + kc)
        cp_async16(skin + (idx - L * kc) * 16, static_cast<const unsigned char *>(a.k) + bg * N * es + (idx - L * kc) * 16);
      else
        cp_async16(sqin + (idx - L * kc - kc) * 16,
                   static_cast<const unsigned char *>(a.q) + bg * N * es + (idx - L * kc - kc) * 16);
    }
    const unsigned char *gv = static_cast<const unsigned char *>(a.ring_v) + bh * L * d * es;
    const int nh = L * vc + vc + L / 4;
    for (int idx = lane; idx < nh; idx += 32) {
      if (idx < L * vc)
        cp_async16(sv + idx * 16, gv + idx * 16);
      else if (idx < L * vc + vc)
        cp_async16(svin + (idx - L * vc) * 16, static_cast<const unsigned char *>(a.v) + bh * d * es + (idx - L * vc) * 16);
      else
        cp_async16(reinterpret_cast<unsigned char *>(sdt) + (idx - L * vc - vc) * 16,
                   reinterpret_cast<const unsigned char *>(a.ring_dt + bh * L) + (idx - L * vc - vc) * 16);
    }
    cp_async_commit();
  }
  const float dt_in = a.dt[bh];
  const float Ai = a.A[i];
  cp_async_wait_all();
  __syncthreads();

  const int h = s_ptr[0], st = s_ptr[1];
  float *wk = a.work + bh * stride;
  const bool valid = h >= 0 && h < L && st >= 0 && st < L;
  if (!valid) {
    if (lane == 0) reinterpret_cast<int *>(wk)[1] = 0;
    if (tid == 0) set_err(a.err, RSSM_EBIT_COUNT_RANGE);
    return;
  }
  const int p = h + 1;
  if (tid == 0 && last_arrival(a.sync, b, a.G)) {
    a.count[b] = (kFuse && p == L) ? 0 : p;  // fused: a filled buffer is folded by this step
    a.flag[b] = (!kFuse && p == L) ? 1 : 0;
  }
  const TI *kring = reinterpret_cast<const TI *>(sk);
  const TI *kin = reinterpret_cast<const TI *>(skin);
  const TI *qin = reinterpret_cast<const TI *>(sqin);
  const TI *vring = reinterpret_cast<const TI *>(sv);
  const TI *vin = reinterpret_cast<const TI *>(svin);

  // k_j^T q for the group: entries spread over the warps, one lane group per entry
  {
    const int col = (lane % LPR) * 4;
    const float4 q4 = load4(qin + col);
    constexpr int RPW = 32 / LPR;
    const int nw = nthreads / 32;
    for (int jb = w * RPW; jb < p; jb += nw * RPW) {
      const int j = jb + lane / LPR;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < p) kv = load4((j < h ? kring + static_cast<size_t>(wrapL(st + j, L)) * N : kin) + col);
      const float m = group_sum<LPR>(dot4(kv, q4));
      if (j < p && (lane % LPR) == 0) s_M[j] = m;
    }
  }
  // decay weights of this warp's head: w_j = Delta_j exp(A sum_{j<m<p} Delta_m), abar = exp(A sum Delta)
  float abar;
  {
    const int slot = wrapL(st + lane, L);
    const float dtj = (lane < h) ? sdt[slot] : (lane == h ? dt_in : 0.f);
    float tot;
    const float ex = excl_suffix_sum(Ai * dtj, lane, tot);
    swt[lane] = (lane < p) ? dtj * expf(ex) : 0.f;
    abar = expf(tot);
  }
  __syncthreads();

  // buffer term of this head; the workspace record
  for (int r = lane; r < d; r += 32) {
    float acc = s_M[h] * swt[h] * load1(vin + r);
    for (int j = 0; j < h; ++j) acc = fmaf(s_M[j] * swt[j], load1(vring + static_cast<size_t>(wrapL(st + j, L)) * d + r), acc);
    wk[4 + L + r] = acc;
  }
  if (lane < L) wk[4 + lane] = swt[lane];
  if (lane == 0) {
    wk[0] = abar;
    reinterpret_cast<int *>(wk)[1] = h | (st << 8) | kInfoValid | ((kFuse && p == L) ? kInfoFold : 0);
  }
  // append this step's entry at slot (start + h) mod L
  const int slot_new = wrapL(st + h, L);
  TI *rv_out = static_cast<TI *>(a.ring_v) + (bh * L + slot_new) * d;
  for (int r = lane; r < d; r += 32) rv_out[r] = vin[r];
  if (lane == 0) a.ring_dt[bh * L + slot_new] = dt_in;
  if (w == 0) {
    TI *rk_out = static_cast<TI *>(a.ring_k) + (bg * L + slot_new) * N;
    for (int c = lane; c < N; c += 32) rk_out[c] = kin[c];
  }
}

// ---------------------------------------------------------------------------
// stream: one CTA per (sequence, head)
// ---------------------------------------------------------------------------
constexpr int kSPass = 8;

template <int N, bool kFuse, typename TI, typename TO>
__global__ void __launch_bounds__(kThreads, 4) m2_stream_kernel(M2Launch a, int stride) {
  constexpr int LPR = N / 4, RPW = 32 / LPR, RPP = kWarps * RPW;
  constexpr int es = sizeof(TI);
  extern __shared__ __align__(16) unsigned char ssm[];  // fold only: [L][d] v ring, [L][N] k ring
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.H, i = blockIdx.x - b * a.H;
  const int d = a.d, L = a.L;
  const size_t bh = static_cast<size_t>(b) * a.H + i;
  const int col = (lane % LPR) * 4;
  const int row0 = warp * RPW + lane / LPR;
  const float *wk = a.work + bh * stride;

  const float *S0 = a.S + bh * d * N;
  float4 s[kSPass];
#pragma unroll
  for (int p = 0; p < kSPass; ++p) {
    const int r = row0 + p * RPP;
    s[p] = (r < d) ? ldg_stream4(S0 + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int g = i / (a.H / a.G);
  const size_t bg = static_cast<size_t>(b) * a.G + g;
  const float4 q4 = load4(static_cast<const TI *>(a.q) + bg * N + col);
  const int info = reinterpret_cast<const int *>(wk)[1];
  const float abar = wk[0];
  if (!(info & kInfoValid)) return;

  float x[kSPass];
#pragma unroll
  for (int pp = 0; pp < kSPass; ++pp) x[pp] = dot4(s[pp], q4);
  TO *y = static_cast<TO *>(a.y) + bh * d;
  if constexpr (kSPass <= LPR) {
    group_sum_multi<LPR, kSPass>(x, lane);
    constexpr int SPAN = LPR / kSPass;
    const int r = row0 + ((lane % LPR) / SPAN) * RPP;
    if ((lane % SPAN) == 0 && r < d) store1(y + r, fmaf(abar, x[0], wk[4 + L + r]));
  } else {
#pragma unroll
    for (int pp = 0; pp < kSPass; ++pp) {
      const float t = group_sum<LPR>(x[pp]);
      const int r = row0 + pp * RPP;
      if ((lane % LPR) == 0 && r < d) store1(y + r, fmaf(abar, t, wk[4 + L + r]));
    }
  }

  if (kFuse && (info & kInfoFold)) {
    // every slot holds an entry: the L - 1 committed ones and this step's
    const int st = (info >> 8) & 0xff;
    unsigned char *sv = ssm;
    unsigned char *sk = ssm + static_cast<size_t>(L) * d * es;
    const unsigned char *gv = static_cast<const unsigned char *>(a.ring_v) + bh * L * d * es;
    const unsigned char *gk = static_cast<const unsigned char *>(a.ring_k) + bg * L * N * es;
    const int nv = L * d * es / 16, nk = L * N * es / 16;
    for (int idx = tid; idx < nv + nk; idx += kThreads) {
      if (idx < nv)
        cp_async16(sv + idx * 16, gv + idx * 16);
      else
        cp_async16(sk + (idx - nv) * 16, gk + (idx - nv) * 16);
    }
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    const TI *vring = reinterpret_cast<const TI *>(sv);
    const TI *kring = reinterpret_cast<const TI *>(sk);
#pragma unroll
    for (int pp = 0; pp < kSPass; ++pp) {
      s[pp].x *= abar;
      s[pp].y *= abar;
      s[pp].z *= abar;
      s[pp].w *= abar;
    }
    for (int j = 0; j < L; ++j) {
      const int sl = wrapL(st + j, L);
      const float4 kv = load4(kring + static_cast<size_t>(sl) * N + col);
      const TI *vj = vring + static_cast<size_t>(sl) * d;
      const float wj = wk[4 + j];
#pragma unroll
      for (int pp = 0; pp < kSPass; ++pp) {
        const int r = row0 + pp * RPP;
        const float wv = (r < d) ? wj * load1(vj + r) : 0.f;
        s[pp].x = fmaf(wv, kv.x, s[pp].x);
        s[pp].y = fmaf(wv, kv.y, s[pp].y);
        s[pp].z = fmaf(wv, kv.z, s[pp].z);
        s[pp].w = fmaf(wv, kv.w, s[pp].w);
      }
    }
    float *S0w = a.S + bh * d * N;
#pragma unroll
    for (int pp = 0; pp < kSPass; ++pp) {
      const int r = row0 + pp * RPP;
      if (r < d) stg_stream4(S0w + static_cast<size_t>(r) * N + col, s[pp]);
    }
  }
}

template <int N, bool kFuse, typename TI, typename TO>
cudaError_t launch_split_n(const M2Launch &a, cudaStream_t stream) {
  constexpr int es = sizeof(TI);
  const int HpG = a.H / a.G;
  const int stride = work_stride_floats(a.d, a.L);
  const size_t head_bytes = static_cast<size_t>(a.L) * a.d * es + static_cast<size_t>(a.d) * es + a.L * 4 + kMaxL * 4;
  const size_t psm = static_cast<size_t>(a.L) * N * es + 2u * N * es + HpG * head_bytes;
  auto prep = m2_prep_kernel<N, kFuse, TI>;
  cudaError_t e;
  if (psm > 48 * 1024 &&
      (e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(psm))) !=
          cudaSuccess)
    return e;
  prep<<<static_cast<unsigned>(a.B) * a.G, 32 * HpG, psm, stream>>>(a, stride);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t ssm = kFuse ? static_cast<size_t>(a.L) * (a.d + N) * es : 0;
  auto strm = m2_stream_kernel<N, kFuse, TI, TO>;
  if (ssm > 48 * 1024 &&
      (e = cudaFuncSetAttribute(strm, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ssm))) !=
          cudaSuccess)
    return e;
  strm<<<static_cast<unsigned>(a.B) * a.H, kThreads, ssm, stream>>>(a, stride);
  return cudaGetLastError();
}

template <bool kFuse, typename TI, typename TO>
cudaError_t launch_split_t(const M2Launch &a, cudaStream_t stream) {
  switch (a.n) {
    case 16: return launch_split_n<16, kFuse, TI, TO>(a, stream);
    case 32: return launch_split_n<32, kFuse, TI, TO>(a, stream);
    case 64: return launch_split_n<64, kFuse, TI, TO>(a, stream);
    case 128: return launch_split_n<128, kFuse, TI, TO>(a, stream);
  }
  return cudaErrorInvalidValue;
}

template <bool kFuse>
cudaError_t launch_split_f(const M2Launch &a, cudaStream_t stream) {
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_F32) return launch_split_t<kFuse, bf16, float>(a, stream);
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_BF16) return launch_split_t<kFuse, bf16, bf16>(a, stream);
  if (a.in_dtype == RSSM_F32 && a.y_dtype == RSSM_F32) return launch_split_t<kFuse, float, float>(a, stream);
  return launch_split_t<kFuse, float, bf16>(a, stream);
}

}  // namespace

bool m2_decode_split_eligible(const M2Launch &a) {
  const int es = a.in_dtype == RSSM_BF16 ? 2 : 4;
  const int rpp = kWarps * (128 / a.n);
  const int HpG = a.H / a.G;
  auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const size_t psm = static_cast<size_t>(a.L) * a.n * es + 2u * a.n * es +
                     static_cast<size_t>(HpG) * (static_cast<size_t>(a.L + 1) * a.d * es + a.L * 4 + kMaxL * 4);
  return a.work != nullptr && a16(a.work) && HpG <= 32 && psm <= 160 * 1024 && a.L % 4 == 0 && a.L <= 255 &&
         (a.d * es) % 16 == 0 &&
         a.d <= kSPass * rpp && a16(a.S) && a16(a.ring_v) && a16(a.ring_k) && a16(a.ring_dt) && a16(a.v) &&
         a16(a.k) && a16(a.q);
}

cudaError_t launch_m2_decode_split(const M2Launch &a, bool fuse_flush, cudaStream_t stream) {
  return fuse_flush ? launch_split_f<true>(a, stream) : launch_split_f<false>(a, stream);
}

}  // namespace rssm
