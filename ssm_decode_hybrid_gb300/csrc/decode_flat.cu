// ReplaySSM decode step for Mamba-2, one CTA per (sequence, head), every
// load issued up front (sm_103a).
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- "Algorithm: Mamba-2 standard
// decode" (output-only decode; "if the buffer is full, flush") and "Kernel
// design details" (ring buffer with in-kernel indexing).
//
// The step is bound by the read of S_0 (the head's d x n fp32 block).  A CTA
// of 256 threads holds the whole block in registers (each thread eight
// 16-byte row slices, coalesced: n/4 lanes cover a row) and, in the same
// breath, copies ALL L ring slots of the head's v, its group's k and the Delta
// ring into shared memory with 16-byte cp.async -- without first reading the
// sequence's pointers, so the CTA waits for memory once.  Slots outside the
// committed window are read and ignored; they are a few KB next to the 32 KB
// of S_0 and sit in L2 (the previous step wrote them).  Then: decay weights
// (suffix scan in one warp), k_j^T q (multi-value shuffle reductions), S_0 q
// from the registers, the buffer term with four threads per row, y and the
// appended entry.  With the flush fused, a head whose buffer fills folds
// S_0 <- abar S_0 + sum_j s_j v_j k_j^T from the registers and writes it back.
// Four CTAs fit an SM, so loads of some overlap the arithmetic of others.
#include "kernels.cuh"

namespace rssm {

namespace {

constexpr int kFlatPass = 8;  // row slices per thread

template <int N, bool kFuse, typename TI, typename TO>
__global__ void __launch_bounds__(kThreads, 4) m2_decode_flat_kernel(M2Launch a) {
  constexpr int LPR = N / 4, RPW = 32 / LPR, RPP = kWarps * RPW;
  constexpr int es = sizeof(TI);
  constexpr int kc = N * es / 16;  // 16-byte chunks per key row
  extern __shared__ __align__(16) unsigned char fsm[];
  __shared__ float s_wt[kMaxL], s_c[kMaxL];
  __shared__ int s_slot[kMaxL];
  __shared__ float s_abar;
  __shared__ int s_ptr[2];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.H, i = blockIdx.x - b * a.H;
  const int HpG = a.H / a.G, g = i / HpG;
  const int d = a.d, L = a.L;
  const int vc = d * es / 16;  // 16-byte chunks per value row
  const size_t bh = static_cast<size_t>(b) * a.H + i;
  const size_t bg = static_cast<size_t>(b) * a.G + g;
  const int col = (lane % LPR) * 4;
  const int row0 = warp * RPW + lane / LPR;

  // shared layout: [L][d] v ring | [L][N] k ring | [L] Delta ring | v | k | q | [d] S_0 q
  unsigned char *sv = fsm;
  unsigned char *sk = sv + static_cast<size_t>(L) * d * es;
  float *sdt = reinterpret_cast<float *>(sk + static_cast<size_t>(L) * N * es);
  unsigned char *svin = reinterpret_cast<unsigned char *>(sdt + L);
  unsigned char *skin = svin + static_cast<size_t>(d) * es;
  unsigned char *sqin = skin + static_cast<size_t>(N) * es;
  float *sdot = reinterpret_cast<float *>(sqin + static_cast<size_t>(N) * es);

  // 1. every load at once: pointers, S_0 into registers, the rest into shared memory
  if (tid == 0) {
    s_ptr[0] = a.count[b];
    s_ptr[1] = a.start[b];
  }
  const float *S0 = a.S + bh * d * N;
  float4 s[kFlatPass];
#pragma unroll
  for (int p = 0; p < kFlatPass; ++p) {
    const int r = row0 + p * RPP;
    s[p] = (r < d) ? ldg_stream4(S0 + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  {
    const unsigned char *gv = static_cast<const unsigned char *>(a.ring_v) + bh * L * d * es;
    const unsigned char *gk = static_cast<const unsigned char *>(a.ring_k) + bg * L * N * es;
    const int nv = L * vc, nk = L * kc, nd = L / 4;
    const int total = nv + nk + nd + vc + 2 * kc;
    for (int idx = tid; idx < total; idx += kThreads) {
      int c = idx;
      if (c < nv) {
        cp_async16(sv + c * 16, gv + c * 16);
        continue;
      }
      c -= nv;
      if (c < nk) {
        cp_async16(sk + c * 16, gk + c * 16);
        continue;
      }
      c -= nk;
      if (c < nd) {
        cp_async16(reinterpret_cast<unsigned char *>(sdt) + c * 16,
                   reinterpret_cast<const unsigned char *>(a.ring_dt + bh * L) + c * 16);
        continue;
      }
      c -= nd;
      if (c < vc) {
        cp_async16(svin + c * 16, static_cast<const unsigned char *>(a.v) + bh * d * es + c * 16);
        continue;
      }
      c -= vc;
      if (c < kc) {
        cp_async16(skin + c * 16, static_cast<const unsigned char *>(a.k) + bg * N * es + c * 16);
        continue;
      }
      c -= kc;
      cp_async16(sqin + c * 16, static_cast<const unsigned char *>(a.q) + bg * N * es + c * 16);
    }
    cp_async_commit();
  }
  const float dt_in = a.dt[bh];
  const float Ai = a.A[i];
  cp_async_wait_all();
  __syncthreads();

  const int h = s_ptr[0], st = s_ptr[1];
  if (h < 0 || h >= L || st < 0 || st >= L) {
    if (tid == 0) set_err(a.err, RSSM_EBIT_COUNT_RANGE);
    return;
  }
  const int p = h + 1;
  if (tid == 0 && last_arrival(a.sync, b, a.H)) {
    a.count[b] = (kFuse && p == L) ? 0 : p;  // fused: a filled buffer is folded by this launch
    a.flag[b] = (!kFuse && p == L) ? 1 : 0;
  }
  const TI *vring = reinterpret_cast<const TI *>(sv);
  const TI *kring = reinterpret_cast<const TI *>(sk);
  const TI *vin = reinterpret_cast<const TI *>(svin);
  const TI *kin = reinterpret_cast<const TI *>(skin);
  const TI *qin = reinterpret_cast<const TI *>(sqin);

  // 2. decay weights (warp 0), k_j^T q (all warps), S_0 q per row (all warps)
  const float4 q4 = load4(qin + col);
  if (warp == 0) {
    const int slot = (st + lane) % L;
    const float dtj = (lane < h) ? sdt[slot] : (lane == h ? dt_in : 0.f);
    float tot;
    const float ex = excl_suffix_sum(Ai * dtj, lane, tot);
    s_wt[lane] = (lane < p) ? dtj * expf(ex) : 0.f;
    s_slot[lane] = slot;
    if (lane == 0) s_abar = expf(tot);
  }
  if constexpr (LPR == 32) {
    float x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = warp + kWarps * u;
      x[u] = 0.f;
      if (j < p) x[u] = dot4(load4((j < h ? kring + static_cast<size_t>((st + j) % L) * N : kin) + col), q4);
    }
    group_sum_multi<32, 4>(x, lane);
    const int j = warp + kWarps * (lane >> 3);
    if ((lane & 7) == 0 && j < p) s_c[j] = x[0];
  } else {
    for (int jb = warp * RPW; jb < p; jb += RPP) {
      const int j = jb + lane / LPR;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < p) kv = load4((j < h ? kring + static_cast<size_t>((st + j) % L) * N : kin) + col);
      const float m = group_sum<LPR>(dot4(kv, q4));
      if (j < p && (lane % LPR) == 0) s_c[j] = m;
    }
  }
  {
    float x[kFlatPass];
#pragma unroll
    for (int pp = 0; pp < kFlatPass; ++pp) x[pp] = dot4(s[pp], q4);
    if constexpr (kFlatPass <= LPR) {
      group_sum_multi<LPR, kFlatPass>(x, lane);
      constexpr int SPAN = LPR / kFlatPass;
      const int r = row0 + ((lane % LPR) / SPAN) * RPP;
      if ((lane % SPAN) == 0 && r < d) sdot[r] = x[0];
    } else {
#pragma unroll
      for (int pp = 0; pp < kFlatPass; ++pp) {
        const float t = group_sum<LPR>(x[pp]);
        const int r = row0 + pp * RPP;
        if ((lane % LPR) == 0 && r < d) sdot[r] = t;
      }
    }
  }
  __syncthreads();
  if (tid < p) s_c[tid] *= s_wt[tid];  // c_j = w_j (k_j^T q)
  __syncthreads();

  // 3. y = abar (S_0 q) + sum_j c_j v_j with four threads per row; appended entry
  const float abar = s_abar;
  TO *y = static_cast<TO *>(a.y) + bh * d;
  const int slot_new = checked_slot((st + h) % L, L, a.err);
  TI *rv_out = static_cast<TI *>(a.ring_v) + (bh * L + slot_new) * d;
  for (int rb = 0; rb < d; rb += kThreads / 4) {
    const int r = rb + (tid >> 2), part = tid & 3;
    float acc = 0.f;
    if (r < d) {
      for (int j = part; j < p; j += 4)
        acc = fmaf(s_c[j], load1((j < h ? vring + static_cast<size_t>(s_slot[j]) * d : vin) + r), acc);
    }
    acc += __shfl_xor_sync(kFull, acc, 1);
    acc += __shfl_xor_sync(kFull, acc, 2);
    if (r < d && part == 0) {
      store1(y + r, fmaf(abar, sdot[r], acc));
      rv_out[r] = vin[r];
    }
  }
  if (tid == 0) a.ring_dt[bh * L + slot_new] = dt_in;
  if (i % HpG == 0) {
    TI *rk_out = static_cast<TI *>(a.ring_k) + (bg * L + slot_new) * N;
    for (int c = tid; c < N; c += kThreads) rk_out[c] = kin[c];
  }

  // 4. fused flush: the buffer is full after this append, fold every entry
  // with this step's weights, S_0 <- abar S_0 + sum_j s_j v_j k_j^T, from the
  // registers, and write S_0 back
  if (kFuse && p == L) {
    float *S0w = a.S + bh * d * N;
#pragma unroll
    for (int pp = 0; pp < kFlatPass; ++pp) {
      s[pp].x *= abar;
      s[pp].y *= abar;
      s[pp].z *= abar;
      s[pp].w *= abar;
    }
    for (int j = 0; j < L; ++j) {
      const bool cur = j == h;
      const float4 kv = load4((cur ? kin : kring + static_cast<size_t>(s_slot[j]) * N) + col);
      const TI *vj = cur ? vin : vring + static_cast<size_t>(s_slot[j]) * d;
      const float w = s_wt[j];
#pragma unroll
      for (int pp = 0; pp < kFlatPass; ++pp) {
        const int r = row0 + pp * RPP;
        const float wv = (r < d) ? w * load1(vj + r) : 0.f;
        s[pp].x = fmaf(wv, kv.x, s[pp].x);
        s[pp].y = fmaf(wv, kv.y, s[pp].y);
        s[pp].z = fmaf(wv, kv.z, s[pp].z);
        s[pp].w = fmaf(wv, kv.w, s[pp].w);
      }
    }
#pragma unroll
    for (int pp = 0; pp < kFlatPass; ++pp) {
      const int r = row0 + pp * RPP;
      if (r < d) stg_stream4(S0w + static_cast<size_t>(r) * N + col, s[pp]);
    }
  }
}

template <int N, bool kFuse, typename TI, typename TO>
cudaError_t launch_flat_n(const M2Launch &a, cudaStream_t stream) {
  constexpr int es = sizeof(TI);
  const size_t sm = static_cast<size_t>(a.L) * (a.d + N) * es + static_cast<size_t>(a.L) * 4 +
                    static_cast<size_t>(a.d + 2 * N) * es + static_cast<size_t>(a.d) * 4;
  auto kern = m2_decode_flat_kernel<N, kFuse, TI, TO>;
  if (sm > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm));
    if (e != cudaSuccess) return e;
  }
  kern<<<static_cast<unsigned>(a.B) * a.H, kThreads, sm, stream>>>(a);
  return cudaGetLastError();
}

template <bool kFuse, typename TI, typename TO>
cudaError_t launch_flat_t(const M2Launch &a, cudaStream_t stream) {
  switch (a.n) {
    case 16: return launch_flat_n<16, kFuse, TI, TO>(a, stream);
    case 32: return launch_flat_n<32, kFuse, TI, TO>(a, stream);
    case 64: return launch_flat_n<64, kFuse, TI, TO>(a, stream);
    case 128: return launch_flat_n<128, kFuse, TI, TO>(a, stream);
  }
  return cudaErrorInvalidValue;
}

template <bool kFuse>
cudaError_t launch_flat_f(const M2Launch &a, cudaStream_t stream) {
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_F32) return launch_flat_t<kFuse, bf16, float>(a, stream);
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_BF16) return launch_flat_t<kFuse, bf16, bf16>(a, stream);
  if (a.in_dtype == RSSM_F32 && a.y_dtype == RSSM_F32) return launch_flat_t<kFuse, float, float>(a, stream);
  return launch_flat_t<kFuse, float, bf16>(a, stream);
}

}  // namespace

bool m2_decode_flat_eligible(const M2Launch &a) {
  const int es = a.in_dtype == RSSM_BF16 ? 2 : 4;
  const int rpp = kWarps * (128 / a.n);  // rows per pass of the CTA
  auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return a.L % 4 == 0 && (a.d * es) % 16 == 0 && a.d <= kFlatPass * rpp && a16(a.S) && a16(a.ring_v) &&
         a16(a.ring_k) && a16(a.ring_dt) && a16(a.v) && a16(a.k) && a16(a.q);
}

cudaError_t launch_m2_decode_flat(const M2Launch &a, bool fuse_flush, cudaStream_t stream) {
  return fuse_flush ? launch_flat_f<true>(a, stream) : launch_flat_f<false>(a, stream);
}

}  // namespace rssm
