// Flush: fold the committed ring entries of flagged sequences into S_0.
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- "Algorithm: Mamba-2 standard
// decode" (flush: S_0 <- abar S_0 + sum_j s_j v_j k_j^T, clear the buffer) and
// the GDN appendix (same history form with the cached corrections u_j).
//
// CUDA-core version: a persistent grid walks the (sequence, head) items; items
// of unflagged sequences cost one flag read.  For a flagged item the c
// weighted vectors (d floats each) and c keys (n floats each) are staged in
// shared memory, and every thread updates the 16-byte column slices of S_0
// it owns: acc = abar * S_0 + sum_j (w_j v_j[r]) k_j[col..col+3].
#include "kernels.cuh"

namespace rssm {

namespace {

constexpr int kPass = 8;

template <int N, typename TV, typename TK>
__global__ void __launch_bounds__(kThreads) flush_kernel(FlushLaunch a) {
  constexpr int LPR = N / 4, RPW = 32 / LPR, RPP = kWarps * RPW;
  extern __shared__ float smem[];  // [L][d] vectors, then [L][N] keys (f32)
  __shared__ float s_wt[kMaxL];
  __shared__ float s_abar;
  __shared__ int s_ptr[3];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d = a.d, L = a.L;
  const int HpG = a.H / a.G;
  float *s_vec = smem;
  float *s_key = smem + static_cast<size_t>(L) * d;
  const int col = (lane % LPR) * 4;
  const int row0 = warp * RPW + lane / LPR;
  const int items = a.B * a.H;

  for (int w = blockIdx.x; w < items; w += gridDim.x) {
    const int b = w / a.H, i = w - b * a.H;
    if (tid == 0) {
      s_ptr[0] = a.flag[b];
      s_ptr[1] = a.count[b];
      s_ptr[2] = a.start[b];
    }
    __syncthreads();
    const int f = s_ptr[0], c = s_ptr[1], st = s_ptr[2];
    __syncthreads();
    if (f == 0) continue;
    if (c < 0 || c > L || st < 0 || st >= L) {
      if (tid == 0) set_err(a.err, RSSM_EBIT_COUNT_RANGE);
      continue;
    }
    if (tid == 0 && last_arrival(a.sync, b, a.H)) {
      a.start[b] = (st + c) % L;
      a.count[b] = 0;
      a.flag[b] = 0;
    }
    const size_t bh = static_cast<size_t>(b) * a.H + i;
    const size_t bg = static_cast<size_t>(b) * a.G + i / HpG;
    float *S0 = a.S0 + bh * d * N;

    // checkpoint loads for the first chunk go out first
    float4 s[kPass];
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int r = row0 + p * RPP;
      s[p] = (r < d) ? ldg_stream4(S0 + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // weights: lane j < c holds entry j+1
    if (warp == 0) {
      float ld = 0.f;
      if (lane < c) ld = a.ring_ld[bh * L + (st + lane) % L];
      const float la = a.mamba2 ? a.A[i] * ld : ld;
      float total;
      const float ex = excl_suffix_sum(lane < c ? la : 0.f, lane, total);
      if (lane < c) s_wt[lane] = (a.mamba2 ? ld : 1.f) * expf(ex);
      if (lane == 0) s_abar = expf(total);
    }
    const TV *vec = static_cast<const TV *>(a.ring_vec) + bh * L * d;
    for (int idx = tid; idx < c * d; idx += kThreads) {
      const int j = idx / d, r = idx - j * d;
      s_vec[idx] = load1(vec + static_cast<size_t>((st + j) % L) * d + r);
    }
    const TK *key = static_cast<const TK *>(a.ring_key) + bg * L * N;
    for (int idx = tid; idx < c * (N / 4); idx += kThreads) {
      const int j = idx / (N / 4), c4 = (idx - j * (N / 4)) * 4;
      store4(s_key + j * N + c4, load4(key + static_cast<size_t>((st + j) % L) * N + c4));
    }
    __syncthreads();
    const float abar = s_abar;
    for (int base = 0; base < d; base += kPass * RPP) {
      if (base > 0) {
#pragma unroll
        for (int p = 0; p < kPass; ++p) {
          const int r = base + row0 + p * RPP;
          s[p] = (r < d) ? ldg_stream4(S0 + static_cast<size_t>(r) * N + col) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int p = 0; p < kPass; ++p) {
        const int r = base + row0 + p * RPP;
        if (r < d) {
          float4 acc = make_float4(abar * s[p].x, abar * s[p].y, abar * s[p].z, abar * s[p].w);
          for (int j = 0; j < c; ++j) {
            const float wv = s_wt[j] * s_vec[j * d + r];
            const float4 kv = *reinterpret_cast<const float4 *>(s_key + j * N + col);
            acc.x = fmaf(wv, kv.x, acc.x);
            acc.y = fmaf(wv, kv.y, acc.y);
            acc.z = fmaf(wv, kv.z, acc.z);
            acc.w = fmaf(wv, kv.w, acc.w);
          }
          stg_stream4(S0 + static_cast<size_t>(r) * N + col, acc);
        }
      }
    }
    __syncthreads();
  }
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
  const long cap = static_cast<long>(a.num_sms > 0 ? a.num_sms : 148) * 8;
  const unsigned grid = static_cast<unsigned>(items < cap ? items : cap);
  kern<<<grid, kThreads, sm, stream>>>(a);
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

}  // namespace

cudaError_t launch_flush(const FlushLaunch &a, cudaStream_t stream) {
  const bool vb = a.vec_dtype == RSSM_BF16, kb = a.key_dtype == RSSM_BF16;
  if (vb && kb) return launch_flush_t<bf16, bf16>(a, stream);
  if (!vb && kb) return launch_flush_t<float, bf16>(a, stream);
  if (vb && !kb) return launch_flush_t<bf16, float>(a, stream);
  return launch_flush_t<float, float>(a, stream);
}

}  // namespace rssm
