// Convolution-state decode step (sm_103a): the causal depthwise convolution
// that produces a Mamba-2 layer's x, B and C (the SSM's v, k and q) from the
// in-projection, one token per sequence.
//
// "Disaggregated Serving for Hybrid SSM Models" -- Mamba state layout: each
// sequence keeps a convolution state of shape (conv_dim, state_len) in the
// DS layout (channel-major), conv_dim = |x| + 2 |B|.  Per channel c, with
// the state's W - 1 columns oldest first and the new input u,
//   z = bias[c] + sum_{w < W-1} weight[c][w] state[c][w] + weight[c][W-1] u
//   out = silu(z) (or z), state <- (state[c][1..W-2], u).
// Each thread takes four (sequence, channel) items a grid-stride apart and
// issues all of their loads before any arithmetic; all of it is a few bytes
// per channel, read and written once.
#include "kernels.cuh"

namespace rssm {

namespace {

constexpr int kConvThreads = 256;
constexpr int kConvPer = 4;  // (sequence, channel) items per thread, a grid-stride apart: all loads in flight together

template <typename T, int W>
__global__ void __launch_bounds__(kConvThreads) conv_step_kernel(ConvLaunch a) {
  const int C = a.dx + 2 * a.dbc;
  const int64_t total = static_cast<int64_t>(a.B) * C;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kConvThreads;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kConvThreads + threadIdx.x;
  float win[kConvPer][W], wt[kConvPer][W], z[kConvPer];
  T u[kConvPer];
  // every load first: consecutive threads take consecutive channels, so each
  // load instruction of a warp reads one contiguous span
#pragma unroll
  for (int j = 0; j < kConvPer; ++j) {
    const int64_t idx = i0 + j * stride;
    if (idx < total) {
      const int c = static_cast<int>(idx % C);
      const T *st = static_cast<const T *>(a.state) + idx * (W - 1);
#pragma unroll
      for (int w = 0; w < W - 1; ++w) win[j][w] = load1(st + w);
      u[j] = static_cast<const T *>(a.u)[idx];
#pragma unroll
      for (int w = 0; w < W; ++w) wt[j][w] = a.weight[static_cast<int64_t>(c) * W + w];
      z[j] = a.bias ? a.bias[c] : 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < kConvPer; ++j) {
    const int64_t idx = i0 + j * stride;
    if (idx < total) {
      const int b = static_cast<int>(idx / C), c = static_cast<int>(idx - static_cast<int64_t>(b) * C);
      win[j][W - 1] = load1(&u[j]);
#pragma unroll
      for (int w = 0; w < W; ++w) z[j] = fmaf(wt[j][w], win[j][w], z[j]);
      if (a.silu) z[j] = z[j] / (1.f + expf(-z[j]));
      // shift the state by one column, then u (stored values come back
      // exactly: every one of them was a T value widened to fp32)
      T *st = static_cast<T *>(a.state) + idx * (W - 1);
#pragma unroll
      for (int w = 0; w < W - 2; ++w) store1(st + w, win[j][w + 1]);
      st[W - 2] = u[j];
      T *out;
      int64_t o;
      if (c < a.dx) {
        out = static_cast<T *>(a.out_x);
        o = static_cast<int64_t>(b) * a.dx + c;
      } else if (c < a.dx + a.dbc) {
        out = static_cast<T *>(a.out_b);
        o = static_cast<int64_t>(b) * a.dbc + (c - a.dx);
      } else {
        out = static_cast<T *>(a.out_c);
        o = static_cast<int64_t>(b) * a.dbc + (c - a.dx - a.dbc);
      }
      store1(out + o, z[j]);
    }
  }
}

template <typename T>
cudaError_t launch_conv_t(const ConvLaunch &a, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(a.B) * (a.dx + 2 * a.dbc);
  const int64_t per_block = static_cast<int64_t>(kConvThreads) * kConvPer;
  const unsigned grid = static_cast<unsigned>((n + per_block - 1) / per_block);
  switch (a.W) {
    case 2: conv_step_kernel<T, 2><<<grid, kConvThreads, 0, stream>>>(a); break;
    case 3: conv_step_kernel<T, 3><<<grid, kConvThreads, 0, stream>>>(a); break;
    case 4: conv_step_kernel<T, 4><<<grid, kConvThreads, 0, stream>>>(a); break;
    case 5: conv_step_kernel<T, 5><<<grid, kConvThreads, 0, stream>>>(a); break;
    case 6: conv_step_kernel<T, 6><<<grid, kConvThreads, 0, stream>>>(a); break;
    case 7: conv_step_kernel<T, 7><<<grid, kConvThreads, 0, stream>>>(a); break;
    case 8: conv_step_kernel<T, 8><<<grid, kConvThreads, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv_step(const ConvLaunch &a, cudaStream_t stream) {
  return a.io_dtype == RSSM_BF16 ? launch_conv_t<bf16>(a, stream) : launch_conv_t<float>(a, stream);
}

}  // namespace rssm
