// Launch descriptors and launcher declarations of libreplayssm (internal).
#pragma once

#include <algorithm>
#include <atomic>

#include "common.cuh"

namespace rssm {

// Number of SMs of the current device, looked up once per device.
inline int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Everything a Mamba-2 kernel launch needs, already validated on the host.
struct M2Launch {
  int B, H, G, d, n, L, T;
  int in_dtype, y_dtype;
  float *S;  // S_0 (replay kernels), S (baseline) or the snapshot slots
  void *ring_v, *ring_k;
  float *ring_dt;
  int32_t *start, *count, *flag, *sync, *err;
  const int32_t *cur;  // snapshot baseline
  const void *v, *k, *q;
  const float *dt, *A;
  void *y;
  float *work;         // workspace of the two-launch decode, or null
  int64_t work_bytes;  // its size
  uint64_t wait_ns;    // limit of the precompute kernels' data wait (0: the wait counts as run out)
};

// Floats per (sequence, head) record of the two-launch decode workspace:
// abar, info, two spare words, the L decay weights, the d-row buffer term,
// rounded up to 16 bytes.
__host__ __device__ constexpr int work_stride_floats(int d, int L) { return (4 + L + d + 3) & ~3; }

enum class M2Kind { Baseline, Decode, DecodeFused, Verify, SnapshotVerify };

cudaError_t launch_m2(M2Kind kind, const M2Launch &a, cudaStream_t stream);

// Two launches through the caller's workspace (decode_split.cu): a precompute
// kernel per (sequence, group), then a kernel streaming S_0 per (sequence, head).
bool m2_decode_split_eligible(const M2Launch &a);
cudaError_t launch_m2_decode_split(const M2Launch &a, bool fuse_flush, cudaStream_t stream);
// Speculative verify through the caller's workspace (decode_split.cu): a
// precompute kernel per (sequence, group), then a kernel streaming S_0 per
// (sequence, head) for all T drafts.  Record per (sequence, head): a 16-float
// header (abar_s, info), then P buffer vectors of d rows, P = 1, 4 or 8 >= T.
constexpr int kM2VerifyHeader = 16;
__host__ __device__ constexpr int m2_verify_stride_floats(int d, int P) { return (kM2VerifyHeader + P * d + 3) & ~3; }
bool m2_verify_split_eligible(const M2Launch &a);
cudaError_t launch_m2_verify_split(const M2Launch &a, cudaStream_t stream);
// Its streaming half as the persistent TMA + tcgen05 pipeline
// (verify_pipe.cu): n = 128, d = 64, two heads of a group per item, bf16
// inputs, 5 <= T (fewer queries stay on the CUDA-core stream).
bool m2_verify_pipe_eligible(const M2Launch &a);
cudaError_t launch_m2_verify_pipe(const M2Launch &a, int stride, cudaStream_t stream);
// One CTA per (sequence, head) with every load issued up front (decode_flat.cu).
// fuse_flush (here and in launch_m2_decode_split): a sequence whose buffer
// fills is folded into S_0 in the same launch (count and flag end at 0)
// instead of being flagged for replay_flush.
bool m2_decode_flat_eligible(const M2Launch &a);
cudaError_t launch_m2_decode_flat(const M2Launch &a, bool fuse_flush, cudaStream_t stream);
cudaError_t launch_replay_commit(int B, int T, int L, const int32_t *accepted, int32_t *count, int32_t *err,
                                 cudaStream_t stream);
cudaError_t launch_snapshot_commit(int B, int T, const int32_t *accepted, int32_t *cur, int32_t *err,
                                   cudaStream_t stream);

// Everything a GDN kernel launch needs.
struct GdnLaunch {
  int B, Hv, Hk, dk, dv, L, T;
  int in_dtype, u_dtype, y_dtype;
  float *S;
  void *ring_u, *ring_k;
  float *ring_g;
  int32_t *start, *count, *flag, *sync, *err;
  const int32_t *cur;
  const void *q, *k, *v;
  const float *beta, *g;
  void *y;
  float *work;         // workspace of the two-launch decode / verify, or null
  int64_t work_bytes;  // its size
  uint64_t wait_ns;    // limit of the precompute kernel's data wait (0: the wait counts as run out)
};

enum class GdnKind { Baseline, Decode, DecodeFused, Verify, SnapshotVerify };

// Window width P of the GDN two-launch kernels for a call with T drafts
// (T = 1 also covers decode), and the floats of one (sequence, value head)
// workspace record: a 180-float header of per-head scalars, then the 2P
// buffer-term vectors of dv rows.
__host__ __device__ constexpr int gdn_window_width(int T) { return T <= 1 ? 1 : (T <= 4 ? 4 : 8); }
// Header of a GDN workspace record (written by the precompute kernel of
// gdn_split.cu, read by the streaming kernels), in floats:
constexpr int kGwAbar = 0;                    // exp(sum_{m<h} g_m)
constexpr int kGwInfo = 1;                    // int: h | start << 8 | flags
constexpr int kGwAbarFold = 2;                // abar e^{g_t} (fused decode's fold); slot 3 unused
constexpr int kGwW = 4;                       // [kMaxL] fold weights, window order
constexpr int kGwEG = kGwW + kMaxL;           // [kMaxT] e^{G_m}
constexpr int kGwBeta = kGwEG + kMaxT;        // [kMaxT] beta_m
constexpr int kGwA = kGwBeta + kMaxT;         // [kMaxT][kMaxT] A[m][m'], m' < m
constexpr int kGwY = kGwA + kMaxT * kMaxT;    // [kMaxT][kMaxT] Y[m][m'], m' <= m
constexpr int kGwBuf = kGwY + kMaxT * kMaxT;  // [2P][dv] buffer vectors
constexpr int kGdnWorkHeader = kGwBuf;
__host__ __device__ constexpr int gdn_work_stride_floats(int dv, int P) {
  return (kGdnWorkHeader + 2 * P * dv + 3) & ~3;
}

// Two launches through the caller's workspace (gdn_split.cu): a precompute
// kernel per (sequence, key head), then a kernel streaming S_0 per (sequence,
// value head, row block).  kind: Decode, DecodeFused or Verify.
bool gdn_split_eligible(GdnKind kind, const GdnLaunch &a);
cudaError_t launch_gdn_split(GdnKind kind, const GdnLaunch &a, cudaStream_t stream);
// The streaming half of the two-launch GDN verify as a persistent,
// warp-specialised TMA + tcgen05 pipeline (verify_pipe.cu): dk = dv = 128,
// bf16 inputs, 2 <= T; it reads the records the precompute kernel left for
// window width P.
bool gdn_verify_pipe_eligible(const GdnLaunch &a);
cudaError_t launch_gdn_verify_pipe(const GdnLaunch &a, int stride, int P, cudaStream_t stream);

cudaError_t launch_gdn(GdnKind kind, const GdnLaunch &a, cudaStream_t stream);

// Convolution-state decode step (conv.cu).
struct ConvLaunch {
  int B, dx, dbc, W, io_dtype, silu;
  void *state;
  const void *u;
  const float *weight, *bias;
  void *out_x, *out_b, *out_c;
};
cudaError_t launch_conv_step(const ConvLaunch &a, cudaStream_t stream);

// Flush of either family.  For Mamba-2 the per-entry log decay is A_i * dt_j
// and the folded vector is dt_j * v_j; for GDN the log decay is g_j and the
// vector u_j.
struct FlushLaunch {
  int B, H, G, d, n, L;
  int vec_dtype;  // dtype of ring_vec
  int key_dtype;  // dtype of ring_key
  bool mamba2;    // true: Mamba-2 (ring_ld holds dt, A given); false: GDN (ring_ld holds g)
  float *S0;
  const void *ring_vec;  // [B][H][L][d]
  const void *ring_key;  // [B][G][L][n]
  const float *ring_ld;  // [B][H][L]
  const float *A;        // [H] (Mamba-2 only)
  int32_t *start, *count, *flag, *sync, *err;
  int num_sms;
};

cudaError_t launch_flush(const FlushLaunch &a, cudaStream_t stream);
// The flush as a persistent TMA + tcgen05 pipeline (flush_pipe.cu): n = 128,
// bf16 keys, d = 64 or 128, L <= 16.
bool flush_pipe_eligible(const FlushLaunch &a);
cudaError_t launch_flush_pipe(const FlushLaunch &a, cudaStream_t stream);
// The tensor-core flush applies (n = 128, bf16 keys, d a multiple of 32).
bool flush_tc_eligible(const FlushLaunch &a);

}  // namespace rssm
