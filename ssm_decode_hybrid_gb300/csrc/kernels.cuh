// Launch descriptors and launcher declarations of libreplayssm (internal).
#pragma once

#include "common.cuh"

namespace rssm {

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
  float *work;  // decode workspace (two-launch decode) or null
};

// Floats per (sequence, head) record of the two-launch decode workspace:
// abar, info, two spare words, the L decay weights, the d-row buffer term,
// rounded up to 16 bytes.
__host__ __device__ constexpr int work_stride_floats(int d, int L) { return (4 + L + d + 3) & ~3; }

enum class M2Kind { Baseline, Decode, DecodeFused, Verify, SnapshotVerify };

cudaError_t launch_m2(M2Kind kind, const M2Launch &a, cudaStream_t stream);

// Persistent bulk-copy pipelined decode step (decode_pipe.cu).  Eligible when
// every bulk copy is 16-byte sized and aligned; `launched` reports whether the
// kernel ran (false: the caller falls back to the per-head kernel).
bool m2_decode_pipe_eligible(const M2Launch &a);
// Two launches through the caller's workspace (decode_split.cu): a precompute
// kernel per (sequence, group), then a kernel streaming S_0 per (sequence, head).
bool m2_decode_split_eligible(const M2Launch &a);
cudaError_t launch_m2_decode_split(const M2Launch &a, bool fuse_flush, cudaStream_t stream);
// One CTA per (sequence, head) with every load issued up front (decode_flat.cu).
bool m2_decode_flat_eligible(const M2Launch &a);
cudaError_t launch_m2_decode_flat(const M2Launch &a, bool fuse_flush, cudaStream_t stream);
// fuse_flush: a sequence whose buffer fills is folded into S_0 in the same
// launch (count and flag end at 0) instead of being flagged for replay_flush.
cudaError_t launch_m2_decode_pipe(const M2Launch &a, bool fuse_flush, cudaStream_t stream, bool *launched);
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
};

enum class GdnKind { Baseline, Decode, Verify, SnapshotVerify };

cudaError_t launch_gdn(GdnKind kind, const GdnLaunch &a, cudaStream_t stream);

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
// The tensor-core flush applies (n = 128, bf16 keys, d a multiple of 32).
bool flush_tc_eligible(const FlushLaunch &a);

}  // namespace rssm
