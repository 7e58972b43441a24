// C-ABI entry points of libreplayssm: argument validation on the host, then
// one kernel launch on the caller's stream.  Nothing here allocates memory or
// synchronises.
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>

#include "kernels.cuh"

namespace {

using namespace rssm;

thread_local char g_last_cuda_error[256] = "";

rssm_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return RSSM_OK;
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return RSSM_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool ok16(const void *p) { return p != nullptr && aligned(p, 16); }
bool ok4(const void *p) { return p != nullptr && aligned(p, 4); }
bool ok_elem(const void *p, int dtype) { return p != nullptr && aligned(p, dtype == RSSM_BF16 ? 2 : 4); }
bool valid_dtype(int t) { return t == RSSM_F32 || t == RSSM_BF16; }
bool supported_n(int n) { return n == 16 || n == 32 || n == 64 || n == 128; }

// Shape checks shared by the Mamba-2 calls.
rssm_status check_m2_dims(const rssm_m2_dims *dm) {
  if (dm == nullptr) return RSSM_ERR_INVALID_ARG;
  const rssm_m2_dims &d = *dm;
  if (d.B < 1 || d.H < 1 || d.G < 1 || d.d < 1 || d.n < 1 || d.L < 1) return RSSM_ERR_INVALID_ARG;
  if (d.H % d.G != 0) return RSSM_ERR_INVALID_ARG;
  if (!valid_dtype(d.in_dtype) || !valid_dtype(d.y_dtype)) return RSSM_ERR_INVALID_ARG;
  if (!supported_n(d.n) || d.d % 4 != 0 || d.d > 256 || d.L > kMaxL) return RSSM_ERR_UNSUPPORTED;
  if (static_cast<long long>(d.B) * d.H > 0x7fffffffLL) return RSSM_ERR_UNSUPPORTED;
  return RSSM_OK;
}

rssm_status check_gdn_dims(const rssm_gdn_dims *dm) {
  if (dm == nullptr) return RSSM_ERR_INVALID_ARG;
  const rssm_gdn_dims &d = *dm;
  if (d.B < 1 || d.Hv < 1 || d.Hk < 1 || d.dk < 1 || d.dv < 1 || d.L < 1) return RSSM_ERR_INVALID_ARG;
  if (d.Hv % d.Hk != 0) return RSSM_ERR_INVALID_ARG;
  if (!valid_dtype(d.in_dtype) || !valid_dtype(d.u_dtype) || !valid_dtype(d.y_dtype)) return RSSM_ERR_INVALID_ARG;
  if (!supported_n(d.dk) || d.dv % 4 != 0 || d.dv > 256 || d.L > kMaxL) return RSSM_ERR_UNSUPPORTED;
  if (static_cast<long long>(d.B) * d.Hv > 0x7fffffffLL) return RSSM_ERR_UNSUPPORTED;
  return RSSM_OK;
}

// Limit of the precompute kernels' data waits: about one second, or the
// value of the environment variable RSSM_WAIT_LIMIT_NS (nanoseconds), read
// at every call.  0 makes every such wait count as run out, which exercises
// the path that gives a sequence up (RSSM_EBIT_TIMEOUT).
uint64_t precompute_wait_ns() {
  const char *e = std::getenv("RSSM_WAIT_LIMIT_NS");
  if (e == nullptr || *e == '\0') return kWaitLimitNs;
  char *end = nullptr;
  const unsigned long long v = std::strtoull(e, &end, 10);
  return (end != nullptr && *end == '\0') ? static_cast<uint64_t>(v) : kWaitLimitNs;
}

M2Launch m2_launch(const rssm_m2_dims &d) {
  M2Launch a;
  std::memset(&a, 0, sizeof(a));
  a.B = d.B;
  a.H = d.H;
  a.G = d.G;
  a.d = d.d;
  a.n = d.n;
  a.L = d.L;
  a.T = 1;
  a.in_dtype = d.in_dtype;
  a.y_dtype = d.y_dtype;
  a.wait_ns = precompute_wait_ns();
  return a;
}

GdnLaunch gdn_launch(const rssm_gdn_dims &d) {
  GdnLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.B = d.B;
  a.Hv = d.Hv;
  a.Hk = d.Hk;
  a.dk = d.dk;
  a.dv = d.dv;
  a.L = d.L;
  a.T = 1;
  a.in_dtype = d.in_dtype;
  a.u_dtype = d.u_dtype;
  a.y_dtype = d.y_dtype;
  a.wait_ns = precompute_wait_ns();
  return a;
}

bool m2_replay_ok(const rssm_m2_dims &d, const rssm_m2_replay *s, bool need_sync) {
  return s != nullptr && ok16(s->S0) && ok_elem(s->ring_v, d.in_dtype) && ok16(s->ring_k) && ok4(s->ring_dt) &&
         ok4(s->start) && ok4(s->count) && ok4(s->flag) && (!need_sync || ok4(s->sync)) &&
         (s->err == nullptr || aligned(s->err, 4)) && (s->work == nullptr || aligned(s->work, 16));
}

bool gdn_replay_ok(const rssm_gdn_dims &d, const rssm_gdn_replay *s, bool need_sync) {
  return s != nullptr && ok16(s->S0) && ok_elem(s->ring_u, d.u_dtype) && ok16(s->ring_k) && ok4(s->ring_g) &&
         ok4(s->start) && ok4(s->count) && ok4(s->flag) && (!need_sync || ok4(s->sync)) &&
         (s->err == nullptr || aligned(s->err, 4)) && (s->work == nullptr || aligned(s->work, 16));
}

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

}  // namespace

extern "C" {

rssm_status conv_state_update(const rssm_conv_dims *dims, void *state, const void *u, const float *weight,
                              const float *bias, void *out_x, void *out_b, void *out_c, rssm_stream_t stream) {
  if (dims == nullptr) return RSSM_ERR_INVALID_ARG;
  const rssm_conv_dims &d = *dims;
  if (d.B < 1 || d.dx < 1 || d.dbc < 0 || d.W < 2 || d.W > 8 || !valid_dtype(d.io_dtype) ||
      (d.silu != 0 && d.silu != 1))
    return RSSM_ERR_INVALID_ARG;
  if (static_cast<long long>(d.B) * (d.dx + 2ll * d.dbc) * d.W > 0x7fffffffLL * 16) return RSSM_ERR_UNSUPPORTED;
  if (!ok_elem(state, d.io_dtype) || !ok_elem(u, d.io_dtype) || !ok4(weight) || (bias && !ok4(bias)) ||
      !ok_elem(out_x, d.io_dtype) || (d.dbc > 0 && (!ok_elem(out_b, d.io_dtype) || !ok_elem(out_c, d.io_dtype))))
    return RSSM_ERR_INVALID_ARG;
  ConvLaunch a;
  a.B = d.B;
  a.dx = d.dx;
  a.dbc = d.dbc;
  a.W = d.W;
  a.io_dtype = d.io_dtype;
  a.silu = d.silu;
  a.state = state;
  a.u = u;
  a.weight = weight;
  a.bias = bias;
  a.out_x = out_x;
  a.out_b = out_b;
  a.out_c = out_c;
  return cuda_status(launch_conv_step(a, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t rssm_version(void) { return 200; }

const char *rssm_status_string(rssm_status s) {
  switch (s) {
    case RSSM_OK: return "ok";
    case RSSM_ERR_INVALID_ARG: return "invalid argument";
    case RSSM_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case RSSM_ERR_CUDA: return "CUDA launch error";
  }
  return "unknown status";
}

const char *rssm_last_cuda_error(void) { return g_last_cuda_error; }

rssm_status rssm_m2_layout_sizes(const rssm_m2_dims *dims, rssm_layout *out) {
  if (out == nullptr) return RSSM_ERR_INVALID_ARG;
  const rssm_status st = check_m2_dims(dims);
  if (st) return st;
  const int64_t B = dims->B;
  out->S0 = B * dims->H * dims->d * dims->n;
  out->ring_vec = B * dims->H * dims->L * dims->d;
  out->ring_k = B * dims->G * dims->L * dims->n;
  out->ring_decay = B * dims->H * dims->L;
  out->per_seq = B;
  return RSSM_OK;
}

rssm_status rssm_gdn_layout_sizes(const rssm_gdn_dims *dims, rssm_layout *out) {
  if (out == nullptr) return RSSM_ERR_INVALID_ARG;
  const rssm_status st = check_gdn_dims(dims);
  if (st) return st;
  const int64_t B = dims->B;
  out->S0 = B * dims->Hv * dims->dv * dims->dk;
  out->ring_vec = B * dims->Hv * dims->L * dims->dv;
  out->ring_k = B * dims->Hk * dims->L * dims->dk;
  out->ring_decay = B * dims->Hv * dims->L;
  out->per_seq = B;
  return RSSM_OK;
}

rssm_status rssm_read_error(const int32_t *err, int32_t *value, rssm_stream_t stream) {
  if (err == nullptr || value == nullptr || !ok4(err)) return RSSM_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(value, err, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

// ------------------------------- Mamba-2 ---------------------------------

int64_t replay_decode_workspace_bytes(const rssm_m2_dims *dims) {
  if (check_m2_dims(dims) != RSSM_OK) return 0;
  return static_cast<int64_t>(dims->B) * dims->H * work_stride_floats(dims->d, dims->L) * 4;
}

int64_t replay_verify_workspace_bytes(const rssm_m2_dims *dims, int32_t T) {
  if (check_m2_dims(dims) != RSSM_OK || T < 1 || T > kMaxT) return 0;
  return static_cast<int64_t>(dims->B) * dims->H * m2_verify_stride_floats(dims->d, gdn_window_width(T)) * 4;
}

// Device bytes one sequence holds per layer, for the concurrency accounting of
// "Results -- speculative decoding" (maximum concurrency at a fixed HBM budget).
int64_t replay_seq_bytes(const rssm_m2_dims *dims, int32_t T, int32_t kind) {
  if (check_m2_dims(dims) != RSSM_OK || T < 0 || T > kMaxT) return 0;
  const rssm_m2_dims &d = *dims;
  const int64_t es = d.in_dtype == RSSM_BF16 ? 2 : 4;
  const int64_t state = 4ll * d.H * d.d * d.n;
  if (kind == RSSM_SEQ_SNAPSHOT) return T == 0 ? state : (T + 1) * state + 4;
  if (kind != RSSM_SEQ_REPLAY) return 0;
  const int64_t ring = static_cast<int64_t>(d.L) * (d.H * d.d * es + d.G * d.n * es + 4ll * d.H);
  int64_t stride = work_stride_floats(d.d, d.L);
  if (T > 0) stride = std::max<int64_t>(stride, m2_verify_stride_floats(d.d, gdn_window_width(T)));
  const int64_t work = 4ll * d.H * stride;
  return state + ring + 4 * 4 + work;
}

int64_t gdn_replay_seq_bytes(const rssm_gdn_dims *dims, int32_t T, int32_t kind) {
  if (check_gdn_dims(dims) != RSSM_OK || T < 0 || T > kMaxT) return 0;
  const rssm_gdn_dims &d = *dims;
  const int64_t es = d.in_dtype == RSSM_BF16 ? 2 : 4, eu = d.u_dtype == RSSM_BF16 ? 2 : 4;
  const int64_t state = 4ll * d.Hv * d.dv * d.dk;
  if (kind == RSSM_SEQ_SNAPSHOT) return T == 0 ? state : (T + 1) * state + 4;
  if (kind != RSSM_SEQ_REPLAY) return 0;
  const int64_t ring = static_cast<int64_t>(d.L) * (d.Hv * d.dv * eu + d.Hk * d.dk * es + 4ll * d.Hv);
  const int64_t work = 4ll * d.Hv * gdn_work_stride_floats(d.dv, gdn_window_width(T < 1 ? 1 : T));
  return state + ring + 4 * 4 + work;
}

rssm_status ssm_state_update_baseline(const rssm_m2_dims *dims, float *S, const void *v, const void *k,
                                      const void *q, const float *dt, const float *A, void *y,
                                      rssm_stream_t stream) {
  rssm_status st = check_m2_dims(dims);
  if (st) return st;
  const rssm_m2_dims &d = *dims;
  if (!ok16(S) || !ok_elem(v, d.in_dtype) || !ok16(k) || !ok16(q) || !ok4(dt) || !ok4(A) || !ok_elem(y, d.y_dtype))
    return RSSM_ERR_INVALID_ARG;
  M2Launch a = m2_launch(d);
  a.S = S;
  a.v = v;
  a.k = k;
  a.q = q;
  a.dt = dt;
  a.A = A;
  a.y = y;
  return cuda_status(launch_m2(M2Kind::Baseline, a, reinterpret_cast<cudaStream_t>(stream)));
}

rssm_status replay_decode_step(const rssm_m2_dims *dims, const rssm_m2_replay *s, const void *v, const void *k,
                               const void *q, const float *dt, const float *A, void *y, rssm_stream_t stream) {
  rssm_status st = check_m2_dims(dims);
  if (st) return st;
  const rssm_m2_dims &d = *dims;
  if (!m2_replay_ok(d, s, true) || !ok_elem(v, d.in_dtype) || !ok16(k) || !ok16(q) || !ok4(dt) || !ok4(A) ||
      !ok_elem(y, d.y_dtype))
    return RSSM_ERR_INVALID_ARG;
  M2Launch a = m2_launch(d);
  a.S = s->S0;
  a.ring_v = s->ring_v;
  a.ring_k = s->ring_k;
  a.ring_dt = s->ring_dt;
  a.start = s->start;
  a.count = s->count;
  a.flag = s->flag;
  a.sync = s->sync;
  a.err = s->err;
  a.v = v;
  a.k = k;
  a.q = q;
  a.dt = dt;
  a.A = A;
  a.y = y;
  a.work = s->work;
  a.work_bytes = s->work_bytes;
  return cuda_status(launch_m2(M2Kind::Decode, a, reinterpret_cast<cudaStream_t>(stream)));
}

static FlushLaunch m2_flush_launch(const rssm_m2_dims &d, const rssm_m2_replay *s, const float *A);

rssm_status replay_decode_step_fused(const rssm_m2_dims *dims, const rssm_m2_replay *s, const void *v,
                                     const void *k, const void *q, const float *dt, const float *A, void *y,
                                     rssm_stream_t stream) {
  rssm_status st = check_m2_dims(dims);
  if (st) return st;
  const rssm_m2_dims &d = *dims;
  if (!m2_replay_ok(d, s, true) || !ok_elem(v, d.in_dtype) || !ok16(k) || !ok16(q) || !ok4(dt) || !ok4(A) ||
      !ok_elem(y, d.y_dtype))
    return RSSM_ERR_INVALID_ARG;
  M2Launch a = m2_launch(d);
  a.S = s->S0;
  a.ring_v = s->ring_v;
  a.ring_k = s->ring_k;
  a.ring_dt = s->ring_dt;
  a.start = s->start;
  a.count = s->count;
  a.flag = s->flag;
  a.sync = s->sync;
  a.err = s->err;
  a.v = v;
  a.k = k;
  a.q = q;
  a.dt = dt;
  a.A = A;
  a.y = y;
  a.work = s->work;
  a.work_bytes = s->work_bytes;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_m2(M2Kind::DecodeFused, a, cs);
  if (e != cudaErrorNotSupported) return cuda_status(e);
  // shapes outside the fused kernels: the decode step, then the flush
  e = launch_m2(M2Kind::Decode, a, cs);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_flush(m2_flush_launch(d, s, A), cs));
}

static FlushLaunch m2_flush_launch(const rssm_m2_dims &d, const rssm_m2_replay *s, const float *A) {
  FlushLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.B = d.B;
  a.H = d.H;
  a.G = d.G;
  a.d = d.d;
  a.n = d.n;
  a.L = d.L;
  a.vec_dtype = d.in_dtype;
  a.key_dtype = d.in_dtype;
  a.mamba2 = true;
  a.S0 = s->S0;
  a.ring_vec = s->ring_v;
  a.ring_key = s->ring_k;
  a.ring_ld = s->ring_dt;
  a.A = A;
  a.start = s->start;
  a.count = s->count;
  a.flag = s->flag;
  a.sync = s->sync;
  a.err = s->err;
  a.num_sms = device_sm_count();
  return a;
}

rssm_status replay_flush(const rssm_m2_dims *dims, const rssm_m2_replay *s, const float *A, rssm_stream_t stream) {
  rssm_status st = check_m2_dims(dims);
  if (st) return st;
  const rssm_m2_dims &d = *dims;
  if (!m2_replay_ok(d, s, true) || !ok4(A)) return RSSM_ERR_INVALID_ARG;
  return cuda_status(launch_flush(m2_flush_launch(d, s, A), reinterpret_cast<cudaStream_t>(stream)));
}

rssm_status replay_spec_verify(const rssm_m2_dims *dims, const rssm_m2_replay *s, int32_t T, const void *v,
                               const void *k, const void *q, const float *dt, const float *A, void *y,
                               rssm_stream_t stream) {
  rssm_status st = check_m2_dims(dims);
  if (st) return st;
  const rssm_m2_dims &d = *dims;
  if (T < 1 || T > d.L) return RSSM_ERR_INVALID_ARG;
  if (T > kMaxT) return RSSM_ERR_UNSUPPORTED;
  if (!m2_replay_ok(d, s, false) || !ok_elem(v, d.in_dtype) || !ok16(k) || !ok16(q) || !ok4(dt) || !ok4(A) ||
      !ok_elem(y, d.y_dtype))
    return RSSM_ERR_INVALID_ARG;
  M2Launch a = m2_launch(d);
  a.T = T;
  a.S = s->S0;
  a.ring_v = s->ring_v;
  a.ring_k = s->ring_k;
  a.ring_dt = s->ring_dt;
  a.start = s->start;
  a.count = s->count;
  a.flag = s->flag;
  a.sync = s->sync;
  a.err = s->err;
  a.v = v;
  a.k = k;
  a.q = q;
  a.dt = dt;
  a.A = A;
  a.y = y;
  a.work = s->work;
  a.work_bytes = s->work_bytes;
  return cuda_status(launch_m2(M2Kind::Verify, a, reinterpret_cast<cudaStream_t>(stream)));
}

rssm_status replay_spec_verify_fused(const rssm_m2_dims *dims, const rssm_m2_replay *s, int32_t T, const void *v,
                                     const void *k, const void *q, const float *dt, const float *A, void *y,
                                     rssm_stream_t stream) {
  rssm_status st = check_m2_dims(dims);
  if (st) return st;
  const rssm_m2_dims &d = *dims;
  if (T < 1 || T > d.L) return RSSM_ERR_INVALID_ARG;
  if (T > kMaxT) return RSSM_ERR_UNSUPPORTED;
  if (!m2_replay_ok(d, s, true) || !ok_elem(v, d.in_dtype) || !ok16(k) || !ok16(q) || !ok4(dt) || !ok4(A) ||
      !ok_elem(y, d.y_dtype))
    return RSSM_ERR_INVALID_ARG;
  M2Launch a = m2_launch(d);
  a.T = T;
  a.S = s->S0;
  a.ring_v = s->ring_v;
  a.ring_k = s->ring_k;
  a.ring_dt = s->ring_dt;
  a.start = s->start;
  a.count = s->count;
  a.flag = s->flag;
  a.sync = s->sync;
  a.err = s->err;
  a.v = v;
  a.k = k;
  a.q = q;
  a.dt = dt;
  a.A = A;
  a.y = y;
  a.work = s->work;
  a.work_bytes = s->work_bytes;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_flush(m2_flush_launch(d, s, A), cs);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_m2(M2Kind::Verify, a, cs));
}

rssm_status replay_spec_commit(int32_t B, int32_t T, int32_t L, const int32_t *accepted, int32_t *count,
                               int32_t *err, rssm_stream_t stream) {
  if (B < 1 || T < 1 || L < 1 || T > L || !ok4(accepted) || !ok4(count) || (err && !aligned(err, 4)))
    return RSSM_ERR_INVALID_ARG;
  return cuda_status(launch_replay_commit(B, T, L, accepted, count, err, reinterpret_cast<cudaStream_t>(stream)));
}

rssm_status ssm_spec_verify_baseline(const rssm_m2_dims *dims, int32_t T, float *slots, const int32_t *cur,
                                     const void *v, const void *k, const void *q, const float *dt, const float *A,
                                     void *y, int32_t *err, rssm_stream_t stream) {
  rssm_status st = check_m2_dims(dims);
  if (st) return st;
  const rssm_m2_dims &d = *dims;
  if (T < 1) return RSSM_ERR_INVALID_ARG;
  if (T > kMaxT) return RSSM_ERR_UNSUPPORTED;
  if (!ok16(slots) || !ok4(cur) || !ok_elem(v, d.in_dtype) || !ok16(k) || !ok16(q) || !ok4(dt) || !ok4(A) ||
      !ok_elem(y, d.y_dtype) || (err && !aligned(err, 4)))
    return RSSM_ERR_INVALID_ARG;
  M2Launch a = m2_launch(d);
  a.T = T;
  a.S = slots;
  a.cur = cur;
  a.err = err;
  a.v = v;
  a.k = k;
  a.q = q;
  a.dt = dt;
  a.A = A;
  a.y = y;
  return cuda_status(launch_m2(M2Kind::SnapshotVerify, a, reinterpret_cast<cudaStream_t>(stream)));
}

rssm_status ssm_spec_commit_baseline(int32_t B, int32_t T, const int32_t *accepted, int32_t *cur, int32_t *err,
                                     rssm_stream_t stream) {
  if (B < 1 || T < 1 || !ok4(accepted) || !ok4(cur) || (err && !aligned(err, 4))) return RSSM_ERR_INVALID_ARG;
  return cuda_status(launch_snapshot_commit(B, T, accepted, cur, err, reinterpret_cast<cudaStream_t>(stream)));
}

// --------------------------------- GDN -----------------------------------

rssm_status gdn_state_update_baseline(const rssm_gdn_dims *dims, float *S, const void *q, const void *k,
                                      const void *v, const float *beta, const float *g, void *y,
                                      rssm_stream_t stream) {
  rssm_status st = check_gdn_dims(dims);
  if (st) return st;
  const rssm_gdn_dims &d = *dims;
  if (!ok16(S) || !ok16(q) || !ok16(k) || !ok_elem(v, d.in_dtype) || !ok4(beta) || !ok4(g) || !ok_elem(y, d.y_dtype))
    return RSSM_ERR_INVALID_ARG;
  GdnLaunch a = gdn_launch(d);
  a.S = S;
  a.q = q;
  a.k = k;
  a.v = v;
  a.beta = beta;
  a.g = g;
  a.y = y;
  return cuda_status(launch_gdn(GdnKind::Baseline, a, reinterpret_cast<cudaStream_t>(stream)));
}

static GdnLaunch gdn_replay_launch(const rssm_gdn_dims &d, const rssm_gdn_replay *s) {
  GdnLaunch a = gdn_launch(d);
  a.S = s->S0;
  a.ring_u = s->ring_u;
  a.ring_k = s->ring_k;
  a.ring_g = s->ring_g;
  a.start = s->start;
  a.count = s->count;
  a.flag = s->flag;
  a.sync = s->sync;
  a.err = s->err;
  a.work = s->work;
  a.work_bytes = s->work_bytes;
  return a;
}

static FlushLaunch gdn_flush_launch(const rssm_gdn_dims &d, const rssm_gdn_replay *s);

rssm_status gdn_replay_decode(const rssm_gdn_dims *dims, const rssm_gdn_replay *s, const void *q, const void *k,
                              const void *v, const float *beta, const float *g, void *y, rssm_stream_t stream) {
  rssm_status st = check_gdn_dims(dims);
  if (st) return st;
  const rssm_gdn_dims &d = *dims;
  if (!gdn_replay_ok(d, s, true) || !ok16(q) || !ok16(k) || !ok_elem(v, d.in_dtype) || !ok4(beta) || !ok4(g) ||
      !ok_elem(y, d.y_dtype))
    return RSSM_ERR_INVALID_ARG;
  GdnLaunch a = gdn_replay_launch(d, s);
  a.q = q;
  a.k = k;
  a.v = v;
  a.beta = beta;
  a.g = g;
  a.y = y;
  return cuda_status(launch_gdn(GdnKind::Decode, a, reinterpret_cast<cudaStream_t>(stream)));
}

rssm_status gdn_replay_decode_fused(const rssm_gdn_dims *dims, const rssm_gdn_replay *s, const void *q,
                                   const void *k, const void *v, const float *beta, const float *g, void *y,
                                   rssm_stream_t stream) {
  rssm_status st = check_gdn_dims(dims);
  if (st) return st;
  const rssm_gdn_dims &d = *dims;
  if (!gdn_replay_ok(d, s, true) || !ok16(q) || !ok16(k) || !ok_elem(v, d.in_dtype) || !ok4(beta) || !ok4(g) ||
      !ok_elem(y, d.y_dtype))
    return RSSM_ERR_INVALID_ARG;
  GdnLaunch a = gdn_replay_launch(d, s);
  a.q = q;
  a.k = k;
  a.v = v;
  a.beta = beta;
  a.g = g;
  a.y = y;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (gdn_split_eligible(GdnKind::DecodeFused, a)) return cuda_status(launch_gdn_split(GdnKind::DecodeFused, a, cs));
  // outside the two-launch kernels: the decode step, then the flush
  cudaError_t e = launch_gdn(GdnKind::Decode, a, cs);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_flush(gdn_flush_launch(d, s), cs));
}

int64_t gdn_replay_workspace_bytes(const rssm_gdn_dims *dims, int32_t T) {
  if (check_gdn_dims(dims) != RSSM_OK || T < 1 || T > kMaxT) return 0;
  return static_cast<int64_t>(dims->B) * dims->Hv * gdn_work_stride_floats(dims->dv, gdn_window_width(T)) * 4;
}

static FlushLaunch gdn_flush_launch(const rssm_gdn_dims &d, const rssm_gdn_replay *s) {
  FlushLaunch a;
  std::memset(&a, 0, sizeof(a));
  a.B = d.B;
  a.H = d.Hv;
  a.G = d.Hk;
  a.d = d.dv;
  a.n = d.dk;
  a.L = d.L;
  a.vec_dtype = d.u_dtype;
  a.key_dtype = d.in_dtype;
  a.mamba2 = false;
  a.S0 = s->S0;
  a.ring_vec = s->ring_u;
  a.ring_key = s->ring_k;
  a.ring_ld = s->ring_g;
  a.A = nullptr;
  a.start = s->start;
  a.count = s->count;
  a.flag = s->flag;
  a.sync = s->sync;
  a.err = s->err;
  a.num_sms = device_sm_count();
  return a;
}

rssm_status gdn_replay_flush(const rssm_gdn_dims *dims, const rssm_gdn_replay *s, rssm_stream_t stream) {
  rssm_status st = check_gdn_dims(dims);
  if (st) return st;
  const rssm_gdn_dims &d = *dims;
  if (!gdn_replay_ok(d, s, true)) return RSSM_ERR_INVALID_ARG;
  return cuda_status(launch_flush(gdn_flush_launch(d, s), reinterpret_cast<cudaStream_t>(stream)));
}

rssm_status gdn_replay_verify(const rssm_gdn_dims *dims, const rssm_gdn_replay *s, int32_t T, const void *q,
                              const void *k, const void *v, const float *beta, const float *g, void *y,
                              rssm_stream_t stream) {
  rssm_status st = check_gdn_dims(dims);
  if (st) return st;
  const rssm_gdn_dims &d = *dims;
  if (T < 1 || T > d.L) return RSSM_ERR_INVALID_ARG;
  if (T > kMaxT) return RSSM_ERR_UNSUPPORTED;
  if (!gdn_replay_ok(d, s, false) || !ok16(q) || !ok16(k) || !ok_elem(v, d.in_dtype) || !ok4(beta) || !ok4(g) ||
      !ok_elem(y, d.y_dtype))
    return RSSM_ERR_INVALID_ARG;
  GdnLaunch a = gdn_replay_launch(d, s);
  a.T = T;
  a.q = q;
  a.k = k;
  a.v = v;
  a.beta = beta;
  a.g = g;
  a.y = y;
  return cuda_status(launch_gdn(GdnKind::Verify, a, reinterpret_cast<cudaStream_t>(stream)));
}

rssm_status gdn_replay_verify_fused(const rssm_gdn_dims *dims, const rssm_gdn_replay *s, int32_t T, const void *q,
                                    const void *k, const void *v, const float *beta, const float *g, void *y,
                                    rssm_stream_t stream) {
  rssm_status st = check_gdn_dims(dims);
  if (st) return st;
  const rssm_gdn_dims &d = *dims;
  if (T < 1 || T > d.L) return RSSM_ERR_INVALID_ARG;
  if (T > kMaxT) return RSSM_ERR_UNSUPPORTED;
  if (!gdn_replay_ok(d, s, true) || !ok16(q) || !ok16(k) || !ok_elem(v, d.in_dtype) || !ok4(beta) || !ok4(g) ||
      !ok_elem(y, d.y_dtype))
    return RSSM_ERR_INVALID_ARG;
  GdnLaunch a = gdn_replay_launch(d, s);
  a.T = T;
  a.q = q;
  a.k = k;
  a.v = v;
  a.beta = beta;
  a.g = g;
  a.y = y;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_flush(gdn_flush_launch(d, s), cs);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_gdn(GdnKind::Verify, a, cs));
}

rssm_status gdn_spec_verify_baseline(const rssm_gdn_dims *dims, int32_t T, float *slots, const int32_t *cur,
                                     const void *q, const void *k, const void *v, const float *beta, const float *g,
                                     void *y, int32_t *err, rssm_stream_t stream) {
  rssm_status st = check_gdn_dims(dims);
  if (st) return st;
  const rssm_gdn_dims &d = *dims;
  if (T < 1) return RSSM_ERR_INVALID_ARG;
  if (T > kMaxT) return RSSM_ERR_UNSUPPORTED;
  if (!ok16(slots) || !ok4(cur) || !ok16(q) || !ok16(k) || !ok_elem(v, d.in_dtype) || !ok4(beta) || !ok4(g) ||
      !ok_elem(y, d.y_dtype) || (err && !aligned(err, 4)))
    return RSSM_ERR_INVALID_ARG;
  GdnLaunch a = gdn_launch(d);
  a.T = T;
  a.S = slots;
  a.cur = cur;
  a.err = err;
  a.q = q;
  a.k = k;
  a.v = v;
  a.beta = beta;
  a.g = g;
  a.y = y;
  return cuda_status(launch_gdn(GdnKind::SnapshotVerify, a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------- fused decode step with a library-owned workspace ----------

namespace {

// Workspace of replay_decode_step_fused_noalloc: module data, so the call
// needs no allocation by anyone.  Every call on a device uses the same array.
constexpr size_t kStaticWorkFloats = size_t(1) << 21;  // 8 MiB
__device__ __align__(256) float g_static_work[kStaticWorkFloats];

// Device address of g_static_work in the current context.  A __device__
// variable's address belongs to the context that loaded the module, so it is
// looked up on every call (a table lookup in the runtime, no allocation):
// after cudaDeviceReset, or under another context, the fresh address is used.
cudaError_t static_work_ptr(float **out) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_work);
  if (e != cudaSuccess) return e;
  *out = static_cast<float *>(p);
  return cudaSuccess;
}

}  // namespace

extern "C" rssm_status replay_decode_step_fused_noalloc(const rssm_m2_dims *dims, const rssm_m2_replay *s,
                                                        const void *v, const void *k, const void *q,
                                                        const float *dt, const float *A, void *y,
                                                        rssm_stream_t stream) {
  rssm_status st = check_m2_dims(dims);
  if (st) return st;
  const rssm_m2_dims &d = *dims;
  if (!m2_replay_ok(d, s, true) || !ok_elem(v, d.in_dtype) || !ok16(k) || !ok16(q) || !ok4(dt) || !ok4(A) ||
      !ok_elem(y, d.y_dtype))
    return RSSM_ERR_INVALID_ARG;
  if (static_cast<size_t>(d.B) * d.H * work_stride_floats(d.d, d.L) > kStaticWorkFloats) return RSSM_ERR_UNSUPPORTED;
  float *work = nullptr;
  cudaError_t e = static_work_ptr(&work);
  if (e != cudaSuccess) return cuda_status(e);
  M2Launch a = m2_launch(d);
  a.S = s->S0;
  a.ring_v = s->ring_v;
  a.ring_k = s->ring_k;
  a.ring_dt = s->ring_dt;
  a.start = s->start;
  a.count = s->count;
  a.flag = s->flag;
  a.sync = s->sync;
  a.err = s->err;
  a.v = v;
  a.k = k;
  a.q = q;
  a.dt = dt;
  a.A = A;
  a.y = y;
  a.work = work;
  a.work_bytes = static_cast<int64_t>(kStaticWorkFloats * sizeof(float));
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  e = launch_m2(M2Kind::DecodeFused, a, cs);
  if (e != cudaErrorNotSupported) return cuda_status(e);
  // shapes outside the fused kernels: the decode step, then the flush
  e = launch_m2(M2Kind::Decode, a, cs);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_flush(m2_flush_launch(d, s, A), cs));
}
