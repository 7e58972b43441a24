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
// Precompute (grid B x G, one warp per head of the group) brings in the
// group's ring entries and this step's inputs with bulk copies, reads the
// pointers, computes k_j^T q for the group, per head the decay weights w_j and
// abar and the buffer term buf[r] = sum_j w_j (k_j^T q) v_j[r], appends this
// step's entry to the ring, and leaves per head in the caller's workspace:
// abar, (h, start, flags), w_1..w_L, buf[0..d).  It does not move the
// pointers: the streaming kernel's block of head 0 does, once every
// precompute block has read them, so no arrival counter is needed.
//
// Stream (grid B x H, 256 threads, launched as a programmatic dependent of the
// precompute so that its S_0 loads overlap the precompute's tail) is then as
// lean as the baseline kernel:
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
// Shared memory, each part 16-byte aligned and filled by one bulk copy:
//   [L][N] group k ring | [N] k | [N] q | [HpG][L][d] v rings | [HpG][d] v |
//   [HpG][L] Delta rings | [HpG][kMaxL] per-slot coefficients
struct PrepSmem {
  uint32_t k_ring, k_in, q_in, v_ring, v_in, dt_ring, coef, total, copied;
  __host__ __device__ PrepSmem(int L, int N, int d, int HpG, int es) {
    k_ring = 0;
    k_in = k_ring + L * N * es;
    q_in = k_in + N * es;
    v_ring = q_in + N * es;
    v_in = v_ring + HpG * L * d * es;
    dt_ring = v_in + HpG * d * es;
    coef = dt_ring + HpG * L * 4;
    copied = coef;
    total = coef + HpG * kMaxL * 4;
  }
};

template <int N, bool kFuse, typename TI>
__global__ void __launch_bounds__(1024) m2_prep_kernel(M2Launch a, int stride) {
  constexpr int LPR = N / 4;
  constexpr int es = sizeof(TI);
  extern __shared__ __align__(128) unsigned char psm[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ float s_M[kMaxL];
  __shared__ int s_ptr[2];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int HpG = a.H / a.G;
  const int b = blockIdx.x / a.G, g = blockIdx.x - b * a.G;
  const int i = g * HpG + w;  // this warp's head
  const int d = a.d, L = a.L;
  const size_t bg = static_cast<size_t>(b) * a.G + g;
  const size_t h0 = static_cast<size_t>(b) * a.H + g * HpG;  // first head of the group
  const size_t bh = h0 + w;
  const PrepSmem lay(L, N, d, HpG, es);

  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, lay.copied);  // the rings now, this step's inputs after the wait
    const unsigned char *ck = static_cast<const unsigned char *>(a.ring_k);
    const unsigned char *cv = static_cast<const unsigned char *>(a.ring_v);
    bulk_g2s(psm + lay.k_ring, ck + bg * L * N * es, lay.k_in - lay.k_ring, &bar);
    bulk_g2s(psm + lay.v_ring, cv + h0 * L * d * es, lay.v_in - lay.v_ring, &bar);
    bulk_g2s(psm + lay.dt_ring, a.ring_dt + h0 * L, lay.coef - lay.dt_ring, &bar);
  }
  // This grid may start while the previous step's streaming grid finishes (it
  // is launched with programmatic serialisation, and that grid lets it start
  // once all its blocks are past their own wait on the previous precompute):
  // the rings copied above are final by then (only precompute grids write
  // them), but the pointers and the workspace records are not, nor need the
  // step's inputs be (the caller may pass that grid's output), so everything
  // below waits for that grid.
  pdl_wait();
  // the streaming kernel may start its S_0 loads now; it waits for this grid
  // before it reads the workspace
  pdl_launch_dependents();
  if (tid == 0) {
    // this step's k, q and v, in flight together with the pointer reads
    bulk_g2s(psm + lay.k_in, static_cast<const unsigned char *>(a.k) + bg * N * es, N * es, &bar);
    bulk_g2s(psm + lay.q_in, static_cast<const unsigned char *>(a.q) + bg * N * es, N * es, &bar);
    bulk_g2s(psm + lay.v_in, static_cast<const unsigned char *>(a.v) + h0 * d * es, lay.dt_ring - lay.v_in, &bar);
    s_ptr[0] = a.count[b];
    s_ptr[1] = a.start[b];
  }
  const float dt_in = a.dt[bh];
  const float Ai = a.A[i];
  float *wk = a.work + bh * stride;
  __syncthreads();  // barrier initialised, pointers read
  const bool arrived = mbar_wait_limit(&bar, 0, a.wait_ns);
  if (__syncthreads_or(!arrived)) {
    // give the sequence up: no valid record, so every streaming block of it
    // skips it and its pointers, S_0 and y stay as they were
    if (lane == 0) reinterpret_cast<int *>(wk)[1] = 0;
    if (tid == 0) {
      set_err(a.err, RSSM_EBIT_TIMEOUT);
      mbar_wait(&bar, 0);  // bounded: the copies must land before shared memory is released
    }
    return;
  }

  const int h = s_ptr[0], st = s_ptr[1];
  if (h < 0 || h >= L || st < 0 || st >= L) {
    if (lane == 0) reinterpret_cast<int *>(wk)[1] = 0;
    if (tid == 0) set_err(a.err, RSSM_EBIT_COUNT_RANGE);
    return;
  }
  const int p = h + 1;
  // start/count/flag are rewritten by the streaming kernel, after every block
  // of this grid has read them
  const TI *kring = reinterpret_cast<const TI *>(psm + lay.k_ring);
  const TI *kin = reinterpret_cast<const TI *>(psm + lay.k_in);
  const TI *qin = reinterpret_cast<const TI *>(psm + lay.q_in);
  TI *vring = reinterpret_cast<TI *>(psm + lay.v_ring) + static_cast<size_t>(w) * L * d;
  const TI *vin = reinterpret_cast<const TI *>(psm + lay.v_in) + static_cast<size_t>(w) * d;
  const float *sdt = reinterpret_cast<const float *>(psm + lay.dt_ring) + w * L;
  float *scoef = reinterpret_cast<float *>(psm + lay.coef) + w * kMaxL;
  const int slot_new = checked_slot(wrapL(st + h, L), L, a.err);

  // k_j^T q for the group, in window order: each lane group of LPR lanes
  // forms V entries at a time and reduces them together
  {
    constexpr int V = LPR >= 4 ? 4 : LPR;
    constexpr int RPW = 32 / LPR;
    const int col = (lane % LPR) * 4;
    const float4 q4 = load4(qin + col);
    const int nw = blockDim.x / 32;
    const int grp = lane / LPR;
    for (int base = w * RPW * V; base < p; base += nw * RPW * V) {
      float x[V];
#pragma unroll
      for (int m = 0; m < V; ++m) {
        const int j = base + grp * V + m;
        x[m] = 0.f;
        if (j < p) x[m] = dot4(load4((j < h ? kring + static_cast<size_t>(wrapL(st + j, L)) * N : kin) + col), q4);
      }
      group_sum_multi<LPR, V>(x, lane);
      const int j = base + grp * V + (lane % LPR) / (LPR / V);
      if ((lane % (LPR / V)) == 0 && j < p) s_M[j] = x[0];
    }
  }
  // decay weights of this warp's head, one entry per lane:
  // w_j = Delta_j exp(A sum_{j<m<p} Delta_m), abar = exp(A sum_{m<p} Delta_m)
  float abar, wj;
  {
    const float dtj = (lane < h) ? sdt[wrapL(st + lane, L)] : (lane == h ? dt_in : 0.f);
    float tot;
    const float ex = excl_suffix_sum(Ai * dtj, lane, tot);
    wj = (lane < p) ? dtj * expf(ex) : 0.f;
    abar = expf(tot);
  }
  // this step's v joins its head's ring copy, so that the window is slots
  // st .. st+h (mod L) of one array
  for (int c = lane; c < d * es / 4; c += 32)
    reinterpret_cast<uint32_t *>(vring + static_cast<size_t>(slot_new) * d)[c] =
        reinterpret_cast<const uint32_t *>(vin)[c];
  __syncthreads();  // s_M complete
  if (lane < p) scoef[wrapL(st + lane, L)] = s_M[lane] * wj;
  if (lane < L) wk[4 + lane] = wj;
  if (lane == 0) {
    wk[0] = abar;
    reinterpret_cast<int *>(wk)[1] = h | (st << 8) | kInfoValid | ((kFuse && p == L) ? kInfoFold : 0);
  }
  __syncwarp();

  // buffer term buf[r] = sum over the window's slots of coef(slot) v_slot[r], two rows per lane
  const int seg1 = min(st + p, L), seg2 = st + p - L;
  for (int r = 2 * lane; r < d; r += 64) {
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int sl = st; sl < seg1; ++sl) {
      const float c = scoef[sl];
      const float2 v2 = load2(vring + static_cast<size_t>(sl) * d + r);
      acc.x = fmaf(c, v2.x, acc.x);
      acc.y = fmaf(c, v2.y, acc.y);
    }
#pragma unroll 4
    for (int sl = 0; sl < seg2; ++sl) {
      const float c = scoef[sl];
      const float2 v2 = load2(vring + static_cast<size_t>(sl) * d + r);
      acc.x = fmaf(c, v2.x, acc.x);
      acc.y = fmaf(c, v2.y, acc.y);
    }
    *reinterpret_cast<float2 *>(wk + 4 + L + r) = acc;
  }

  // append this step's entry at slot (start + h) mod L
  {
    uint32_t *rv_out = reinterpret_cast<uint32_t *>(static_cast<TI *>(a.ring_v) + (bh * L + slot_new) * d);
    for (int c = lane; c < d * es / 4; c += 32) rv_out[c] = reinterpret_cast<const uint32_t *>(vin)[c];
    if (lane == 0) a.ring_dt[bh * L + slot_new] = dt_in;
    if (w == 0) {
      uint32_t *rk_out = reinterpret_cast<uint32_t *>(static_cast<TI *>(a.ring_k) + (bg * L + slot_new) * N);
      for (int c = lane; c < N * es / 4; c += 32) rk_out[c] = reinterpret_cast<const uint32_t *>(kin)[c];
    }
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
  pdl_wait();  // the precompute grid has finished: workspace, ring and pointers are final
  // the next step's precompute may start its ring copies once every block is
  // past this wait (it waits for this grid before it touches the pointers or
  // the workspace)
  pdl_launch_dependents();
  const int info = reinterpret_cast<const int *>(wk)[1];
  const float abar = wk[0];
  if (!(info & kInfoValid)) return;

  // y: written whatever the other groups' precompute blocks did (outputs of a
  // sequence that is given up are undefined)
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
  // a block that changes the sequence's state (S_0 by a fold, its pointers)
  // first makes sure that every group's precompute block of the sequence
  // finished, so that a sequence given up keeps its state whole
  const float *first = a.work + static_cast<size_t>(b) * a.H * stride;
  const int HpG = a.H / a.G;
  bool checked = false;

  if (kFuse && (info & kInfoFold) && rssm_check(((info >> 8) & 0xff) < L && (info & 0xff) + 1 == L, a.err)) {
    if (!sequence_records_valid(first, a.G, HpG, stride, 1, kInfoValid)) return;
    checked = true;
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
  if (i == 0 && warp == 0 && (checked || sequence_records_valid(first, a.G, HpG, stride, 1, kInfoValid)) &&
      lane == 0) {
    // every precompute block has read this sequence's pointers: advance them
    const int p = (info & 0xff) + 1;
    a.count[b] = (kFuse && p == L) ? 0 : p;  // fused: a filled buffer is folded above
    a.flag[b] = (!kFuse && p == L) ? 1 : 0;
  }
}

template <int N, bool kFuse, typename TI, typename TO>
cudaError_t launch_split_n(const M2Launch &a, cudaStream_t stream) {
  constexpr int es = sizeof(TI);
  const int HpG = a.H / a.G;
  const int stride = work_stride_floats(a.d, a.L);
  const size_t psm = PrepSmem(a.L, N, a.d, HpG, es).total;
  auto prep = m2_prep_kernel<N, kFuse, TI>;
  cudaError_t e;
  if (psm > 48 * 1024 &&
      (e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(psm))) !=
          cudaSuccess)
    return e;
  // programmatic dependent launches: the precompute's ring copies overlap the
  // previous step's S_0 stream tail, and this step's S_0 stream the
  // precompute's tail
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t pcfg = {};
  pcfg.gridDim = dim3(static_cast<unsigned>(a.B) * a.G);
  pcfg.blockDim = dim3(32 * HpG);
  pcfg.dynamicSmemBytes = psm;
  pcfg.stream = stream;
  pcfg.attrs = attr;
  pcfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&pcfg, prep, a, stride)) != cudaSuccess) return e;
  const size_t ssm = kFuse ? static_cast<size_t>(a.L) * (a.d + N) * es : 0;
  auto strm = m2_stream_kernel<N, kFuse, TI, TO>;
  if (ssm > 48 * 1024 &&
      (e = cudaFuncSetAttribute(strm, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ssm))) !=
          cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B) * a.H);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = ssm;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, strm, a, stride);
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

// ---------------------------------------------------------------------------
// speculative verify of T drafts ("Algorithm -- speculative decoding"):
//   Y_s = abar_s (S_0 q_s) + sum_{j <= p_s} w_{j,s} (k_j^T q_s) v_j,  p_s = h + s,
// with the drafts' (v, k, Delta) written tentatively after the committed window.
// The precompute kernel (per sequence and group) forms abar_s and the buffer
// vectors buf_s[r] = sum_j w_{j,s} (k_j^T q_s) v_j[r] for every draft s; the
// streaming kernel (per sequence and head) reads S_0 once for all T queries.
// Workspace record per (sequence, head): abar_s [kMaxT], info, pad, then
// buf [P][d] (P = 1, 4 or 8 >= T).
// ---------------------------------------------------------------------------
constexpr int kVwInfo = kMaxT;
constexpr int kVwBuf = kM2VerifyHeader;

struct VPrepSmem {
  uint32_t k_ring, v_ring, dt_ring, k_in, q_in, v_in, dots, coef, total;
  __host__ __device__ VPrepSmem(int L, int N, int d, int HpG, int P, int es) {
    k_ring = 0;
    v_ring = k_ring + L * N * es;
    dt_ring = v_ring + HpG * L * d * es;
    k_in = dt_ring + HpG * L * 4;
    q_in = k_in + P * N * es;
    v_in = q_in + P * N * es;            // [P][HpG][d]
    dots = v_in + P * HpG * d * es;      // float [P][kMaxL]: k_e . q_s over the committed and draft keys
    coef = dots + P * kMaxL * 4;         // float [HpG][P][kMaxL]
    total = coef + HpG * P * kMaxL * 4;
  }
};

template <int N, int NT, typename TI>
__global__ void __launch_bounds__(1024) m2_vprep_kernel(M2Launch a, int stride) {
  constexpr int LPR = N / 4;
  constexpr int es = sizeof(TI);
  extern __shared__ __align__(128) unsigned char psm[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_ptr[2];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int HpG = a.H / a.G;
  const int b = blockIdx.x / a.G, g = blockIdx.x - b * a.G;
  const int i = g * HpG + w;
  const int d = a.d, L = a.L, T = a.T;
  const size_t bg = static_cast<size_t>(b) * a.G + g;
  const size_t h0 = static_cast<size_t>(b) * a.H + g * HpG;
  const size_t bh = h0 + w;
  const VPrepSmem lay(L, N, d, HpG, NT, es);

  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    // the Delta rings and the drafts' k, q, v first; then, once the pointers
    // are in, the committed slots of the k and v rings (at their own slot
    // positions in shared memory)
    mbar_expect_tx(&bar, (lay.k_in - lay.dt_ring) + static_cast<uint32_t>(T) * (2 * N + HpG * d) * es);
    bulk_g2s(psm + lay.dt_ring, a.ring_dt + h0 * L, lay.k_in - lay.dt_ring, &bar);
    for (int m = 0; m < T; ++m) {
      const size_t kq = ((static_cast<size_t>(b) * T + m) * a.G + g) * N * es;
      bulk_g2s(psm + lay.k_in + m * N * es, static_cast<const unsigned char *>(a.k) + kq, N * es, &bar);
      bulk_g2s(psm + lay.q_in + m * N * es, static_cast<const unsigned char *>(a.q) + kq, N * es, &bar);
      const size_t vo = ((static_cast<size_t>(b) * T + m) * a.H + g * HpG) * d * es;
      bulk_g2s(psm + lay.v_in + m * HpG * d * es, static_cast<const unsigned char *>(a.v) + vo, HpG * d * es, &bar);
    }
    const int hc = a.count[b], sc = a.start[b];
    s_ptr[0] = hc;
    s_ptr[1] = sc;
    if (hc >= 1 && hc <= L && sc >= 0 && sc < L) {
      const int n1 = min(hc, L - sc), n2 = hc - n1;
      mbar_expect_tx(&bar, static_cast<uint32_t>(hc) * (N * es + HpG * d * es));
      const unsigned char *gk = static_cast<const unsigned char *>(a.ring_k) + bg * L * N * es;
      bulk_g2s(psm + lay.k_ring + sc * N * es, gk + static_cast<size_t>(sc) * N * es, n1 * N * es, &bar);
      if (n2 > 0) bulk_g2s(psm + lay.k_ring, gk, n2 * N * es, &bar);
      for (int hw = 0; hw < HpG; ++hw) {
        const unsigned char *gv = static_cast<const unsigned char *>(a.ring_v) + (h0 + hw) * L * d * es;
        unsigned char *sv = psm + lay.v_ring + static_cast<size_t>(hw) * L * d * es;
        bulk_g2s(sv + static_cast<size_t>(sc) * d * es, gv + static_cast<size_t>(sc) * d * es, n1 * d * es, &bar);
        if (n2 > 0) bulk_g2s(sv, gv, n2 * d * es, &bar);
      }
    }
    mbar_arrive(&bar);
  }
  pdl_launch_dependents();
  const float Ai = a.A[i];
  const float dt_draft = (lane < T) ? a.dt[(static_cast<size_t>(b) * T + lane) * a.H + i] : 0.f;
  float *wk = a.work + bh * stride;
  __syncthreads();  // barrier initialised, pointers read
  bool arrived = true;
  if (w == 0) arrived = mbar_wait_limit(&bar, 0, a.wait_ns);
  if (__syncthreads_or(!arrived)) {
    // give the sequence up: no valid record, so the streaming kernel skips it
    if (lane == 0) reinterpret_cast<int *>(wk)[kVwInfo] = 0;
    if (tid == 0) {
      set_err(a.err, RSSM_EBIT_TIMEOUT);
      mbar_wait(&bar, 0);  // bounded: the copies must land before shared memory is released
    }
    return;
  }
  const int h = s_ptr[0], st = s_ptr[1];
  if (h < 0 || st < 0 || st >= L || h + T > L) {
    if (lane == 0) reinterpret_cast<int *>(wk)[kVwInfo] = 0;
    if (tid == 0) set_err(a.err, RSSM_EBIT_WINDOW);
    return;
  }
  const int ne = h + T;  // committed entries, then the drafts
  const TI *kring = reinterpret_cast<const TI *>(psm + lay.k_ring);
  const TI *kin = reinterpret_cast<const TI *>(psm + lay.k_in);
  const TI *qin = reinterpret_cast<const TI *>(psm + lay.q_in);
  const TI *vring = reinterpret_cast<const TI *>(psm + lay.v_ring) + static_cast<size_t>(w) * L * d;
  const TI *vin = reinterpret_cast<const TI *>(psm + lay.v_in);
  const float *sdt = reinterpret_cast<const float *>(psm + lay.dt_ring) + w * L;
  float *sM = reinterpret_cast<float *>(psm + lay.dots);
  float *scoef = reinterpret_cast<float *>(psm + lay.coef) + w * NT * kMaxL;

  // k_e . q_s for every entry e and draft s
  if constexpr (sizeof(TI) == 2) {
    // bf16: D[e][s] on the tensor cores, one warp per 16 entries.  Row e of A
    // is key e (a committed slot or a draft), column s of B is query s; rows
    // past the last entry and columns past the last draft read entry 0 and
    // query 0 and are not stored.
    const int nw = blockDim.x / 32;
    for (int mt = w; mt * 16 < ne; mt += nw) {
      const int e = mt * 16 + (lane & 15), ec = e < ne ? e : 0;
      const TI *key = ec < h ? kring + static_cast<size_t>(wrapL(st + ec, L)) * N : kin + (ec - h) * N;
      const int sq = lane & 7;
      const uint32_t aaddr = smem_addr(key + (lane >> 4) * 8);
      const uint32_t baddr = smem_addr(qin + (sq < T ? sq : 0) * N + ((lane >> 3) & 1) * 8);
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
        const int er = mt * 16 + (lane >> 2) + (j >> 1) * 8, sc = 2 * (lane & 3) + (j & 1);
        if (er < ne && sc < T) sM[sc * kMaxL + er] = c[j];
      }
    }
  } else {
    constexpr int V = LPR >= 4 ? 4 : LPR;
    constexpr int RPW = 32 / LPR;
    const int col = (lane % LPR) * 4;
    const int nw = blockDim.x / 32, grp = lane / LPR;
    const int npair = ne * T;
    for (int base = w * RPW * V; base < npair; base += nw * RPW * V) {
      float x[V];
#pragma unroll
      for (int m = 0; m < V; ++m) {
        const int pi = base + grp * V + m;
        x[m] = 0.f;
        if (pi < npair) {
          const int e = pi / T, sq = pi - e * T;
          const TI *key = e < h ? kring + static_cast<size_t>(wrapL(st + e, L)) * N : kin + (e - h) * N;
          x[m] = dot4(load4(key + col), load4(qin + sq * N + col));
        }
      }
      group_sum_multi<LPR, V>(x, lane);
      const int pi = base + grp * V + (lane % LPR) / (LPR / V);
      if ((lane % (LPR / V)) == 0 && pi < npair) {
        const int e = pi / T, sq = pi - e * T;
        sM[sq * kMaxL + e] = x[0];
      }
    }
  }
  // decay of this head for each draft s: w_{e,s} = Delta_e exp(A sum_{e<m<p_s} Delta_m),
  // p_s = h + s + 1, from one prefix sum C_e = sum_{m<=e} A Delta_m of entry
  // `lane`: the exponent is C_{p_s - 1} - C_e and abar_s = exp(C_{p_s - 1})
  const float dd = __shfl_sync(kFull, dt_draft, (lane - h) & 31);
  const float dte = (lane < h) ? sdt[wrapL(st + lane, L)] : (lane < ne ? dd : 0.f);
  float cs = Ai * dte;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(kFull, cs, o);
    if (lane >= o) cs += t;
  }
  __syncthreads();  // sM complete
#pragma unroll
  for (int sq = 0; sq < NT; ++sq) {
    const int p = h + sq + 1;
    const float cp = __shfl_sync(kFull, cs, (p - 1) & 31);
    if (sq < T) {
      scoef[lane * NT + sq] = (lane < p) ? dte * expf(cp - cs) * sM[sq * kMaxL + lane] : 0.f;
      if (lane == 0) wk[sq] = expf(cp);
    }
  }
  if (lane == 0)
    reinterpret_cast<int *>(wk)[kVwInfo] = h | (st << 8) | kInfoValid;
  __syncwarp();

  // buffer vectors of this head, two rows per lane: the committed entries from
  // the ring (slot by slot), then the drafts
  for (int r = 2 * lane; r < d; r += 64) {
    float2 acc[NT];
#pragma unroll
    for (int sq = 0; sq < NT; ++sq) acc[sq] = make_float2(0.f, 0.f);
    auto add = [&](int e, float2 v2) {
      float c[NT];
      if constexpr (NT % 4 == 0) {
#pragma unroll
        for (int q4 = 0; q4 < NT; q4 += 4) {
          const float4 c4 = *reinterpret_cast<const float4 *>(scoef + e * NT + q4);
          c[q4] = c4.x;
          c[q4 + 1] = c4.y;
          c[q4 + 2] = c4.z;
          c[q4 + 3] = c4.w;
        }
      } else {
#pragma unroll
        for (int sq = 0; sq < NT; ++sq) c[sq] = scoef[e * NT + sq];
      }
#pragma unroll
      for (int sq = 0; sq < NT; ++sq) {
        acc[sq].x = fmaf(c[sq], v2.x, acc[sq].x);
        acc[sq].y = fmaf(c[sq], v2.y, acc[sq].y);
      }
    };
    int sl = st;
    for (int e = 0; e < h; ++e) {
      add(e, load2(vring + static_cast<size_t>(sl) * d + r));
      sl = sl + 1 == L ? 0 : sl + 1;
    }
    for (int m = 0; m < T; ++m) add(h + m, load2(vin + static_cast<size_t>(m * HpG + w) * d + r));
#pragma unroll
    for (int sq = 0; sq < NT; ++sq)
      if (sq < T) *reinterpret_cast<float2 *>(wk + kVwBuf + sq * d + r) = acc[sq];
  }

  // the drafts' entries, tentatively, at slots (start + h + m) mod L
  int sd = wrapL(st + h, L);
  for (int m = 0; m < T; ++m, sd = sd + 1 == L ? 0 : sd + 1) {
    const int sl = checked_slot(sd, L, a.err);
    uint32_t *rv = reinterpret_cast<uint32_t *>(static_cast<TI *>(a.ring_v) + (bh * L + sl) * d);
    const uint32_t *sv = reinterpret_cast<const uint32_t *>(vin + static_cast<size_t>(m * HpG + w) * d);
    for (int c = lane; c < d * es / 4; c += 32) rv[c] = sv[c];
    const float dtm = __shfl_sync(kFull, dt_draft, m);
    if (lane == 0) a.ring_dt[bh * L + sl] = dtm;
    if (w == 0) {
      uint32_t *rk = reinterpret_cast<uint32_t *>(static_cast<TI *>(a.ring_k) + (bg * L + sl) * N);
      const uint32_t *sk = reinterpret_cast<const uint32_t *>(kin + m * N);
      for (int c = lane; c < N * es / 4; c += 32) rk[c] = sk[c];
    }
  }
}

template <int N, int NT, typename TI, typename TO>
__global__ void __launch_bounds__(kThreads, NT == 8 ? 2 : (NT == 1 ? 5 : 4)) m2_vstream_kernel(M2Launch a, int stride) {
  constexpr int LPR = N / 4, RPW = 32 / LPR, RPP = kWarps * RPW;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.H, i = blockIdx.x - b * a.H;
  const int d = a.d, L = a.L, T = a.T;
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
  float4 xv[NT];
#pragma unroll
  for (int sq = 0; sq < NT; ++sq)
    xv[sq] = (sq < T) ? load4(static_cast<const TI *>(a.q) + ((static_cast<size_t>(b) * T + sq) * a.G + g) * N + col)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
  pdl_wait();  // the precompute grid has finished
  const int info = reinterpret_cast<const int *>(wk)[kVwInfo];
  const int HpG = a.H / a.G;
  if (!(info & kInfoValid)) return;
  const float *first = a.work + static_cast<size_t>(b) * a.H * stride;

  // S_0 q_s, PB passes x NT drafts reduced together; the reducing lane writes y
  static_assert(NT <= LPR, "drafts per lane group");
  constexpr int PB = (kSPass * NT <= LPR) ? kSPass : LPR / NT;
  TO *y = static_cast<TO *>(a.y);
#pragma unroll
  for (int p0 = 0; p0 < kSPass; p0 += PB) {
    float x[PB * NT];
#pragma unroll
    for (int pp = 0; pp < PB; ++pp)
#pragma unroll
      for (int sq = 0; sq < NT; ++sq) x[pp * NT + sq] = dot4(s[p0 + pp], xv[sq]);
    group_sum_multi<LPR, PB * NT>(x, lane);
    constexpr int SPAN = LPR / (PB * NT);
    const int idx = (lane % LPR) / SPAN;
    const int pp = idx / NT, sq = idx - pp * NT;
    const int r = row0 + (p0 + pp) * RPP;
    if ((lane % SPAN) == 0 && r < d && sq < T)
      store1(y + ((static_cast<size_t>(b) * T + sq) * a.H + i) * d + r, fmaf(wk[sq], x[0], wk[kVwBuf + sq * d + r]));
  }
  // the flag, once every group's precompute block of the sequence finished,
  // so that a sequence given up keeps its state whole
  if (i == 0 && warp == 0 && sequence_records_valid(first, a.G, HpG, stride, kVwInfo, kInfoValid) && lane == 0)
    a.flag[b] = ((info & 0xff) + 2 * T > L) ? 1 : 0;  // early flush, one window ahead
}

template <int N, int NT, typename TI, typename TO>
cudaError_t launch_vsplit(const M2Launch &a, cudaStream_t stream) {
  constexpr int es = sizeof(TI);
  const int HpG = a.H / a.G;
  const int stride = m2_verify_stride_floats(a.d, NT);
  const size_t psm = VPrepSmem(a.L, N, a.d, HpG, NT, es).total;
  auto prep = m2_vprep_kernel<N, NT, TI>;
  cudaError_t e;
  if (psm > 48 * 1024 &&
      (e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(psm))) !=
          cudaSuccess)
    return e;
  prep<<<static_cast<unsigned>(a.B) * a.G, 32 * HpG, psm, stream>>>(a, stride);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (m2_verify_pipe_eligible(a)) return launch_m2_verify_pipe(a, stride, stream);
  auto strm = m2_vstream_kernel<N, NT, TI, TO>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B) * a.H);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, strm, a, stride);
}

template <int N, typename TI, typename TO>
cudaError_t launch_vsplit_t(const M2Launch &a, cudaStream_t stream) {
  switch (gdn_window_width(a.T)) {
    case 1: return launch_vsplit<N, 1, TI, TO>(a, stream);
    case 4: return launch_vsplit<N, 4, TI, TO>(a, stream);
    default: return launch_vsplit<N, 8, TI, TO>(a, stream);
  }
}

template <typename TI, typename TO>
cudaError_t launch_vsplit_n(const M2Launch &a, cudaStream_t stream) {
  switch (a.n) {
    case 32: return launch_vsplit_t<32, TI, TO>(a, stream);
    case 64: return launch_vsplit_t<64, TI, TO>(a, stream);
    case 128: return launch_vsplit_t<128, TI, TO>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool m2_verify_split_eligible(const M2Launch &a) {
  if (a.T < 1 || a.T > kMaxT || (a.n != 32 && a.n != 64 && a.n != 128)) return false;
  const int es = a.in_dtype == RSSM_BF16 ? 2 : 4;
  const int rpp = kWarps * (128 / a.n);
  const int HpG = a.H / a.G;
  const int P = gdn_window_width(a.T);
  auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (HpG > 32 || P > a.n / 4) return false;
  const int64_t need = static_cast<int64_t>(a.B) * a.H * m2_verify_stride_floats(a.d, P) * 4;
  return a.work != nullptr && a.work_bytes >= need && a16(a.work) && a.L % 4 == 0 && (a.d * es) % 16 == 0 &&
         a.d % 2 == 0 && a.d <= kSPass * rpp && VPrepSmem(a.L, a.n, a.d, HpG, P, es).total <= 160u * 1024u &&
         a16(a.S) && a16(a.ring_v) && a16(a.ring_k) && a16(a.ring_dt) && a16(a.v) && a16(a.k) && a16(a.q);
}

cudaError_t launch_m2_verify_split(const M2Launch &a, cudaStream_t stream) {
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_F32) return launch_vsplit_n<bf16, float>(a, stream);
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_BF16) return launch_vsplit_n<bf16, bf16>(a, stream);
  if (a.in_dtype == RSSM_F32 && a.y_dtype == RSSM_F32) return launch_vsplit_n<float, float>(a, stream);
  return launch_vsplit_n<float, bf16>(a, stream);
}

bool m2_decode_split_eligible(const M2Launch &a) {
  const int es = a.in_dtype == RSSM_BF16 ? 2 : 4;
  const int rpp = kWarps * (128 / a.n);
  const int HpG = a.H / a.G;
  auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (HpG > 32) return false;
  const size_t psm = PrepSmem(a.L, a.n, a.d, HpG, es).total;
  const int64_t need = static_cast<int64_t>(a.B) * a.H * work_stride_floats(a.d, a.L) * 4;
  return a.work != nullptr && a.work_bytes >= need && a16(a.work) && HpG <= 32 && psm <= 160 * 1024 && a.L % 4 == 0 && a.L <= 255 &&
         (a.d * es) % 16 == 0 &&
         a.d <= kSPass * rpp && a16(a.S) && a16(a.ring_v) && a16(a.ring_k) && a16(a.ring_dt) && a16(a.v) &&
         a16(a.k) && a16(a.q);
}

cudaError_t launch_m2_decode_split(const M2Launch &a, bool fuse_flush, cudaStream_t stream) {
  return fuse_flush ? launch_split_f<true>(a, stream) : launch_split_f<false>(a, stream);
}

}  // namespace rssm
