// Pipelined ReplaySSM decode step for Mamba-2 (sm_103a): a persistent kernel
// that streams each (sequence, head) work item's checkpoint tile and ring
// entries into shared memory with bulk asynchronous copies (TMA engine,
// cp.async.bulk) through a multi-stage mbarrier pipeline.
//
// "ReplaySSM: Cache SSM Inputs, Not State" -- "Algorithm: Mamba-2 standard
// decode" (output-only decode; "if the buffer is full, flush") and "Kernel
// design details" (ring buffer with in-kernel indexing).
//
// Roles.  Warp 0 is the producer: per item, one lane waits for a free stage
// and issues a single bulk copy, the item's d x n fp32 block of S_0 (one
// contiguous region).  One request per item keeps the TMA engine streaming;
// every other byte of the item -- the committed ring slots of v and k, the
// Delta ring, this step's v, k, q -- is fetched by the consumer group itself
// with 16-byte cp.async copies into its private double buffer, one item
// ahead (while it computes the current item).  The producer warp also reads
// the per-item metadata (start, count, this step's Delta, A) 32 items at a
// time and counts the items' arrivals for the pointer update.  kGroups
// consumer groups of four warps take items in turn: decay weights (suffix
// scan over <= 32 entries in one warp), k_j^T q (one lane group per entry),
// the buffer term, S_0 q from the shared-memory tile; then y and the appended
// ring entry go to HBM.  With the flush fused, an item whose buffer fills is
// folded into S_0 from the same shared-memory data.
//
// Work split.  Items are numbered head-major, item = i * B + b, and CTA c
// takes a contiguous run of them.  Each item's S_0 block is one contiguous
// 16-byte aligned region, so the order costs no DRAM efficiency, and the
// items of a sequence (which share its fill level, hence its flush) spread
// over many CTAs.  The pointer update of a sequence is handed to the last of
// its items to arrive on the per-sequence counter.
#include "kernels.cuh"
#include "tc05.cuh"

namespace rssm {

namespace {

constexpr int kGroups = 3;
constexpr int kGroupWarps = 4;
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr int kPipeThreads = 32 + kGroups * kGroupThreads;
constexpr int kMaxStages = 8;
constexpr int kMaxRows = 256;
constexpr int kItemMax = 256;  // items per CTA (metadata table size)

struct ItemMeta {
  int h, st;
  float dt, A;
};

struct GroupScratch {
  float wt[kMaxL];
  float M[kMaxL];
  int slot[kMaxL];
  float abar, pad[3];
  float dot[kMaxRows];
  float buf[kMaxRows];
};

struct PipeGeom {
  int stages, items_per_cta;
  uint32_t stage_bytes;  // S_0 tile of one item
  // per-group double buffer of the item's small data: offsets inside one buffer
  uint32_t pbuf_bytes, off_vring, off_kring, off_dtring, off_vin, off_kin, off_qin;
  uint32_t off_pbufs, off_meta;
  // tensor-core fold unit (fused flush): offsets from the end of the stages
  uint32_t off_fold, off_opA, off_opB, ke, ncols;
};

// One tensor-core fold unit per CTA, shared by the consumer groups under a
// lock (a fold touches one item in L): TMEM accumulator, its mbarrier, the
// operand buffers.
struct FoldUnit {
  uint64_t bar;
  uint32_t tmem;
  int lock;
  uint32_t phase;
  int pad[3];
};

__device__ __forceinline__ int wrap(int s, int L) { return s >= L ? s - L : s; }

// Tensor-core fold of one full buffer (n = 128, bf16 entries), by the 128
// threads of one consumer group holding the CTA's fold unit.  Transposed
// form: D^T[c][r] = sum_s k_s[c] (w_s v_s[r]) with M = n = 128 state columns
// (TMEM lanes), N = d rows of S_0, K = the L ring slots (every slot holds a
// committed entry when the buffer is full; the order over slots is irrelevant
// to the sum).  The weighted vectors are split into three bf16 terms
// (hi + mid + lo, about 2^-25 relative) and accumulated by three MMAs over the
// same key operand, so the fold keeps fp32 accuracy.  Thread (warp w, lane l)
// owns state column c = 32 (w % 4) + l, the TMEM lane its warp may access,
// and writes S_0[r][c] = abar S_0[r][c] + D^T[c][r] row by row, coalesced.
template <int N, typename TI>
__device__ __forceinline__ void fold_tc(const M2Launch &a, const PipeGeom &geo, FoldUnit *fu,
                                        const GroupScratch &sc, int gi, int gtid, int warp, int lane,
                                        const float *s0, const TI *kring, const TI *vring, const TI *kin,
                                        const TI *vin, int st, int h, float abar, float *S0g) {
  static_assert(N == 128, "the tensor-core fold maps the 128 state columns to TMEM lanes");
  const int d = a.d, L = a.L, KE = static_cast<int>(geo.ke);
  unsigned char *base = reinterpret_cast<unsigned char *>(fu);
  unsigned char *opA = base + (geo.off_opA - geo.off_fold);
  unsigned char *opB = base + (geo.off_opB - geo.off_fold);
  const int c = 32 * (warp & 3) + lane;
  const int cur = (st + h) % L;

  // acquire the unit (bounded)
  int got = 1;
  if (gtid == 0) {
    const uint64_t t0 = global_ns();
    while (atomicCAS(&fu->lock, 0, 1) != 0) {
      if (global_ns() - t0 > kWaitLimitNs) {
        got = 0;
        break;
      }
      __nanosleep(64);
    }
  }
  if (named_bar_or(1 + gi, kGroupThreads, gtid == 0 && !got)) {
    if (gtid == 0) set_err(a.err, RSSM_EBIT_TIMEOUT);
    return;
  }
  tc05::fence_after_sync();
  const uint32_t phase = fu->phase;

  // A: row c = state column, K = slot (keys are exact in bf16)
  for (int sl = 0; sl < KE; sl += 2) {
    __nv_bfloat162 pr;
    pr.x = (sl < L) ? (sl == cur ? kin[c] : kring[static_cast<size_t>(sl) * N + c]) : __float2bfloat16_rn(0.f);
    pr.y = (sl + 1 < L) ? (sl + 1 == cur ? kin[c] : kring[static_cast<size_t>(sl + 1) * N + c])
                        : __float2bfloat16_rn(0.f);
    *reinterpret_cast<__nv_bfloat162 *>(opA + tc05::kmajor_offset(N, c, sl)) = pr;
  }
  // B: three terms of w_s v_s[r], row r of S_0, K = slot
  const uint32_t term_bytes = static_cast<uint32_t>(d) * KE * 2u;
  for (int idx = gtid; idx < d * (KE / 2); idx += kGroupThreads) {
    const int sp = idx / d, r = idx - sp * d, s_0 = 2 * sp;
    float w[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int sl = s_0 + u;
      w[u] = 0.f;
      if (sl < L) {
        int e = sl - st;
        if (e < 0) e += L;
        const float vv = (sl == cur) ? load1(vin + r) : load1(vring + static_cast<size_t>(sl) * d + r);
        w[u] = sc.wt[e] * vv;
      }
    }
    __nv_bfloat162 t3[3];
    tc05::split3_bf16(w[0], t3[0].x, t3[1].x, t3[2].x);
    tc05::split3_bf16(w[1], t3[0].y, t3[1].y, t3[2].y);
#pragma unroll
    for (int t = 0; t < 3; ++t)
      *reinterpret_cast<__nv_bfloat162 *>(opB + t * term_bytes + tc05::kmajor_offset(d, r, s_0)) = t3[t];
  }
  tc05::fence_proxy_async_smem();
  named_bar(1 + gi, kGroupThreads);
  if (gtid == 0) {
    tc05::fence_after_sync();
    const uint32_t idesc = tc05::idesc_bf16_f32(N, d);
    bool acc = false;
    for (int t = 0; t < 3; ++t)
      for (int ks = 0; ks < KE / 16; ++ks) {
        tc05::mma_bf16(fu->tmem, tc05::smem_desc(opA + ks * N * 32, tc05::kLBO, tc05::kSBO),
                       tc05::smem_desc(opB + t * term_bytes + ks * d * 32, tc05::kLBO, tc05::kSBO), idesc, acc);
        acc = true;
      }
    tc05::commit(&fu->bar);
  }
  const bool timed_out = !mbar_wait(&fu->bar, phase);
  const bool fail = named_bar_or(1 + gi, kGroupThreads, timed_out);
  if (!fail) {
    tc05::fence_after_sync();
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    for (int r0 = 0; r0 < d; r0 += 32) {
      float dv[32];
      tc05::ld_32x32b_x32(fu->tmem + lane_base + static_cast<uint32_t>(r0), dv);
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const int r = r0 + u;
        __stcs(S0g + static_cast<size_t>(r) * N + c, fmaf(abar, s0[static_cast<size_t>(r) * N + c], dv[u]));
      }
    }
  } else if (gtid == 0) {
    set_err(a.err, RSSM_EBIT_TIMEOUT);
  }
  // release the unit
  tc05::fence_before_sync();
  named_bar(1 + gi, kGroupThreads);
  if (gtid == 0) {
    fu->phase = phase ^ 1u;
    __threadfence_block();
    atomicExch(&fu->lock, 0);
  }
}

// Consumer-side fetch of one item's small data into a group buffer: the
// committed ring slots of v and k (at their slot positions), the Delta ring,
// and this step's v, k, q, as 16-byte cp.async copies spread over the group.
template <int N, typename TI>
__device__ __forceinline__ void prefetch_item(const M2Launch &a, const PipeGeom &geo, const ItemMeta &m, int item,
                                              unsigned char *pb, int gtid) {
  const int B = a.B, H = a.H, d = a.d, L = a.L;
  if (!(m.h >= 0 && m.h < L && m.st >= 0 && m.st < L)) return;
  constexpr int es = sizeof(TI);
  constexpr int kc = N * es / 16;  // 16-byte chunks per key slot (a power of two)
  const int i = item / B, b = item - i * B, g = i / (H / a.G);
  const size_t bh = static_cast<size_t>(b) * H + i, bg = static_cast<size_t>(b) * a.G + g;
  const int h = m.h, st = m.st;
  const int vc = d * es / 16;
  const unsigned char *rv = static_cast<const unsigned char *>(a.ring_v) + bh * L * d * es;
  const unsigned char *rk = static_cast<const unsigned char *>(a.ring_k) + bg * L * N * es;
  // keys: thread t takes chunk t % kc of entries t / kc, t / kc + 128 / kc, ...
  {
    const int c = gtid % kc;
    for (int j = gtid / kc; j < h; j += kGroupThreads / kc) {
      const int off = (wrap(st + j, L) * kc + c) * 16;
      cp_async16(pb + geo.off_kring + off, rk + off);
    }
  }
  // values: rows of vc chunks, walked with a running (entry, chunk) pair
  {
    int j = gtid / vc, c = gtid - (gtid / vc) * vc;
    const int jstep = kGroupThreads / vc, cstep = kGroupThreads - jstep * vc;
    for (; j < h;) {
      const int off = (wrap(st + j, L) * vc + c) * 16;
      cp_async16(pb + geo.off_vring + off, rv + off);
      j += jstep;
      c += cstep;
      if (c >= vc) {
        c -= vc;
        ++j;
      }
    }
  }
  // Delta ring, this step's v, k, q
  const int dc = L / 4;
  if (gtid < dc) {
    cp_async16(pb + geo.off_dtring + gtid * 16, reinterpret_cast<const unsigned char *>(a.ring_dt + bh * L) + gtid * 16);
  } else if (gtid < dc + vc) {
    const int c = gtid - dc;
    cp_async16(pb + geo.off_vin + c * 16, static_cast<const unsigned char *>(a.v) + bh * d * es + c * 16);
  } else if (gtid < dc + vc + kc) {
    const int c = gtid - dc - vc;
    cp_async16(pb + geo.off_kin + c * 16, static_cast<const unsigned char *>(a.k) + bg * N * es + c * 16);
  } else if (gtid < dc + vc + 2 * kc) {
    const int c = gtid - dc - vc - kc;
    cp_async16(pb + geo.off_qin + c * 16, static_cast<const unsigned char *>(a.q) + bg * N * es + c * 16);
  }
}

template <int N, bool kFuse, bool kTc, typename TI, typename TO>
__global__ void __launch_bounds__(kPipeThreads, 1) m2_decode_pipe_kernel(M2Launch a, PipeGeom geo) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int NS = geo.stages;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(NS) * geo.stage_bytes);
  uint64_t *empty = full + kMaxStages;
  int *ticket = reinterpret_cast<int *>(empty + kMaxStages);  // next item to start
  GroupScratch *scratch = reinterpret_cast<GroupScratch *>(ticket + 4);
  unsigned char *pbufs = smem + geo.off_pbufs;
  ItemMeta *meta = reinterpret_cast<ItemMeta *>(smem + geo.off_meta);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = a.B, H = a.H, d = a.d, L = a.L;
  const int HpG = H / a.G;
  const int total = B * H;
  const int it0 = blockIdx.x * geo.items_per_cta;
  const int it1 = min(total, it0 + geo.items_per_cta);
  const int n_items = max(0, it1 - it0);

  FoldUnit *fu = reinterpret_cast<FoldUnit *>(smem + geo.off_fold);
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kGroupWarps);
    }
    if (kTc) {
      mbar_init(&fu->bar, 1);
      fu->lock = 0;
      fu->phase = 0;
    }
    *ticket = 0;
    fence_mbar_init();
  }
  if (kTc && warp == 1) {
    tc05::alloc(&fu->tmem, geo.ncols);
    tc05::relinquish();
  }
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    // Metadata of items [32k, 32k+32): one lane per item reads the pointers of
    // its sequence, this step's Delta and A, then counts the item's arrival;
    // the last arrival of a sequence advances its pointers (it runs after
    // every item of the sequence, in every CTA, has read them).
    auto meta_batch = [&](int k) {
      const int it = 32 * k + lane;
      if (it < n_items) {
        const int item = it0 + it;
        const int i = item / B, b = item - i * B;
        ItemMeta m;
        m.h = a.count[b];
        m.st = a.start[b];
        m.dt = a.dt[static_cast<size_t>(b) * H + i];
        m.A = a.A[i];
        meta[it] = m;
        if (m.h >= 0 && m.h < L && m.st >= 0 && m.st < L && last_arrival(a.sync, b, H)) {
          a.count[b] = (kFuse && m.h + 1 == L) ? 0 : m.h + 1;  // fused: a filled buffer is folded now
          a.flag[b] = (!kFuse && m.h + 1 == L) ? 1 : 0;
        }
      }
      __syncwarp();
    };
    meta_batch(0);
    for (int it = 0; it < n_items; ++it) {
      if ((it & 31) == 0 && it + 32 < n_items) meta_batch(it / 32 + 1);
      const int stage = it % NS;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(empty + stage, ((it / NS) & 1) ^ 1) ? 1 : 0;
      ok = __shfl_sync(kFull, ok, 0);
      if (!ok) {
        if (lane == 0) set_err(a.err, RSSM_EBIT_TIMEOUT);
        break;
      }
      if (lane == 0) {
        const ItemMeta m = meta[it];
        const int item = it0 + it;
        const int i = item / B, b = item - i * B;
        uint64_t *bar = full + stage;
        if (m.h >= 0 && m.h < L && m.st >= 0 && m.st < L) {
          const size_t bh = static_cast<size_t>(b) * H + i;
          mbar_arrive_expect_tx(bar, static_cast<uint32_t>(d) * N * 4u);
          bulk_g2s(smem + static_cast<size_t>(stage) * geo.stage_bytes, a.S + bh * d * N,
                   static_cast<uint32_t>(d) * N * 4u, bar);
        } else {
          set_err(a.err, RSSM_EBIT_COUNT_RANGE);
          mbar_arrive(bar);
        }
      }
      __syncwarp();
    }
    return;
  }

  // ------------------------------ consumers -------------------------------
  constexpr int LPR = N / 4;
  constexpr int RPW = 32 / LPR;
  constexpr int RPP = kGroupWarps * RPW;
  const int gi = (warp - 1) / kGroupWarps;
  const int wg = (warp - 1) - gi * kGroupWarps;
  const int gtid = tid - 32 - gi * kGroupThreads;
  GroupScratch &sc = scratch[gi];
  const int col = (lane % LPR) * 4;

  int j_iter = 0;
  for (int it = gi; it < n_items; it += kGroups, ++j_iter) {
    const int stage = it % NS;
    // Items are started in order: every thread of the group waits for this
    // item's stage only after the previous item's fill has been observed
    // (ticket == it).  Then the previous use of this stage has landed, the
    // barrier sits in this use's phase or the one after it, and one parity
    // wait is exact.  (Without the ticket a group running ahead could meet the
    // stage one phase early, where a parity wait passes at once.)
    bool timed_out = false;
    {
      const uint64_t t0 = global_ns();
      while (ld_volatile(ticket) != it)
        if (global_ns() - t0 > kWaitLimitNs) {
          timed_out = true;
          break;
        }
    }
    if (!timed_out) timed_out = !mbar_wait(full + stage, static_cast<uint32_t>(it / NS) & 1u);
    // this item's small data: fetched during the previous item (or now, for
    // the group's first item)
    unsigned char *pb = pbufs + static_cast<size_t>(2 * gi + (j_iter & 1)) * geo.pbuf_bytes;
    unsigned char *pb_next = pbufs + static_cast<size_t>(2 * gi + ((j_iter + 1) & 1)) * geo.pbuf_bytes;
    const ItemMeta m = meta[it];  // written before the producer released this item
    if (j_iter == 0 && !timed_out) {
      prefetch_item<N, TI>(a, geo, m, it0 + it, pb, gtid);
      cp_async_commit();
    }
    cp_async_wait_all();
    if (named_bar_or(1 + gi, kGroupThreads, timed_out)) {  // same decision in the whole group
      if (gtid == 0) set_err(a.err, RSSM_EBIT_TIMEOUT);
      break;
    }
    if (gtid == 0) st_volatile(ticket, it + 1);

    const unsigned char *sb = smem + static_cast<size_t>(stage) * geo.stage_bytes;
    bool released = false;
    if (m.h >= 0 && m.h < L && m.st >= 0 && m.st < L) {
      const int item = it0 + it;
      const int i = item / B, b = item - i * B, g = i / HpG;
      const int h = m.h, st = m.st, p = h + 1;
      const float *s0 = reinterpret_cast<const float *>(sb);
      const TI *vring = reinterpret_cast<const TI *>(pb + geo.off_vring);
      const TI *kring = reinterpret_cast<const TI *>(pb + geo.off_kring);
      const float *dtring = reinterpret_cast<const float *>(pb + geo.off_dtring);
      const TI *vin = reinterpret_cast<const TI *>(pb + geo.off_vin);
      const TI *kin = reinterpret_cast<const TI *>(pb + geo.off_kin);
      const TI *qin = reinterpret_cast<const TI *>(pb + geo.off_qin);
      const bool fold = kFuse && p == L;

      // phase 1: S_0 q per row first (all warps) so that each warp can hand
      // its share of the stage back at once, then k_j^T q (all warps) and the
      // decay weights and ring slots (warp 0) -- independent of each other
      const float4 q4 = load4(qin + col);
      // rows in batches of RB per lane group: RB independent shared-memory
      // loads in flight, then one multi-value reduction (RB - 1 + log2(LPR/RB)
      // shuffles), which keeps this latency-bound phase short
      constexpr int RB = LPR >= 16 ? 16 : 8;
      for (int base = 0; base < d; base += RB * RPP) {
        float x[RB];
#pragma unroll
        for (int pp = 0; pp < RB; ++pp) {
          const int r = base + wg * RPW + lane / LPR + pp * RPP;
          x[pp] = (r < d) ? dot4(*reinterpret_cast<const float4 *>(s0 + static_cast<size_t>(r) * N + col), q4) : 0.f;
        }
        if constexpr (RB <= LPR) {
          group_sum_multi<LPR, RB>(x, lane);
          constexpr int SPAN = LPR / RB;
          const int pp = (lane % LPR) / SPAN;
          const int r = base + wg * RPW + lane / LPR + pp * RPP;
          if ((lane % SPAN) == 0 && r < d) sc.dot[r] = x[0];
        } else {
#pragma unroll
          for (int pp = 0; pp < RB; ++pp) {
            const float t = group_sum<LPR>(x[pp]);
            const int r = base + wg * RPW + lane / LPR + pp * RPP;
            if ((lane % LPR) == 0 && r < d) sc.dot[r] = t;
          }
        }
      }
      if (!fold) {
        __syncwarp();  // this warp's rows of S_0 are read
        if (lane == 0) mbar_arrive(empty + stage);
        released = true;
      }
      // the next item's small data goes out now, into the other buffer
      if (it + kGroups < n_items) {
        prefetch_item<N, TI>(a, geo, meta[it + kGroups], it0 + it + kGroups, pb_next, gtid);
        cp_async_commit();
      }
      if constexpr (LPR == 32) {
        // four entries per warp per pass, reduced together
        for (int jb = wg; jb < p; jb += 4 * kGroupWarps) {
          float x[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = jb + u * kGroupWarps;
            x[u] = 0.f;
            if (j < p) x[u] = dot4(load4((j < h ? kring + static_cast<size_t>(wrap(st + j, L)) * N : kin) + col), q4);
          }
          group_sum_multi<32, 4>(x, lane);
          const int j = jb + (lane >> 3) * kGroupWarps;
          if ((lane & 7) == 0 && j < p) sc.M[j] = x[0];
        }
      } else {
        for (int jb = wg * RPW; jb < p; jb += RPP) {
          const int j = jb + lane / LPR;
          float4 kv = make_float4(0.f, 0.f, 0.f, 0.f);
          if (j < p) kv = load4((j < h ? kring + static_cast<size_t>(wrap(st + j, L)) * N : kin) + col);
          const float mm = group_sum<LPR>(dot4(kv, q4));
          if (j < p && (lane % LPR) == 0) sc.M[j] = mm;
        }
      }
      if (wg == 0) {
        const int slot = wrap(st + lane, L);
        const float dtj = (lane < h) ? dtring[slot] : (lane == h ? m.dt : 0.f);
        float tot;
        const float ex = excl_suffix_sum(m.A * dtj, lane, tot);
        sc.wt[lane] = (lane < p) ? dtj * expf(ex) : 0.f;
        sc.slot[lane] = slot;
        if (lane == 0) sc.abar = expf(tot);
      }
      named_bar(1 + gi, kGroupThreads);
      if (gtid < p) sc.M[gtid] *= sc.wt[gtid];  // c_j = w_j (k_j^T q), read after the next barrier

      // phase 2: y = abar (S_0 q) + sum_j c_j v_j; the appended entry
      named_bar(1 + gi, kGroupThreads);
      const float abar = sc.abar;
      const size_t bh = static_cast<size_t>(b) * H + i;
      const int slot = checked_slot(wrap(st + h, L), L, a.err);
      TO *y = static_cast<TO *>(a.y) + bh * d;
      TI *rv_out = static_cast<TI *>(a.ring_v) + (bh * L + slot) * d;
      // two adjacent lanes per row, each summing every other entry
      for (int rb = 0; rb < d; rb += kGroupThreads / 2) {
        const int r = rb + (gtid >> 1), par = gtid & 1;
        float acc0 = 0.f, acc1 = 0.f;
        if (r < d) {
          if (par == 0) acc0 = sc.M[h] * load1(vin + r);
          int j = par;
          for (; j + 2 < h; j += 4) {
            acc0 = fmaf(sc.M[j], load1(vring + static_cast<size_t>(sc.slot[j]) * d + r), acc0);
            acc1 = fmaf(sc.M[j + 2], load1(vring + static_cast<size_t>(sc.slot[j + 2]) * d + r), acc1);
          }
          for (; j < h; j += 2) acc0 = fmaf(sc.M[j], load1(vring + static_cast<size_t>(sc.slot[j]) * d + r), acc0);
        }
        float acc = acc0 + acc1;
        acc += __shfl_xor_sync(kFull, acc, 1);
        if (r < d && par == 0) {
          store1(y + r, fmaf(abar, sc.dot[r], acc));
          rv_out[r] = vin[r];
        }
      }
      if (gtid == 0) a.ring_dt[bh * L + slot] = m.dt;
      if (i % HpG == 0) {
        TI *rk_out = static_cast<TI *>(a.ring_k) + ((static_cast<size_t>(b) * a.G + g) * L + slot) * N;
        for (int c = gtid; c < N; c += kGroupThreads) rk_out[c] = kin[c];
      }
      if constexpr (kTc) {
        if (fold) {
          // The buffer is full after this append: fold all L entries into S_0
          // with this step's weights on the tensor core (see fold_tc).
          fold_tc<N, TI>(a, geo, fu, sc, gi, gtid, warp, lane, s0, kring, vring, kin, vin, st, h, abar,
                         a.S + bh * d * N);
        }
      } else if (fold) {
        // The buffer is full after this append: fold all L entries into S_0
        // with this step's weights, S_0 <- abar S_0 + sum_j s_j v_j k_j^T,
        // reading S_0 and the entries from shared memory.
        float *S0g = a.S + bh * d * N;
        constexpr int CG = N / 4;                  // column groups of 4
        constexpr int RSTEP = kGroupThreads / CG;  // rows covered per pass
        const int c4 = (gtid % CG) * 4;
        for (int r0 = gtid / CG; r0 < d; r0 += 4 * RSTEP) {
          float4 acc[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = r0 + u * RSTEP;
            const float4 sv = (r < d) ? *reinterpret_cast<const float4 *>(s0 + static_cast<size_t>(r) * N + c4)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            acc[u] = make_float4(abar * sv.x, abar * sv.y, abar * sv.z, abar * sv.w);
          }
          for (int j = 0; j < L; ++j) {
            const bool cur = j == h;
            const size_t sl = static_cast<size_t>(sc.slot[j]);
            const float4 kv = load4((cur ? kin : kring + sl * N) + c4);
            const TI *vj = cur ? vin : vring + sl * d;
            const float w = sc.wt[j];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int r = r0 + u * RSTEP;
              const float wv = (r < d) ? w * load1(vj + r) : 0.f;
              acc[u].x = fmaf(wv, kv.x, acc[u].x);
              acc[u].y = fmaf(wv, kv.y, acc[u].y);
              acc[u].z = fmaf(wv, kv.z, acc[u].z);
              acc[u].w = fmaf(wv, kv.w, acc[u].w);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = r0 + u * RSTEP;
            if (r < d) stg_stream4(S0g + static_cast<size_t>(r) * N + c4, acc[u]);
          }
        }
      }
      // phase 2 reads sc.* and the group buffer; the next item overwrites
      // them only after its own vote barrier, which every thread reaches
      // after finishing this item
    }
    else if (it + kGroups < n_items) {
      prefetch_item<N, TI>(a, geo, meta[it + kGroups], it0 + it + kGroups, pb_next, gtid);
      cp_async_commit();
    }
    if (!released) {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + stage);
    }
  }
  cp_async_wait_all();  // no copy of this thread outlives the kernel
  if (kTc) {
    // every consumer warp is done with TMEM before warp 1 releases it
    tc05::fence_before_sync();
    named_bar(15, kGroups * kGroupThreads);
    tc05::fence_after_sync();
    if (warp == 1) tc05::dealloc(fu->tmem, geo.ncols);
  }
}

template <int N, bool kFuse, typename TI, typename TO>
cudaError_t launch_pipe_n(const M2Launch &a, cudaStream_t stream, bool *launched) {
  *launched = false;
  int dev = 0, sms = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
  const uint32_t es = sizeof(TI);
  auto al = [](uint32_t x) { return (x + 127u) & ~127u; };
  PipeGeom geo;
  geo.stage_bytes = al(static_cast<uint32_t>(a.d) * N * 4u);
  // one group buffer: v ring, k ring, Delta ring, v, k, q (16-byte aligned pieces)
  auto a16 = [](uint32_t x) { return (x + 15u) & ~15u; };
  uint32_t off = 0;
  geo.off_vring = off;
  off = a16(off + static_cast<uint32_t>(a.L) * a.d * es);
  geo.off_kring = off;
  off = a16(off + static_cast<uint32_t>(a.L) * N * es);
  geo.off_dtring = off;
  off = a16(off + static_cast<uint32_t>(a.L) * 4u);
  geo.off_vin = off;
  off = a16(off + static_cast<uint32_t>(a.d) * es);
  geo.off_kin = off;
  off = a16(off + N * es);
  geo.off_qin = off;
  geo.pbuf_bytes = al(off + N * es);
  constexpr bool tc = kFuse && N == 128 && sizeof(TI) == 2;
  const bool use_tc = tc && a.d % 32 == 0 && a.d <= 256 && a.L <= kMaxL;
  geo.ke = a.L <= 16 ? 16u : 32u;
  geo.ncols = 32;
  while (geo.ncols < static_cast<uint32_t>(a.d)) geo.ncols <<= 1;
  const uint32_t fold_bytes =
      use_tc ? al(sizeof(FoldUnit)) + 128u * geo.ke * 2u + 3u * static_cast<uint32_t>(a.d) * geo.ke * 2u : 0u;
  const uint32_t bars = al(2u * kMaxStages * 8u + 16u + kGroups * sizeof(GroupScratch));
  const uint32_t pbufs = 2u * kGroups * geo.pbuf_bytes;
  const uint32_t metas = al(kItemMax * sizeof(ItemMeta));
  const uint32_t fixed = bars + pbufs + metas + fold_bytes;
  if (static_cast<uint32_t>(optin) <= fixed) return cudaSuccess;
  const int stages = static_cast<int>((static_cast<uint32_t>(optin) - fixed) / geo.stage_bytes);
  if (stages < kGroups) return cudaSuccess;  // not launched: the caller uses the per-head kernel
  geo.stages = stages < kMaxStages ? stages : kMaxStages;
  const uint32_t head = static_cast<uint32_t>(geo.stages) * geo.stage_bytes;
  geo.off_pbufs = head + bars;
  geo.off_meta = geo.off_pbufs + pbufs;
  geo.off_fold = geo.off_meta + metas;
  geo.off_opA = geo.off_fold + al(sizeof(FoldUnit));
  geo.off_opB = geo.off_opA + 128u * geo.ke * 2u;
  const int total = a.B * a.H;
  int grid = total < sms ? total : sms;
  geo.items_per_cta = (total + grid - 1) / grid;
  if (geo.items_per_cta > kItemMax) geo.items_per_cta = kItemMax;
  grid = (total + geo.items_per_cta - 1) / geo.items_per_cta;
  const size_t smem = static_cast<size_t>(head) + fixed;
  auto kern = use_tc ? m2_decode_pipe_kernel<N, kFuse, tc, TI, TO> : m2_decode_pipe_kernel<N, kFuse, false, TI, TO>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) !=
      cudaSuccess)
    return e;
  kern<<<grid, kPipeThreads, smem, stream>>>(a, geo);
  *launched = true;
  return cudaGetLastError();
}

template <bool kFuse, typename TI, typename TO>
cudaError_t launch_pipe_t(const M2Launch &a, cudaStream_t stream, bool *launched) {
  switch (a.n) {
    case 16: return launch_pipe_n<16, kFuse, TI, TO>(a, stream, launched);
    case 32: return launch_pipe_n<32, kFuse, TI, TO>(a, stream, launched);
    case 64: return launch_pipe_n<64, kFuse, TI, TO>(a, stream, launched);
    case 128: return launch_pipe_n<128, kFuse, TI, TO>(a, stream, launched);
  }
  *launched = false;
  return cudaSuccess;
}

template <bool kFuse>
cudaError_t launch_pipe_f(const M2Launch &a, cudaStream_t stream, bool *launched) {
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_F32) return launch_pipe_t<kFuse, bf16, float>(a, stream, launched);
  if (a.in_dtype == RSSM_BF16 && a.y_dtype == RSSM_BF16) return launch_pipe_t<kFuse, bf16, bf16>(a, stream, launched);
  if (a.in_dtype == RSSM_F32 && a.y_dtype == RSSM_F32) return launch_pipe_t<kFuse, float, float>(a, stream, launched);
  if (a.in_dtype == RSSM_F32 && a.y_dtype == RSSM_BF16) return launch_pipe_t<kFuse, float, bf16>(a, stream, launched);
  *launched = false;
  return cudaSuccess;
}

}  // namespace

bool m2_decode_pipe_eligible(const M2Launch &a) {
  const int es = a.in_dtype == RSSM_BF16 ? 2 : 4;
  auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  // one 16-byte chunk per thread covers the Delta ring and this step's v, k, q
  const bool small_fits = a.L / 4 + a.d * es / 16 + 2 * a.n * es / 16 <= kGroupThreads;
  return a.L % 4 == 0 && (a.d * es) % 16 == 0 && a.d <= kMaxRows && a.d * a.n * 4 <= 96 * 1024 && small_fits && a16(a.S) &&
         a16(a.ring_v) && a16(a.ring_k) && a16(a.ring_dt) && a16(a.v) && a16(a.k) && a16(a.q);
}

cudaError_t launch_m2_decode_pipe(const M2Launch &a, bool fuse_flush, cudaStream_t stream, bool *launched) {
  return fuse_flush ? launch_pipe_f<true>(a, stream, launched) : launch_pipe_f<false>(a, stream, launched);
}

}  // namespace rssm
