"""fp64 oracle for the Mamba-2 decode step: the plain recurrence, the ReplaySSM
ring buffer (output-only decode, flush, speculative verify and commit) and the
per-draft snapshot baseline.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Readings of the page "ReplaySSM: Cache SSM Inputs, Not State" that this file
fixes where the text is silent:

* head i reads the k and q of group ``i // (H // G)`` (contiguous groups);
* a buffer is "full" when ``count == L`` after the append; the flush then
  folds all ``count`` entries, the current one included;
* flushing moves the ring's start past the folded entries,
  ``start <- (start + count) mod L``, and sets ``count <- 0``;
* speculative verify decides the early flush on the committed count h before
  the round: ``flag = (h + 2T > L)``; commit adds the accepted count; the
  flush then folds the ``h + accepted`` committed entries;
* Delta arrives after its softplus; there is no D skip term and no z gate.
"""
from __future__ import annotations

import numpy as np

# error bits, shared meaning with the C ABI's sticky error word
ERR_COUNT_RANGE = 1  # committed count outside [0, L-1] at a decode step
ERR_WINDOW = 2  # count + T > L at a verify round
ERR_ACCEPTED = 4  # accepted outside [0, T] or count + accepted > L at commit
ERR_CUR = 8  # snapshot slot index outside [0, T]


def head_group(H: int, G: int) -> np.ndarray:
    """Group (k/q index) of every head: heads share k and q within a group
    (page: "Background — memory bound", shapes paragraph); contiguous mapping."""
    if H % G:
        raise ValueError("H must be a multiple of G")
    return np.arange(H) // (H // G)


def recurrence_step(S, v, k, q, dt, A):
    """One token of the Mamba-2 recurrence for a batch of sequences.

    Page "Background — memory bound", Mamba-2 recurrence:
        a_t = exp(A * Delta_t)
        S_t = a_t S_{t-1} + Delta_t v_t k_t^T        (update)
        y_t = S_t q_t                                (read)

    S [B,H,d,n]; v [B,H,d]; k, q [B,G,n]; dt [B,H]; A [H].  Returns (S_t, y_t).
    This is also exactly what the baseline decode kernel computes
    ("Algorithm — Mamba-2 standard decode", baseline).
    """
    S = np.asarray(S, np.float64)
    H = S.shape[1]
    grp = head_group(H, k.shape[1])
    kh = np.asarray(k, np.float64)[:, grp, :]
    qh = np.asarray(q, np.float64)[:, grp, :]
    v = np.asarray(v, np.float64)
    dt = np.asarray(dt, np.float64)
    a = np.exp(np.asarray(A, np.float64)[None, :] * dt)
    S_next = a[:, :, None, None] * S + dt[:, :, None, None] * (v[:, :, :, None] * kh[:, :, None, :])
    y = np.einsum("bhdn,bhn->bhd", S_next, qh)
    return S_next, y


class Mamba2Replay:
    """ReplaySSM state of a batch of sequences: checkpoint S_0 plus a ring buffer
    of the last inputs (v, Delta, k) with per-sequence start/count/flag.

    Page "Core idea: cache recent inputs instead of storing the state" and
    "Algorithm — Mamba-2 standard decode / speculative decoding";
    ring buffer with in-kernel indexing from "Kernel design details".
    Entry j (1-based) of sequence b's window sits in slot (start + j - 1) mod L.
    """

    def __init__(self, S0, A, ring_v, ring_k, ring_dt, start, count):
        self.S0 = np.array(S0, dtype=np.float64)
        self.A = np.array(A, dtype=np.float64)
        self.ring_v = np.array(ring_v, dtype=np.float64)  # [B,H,L,d]
        self.ring_k = np.array(ring_k, dtype=np.float64)  # [B,G,L,n]
        self.ring_dt = np.array(ring_dt, dtype=np.float64)  # [B,H,L]
        self.B, self.H, self.d, self.n = self.S0.shape
        self.G = self.ring_k.shape[1]
        self.L = self.ring_v.shape[2]
        self.grp = head_group(self.H, self.G)
        self.start = np.array(start, dtype=np.int64)
        self.count = np.array(count, dtype=np.int64)
        self.flag = np.zeros(self.B, dtype=np.int64)
        self.err = 0

    # -- ring indexing -----------------------------------------------------
    def slot(self, b: int, j: int) -> int:
        """Ring slot of the j-th (1-based) entry of sequence b's window."""
        return int((self.start[b] + j - 1) % self.L)

    def _append(self, b, j, v, k, dt):
        s = self.slot(b, j)
        self.ring_v[b, :, s, :] = v
        self.ring_k[b, :, s, :] = k
        self.ring_dt[b, :, s] = dt

    # -- decay weights -----------------------------------------------------
    def weights(self, b: int, p: int):
        """Decay weights over the first p window entries, per head.

        abar = prod_{i=1}^{p} a_i and s_j = Delta_j prod_{i=j+1}^{p} a_i with
        a_i = exp(A Delta_i): the coefficients of the history route
        ("Core idea", unrolled sum) seen from the checkpoint S_0.
        Products are taken as products, one factor at a time.
        """
        a = [np.exp(self.A * self.ring_dt[b, :, self.slot(b, i)]) for i in range(1, p + 1)]
        abar = np.ones(self.H)
        for ai in a:
            abar = abar * ai
        s = []
        for j in range(1, p + 1):
            w = self.ring_dt[b, :, self.slot(b, j)].copy()
            for i in range(j + 1, p + 1):
                w = w * a[i - 1]
            s.append(w)
        return abar, s

    # -- the three routes to the output/state ------------------------------
    def output(self, b: int, p: int, q_b):
        """Output-only decode over the first p window entries ("Relaxed
        requirement: output-only decode"):
            y = abar (S_0 q) + sum_{j=1}^{p} s_j v_j (k_j^T q)
        q_b [G,n]; returns y [H,d].
        """
        abar, s = self.weights(b, p)
        qh = np.asarray(q_b, np.float64)[self.grp]  # [H,n]
        y = abar[:, None] * np.einsum("hdn,hn->hd", self.S0[b], qh)
        for j in range(1, p + 1):
            sl = self.slot(b, j)
            kj = self.ring_k[b, self.grp, sl, :]  # [H,n]
            vj = self.ring_v[b, :, sl, :]  # [H,d]
            kq = np.sum(kj * qh, axis=-1)  # [H]
            y = y + (s[j - 1] * kq)[:, None] * vj
        return y

    def state(self, b: int, p: int | None = None):
        """State after the first p window entries by the history route
        ("Core idea"): S = abar S_0 + sum_j s_j v_j k_j^T.  p defaults to the
        committed count.  Returns [H,d,n]."""
        if p is None:
            p = int(self.count[b])
        abar, s = self.weights(b, p)
        S = abar[:, None, None] * self.S0[b]
        for j in range(1, p + 1):
            sl = self.slot(b, j)
            vj = self.ring_v[b, :, sl, :]
            kj = self.ring_k[b, self.grp, sl, :]
            S = S + s[j - 1][:, None, None] * (vj[:, :, None] * kj[:, None, :])
        return S

    # -- the decode step and the flush -------------------------------------
    def decode_step(self, v, k, q, dt):
        """One ReplaySSM decode step ("Algorithm — Mamba-2 standard decode"):
        append (v, Delta, k), compute y from S_0 and the buffer, then
        count <- h + 1 and flag <- (count == L).  The flush is a separate call.
        v [B,H,d]; k, q [B,G,n]; dt [B,H].  Returns y [B,H,d]."""
        y = np.zeros((self.B, self.H, self.d))
        for b in range(self.B):
            h = int(self.count[b])
            if not (0 <= h < self.L):
                self.err |= ERR_COUNT_RANGE
                continue
            self._append(b, h + 1, v[b], k[b], dt[b])
            y[b] = self.output(b, h + 1, q[b])
            self.count[b] = h + 1
            self.flag[b] = int(self.count[b] == self.L)
        return y

    def flush(self):
        """Fold the committed entries of every flagged sequence into S_0
        ("Algorithm — Mamba-2 standard decode", flush):
            S_0 <- abar S_0 + sum_j s_j v_j k_j^T
        then clear the buffer: start <- (start + count) mod L, count <- 0."""
        for b in range(self.B):
            if not self.flag[b]:
                continue
            c = int(self.count[b])
            self.S0[b] = self.state(b, c)
            self.start[b] = (self.start[b] + c) % self.L
            self.count[b] = 0
            self.flag[b] = 0

    # -- speculative decoding ----------------------------------------------
    def spec_verify(self, v, k, q, dt):
        """Verify T draft tokens ("Algorithm — speculative decoding"): append
        all drafts to the buffer, then for draft s (p_s = h + s)
            Y_s = abar_s (S_0 q_s) + sum_{j <= p_s} w_{j,s} (k_j^T q_s) v_j.
        The committed count is left unchanged; flag <- (h + 2T > L), the early
        flush rule ("flush decision").  v [B,T,H,d]; k, q [B,T,G,n];
        dt [B,T,H].  Returns Y [B,T,H,d]."""
        T = v.shape[1]
        Y = np.zeros((self.B, T, self.H, self.d))
        for b in range(self.B):
            h = int(self.count[b])
            if not (0 <= h and h + T <= self.L):
                self.err |= ERR_WINDOW
                continue
            for s in range(1, T + 1):
                self._append(b, h + s, v[b, s - 1], k[b, s - 1], dt[b, s - 1])
            for s in range(1, T + 1):
                Y[b, s - 1] = self.output(b, h + s, q[b, s - 1])
            self.flag[b] = int(h + 2 * T > self.L)
        return Y

    def commit(self, accepted, T: int):
        """Device-side commit ("CUDA Graph supplementary design"): advance the
        committed count by the accepted drafts; rejected drafts stay in slots
        past the window and are overwritten later, so rollback is a pointer move."""
        for b in range(self.B):
            acc = int(accepted[b])
            if acc < 0 or acc > T or self.count[b] + acc > self.L:
                self.err |= ERR_ACCEPTED
                continue
            self.count[b] += acc


class Mamba2SnapshotBaseline:
    """Baseline speculative path ("Algorithm — speculative decoding", baseline):
    update the state serially per draft and store a full snapshot per draft.

    Each sequence owns T+1 state slots and a current index cur; draft s of a
    round is written to slot (cur + s) mod (T+1), and commit moves cur to the
    slot of the last accepted draft.
    """

    def __init__(self, S_init, A, T: int):
        S_init = np.asarray(S_init, np.float64)
        self.B = S_init.shape[0]
        self.T = T
        self.A = np.asarray(A, np.float64)
        self.slots = np.zeros((self.B, T + 1) + S_init.shape[1:])
        self.slots[:, 0] = S_init
        self.cur = np.zeros(self.B, dtype=np.int64)
        self.err = 0

    def verify(self, v, k, q, dt):
        T = self.T
        B, _, H, d = v.shape
        Y = np.zeros((B, T, H, d))
        for b in range(B):
            c = int(self.cur[b])
            if not (0 <= c <= T):
                self.err |= ERR_CUR
                continue
            S = self.slots[b, c][None]
            for s in range(1, T + 1):
                S, y = recurrence_step(S, v[b:b + 1, s - 1], k[b:b + 1, s - 1], q[b:b + 1, s - 1],
                                       dt[b:b + 1, s - 1], self.A)
                self.slots[b, (c + s) % (T + 1)] = S[0]
                Y[b, s - 1] = y[0]
        return Y

    def commit(self, accepted):
        for b in range(self.B):
            acc = int(accepted[b])
            if acc < 0 or acc > self.T:
                self.err |= ERR_ACCEPTED
                continue
            self.cur[b] = (self.cur[b] + acc) % (self.T + 1)

    def state(self, b: int):
        return self.slots[b, int(self.cur[b])]
