"""fp64 oracle for the Gated DeltaNet (GDN) decode step: the Householder-form
recurrence, its rank-1 correction form, the ReplaySSM ring buffer of cached
corrections (decode, flush, chunked speculative verify, commit) and the
per-draft snapshot baseline.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Readings of the page "ReplaySSM: Cache SSM Inputs, Not State" that this file
fixes where the text is silent:

* value head i reads the k and q of key head ``i // (Hv // Hk)``;
* alpha_t = exp(g_t); g arrives as a log decay, beta in (0, 1); k and q arrive
  already L2-normalised (no in-kernel normalisation or 1/sqrt(d_k) scale);
* the appendix writes the baseline correction as u = beta (v - S k) with S the
  already-decayed state alpha S_{t-1}; that is the same quantity as the
  replay form beta (v - alpha S_h k);
* the buffer stores u in a stated storage dtype (float32 by default); the
  oracle rounds what it stores to that dtype exactly as the buffer would, and
  computes everything else in float64;
* full-buffer, early-flush and ring-reset rules are those of the Mamba-2 path.
"""
from __future__ import annotations

import numpy as np

from .mamba2 import ERR_ACCEPTED, ERR_COUNT_RANGE, ERR_CUR, ERR_WINDOW  # noqa: F401


def key_head(Hv: int, Hk: int) -> np.ndarray:
    if Hv % Hk:
        raise ValueError("Hv must be a multiple of Hk")
    return np.arange(Hv) // (Hv // Hk)


def round_storage(x, dtype: str):
    """Round float64 values to the buffer's storage dtype ('f32' or 'bf16',
    round to nearest even; 'f64' keeps them) and return them as float64."""
    x = np.asarray(x, np.float64)
    if dtype == "f64":
        return x.copy()
    f = x.astype(np.float32)
    if dtype == "f32":
        return f.astype(np.float64)
    if dtype != "bf16":
        raise ValueError(dtype)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return (r.astype(np.uint32)).view(np.float32).astype(np.float64)


def householder_step(S, q, k, v, beta, g):
    """One token of the GDN recurrence in its Householder form
    (page "Background — memory bound", delta-rule family):
        S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
        y_t = S_t q_t
    The d_k x d_k Householder matrix is built explicitly (small shapes only).
    S [B,Hv,dv,dk]; q, k [B,Hk,dk]; v [B,Hv,dv]; beta, g [B,Hv]."""
    S = np.asarray(S, np.float64)
    B, Hv, dv, dk = S.shape
    kh_ = key_head(Hv, k.shape[1])
    kh = np.asarray(k, np.float64)[:, kh_, :]
    qh = np.asarray(q, np.float64)[:, kh_, :]
    beta = np.asarray(beta, np.float64)
    g = np.asarray(g, np.float64)
    v = np.asarray(v, np.float64)
    P = np.eye(dk)[None, None] - beta[:, :, None, None] * (kh[:, :, :, None] * kh[:, :, None, :])
    S_next = np.exp(g)[:, :, None, None] * np.matmul(S, P) + beta[:, :, None, None] * (
        v[:, :, :, None] * kh[:, :, None, :])
    y = np.einsum("bhvk,bhk->bhv", S_next, qh)
    return S_next, y


def rank1_step(S, q, k, v, beta, g):
    """One token of the GDN recurrence in correction form (appendix "GDN —
    standard decode", baseline):
        alpha = e^{g};  u = beta (v - alpha S_{t-1} k);  S_t = alpha S_{t-1} + u k^T;  y = S_t q
    Returns (S_t, y_t, u_t).  This is what the baseline GDN kernel computes."""
    S = np.asarray(S, np.float64)
    Hv = S.shape[1]
    kh_ = key_head(Hv, k.shape[1])
    kh = np.asarray(k, np.float64)[:, kh_, :]
    qh = np.asarray(q, np.float64)[:, kh_, :]
    alpha = np.exp(np.asarray(g, np.float64))
    beta = np.asarray(beta, np.float64)
    Sk = np.einsum("bhvk,bhk->bhv", S, kh)
    u = beta[:, :, None] * (np.asarray(v, np.float64) - alpha[:, :, None] * Sk)
    S_next = alpha[:, :, None, None] * S + u[:, :, :, None] * kh[:, :, None, :]
    y = np.einsum("bhvk,bhk->bhv", S_next, qh)
    return S_next, y, u


class GdnReplay:
    """ReplaySSM state for GDN: checkpoint S_0 plus a ring buffer of cached
    corrections (u, k, g) (appendix "GDN — standard decode": cache u; once
    u_t is known the update S_t = alpha_t S_{t-1} + u_t k_t^T has the Mamba-2
    history form)."""

    def __init__(self, S0, ring_u, ring_k, ring_g, start, count, u_dtype: str = "f32"):
        self.S0 = np.array(S0, dtype=np.float64)  # [B,Hv,dv,dk]
        self.ring_u = np.array(ring_u, dtype=np.float64)  # [B,Hv,L,dv]
        self.ring_k = np.array(ring_k, dtype=np.float64)  # [B,Hk,L,dk]
        self.ring_g = np.array(ring_g, dtype=np.float64)  # [B,Hv,L]
        self.B, self.Hv, self.dv, self.dk = self.S0.shape
        self.Hk = self.ring_k.shape[1]
        self.L = self.ring_u.shape[2]
        self.kh = key_head(self.Hv, self.Hk)
        self.u_dtype = u_dtype
        self.start = np.array(start, dtype=np.int64)
        self.count = np.array(count, dtype=np.int64)
        self.flag = np.zeros(self.B, dtype=np.int64)
        self.err = 0

    def slot(self, b: int, j: int) -> int:
        return int((self.start[b] + j - 1) % self.L)

    def _append(self, b, j, u, k, g):
        s = self.slot(b, j)
        self.ring_u[b, :, s, :] = round_storage(u, self.u_dtype)
        self.ring_k[b, :, s, :] = k
        self.ring_g[b, :, s] = g

    def state(self, b: int, p: int | None = None):
        """S_h after the first p window entries, materialised (appendix "GDN —
        standard decode", state-and-output route):
            S_h = (prod_j alpha_j) S_0 + sum_j (prod_{i>j} alpha_i) u_j k_j^T
        Products of alpha_i = exp(g_i) are taken one factor at a time."""
        if p is None:
            p = int(self.count[b])
        al = [np.exp(self.ring_g[b, :, self.slot(b, i)]) for i in range(1, p + 1)]
        abar = np.ones(self.Hv)
        for a in al:
            abar = abar * a
        S = abar[:, None, None] * self.S0[b]
        for j in range(1, p + 1):
            w = np.ones(self.Hv)
            for i in range(j + 1, p + 1):
                w = w * al[i - 1]
            sl = self.slot(b, j)
            uj = self.ring_u[b, :, sl, :]
            kj = self.ring_k[b, self.kh, sl, :]
            S = S + w[:, None, None] * (uj[:, :, None] * kj[:, None, :])
        return S

    def decode_step(self, q, k, v, beta, g):
        """One GDN replay decode step (appendix "GDN — standard decode"):
        rebuild S_h, then u = beta (v - alpha (S_h k)), y = alpha (S_h q) + u (k . q);
        append (u, k, g); count <- h + 1; flag <- (count == L).
        q, k [B,Hk,dk]; v [B,Hv,dv]; beta, g [B,Hv].  Returns y [B,Hv,dv]."""
        y = np.zeros((self.B, self.Hv, self.dv))
        for b in range(self.B):
            h = int(self.count[b])
            if not (0 <= h < self.L):
                self.err |= ERR_COUNT_RANGE
                continue
            Sh = self.state(b, h)
            kb = np.asarray(k[b], np.float64)[self.kh]  # [Hv,dk]
            qb = np.asarray(q[b], np.float64)[self.kh]
            alpha = np.exp(np.asarray(g[b], np.float64))
            Shk = np.einsum("hvk,hk->hv", Sh, kb)
            Shq = np.einsum("hvk,hk->hv", Sh, qb)
            u = np.asarray(beta[b], np.float64)[:, None] * (np.asarray(v[b], np.float64) - alpha[:, None] * Shk)
            y[b] = alpha[:, None] * Shq + u * np.sum(kb * qb, axis=-1)[:, None]
            self._append(b, h + 1, u, k[b], g[b])
            self.count[b] = h + 1
            self.flag[b] = int(self.count[b] == self.L)
        return y

    def flush(self):
        """Fold every flagged sequence's committed entries into S_0 (same as the
        Mamba-2 history route with u_j in place of Delta_j v_j), then reset the
        ring pointers as in the Mamba-2 flush."""
        for b in range(self.B):
            if not self.flag[b]:
                continue
            c = int(self.count[b])
            self.S0[b] = self.state(b, c)
            self.start[b] = (self.start[b] + c) % self.L
            self.count[b] = 0
            self.flag[b] = 0

    def verify(self, q, k, v, beta, g):
        """Verify T drafts with the chunked form (appendix "GDN — speculative
        decoding"): unrolling the recurrence over the window gives
            u_s = R_s - sum_{s' < s} A_{s,s'} u_{s'}
        with G_s = sum_{r <= s} g_r,
            R_s       = beta_s (v_s - e^{G_s} S_h k_s),
            A_{s,s'}  = beta_s e^{G_s - G_{s'}} (k_s . k_{s'})      (s' < s),
        a strictly lower-triangular T x T system solved by forward
        substitution, and outputs
            y_s = e^{G_s} S_h q_s + sum_{s' <= s} e^{G_s - G_{s'}} (k_{s'} . q_s) u_{s'}.
        Drafts are appended tentatively; count is unchanged;
        flag <- (h + 2T > L).  q, k [B,T,Hk,dk]; v [B,T,Hv,dv]; beta, g [B,T,Hv].
        Returns Y [B,T,Hv,dv]."""
        T = v.shape[1]
        Y = np.zeros((self.B, T, self.Hv, self.dv))
        for b in range(self.B):
            h = int(self.count[b])
            if not (0 <= h and h + T <= self.L):
                self.err |= ERR_WINDOW
                continue
            Sh = self.state(b, h)
            kb = np.asarray(k[b], np.float64)[:, self.kh]  # [T,Hv,dk]
            qb = np.asarray(q[b], np.float64)[:, self.kh]
            vb = np.asarray(v[b], np.float64)  # [T,Hv,dv]
            bb = np.asarray(beta[b], np.float64)  # [T,Hv]
            Gc = np.cumsum(np.asarray(g[b], np.float64), axis=0)  # [T,Hv]
            R = np.zeros((T, self.Hv, self.dv))
            for s in range(T):
                R[s] = bb[s][:, None] * (vb[s] - np.exp(Gc[s])[:, None] * np.einsum("hvk,hk->hv", Sh, kb[s]))
            Amat = np.zeros((self.Hv, T, T))
            for s in range(T):
                for sp in range(s):
                    Amat[:, s, sp] = bb[s] * np.exp(Gc[s] - Gc[sp]) * np.sum(kb[s] * kb[sp], axis=-1)
            U = np.zeros((T, self.Hv, self.dv))
            for s in range(T):
                acc = R[s].copy()
                for sp in range(s):
                    acc = acc - Amat[:, s, sp][:, None] * U[sp]
                U[s] = acc
            for s in range(T):
                ys = np.exp(Gc[s])[:, None] * np.einsum("hvk,hk->hv", Sh, qb[s])
                for sp in range(s + 1):
                    ys = ys + (np.exp(Gc[s] - Gc[sp]) * np.sum(kb[sp] * qb[s], axis=-1))[:, None] * U[sp]
                Y[b, s] = ys
            for s in range(T):
                self._append(b, h + s + 1, U[s], k[b, s], g[b, s])
            self.flag[b] = int(h + 2 * T > self.L)
        return Y

    def commit(self, accepted, T: int):
        for b in range(self.B):
            acc = int(accepted[b])
            if acc < 0 or acc > T or self.count[b] + acc > self.L:
                self.err |= ERR_ACCEPTED
                continue
            self.count[b] += acc


class GdnSnapshotBaseline:
    """Baseline GDN speculative path: serial correction-form updates per draft,
    with a full state snapshot stored per draft (T+1 slots and a current index,
    as in the Mamba-2 snapshot baseline)."""

    def __init__(self, S_init, T: int):
        S_init = np.asarray(S_init, np.float64)
        self.B = S_init.shape[0]
        self.T = T
        self.slots = np.zeros((self.B, T + 1) + S_init.shape[1:])
        self.slots[:, 0] = S_init
        self.cur = np.zeros(self.B, dtype=np.int64)
        self.err = 0

    def verify(self, q, k, v, beta, g):
        T = self.T
        B, _, Hv, dv = v.shape
        Y = np.zeros((B, T, Hv, dv))
        for b in range(B):
            c = int(self.cur[b])
            if not (0 <= c <= T):
                self.err |= ERR_CUR
                continue
            S = self.slots[b, c][None]
            for s in range(1, T + 1):
                S, y, _ = rank1_step(S, q[b:b + 1, s - 1], k[b:b + 1, s - 1], v[b:b + 1, s - 1],
                                     beta[b:b + 1, s - 1], g[b:b + 1, s - 1])
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
