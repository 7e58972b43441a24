"""fp64 oracle for the convolution-state step that precedes the SSM in a
Mamba-2 layer's decode.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the pages fix ("Disaggregated Serving for Hybrid SSM Models", section on
the Mamba state layout): besides the SSM state, every Mamba layer keeps a
convolution state of shape (conv_dim, state_len) per sequence, e.g.
(3072, 3) in bf16, stored in the "DS" layout (dim, state_len) so that the x,
B and C sub-projections are each contiguous; conv_dim = |x| + 2 |B|.

What they leave open, and the plainest reading taken here: the state holds
the last state_len inputs of a causal depthwise convolution of width
W = state_len + 1, oldest first.  A decode step with a new input column u
(one value per channel) computes, per channel c,

    z[c] = bias[c] + sum_{w < W-1} weight[c][w] state[c][w] + weight[c][W-1] u[c]
    out[c] = silu(z[c]) = z[c] / (1 + exp(-z[c]))     (or z[c] without activation)

and shifts the state left by one column, appending u.  The output splits, in
channel order, into x (the SSM's v, H heads x d), B (its k, G groups x n) and
C (its q).  Over a whole sequence this is the cross-correlation of each
channel's input with its weight row, which the pins check against
numpy.convolve.
"""
from __future__ import annotations

import numpy as np


def silu(z):
    """z * sigmoid(z), in float64."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def conv_state_step(state, u, weight, bias=None, activation=True):
    """One decode step of the convolution state for a batch.

    state  [B, C, W-1]  (DS layout: channel-major, oldest entry first)
    u      [B, C]       the new input column
    weight [C, W], bias [C] or None
    Returns (new_state [B, C, W-1], out [B, C]); inputs are not modified.
    """
    state = np.asarray(state, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    B, C, Wm1 = state.shape
    W = Wm1 + 1
    if weight.shape != (C, W) or u.shape != (B, C):
        raise ValueError("shape mismatch")
    out = np.empty((B, C))
    new_state = np.empty_like(state)
    for b in range(B):
        for c in range(C):
            window = list(state[b, c]) + [u[b, c]]  # oldest .. newest
            z = 0.0 if bias is None else float(bias[c])
            for w in range(W):
                z += float(weight[c, w]) * window[w]
            out[b, c] = silu(z) if activation else z
            new_state[b, c] = window[1:]
    return new_state, out


def split_xbc(out, dx, dbc):
    """The x, B and C sub-projections of a step's output [B, dx + 2 dbc]."""
    out = np.asarray(out)
    if out.shape[1] != dx + 2 * dbc:
        raise ValueError("channel count is not dx + 2 dbc")
    return out[:, :dx], out[:, dx:dx + dbc], out[:, dx + dbc:]
