"""The layers around the KDA recurrence, in fp64 NumPy -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may use this
module; the product never does. Definitions (Kimi K3 wiki):

* "Notations mathématiques", table "Fonctions": Sigmoid(x) = 1 / (1 + e^-x);
  L2Norm(x) = x / ||x||_2; RMSNorm(x) = x / sqrt(mean_i x_i^2 + eps) (*) g with a learned
  per-channel weight g; ShortConv = causal convolution with a kernel of size 4.
* table "Attention et KDA": q_t, k_t are L2-normalised; g_t in (g_min, 0)^{d_k}; A_h is a
  learned per-head log scale; b_alpha^h a per-head decay bias in R^{d_k}; z_t the decay logit in
  R^{d_k}; o~_t the raw output, before the gate.
* "Glossaire", entry "Décroissance bornée": g = g_min sigma(e^A z), g_min = -5.
* "Tableau des spécifications": ShortConv kernel 4 on KDA; RMSNorm epsilon 1e-5; "full-rank KDA
  gate: yes". Chapter 03: RMSNorm on the recurrent output of KDA; L2Norm on KDA's queries and
  keys.

Readings of what the pages leave open:

* gate: g = g_min * sigma(e^{A_h} z + b_alpha^h) -- the bias of the notation table added to the
  scaled logit of the glossary's formula;
* ShortConv: depthwise (one 4-tap filter per channel of each of q, k, v), causal with zeros
  before the first token of each sequence, no activation after it:
  y_t[c] = sum_{j=0..3} w[c, j] x_{t-j}[c];
* post-core: y_t = RMSNorm(o~_t) (*) sigma(u_t), u_t the output of the full-rank gate projection
  (an input here), RMSNorm over the d_v channels of each head with one weight vector shared by
  the heads.
"""
from __future__ import annotations

import numpy as np

G_MIN = -5.0
RMS_EPS = 1e-5


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-np.asarray(x, dtype=np.float64)))


def l2norm(x):
    """x / ||x||_2 over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True))


def rmsnorm(x, w, eps=RMS_EPS):
    """x / sqrt(mean(x^2) + eps) * w over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def decay_gate(z, A, b, g_min=G_MIN):
    """g = g_min * sigma(e^{A_h} z + b_h). z: [..., H, d_k]; A: [H]; b: [H, d_k]."""
    z = np.asarray(z, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return g_min * sigmoid(np.exp(A)[:, None] * z + b)


def short_conv(x, w, cu_seqlens=None):
    """Causal depthwise convolution along T with 4 taps, zeros before each sequence's start.

    x: [B, T, H, d]; w: [H, d, 4] with w[..., j] multiplying the token j steps back.
    cu_seqlens (packed batches, B = 1): the convolution restarts at every sequence start.
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    B, T = x.shape[:2]
    starts = np.zeros(T, dtype=np.int64)  # first token of the sequence each token belongs to
    if cu_seqlens is not None:
        cu = [int(c) for c in cu_seqlens]
        for s in range(len(cu) - 1):
            starts[cu[s]:cu[s + 1]] = cu[s]
    y = np.zeros_like(x)
    for t in range(T):
        for j in range(4):
            src = t - j
            if src < starts[t]:
                break
            y[:, t] += w[None, :, :, j] * x[:, src]
    return y


def pre_core(q_raw, k_raw, v_raw, z, conv_q, conv_k, conv_v, A, b, cu_seqlens=None):
    """The inputs of the recurrence from the raw projections: q, k = L2Norm(ShortConv(.)),
    v = ShortConv(v_raw), g = the bounded decay gate of z."""
    q = l2norm(short_conv(q_raw, conv_q, cu_seqlens))
    k = l2norm(short_conv(k_raw, conv_k, cu_seqlens))
    v = short_conv(v_raw, conv_v, cu_seqlens)
    g = decay_gate(z, A, b)
    return q, k, v, g


def post_core(o_raw, u, w, eps=RMS_EPS):
    """y = RMSNorm(o~) * sigma(u), per token and head over the d_v channels."""
    return rmsnorm(o_raw, w, eps) * sigmoid(u)
