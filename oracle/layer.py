"""fp64 oracle of the element-wise operations around the rule in a
GatedDeltaNet layer.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle``).

The pages name these operations only through the layer's buffers (the "qkvz"
activations [B, T, H, D] of PR "Shard the GatedDeltaNet sequence under
ici_context_parallelism", description): q and k enter the rule normalised, the
gates come from logits, and z gates the output.  The plain forms taken here:

    q_n = q / sqrt(sum(q^2) + eps)  (per token and head, eps = 1e-6; k alike)
    beta = sigmoid(b),  g = -softplus(a)
    y = o * silu(z),  silu(z) = z * sigmoid(z)

Each backward is the derivative of its forward, written out:
    d/dq of q_n:   dq = (dq_n - q_n (q_n . dq_n)) / sqrt(sum(q^2) + eps)
    d/da of g:     da = -sigmoid(a) dg
    d/db of beta:  db = sigmoid(b) (1 - sigmoid(b)) dbeta
    d/do, d/dz:    do = dy silu(z),  dz = dy o sigmoid(z) (1 + z (1 - sigmoid(z)))
"""
from __future__ import annotations

import numpy as np
import torch

EPS = 1e-6


def sigmoid(x):
    """1 / (1 + exp(-x)), evaluated as exp(x) / (1 + exp(x)) for x < 0 so that
    the tail keeps its relative accuracy."""
    x = np.asarray(x, np.float64)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def softplus(x):
    x = np.asarray(x, np.float64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def l2norm(x, eps=EPS):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def l2norm_bwd(x, dy, eps=EPS):
    x = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
    y = x * r
    return r * (dy - y * np.sum(y * dy, axis=-1, keepdims=True))


def gates(a, b):
    """(g, beta) from the logits."""
    return -softplus(a), sigmoid(b)


def gates_bwd(a, b, dg, dbeta):
    """(da, db) from the cotangents of g and beta."""
    sb = sigmoid(b)
    return -sigmoid(a) * np.asarray(dg, np.float64), sb * (1.0 - sb) * np.asarray(dbeta, np.float64)


def silu(z):
    z = np.asarray(z, np.float64)
    return z * sigmoid(z)


def out_gate(o, z):
    return np.asarray(o, np.float64) * silu(z)


def out_gate_bwd(o, z, dy):
    """(do, dz) from the cotangent of y = o * silu(z)."""
    o = np.asarray(o, np.float64)
    z = np.asarray(z, np.float64)
    dy = np.asarray(dy, np.float64)
    s = sigmoid(z)
    return dy * z * s, dy * o * s * (1.0 + z * (1.0 - s))


def rule_inputs(raw):
    """The rule's inputs from a layer's raw inputs: ``raw`` is an Inputs whose
    q, k are unnormalised and whose g, beta hold the logits a, b.  q_n and k_n
    are formed in fp64 and rounded to bf16 (the precision the rule takes them
    in); g and beta are formed in fp64 and rounded to fp32."""
    from linear_attention_rnn_gb300.inputs import Inputs
    f64 = lambda t: t.detach().cpu().to(torch.float64).numpy()
    qn = torch.from_numpy(l2norm(f64(raw.q))).to(torch.bfloat16)
    kn = torch.from_numpy(l2norm(f64(raw.k))).to(torch.bfloat16)
    g, beta = gates(f64(raw.g), f64(raw.beta))
    return Inputs(raw.wl, qn, kn, raw.v, torch.from_numpy(g.astype(np.float32)),
                  torch.from_numpy(beta.astype(np.float32)), raw.h0, raw.dO, raw.dhT)
