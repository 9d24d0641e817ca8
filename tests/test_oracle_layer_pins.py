"""Pins of the layer oracle (oracle/layer.py) to facts other than itself:
library routines for the activations, closed forms, and central differences
(fp64) of each forward against its written-out backward, alone and through
the whole layer (normalised q/k, gate logits, the rule by the chunked route,
output gate)."""
import numpy as np
import scipy.special

from oracle import chunked
from oracle import layer as ol


def test_activations_match_library_routines():
    x = np.linspace(-40.0, 40.0, 801)
    assert np.allclose(ol.sigmoid(x), scipy.special.expit(x), rtol=1e-14, atol=1e-300)
    assert np.allclose(ol.softplus(x), np.logaddexp(0.0, x), rtol=1e-14, atol=1e-300)
    assert ol.sigmoid(0.0) == 0.5
    assert abs(ol.softplus(0.0) - np.log(2.0)) < 1e-15
    assert ol.silu(0.0) == 0.0
    # the decay of a logit: exp(-softplus(a)) = 1 / (1 + exp(a)) = sigmoid(-a)
    g, _ = ol.gates(x, x)
    assert np.allclose(np.exp(g), scipy.special.expit(-x), rtol=1e-13, atol=1e-300)


def test_l2norm_gives_unit_rows_and_keeps_direction():
    rng = np.random.default_rng(30)
    x = rng.standard_normal((7, 3, 128)) * 5.0
    y = ol.l2norm(x, eps=0.0)
    assert np.allclose(np.linalg.norm(y, axis=-1), 1.0, atol=1e-14)
    assert np.allclose(y * np.linalg.norm(x, axis=-1, keepdims=True), x, atol=1e-12)


def _fd_check(f, fb, xs, seed, rtol=1e-7):
    """Central differences of the scalar <f(xs), w> along random directions
    against <fb(xs, w), d> for each argument."""
    rng = np.random.default_rng(seed)
    out = f(*xs)
    outs = out if isinstance(out, tuple) else (out,)
    ws = [rng.standard_normal(o.shape) for o in outs]
    grads = fb(*xs, *ws)
    grads = grads if isinstance(grads, tuple) else (grads,)
    for i, (x, gx) in enumerate(zip(xs, grads)):
        d = rng.standard_normal(x.shape)
        h = 1e-6 * (1 + np.max(np.abs(x)))
        xp, xm = list(xs), list(xs)
        xp[i] = x + h * d
        xm[i] = x - h * d
        fp, fm = f(*xp), f(*xm)
        fp = fp if isinstance(fp, tuple) else (fp,)
        fm = fm if isinstance(fm, tuple) else (fm,)
        fd = sum(np.sum((a - b) * w) for a, b, w in zip(fp, fm, ws)) / (2 * h)
        an = float(np.sum(gx * d))
        assert abs(fd - an) <= rtol * max(1.0, abs(an)), (i, fd, an)


def test_elementwise_backwards_match_finite_differences():
    rng = np.random.default_rng(31)
    x = rng.standard_normal((5, 2, 16)) * 2.0
    _fd_check(lambda x_: ol.l2norm(x_), lambda x_, w: ol.l2norm_bwd(x_, w), [x], 32)
    a = rng.standard_normal((9, 3)) * 3.0
    b = rng.standard_normal((9, 3)) * 3.0
    _fd_check(lambda a_, b_: ol.gates(a_, b_), lambda a_, b_, wg, wb: ol.gates_bwd(a_, b_, wg, wb),
              [a, b], 33)
    o = rng.standard_normal((6, 8))
    z = rng.standard_normal((6, 8)) * 3.0
    _fd_check(lambda o_, z_: ol.out_gate(o_, z_), lambda o_, z_, w: ol.out_gate_bwd(o_, z_, w),
              [o, z], 34)


def test_layer_backward_matches_finite_differences():
    """The whole layer on one head: y = out_gate(rule(l2norm(q), l2norm(k), v,
    -softplus(a), sigmoid(b), h0), z), loss <y, dy> + <hT, dhT>; the composed
    backward (gate, rule by the chunked route, activations, normalisation)
    against central differences in every input."""
    rng = np.random.default_rng(35)
    T, dk, dv = 20, 6, 5
    q = rng.standard_normal((T, dk)) * 2
    k = rng.standard_normal((T, dk)) * 2
    v = rng.standard_normal((T, dv))
    a = rng.standard_normal(T) - 1.0
    b = rng.standard_normal(T)
    z = rng.standard_normal((T, dv))
    h0 = rng.standard_normal((dk, dv)) * 0.5
    dy = rng.standard_normal((T, dv))
    dhT = rng.standard_normal((dk, dv)) * 0.3

    def loss(q_, k_, v_, a_, b_, z_, h_):
        g, beta = ol.gates(a_, b_)
        o, hT = chunked.head_fwd(ol.l2norm(q_), ol.l2norm(k_), v_, g, beta, h_, 4)
        return float(np.sum(ol.out_gate(o, z_) * dy) + np.sum(hT * dhT))

    g, beta = ol.gates(a, b)
    qn, kn = ol.l2norm(q), ol.l2norm(k)
    o, _ = chunked.head_fwd(qn, kn, v, g, beta, h0, 4)
    do, dz = ol.out_gate_bwd(o, z, dy)
    dqn, dkn, dvv, dg, dbeta, dh0, _ = chunked.head_bwd(qn, kn, v, g, beta, h0, do, dhT, 4)
    da, db = ol.gates_bwd(a, b, dg, dbeta)
    grads = [ol.l2norm_bwd(q, dqn), ol.l2norm_bwd(k, dkn), dvv, da, db, dz, dh0]
    args = [q, k, v, a, b, z, h0]
    for i, (x, gx) in enumerate(zip(args, grads)):
        d = rng.standard_normal(x.shape)
        h = 1e-6 * (1 + np.max(np.abs(x)))
        ap, am = list(args), list(args)
        ap[i] = x + h * d
        am[i] = x - h * d
        fd = (loss(*ap) - loss(*am)) / (2 * h)
        an = float(np.sum(gx * d))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (i, fd, an)
