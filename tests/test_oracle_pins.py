"""Pins of the fp64 oracle to facts other than itself (CPU only).

Each test ties the oracle (the per-token C reference and its adjoint, and the
chunked numpy form) to something it does not compute itself: hand-derived
worked examples, closed forms, a textbook routine, invariants of the rule,
brute force across two independent routes, and finite differences.
"""
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.signal

import oracle
from oracle import chunked
from conftest import as64, from_arrays, head, random_small, relmax

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(":", 1)
            vals[key.strip()] = np.array([float(x) for x in rest.split()])
    return vals


# --------------------------------------------------------------- worked examples
def test_scalar_worked_example():
    gd = _read_golden("scalar_rule_worked_example.txt")
    T = len(gd["k"])
    inp = from_arrays(gd["q"].reshape(1, T, 1, 1), gd["k"].reshape(1, T, 1, 1),
                      gd["v"].reshape(1, T, 1, 1), gd["g"].reshape(1, T, 1),
                      gd["beta"].reshape(1, T, 1), gd["h0"].reshape(1, 1, 1, 1))
    o, hT = oracle.fwd(inp)
    assert np.max(np.abs(o[0, :, 0] - gd["o"])) <= gd["tol"][0]
    assert np.max(np.abs(hT.ravel() - gd["hT"])) <= gd["tol"][0]
    # the chunked route, every chunk size
    for C in (1, 2, 3):
        oc, hc = chunked.head_fwd(*head(inp, 0, 0), C)
        assert np.max(np.abs(oc[:, 0] - gd["o"])) <= gd["tol"][0]
        assert np.max(np.abs(hc.ravel() - gd["hT"])) <= gd["tol"][0]


def test_basis_overwrite_worked_example():
    gd = _read_golden("basis_overwrite_worked_example.txt")
    T = len(gd["g"])
    inp = from_arrays(gd["q"].reshape(1, T, 1, 2), gd["k"].reshape(1, T, 1, 2),
                      gd["v"].reshape(1, T, 1, 2), gd["g"].reshape(1, T, 1),
                      gd["beta"].reshape(1, T, 1), gd["h0"].reshape(1, 1, 2, 2))
    o, hT = oracle.fwd(inp)
    assert np.array_equal(o[0].ravel(), gd["o"])
    assert np.array_equal(hT.ravel(), gd["hT"])
    oc, hc = chunked.head_fwd(*head(inp, 0, 0), 2)
    assert np.allclose(oc.ravel(), gd["o"], atol=1e-14)
    assert np.allclose(hc.ravel(), gd["hT"], atol=1e-14)


# ------------------------------------------------------------------ closed forms
def test_beta_zero_is_pure_decay():
    """beta = 0: h_T = exp(sum g) h0 and o_t = exp(G_t) h0^T q_t."""
    inp = random_small(T=37, dk=8, dv=6, seed=1)
    inp.beta.zero_()
    o, hT = oracle.fwd(inp)
    q, k, v, g, beta, h0 = head(inp, 0, 0)
    G = np.cumsum(g)
    assert relmax(hT[0], np.exp(G[-1]) * h0) < 1e-13
    ref_o = np.exp(G)[:, None] * (q @ h0)
    assert relmax(o[0], ref_o) < 1e-13


def test_scalar_case_is_first_order_filter():
    """d_k = 1, k = q = 1, constant a and beta: h_t = a (1 - beta) h_{t-1} +
    beta v_t, a first-order IIR filter (scipy.signal.lfilter)."""
    T = 50
    rng = np.random.default_rng(3)
    v = rng.standard_normal(T)
    a, bt = 0.9, 0.3
    ones = np.ones((1, T, 1, 1))
    inp = from_arrays(ones, ones, v.reshape(1, T, 1, 1),
                      np.full((1, T, 1), np.log(a)), np.full((1, T, 1), bt),
                      np.full((1, 1, 1, 1), 0.75))
    o, hT = oracle.fwd(inp)
    vv = as64(inp, "v").ravel()
    af = float(np.exp(np.float64(inp.g[0, 0, 0])))
    bf = float(inp.beta[0, 0, 0])
    c = af * (1 - bf)
    zi = np.array([c * 0.75])
    ref, _ = scipy.signal.lfilter([bf], [1.0, -c], vv, zi=zi)
    assert relmax(o[0, :, 0], ref) < 1e-13
    assert abs(hT.ravel()[0] - ref[-1]) < 1e-13 * max(1, abs(ref[-1]))


def test_unit_key_write_is_retrieved_exactly():
    """beta = 1 and |k| = 1: k_t^T h_t = v_t^T whatever the gate, because
    k^T (I - k k^T) = 0.  Keys with four entries of +-1/2 are exact in bf16."""
    rng = np.random.default_rng(4)
    T, d = 30, 16
    k = np.zeros((1, T, 1, d))
    for t in range(T):
        idx = rng.choice(d, 4, replace=False)
        k[0, t, 0, idx] = 0.5 * rng.choice([-1, 1], 4)
    v = rng.standard_normal((1, T, 1, d))
    g = -rng.uniform(0, 2, (1, T, 1))
    inp = from_arrays(k, k, v, g, np.ones((1, T, 1)), rng.standard_normal((1, 1, d, d)))
    o, _ = oracle.fwd(inp)  # q_t = k_t, so o_t = h_t^T k_t
    assert np.max(np.abs(o[0] - as64(inp, "v")[0, :, 0])) < 1e-12


def test_ladder_all_ones_closed_form():
    """S = strictly-lower ones: (I + S) is the lower ones matrix, whose inverse
    is I minus the first subdiagonal."""
    for C in (2, 16, 128):
        S = np.tril(np.ones((C, C)), -1)
        ref = np.eye(C) - np.eye(C, k=-1)
        assert np.array_equal(chunked.ut_ladder(S), ref)
        assert np.array_equal(chunked.ut_forward_substitution(S), ref)


@pytest.mark.parametrize("kind", ["random", "gaussian_unnormalised", "workload"])
def test_ladder_matches_library_solve(kind):
    rng = np.random.default_rng(5)
    C = 128
    if kind == "random":
        S = np.tril(rng.uniform(-0.1, 0.1, (C, C)), -1)
    elif kind == "gaussian_unnormalised":
        S = np.tril(rng.standard_normal((C, C)), -1)
    else:
        inp = random_small(T=C, dk=128, dv=8, seed=6)
        q, k, v, g, beta, _ = head(inp, 0, 0)
        S = chunked.chunk_intermediates(q, k, v, g, beta)["S"]
    I = np.eye(C)
    ref = scipy.linalg.solve_triangular(I + S, I, lower=True, unit_diagonal=True)
    lad = chunked.ut_ladder(S)
    fs = chunked.ut_forward_substitution(S)
    scale = np.max(np.abs(ref))
    assert np.max(np.abs(lad - ref)) <= 1e-12 * scale
    assert np.max(np.abs(fs - ref)) <= 1e-12 * scale
    if kind != "gaussian_unnormalised":  # inverse of order 1: residual is absolute
        assert np.max(np.abs((I + S) @ lad - I)) < 1e-13


def test_ladder_non_power_of_two():
    rng = np.random.default_rng(7)
    for C in (3, 5, 100):
        S = np.tril(rng.uniform(-0.3, 0.3, (C, C)), -1)
        I = np.eye(C)
        assert np.max(np.abs((I + S) @ chunked.ut_ladder(S) - I)) < 1e-13


def test_chunk_size_one_reduces_to_rule():
    """C = 1: S is empty, T = I, and one chunk step is one token of the rule."""
    inp = random_small(T=9, dk=4, dv=3, seed=8)
    it = chunked.chunk_intermediates(*[x[:1] for x in head(inp, 0, 0)[:5]])
    assert np.array_equal(it["T"], np.eye(1))
    o, hT = oracle.fwd(inp)
    oc, hc = chunked.head_fwd(*head(inp, 0, 0), 1)
    assert relmax(oc, o[0]) < 1e-13 and relmax(hc, hT[0]) < 1e-13


# ---------------------------------------------- two routes: chunked vs per-token
@pytest.mark.parametrize("C", [1, 2, 4, 16, 64, 128])
def test_chunked_equals_per_token(C):
    for (dk, dv, T, shift) in ((4, 4, 61, 0.0), (8, 8, 200, -3.0), (128, 128, 300, 1.0)):
        inp = random_small(B=1, T=T, Hk=1, Hv=2, dk=dk, dv=dv, seed=C + dk, gate_shift=shift)
        o, hT = oracle.fwd(inp)
        for j in range(2):
            oc, hc = chunked.head_fwd(*head(inp, 0, j), C)
            assert relmax(oc, o[j]) < 1e-10, (C, dk, j)
            assert relmax(hc, hT[j]) < 1e-10, (C, dk, j)


def test_ladder_and_substitution_routes_agree_in_the_chunk_form():
    inp = random_small(T=256, dk=16, dv=16, seed=9, gate_shift=-4.0)
    args = head(inp, 0, 0)
    o1, h1 = chunked.head_fwd(*args, 64, use_ladder=True)
    o2, h2 = chunked.head_fwd(*args, 64, use_ladder=False)
    assert relmax(o1, o2) < 1e-12 and relmax(h1, h2) < 1e-12


# ---------------------------------------------------------------- invariants
def test_linear_in_values_and_initial_state():
    """o and h_T are jointly linear in (v, h0): superposition."""
    inp = random_small(T=70, dk=8, dv=8, seed=10)
    o, hT = oracle.fwd(inp)
    a = random_small(T=70, dk=8, dv=8, seed=10)
    a.h0.zero_()
    b = random_small(T=70, dk=8, dv=8, seed=10)
    b.v.zero_()
    oa, ha = oracle.fwd(a)
    ob, hb = oracle.fwd(b)
    assert relmax(oa + ob, o) < 1e-13 and relmax(ha + hb, hT) < 1e-13


def test_value_column_permutation():
    inp = random_small(T=40, dk=8, dv=8, seed=11)
    perm = np.random.default_rng(0).permutation(8)
    o, hT = oracle.fwd(inp)
    p = random_small(T=40, dk=8, dv=8, seed=11)
    p.v = p.v[..., perm].contiguous()
    p.h0 = p.h0[..., perm].contiguous()
    op, hp = oracle.fwd(p)
    assert np.array_equal(op, o[..., perm]) and np.array_equal(hp, hT[..., perm])


def test_gqa_shared_key_equals_repeated_key():
    """Hk=1 shared by Hv=2 equals Hk=Hv=2 with the key/query head repeated."""
    inp = random_small(B=2, T=33, Hk=1, Hv=2, dk=8, dv=8, seed=12)
    o, hT = oracle.fwd(inp)
    rep = random_small(B=2, T=33, Hk=1, Hv=2, dk=8, dv=8, seed=12)
    rep.q = rep.q.repeat(1, 1, 2, 1).contiguous()
    rep.k = rep.k.repeat(1, 1, 2, 1).contiguous()
    rep.wl = rep.wl.replace(Hk=2)
    o2, h2 = oracle.fwd(rep)
    assert np.array_equal(o, o2) and np.array_equal(hT, h2)


# ------------------------------------------------------- composition / segments
def _rand_map(rng, d, dv, scale=0.3):
    return rng.standard_normal((d, d)) * scale, rng.standard_normal((d, dv))


def test_compose_is_associative_with_identity():
    rng = np.random.default_rng(13)
    m1, m2, m3 = (_rand_map(rng, 6, 5) for _ in range(3))
    l = chunked.compose(m3, chunked.compose(m2, m1))
    r = chunked.compose(chunked.compose(m3, m2), m1)
    assert relmax(l[0], r[0]) < 1e-14 and relmax(l[1], r[1]) < 1e-14
    I = chunked.identity_map(6, 5)
    for x in (chunked.compose(I, m1), chunked.compose(m1, I)):
        assert np.array_equal(x[0], m1[0]) and np.array_equal(x[1], m1[1])
    # applying the composition equals applying the maps in turn
    h = rng.standard_normal((6, 5))
    seq = m3[0] @ (m2[0] @ (m1[0] @ h + m1[1]) + m2[1]) + m3[1]
    assert relmax(l[0] @ h + l[1], seq) < 1e-14


def test_chunk_affine_map_reproduces_chunk_step():
    inp = random_small(T=64, dk=8, dv=8, seed=14)
    q, k, v, g, beta, h0 = head(inp, 0, 0)
    it = chunked.chunk_intermediates(q, k, v, g, beta)
    A, B = chunked.chunk_affine(it)
    _, hT = oracle.fwd(inp)
    assert relmax(A @ h0 + B, hT[0]) < 1e-12


@pytest.mark.parametrize("n_seg", [1, 2, 7, 148])
def test_segment_scan_equals_sequential_walk(n_seg):
    # slow decay so that the incoming state matters across segments
    inp = random_small(T=600, dk=8, dv=8, seed=15, gate_shift=-6.0)
    o, hT = oracle.fwd(inp)
    os_, hs, _ = chunked.head_fwd_segmented(*head(inp, 0, 0), 4, n_seg)
    assert relmax(os_, o[0]) < 1e-10 and relmax(hs, hT[0]) < 1e-10


def test_segment_scan_negative_control():
    """Replaying every segment from a zero state (dropping the incoming
    state) must fail the same tolerance."""
    inp = random_small(T=600, dk=8, dv=8, seed=15, gate_shift=-6.0)
    o, hT = oracle.fwd(inp)
    bad, _, _ = chunked.head_fwd_segmented(*head(inp, 0, 0), 4, 7, drop_incoming=True)
    assert relmax(bad, o[0]) > 1e-2


def test_inclusive_prefix_matches_pairwise_folds():
    rng = np.random.default_rng(16)
    maps = [_rand_map(rng, 5, 4) for _ in range(9)]
    As, Bs = chunked.inclusive_prefix([m[0] for m in maps], [m[1] for m in maps])
    h = rng.standard_normal((5, 4))
    x = h
    for i, (A, B) in enumerate(maps):
        x = A @ x + B
        assert relmax(As[i] @ h + Bs[i], x) < 1e-13


# ---------------------------------------------------------------- gradients
def test_finite_differences_match_adjoint():
    """Central differences in fp64 along random directions.  The bf16 inputs
    (q, k, v) are replaced by a fp64 evaluation through the chunked route
    (continuous in every input); g, beta and h0 go through the C rule."""
    base = dict(B=1, T=24, Hk=1, Hv=1, dk=6, dv=5, seed=17, bwd=True)
    inp = random_small(**base)
    res = oracle.bwd(inp, ckpt=5)
    q, k, v, g, beta, h0 = head(inp, 0, 0)
    dO = as64(inp, "dO")[0, :, 0]
    dhT = as64(inp, "dhT")[0, 0]

    def L(q_, k_, v_, g_, b_, h_):
        o, hT = chunked.head_fwd(q_, k_, v_, g_, b_, h_, 4)
        return float(np.sum(o * dO) + np.sum(hT * dhT))

    rng = np.random.default_rng(18)
    args = [q, k, v, g, beta, h0]
    grads = [res["dq_v"][0], res["dk_v"][0], res["dv"][0], res["dg"][0],
             res["dbeta"][0], res["dh0"][0]]
    for i, (x, gx) in enumerate(zip(args, grads)):
        d = rng.standard_normal(x.shape)
        h = 1e-6 * (1 + np.max(np.abs(x)))
        ap = list(args)
        am = list(args)
        ap[i] = x + h * d
        am[i] = x - h * d
        fd = (L(*ap) - L(*am)) / (2 * h)
        an = float(np.sum(gx * d))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (i, fd, an)


def test_adjoint_dot_product_identity():
    """For the map L(v, h0) = (o, hT) at fixed q, k, g, beta (linear):
    <dO, o> + <dhT, hT> = <dv, v> + <dh0, h0> exactly (up to rounding)."""
    inp = random_small(B=1, T=50, Hk=1, Hv=1, dk=8, dv=8, seed=19, bwd=True)
    o, hT = oracle.fwd(inp)
    res = oracle.bwd(inp, ckpt=7)
    lhs = np.sum(o[0] * as64(inp, "dO")[0, :, 0]) + np.sum(hT[0] * as64(inp, "dhT")[0, 0])
    rhs = np.sum(res["dv"][0] * as64(inp, "v")[0, :, 0]) + np.sum(res["dh0"][0] * as64(inp, "h0")[0, 0])
    assert abs(lhs - rhs) < 1e-12 * max(1, abs(lhs))


def test_checkpoint_interval_does_not_change_adjoint():
    inp = random_small(B=1, T=45, Hk=1, Hv=2, dk=8, dv=8, seed=20, bwd=True)
    a = oracle.bwd(inp, ckpt=1)
    b = oracle.bwd(inp, ckpt=16)
    for key in ("dq_v", "dk_v", "dv", "dg", "dbeta", "dh0"):
        assert relmax(a[key], b[key]) < 1e-13


@pytest.mark.parametrize("C", [4, 16, 64])
def test_chunked_backward_equals_per_token_adjoint(C):
    for dk, dv, shift in ((8, 8, 0.0), (16, 12, -4.0)):
        inp = random_small(B=1, T=150, Hk=1, Hv=2, dk=dk, dv=dv, seed=21 + C,
                           gate_shift=shift, bwd=True)
        res = oracle.bwd(inp)
        for j in range(2):
            q, k, v, g, beta, h0 = head(inp, 0, j)
            dq, dk_, dv_, dg, db, dh0, _ = chunked.head_bwd(
                q, k, v, g, beta, h0, as64(inp, "dO")[0, :, j], as64(inp, "dhT")[0, j], C)
            for a, r in ((dq, res["dq_v"][j]), (dk_, res["dk_v"][j]), (dv_, res["dv"][j]),
                         (dg, res["dg"][j]), (db, res["dbeta"][j]), (dh0, res["dh0"][j])):
                assert relmax(a, r) < 1e-9


def test_key_head_gradient_sums():
    inp = random_small(B=1, T=20, Hk=1, Hv=2, dk=4, dv=4, seed=22, bwd=True)
    res = oracle.bwd(inp)
    kg = oracle.key_head_grads(inp.wl, res)
    dq, dk = kg[(0, 0)]
    assert np.array_equal(dq, res["dq_v"][0] + res["dq_v"][1])
    assert np.array_equal(dk, res["dk_v"][0] + res["dk_v"][1])
