"""GPU parity of the backward path against the fp64 per-token adjoint.

Tolerance: max|dx - dx_ref| <= 3e-2 max|dx_ref| for every gradient tensor
(dq and dk summed over the value heads of each key head)."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_rnn_gb300.inputs import WORKLOADS, make_host
from conftest import assert_rel

pytestmark = pytest.mark.gpu

G_TOL = 3e-2


def _check_bwd(gdn, inp, n_segments=0, key_heads=None, record=False):
    """Device backward against the per-token adjoint on the given (b, kh) key
    heads and their value heads (default: all), with the oracle run once over
    all of them; record=True enters the errors in the margin table."""
    wl = inp.wl
    d = inp.to("cuda")
    dq, dk, dv, dg, db, dh0 = gdn.chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.dO, d.dhT,
                                            n_segments=n_segments)
    torch.cuda.synchronize()
    dq, dk, dv = (x.float().cpu().numpy() for x in (dq, dk, dv))
    dg, db, dh0 = (x.cpu().numpy() for x in (dg, db, dh0))
    key_heads = key_heads or [(b, kh) for b in range(wl.B) for kh in range(wl.Hk)]
    grp = wl.Hv // wl.Hk
    heads = [(b, kh * grp + r) for b, kh in key_heads for r in range(grp)]
    res = oracle.bwd(inp, heads=heads)
    kq = oracle.key_head_grads(wl, res)
    idx = {h: i for i, h in enumerate(res["heads"])}
    m = (lambda t: (wl.name, t)) if record else (lambda t: None)
    worst = {}
    for b, kh in key_heads:
        e = [assert_rel(dq[b, :, kh], kq[(b, kh)][0], G_TOL, f"dq[{b},{kh}]", m("dq")),
             assert_rel(dk[b, :, kh], kq[(b, kh)][1], G_TOL, f"dk[{b},{kh}]", m("dk"))]
        for r in range(grp):
            j = kh * grp + r
            i = idx[(b, j)]
            e += [assert_rel(dv[b, :, j], res["dv"][i], G_TOL, f"dv[{b},{j}]", m("dv")),
                  assert_rel(dg[b, :, j], res["dg"][i], G_TOL, f"dg[{b},{j}]", m("dg")),
                  assert_rel(db[b, :, j], res["dbeta"][i], G_TOL, f"dbeta[{b},{j}]", m("dbeta")),
                  assert_rel(dh0[b, j], res["dh0"][i], G_TOL, f"dh0[{b},{j}]", m("dh0"))]
        worst[(b, kh)] = max(e)
    return worst


def _small(T, Hk=1, Hv=2, shift=0.0, h0=0.3, seed=0, B=1):
    return make_host(WORKLOADS["tiny_t1024"].replace(B=B, T=T, Hk=Hk, Hv=Hv, gate_shift=shift,
                                                    h0_std=h0, seed=seed, backward=True))


@pytest.mark.parametrize("T", [128, 256, 300])
def test_small_bwd(gdn_lib, T):
    _check_bwd(gdn_lib, _small(T, seed=T))


def test_bwd_slow_decay(gdn_lib):
    _check_bwd(gdn_lib, _small(640, shift=-4.0, h0=0.5, seed=2))


@pytest.mark.parametrize("shift", [4.0, 8.0])
def test_bwd_fast_decay(gdn_lib, shift):
    # g about -4 and -8 per token: G drops by more than 100 (base 2) inside
    # some (4.0) or all (8.0) 16-token blocks, so the kernels take the direct
    # exponentials there instead of the factored decays
    _check_bwd(gdn_lib, _small(300, shift=shift, h0=0.5, seed=int(shift) + 40))


@pytest.mark.parametrize("T", [1, 77, 129])
def test_bwd_ragged_and_tiny(gdn_lib, T):
    _check_bwd(gdn_lib, _small(T, Hk=2, Hv=4, seed=100 + T))


@pytest.mark.parametrize("B,T,Hk,Hv", [(3, 333, 3, 6), (1, 40 * 128, 1, 4)])
def test_bwd_unit_ranges(gdn_lib, B, T, Hk, Hv):
    """Preparation ranges that start inside a key head's group or cut it (see
    the forward test of the same name), through the backward path."""
    _check_bwd(gdn_lib, _small(T, Hk=Hk, Hv=Hv, seed=T + Hv, B=B))


@pytest.mark.parametrize("S", [2, 3, 7])
def test_bwd_segment_counts(gdn_lib, S):
    _check_bwd(gdn_lib, _small(1024 + 50, shift=-5.0, h0=0.5, seed=5), n_segments=S)


def test_bwd_no_initial_state_no_final_cotangent(gdn_lib):
    inp = _small(256, seed=9, h0=0.0)
    inp.dhT = None
    d = inp.to("cuda")
    out = gdn_lib.chunk_bwd(d.q, d.k, d.v, d.g, d.beta, None, d.dO, None)
    res = oracle.bwd(inp)
    assert_rel(out[2][0, :, 0].float().cpu().numpy(), res["dv"][0], G_TOL, "dv")
    assert_rel(out[5][0, 0].cpu().numpy(), res["dh0"][0], G_TOL, "dh0")


def test_bwd_empty_sequence(gdn_lib):
    inp = _small(0, seed=1)
    d = inp.to("cuda")
    dq, dk, dv, dg, db, dh0 = gdn_lib.chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.dO, d.dhT)
    assert torch.equal(dh0.cpu(), inp.dhT)


def test_layer_workload_bwd(gdn_lib):
    """T=4096, 16 key heads shared by 32 value heads: every gradient of every
    head against the per-token adjoint."""
    inp = make_host(WORKLOADS["layer_t4096"])
    _check_bwd(gdn_lib, inp, record=True)


def test_batched_workload_bwd(gdn_lib):
    """B=2, T=8192, 16 key heads shared by 32 value heads: every gradient of
    every head of both batch rows against the per-token adjoint."""
    inp = make_host(WORKLOADS["batched_b2_t8192"])
    _check_bwd(gdn_lib, inp, record=True)


# ------------------------------------------- forward keeps w, u, P, T for the backward
@pytest.mark.parametrize("name,T,S", [("layer_t4096", 4096, 1), ("tiny_t1024", 300, 1),
                                      ("tiny_t1024", 1024 + 50, 3), ("tiny_t1024", 128, 1),
                                      ("tiny_t1024", 129, 1), ("tiny_t1024", 256 + 7, 2),
                                      ("tiny_t1024", 1024 + 50, 9)])
def test_saved_chunk_quantities(gdn_lib, name, T, S):
    """The forward that keeps w, u, P, T, the entering states and Delta
    (gdn_chunk_fwd_ex with a saved buffer) gives the plain forward's o and hT
    bit for bit; the backward that reads them (gdn_chunk_bwd_ex: the reverse
    walk alone, no preparation, no recompute) matches the per-token adjoint on
    every head, as the plain backward does.  The segment lengths cover walks
    of one, two and three or more chunks (the reverse walk requests each
    chunk's dO slice from the second chunk on), with a last chunk of one row."""
    wl = WORKLOADS[name].replace(T=T, backward=True, h0_std=0.2, gate_shift=-2.0 if S > 1 else 0.0,
                                 seed=70 + S)
    inp = make_host(wl)
    d = inp.to("cuda")
    sv = torch.empty(gdn_lib.saved_bytes(wl.B, wl.T, wl.Hk, wl.Hv, n_segments=S), dtype=torch.uint8,
                     device="cuda")
    o1, h1 = gdn_lib.chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, n_segments=S, saved=sv)
    o2, h2 = gdn_lib.chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, n_segments=S)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    ws = torch.empty(gdn_lib.bwd_workspace_bytes(wl.B, wl.T, wl.Hk, wl.Hv, n_segments=S),
                     dtype=torch.uint8, device="cuda")
    g1 = gdn_lib.chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.dO, d.dhT, n_segments=S, saved=sv,
                           workspace=ws)
    assert gdn_lib.workspace_status(ws) == 0
    g2 = gdn_lib.chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.dO, d.dhT, n_segments=S)
    torch.cuda.synchronize()
    for name_, a, b in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), g1, g2):
        assert_rel(a.float().cpu().numpy(), b.float().cpu().numpy(), G_TOL, f"{name_}: saved vs plain")
    # the saved path against the oracle on every head
    res = oracle.bwd(inp)
    kq = oracle.key_head_grads(wl, res)
    dq, dk, dv = (x.float().cpu().numpy() for x in g1[:3])
    dg, db, dh0 = (x.cpu().numpy() for x in g1[3:])
    tag = f"{name} (saved tiles)" if name == "layer_t4096" else None
    m = (lambda t: (tag, t)) if tag else (lambda t: None)
    grp = wl.Hv // wl.Hk
    for (b, kh), (rq, rk) in kq.items():
        assert_rel(dq[b, :, kh], rq, G_TOL, f"dq[{b},{kh}]", m("dq"))
        assert_rel(dk[b, :, kh], rk, G_TOL, f"dk[{b},{kh}]", m("dk"))
    for i, (b, j) in enumerate(res["heads"]):
        assert_rel(dv[b, :, j], res["dv"][i], G_TOL, f"dv[{b},{j}]", m("dv"))
        assert_rel(dg[b, :, j], res["dg"][i], G_TOL, f"dg[{b},{j}]", m("dg"))
        assert_rel(db[b, :, j], res["dbeta"][i], G_TOL, f"dbeta[{b},{j}]", m("dbeta"))
        assert_rel(dh0[b, j], res["dh0"][i], G_TOL, f"dh0[{b},{j}]", m("dh0"))
    assert grp >= 1


def test_saved_buffer_too_small_is_refused(gdn_lib):
    wl = WORKLOADS["tiny_t1024"].replace(T=256, backward=True)
    d = make_host(wl).to("cuda")
    sv = torch.empty(gdn_lib.saved_bytes(wl.B, wl.T, wl.Hk, wl.Hv) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(gdn_lib.GDNError):
        gdn_lib.chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, saved=sv)
    with pytest.raises(gdn_lib.GDNError):
        gdn_lib.chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.dO, d.dhT, saved=sv)
