"""Full-size workloads on the GPU, in the launch configuration the bench
uses (148 segments for the long sequences).  The oracle checks sampled heads
exactly (its per-token walk over the whole sequence); properties that hold at
any size (segment-count invariance) are checked on every head.

Inputs are generated on the device (torch generator, same distributions as
the host recipe) because host generation takes minutes at these sizes.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_rnn_gb300.inputs import WORKLOADS, Inputs, make_device
from conftest import assert_rel

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

O_TOL, H_TOL, G_TOL = 2e-2, 1e-2, 3e-2


def heads_slice(inp, b, key_heads):
    """Host copy of batch row b restricted to the given key heads and their
    value heads (the oracle's input for those heads)."""
    wl = inp.wl
    grp = wl.Hv // wl.Hk
    vh = [kh * grp + r for kh in key_heads for r in range(grp)]
    kidx = torch.tensor(key_heads, device=inp.q.device)
    vidx = torch.tensor(vh, device=inp.q.device)
    sel = lambda x, idx: None if x is None else x[b:b + 1].index_select(2, idx).contiguous().cpu()
    sel_s = lambda x: None if x is None else x[b:b + 1].index_select(1, vidx).contiguous().cpu()
    sub = Inputs(wl.replace(B=1, Hk=len(key_heads), Hv=len(vh)), sel(inp.q, kidx),
                 sel(inp.k, kidx), sel(inp.v, vidx), sel(inp.g, vidx), sel(inp.beta, vidx),
                 sel_s(inp.h0), sel(inp.dO, vidx), sel_s(inp.dhT))
    return sub, vh


def _fwd_check(gdn, wl, key_heads, check_o=True):
    inp = make_device(wl, "cuda", backward=False)
    o, hT = gdn.chunk_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0,
                          n_segments=wl.n_segments)
    torch.cuda.synchronize()
    assert torch.isfinite(hT).all()
    sub, vh = heads_slice(inp, 0, key_heads)
    ro, rh = oracle.fwd(sub, want_o=check_o)
    for i, j in enumerate(vh):
        assert_rel(hT[0, j].cpu().numpy(), rh[i], H_TOL, f"hT[{j}]", (wl.name, "hT"))
        if check_o:
            assert_rel(o[0, :, j].float().cpu().numpy(), ro[i], O_TOL, f"o[{j}]", (wl.name, "o"))
    return inp, o, hT


def test_long_sequence_forward_148_segments(gdn_lib):
    wl = WORKLOADS["long_t262144"]
    inp, o, hT = _fwd_check(gdn_lib, wl, list(range(wl.Hk)))  # every head
    # the same result from a single sequential walk (every head)
    o1, h1 = gdn_lib.chunk_fwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, n_segments=1)
    assert_rel(o.float().cpu().numpy(), o1.float().cpu().numpy(), O_TOL, "o: 148 vs 1 segments")
    assert_rel(hT.cpu().numpy(), h1.cpu().numpy(), H_TOL, "hT: 148 vs 1 segments")


def test_long_sequence_backward_148_segments(gdn_lib):
    wl = WORKLOADS["long_t262144"]
    inp = make_device(wl, "cuda", backward=True)
    dq, dk, dv, dg, db, dh0 = gdn_lib.chunk_bwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0,
                                                inp.dO, inp.dhT, n_segments=wl.n_segments)
    torch.cuda.synchronize()
    key_heads = [0, 7, 12, 15]
    sub, vh = heads_slice(inp, 0, key_heads)
    res = oracle.bwd(sub, ckpt=256)
    kq = oracle.key_head_grads(sub.wl, res)
    m = lambda t: (wl.name, t)
    for i, kh in enumerate(key_heads):
        assert_rel(dq[0, :, kh].float().cpu().numpy(), kq[(0, i)][0], G_TOL, f"dq[{kh}]", m("dq"))
        assert_rel(dk[0, :, kh].float().cpu().numpy(), kq[(0, i)][1], G_TOL, f"dk[{kh}]", m("dk"))
    for i, j in enumerate(vh):
        assert_rel(dv[0, :, j].float().cpu().numpy(), res["dv"][i], G_TOL, f"dv[{j}]", m("dv"))
        assert_rel(dg[0, :, j].cpu().numpy(), res["dg"][i], G_TOL, f"dg[{j}]", m("dg"))
        assert_rel(db[0, :, j].cpu().numpy(), res["dbeta"][i], G_TOL, f"dbeta[{j}]", m("dbeta"))
        assert_rel(dh0[0, j].cpu().numpy(), res["dh0"][i], G_TOL, f"dh0[{j}]", m("dh0"))
    # segment-count invariance of the backward on every head
    g1 = gdn_lib.chunk_bwd(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.h0, inp.dO, inp.dhT,
                           n_segments=1)
    for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"),
                          (dq, dk, dv, dg, db, dh0), g1):
        assert_rel(a.float().cpu().numpy(), b.float().cpu().numpy(), G_TOL, f"{name}: 148 vs 1")


@pytest.mark.parametrize("name", ["million_t1048576", "million_t1048576_slow"])
def test_million_token_forward_148_segments(gdn_lib, name):
    wl = WORKLOADS[name]
    _fwd_check(gdn_lib, wl, [0, 5, 10, 15])
