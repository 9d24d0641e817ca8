"""GPU parity of the layer entry points (gdn_layer_fwd / gdn_layer_bwd)
against the fp64 oracle: q and k normalised per token, gate logits
(g = -softplus(a), beta = sigmoid(b)) applied where the rule's kernels load
the gates, and the output gate y = o * silu(z).  The forward normalises q and
k inside its kernels (the rows stay raw, their 1/||.|| scale the products), so
its reference runs the chunked route on fp64 unit rows; the backward takes
bf16 normalised copies, so its reference forms them the same way (rounded to
bf16), runs the per-token adjoint, and applies the written-out backwards of
the element-wise operations (oracle/layer.py).  Tolerances as for the rule:
2e-2 on y and o, 1e-2 on hT, 3e-2 on every gradient."""
import numpy as np
import pytest
import torch

import oracle
from oracle import chunked
from oracle import layer as ol
from linear_attention_rnn_gb300.inputs import WORKLOADS, make_layer_host
from conftest import assert_rel

pytestmark = pytest.mark.gpu

O_TOL, H_TOL, G_TOL = 2e-2, 1e-2, 3e-2


def _f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def _check_layer(gdn, raw, gate=True, record=None):
    """Every output tensor against the oracle, each compared as a whole
    (max|x - ref| <= tol max|ref| per tensor)."""
    wl = raw.wl
    d = raw.to("cuda")
    z = d.z if gate else None
    y, o, hT = gdn.layer_fwd(d.q, d.k, d.v, d.a, d.b, z, d.h0)
    grads = gdn.layer_bwd(d.q, d.k, d.v, d.a, d.b, z, d.h0, o, d.dy, d.dhT)
    torch.cuda.synchronize()
    dq, dk, dv, da, db, dz, dh0 = grads
    m = (lambda t: (record, t)) if record else (lambda t: None)
    heads = [(b_, j) for b_ in range(wl.B) for j in range(wl.Hv)]

    def full(per_head, tail):  # [n_heads, ...] oracle arrays -> [B, T, Hv, ...] / [B, Hv, ...]
        out = np.zeros((wl.B, wl.Hv) + tail)
        for i, (b_, j) in enumerate(heads):
            out[b_, j] = per_head[i]
        return out

    # oracle forward: the forward normalises q and k inside its kernels without
    # rounding the unit rows, so the reference takes them in fp64 (the chunked
    # route, pinned to the per-token rule) on fp64 gates from the fp32 logits
    from linear_attention_rnn_gb300.inputs import Inputs
    qn, kn = ol.l2norm(_f64(raw.q)), ol.l2norm(_f64(raw.k))
    g64, b64 = ol.gates(_f64(raw.a), _f64(raw.b))
    grp = wl.Hv // wl.Hk
    h0 = None if raw.h0 is None else _f64(raw.h0)
    o_ref = np.zeros((wl.B, wl.T, wl.Hv, wl.dv))
    h_ref = np.zeros((wl.B, wl.Hv, wl.dk, wl.dv))
    for b_, j in heads:
        o_ref[b_, :, j], h_ref[b_, j] = chunked.head_fwd(
            qn[b_, :, j // grp], kn[b_, :, j // grp], _f64(raw.v)[b_, :, j], g64[b_, :, j], b64[b_, :, j],
            None if h0 is None else h0[b_, j], 128)
    # the backward takes bf16 normalised copies of q and k: its reference rounds them too
    ri = ol.rule_inputs(Inputs(wl, raw.q, raw.k, raw.v, raw.a, raw.b, raw.h0))
    zz = _f64(raw.z)
    y_ref = ol.out_gate(o_ref, zz) if gate else o_ref
    assert_rel(_f64(y), y_ref, O_TOL, "y", m("y"))
    assert_rel(hT.cpu().numpy(), h_ref, H_TOL, "hT", m("hT"))
    if gate:
        assert_rel(_f64(o), o_ref, O_TOL, "o (ungated)", m("o (ungated)"))

    # oracle backward: gate, rule adjoint, activations, normalisation
    dyy = _f64(raw.dy)
    do_ref, dz_ref = ol.out_gate_bwd(o_ref, zz, dyy) if gate else (dyy, None)
    ri.dO = torch.from_numpy(do_ref.astype(np.float32)).to(torch.bfloat16)
    ri.dhT = raw.dhT
    res = oracle.bwd(ri)
    kq = oracle.key_head_grads(wl, res)
    dqn = np.zeros((wl.B, wl.T, wl.Hk, wl.dk))
    dkn = np.zeros_like(dqn)
    for (b_, kh), (x, y_) in kq.items():
        dqn[b_, :, kh], dkn[b_, :, kh] = x, y_
    dg = np.moveaxis(full(res["dg"], (wl.T,)), 1, 2)
    dbeta = np.moveaxis(full(res["dbeta"], (wl.T,)), 1, 2)
    da_ref, db_ref = ol.gates_bwd(_f64(raw.a), _f64(raw.b), dg, dbeta)
    assert_rel(_f64(dq), ol.l2norm_bwd(_f64(raw.q), dqn), G_TOL, "dq", m("dq"))
    assert_rel(_f64(dk), ol.l2norm_bwd(_f64(raw.k), dkn), G_TOL, "dk", m("dk"))
    assert_rel(_f64(dv), np.moveaxis(full(res["dv"], (wl.T, wl.dv)), 1, 2), G_TOL, "dv", m("dv"))
    assert_rel(da.cpu().numpy(), da_ref, G_TOL, "da", m("da"))
    assert_rel(db.cpu().numpy(), db_ref, G_TOL, "db", m("db"))
    assert_rel(dh0.cpu().numpy(), full(res["dh0"], (wl.dk, wl.dv)), G_TOL, "dh0", m("dh0"))
    if gate:
        assert_rel(_f64(dz), dz_ref, G_TOL, "dz", m("dz"))


@pytest.mark.parametrize("T", [1, 300])
def test_layer_small(gdn_lib, T):
    wl = WORKLOADS["tiny_t1024"].replace(T=T, Hk=2, Hv=4, h0_std=0.2, seed=60 + T)
    _check_layer(gdn_lib, make_layer_host(wl))


def test_layer_without_gate(gdn_lib):
    wl = WORKLOADS["tiny_t1024"].replace(T=256, Hk=1, Hv=2, h0_std=0.3, seed=62)
    _check_layer(gdn_lib, make_layer_host(wl), gate=False)


def test_layer_shape_t4096(gdn_lib):
    """The layer workload's shape (B=1, T=4096, 16 key heads shared by 32 value
    heads), every head."""
    wl = WORKLOADS["layer_t4096"].replace(gate_shift=1.0, seed=63)
    _check_layer(gdn_lib, make_layer_host(wl), record="layer_t4096 (layer entry points)")


def test_layer_matches_rule_on_normalised_inputs(gdn_lib):
    """With q, k already unit rows and the logits of given gates, the layer
    forward (no gate) equals gdn_chunk_fwd on the same rule inputs bit for bit
    except for the normalisation's rounding: compared at the rule's tolerance."""
    wl = WORKLOADS["tiny_t1024"].replace(T=384, Hk=1, Hv=2, h0_std=0.1, seed=64)
    raw = make_layer_host(wl)
    d = raw.to("cuda")
    y, _, hT = gdn_lib.layer_fwd(d.q, d.k, d.v, d.a, d.b, None, d.h0)
    from linear_attention_rnn_gb300.inputs import Inputs
    ri = ol.rule_inputs(Inputs(wl, raw.q, raw.k, raw.v, raw.a, raw.b, raw.h0)).to("cuda")
    o2, h2 = gdn_lib.chunk_fwd(ri.q, ri.k, ri.v, ri.g, ri.beta, ri.h0)
    torch.cuda.synchronize()
    assert_rel(_f64(y), _f64(o2), O_TOL, "layer y vs rule o")
    assert_rel(hT.cpu().numpy(), h2.cpu().numpy(), H_TOL, "layer hT vs rule hT")
