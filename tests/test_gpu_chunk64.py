"""GPU parity of the forward with 64-token chunks (chunk = 64) against the
fp64 oracle, through the C ABI.

The rule's result does not depend on the chunk size, so the per-token oracle
is the reference for o and hT; the per-chunk quantities (S, T, w, u of each
64-token chunk) and the segment maps are checked against the oracle's chunked
route run with C = 64.  Tolerances as for 128-token chunks: 2e-2 on o, 1e-2 on
hT and the segment maps, ladder residual max|(I + S) T - I| <= 1e-4.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import chunked
from oracle import layer as ol
from linear_attention_rnn_gb300.inputs import WORKLOADS, make_host, make_layer_host
from conftest import as64, assert_rel, head, record_margin

pytestmark = pytest.mark.gpu

O_TOL, H_TOL, RES_TOL = 2e-2, 1e-2, 1e-4
C = 64


def _check(gdn, inp, n_segments=0, heads=None, record=None):
    d = inp.to("cuda")
    o, hT = gdn.chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, chunk=C, n_segments=n_segments)
    torch.cuda.synchronize()
    o = o.float().cpu().numpy()
    hT = hT.cpu().numpy()
    heads = heads or [(b, j) for b in range(inp.wl.B) for j in range(inp.wl.Hv)]
    ro, rh = oracle.fwd(inp, heads=heads)
    mo = (record, "o") if record else None
    mh = (record, "hT") if record else None
    for i, (b, j) in enumerate(heads):
        assert_rel(o[b, :, j], ro[i], O_TOL, f"o[{b},{j}] (chunk 64)", mo)
        assert_rel(hT[b, j], rh[i], H_TOL, f"hT[{b},{j}] (chunk 64)", mh)
    return o, hT


def test_chunk64_tiny_workload(gdn_lib):
    _check(gdn_lib, make_host(WORKLOADS["tiny_t1024"]), record="tiny_t1024 (chunk 64)")


def test_chunk64_layer_workload_all_heads(gdn_lib):
    inp = make_host(WORKLOADS["layer_t4096"], backward=False)
    o64, h64 = _check(gdn_lib, inp, record="layer_t4096 (chunk 64)")
    # the same result as with 128-token chunks, up to rounding
    d = inp.to("cuda")
    o128, h128 = gdn_lib.chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0)
    assert_rel(o64, o128.float().cpu().numpy(), O_TOL, "o: chunk 64 vs 128")
    assert_rel(h64, h128.cpu().numpy(), H_TOL, "hT: chunk 64 vs 128")


@pytest.mark.parametrize("T", [1, 5, 63, 64, 65, 127, 128, 129, 191, 300, 1000])
def test_chunk64_ragged_lengths(gdn_lib, T):
    """Lengths that end inside the first or second chunk of a 128-row tile,
    on a tile boundary, and one past it."""
    _check(gdn_lib, make_host(WORKLOADS["tiny_t1024"].replace(T=T, Hk=2, Hv=4, h0_std=0.1, seed=200 + T)))


@pytest.mark.parametrize("B,T,Hk,Hv", [(2, 384, 1, 4), (2, 384, 3, 6), (3, 333, 3, 6)])
def test_chunk64_head_groupings_and_unit_ranges(gdn_lib, B, T, Hk, Hv):
    _check(gdn_lib, make_host(WORKLOADS["tiny_t1024"].replace(B=B, T=T, Hk=Hk, Hv=Hv, h0_std=0.2,
                                                             seed=T + Hv + 7)))


@pytest.mark.parametrize("shift", [4.0, 8.0])
def test_chunk64_fast_decay(gdn_lib, shift):
    _check(gdn_lib, make_host(WORKLOADS["tiny_t1024"].replace(T=300, Hk=1, Hv=2, gate_shift=shift,
                                                             h0_std=0.5, seed=int(shift) + 230)))


@pytest.mark.parametrize("S", [1, 2, 3, 7, 33])
def test_chunk64_segment_counts_slow_decay(gdn_lib, S):
    """Slow decay so every segment's incoming state matters; segments of
    whole 64-token chunks (33 segments of the 33 chunks: one chunk each)."""
    inp = make_host(WORKLOADS["tiny_t1024"].replace(T=2048 + 13, Hk=1, Hv=2, gate_shift=-3.0,
                                                   h0_std=0.5, seed=211))
    _check(gdn_lib, inp, n_segments=S)


@pytest.mark.parametrize("name", ["tiny_t1024", "layer_t4096"])
def test_chunk64_ut_intermediates_and_ladder_residual(gdn_lib, name):
    """S, T, w, u of every 64-token chunk of every head against the oracle's
    chunk quantities with C = 64; the device's 128-row tiles are exactly
    block diagonal."""
    wl = WORKLOADS[name]
    inp = make_host(wl, backward=False)
    d = inp.to("cuda")
    St, Tt, _, _ = gdn_lib.debug_ut(d.k, d.v, d.g, d.beta, chunk=C, tiles=True)
    S, T, w, u = gdn_lib.debug_ut(d.k, d.v, d.g, d.beta, chunk=C)
    torch.cuda.synchronize()
    for x in (St, Tt):
        assert torch.count_nonzero(x[..., 64:, :64]) == 0 and torch.count_nonzero(x[..., :64, 64:]) == 0
    S, T, w, u = (x.float().cpu().numpy() for x in (S, T, w, u))
    I = np.eye(C)
    worst = 0.0
    for b in range(wl.B):
        for j in range(wl.Hv):
            q, k, v, g, beta, _ = head(inp, b, j)
            for c in range(wl.T // C):
                sl = slice(c * C, (c + 1) * C)
                it = chunked.chunk_intermediates(q[sl], k[sl], v[sl], g[sl], beta[sl])
                m = f"{name} (chunk 64)"
                assert_rel(S[b, j, c], it["S"], 1e-4, f"S[{b},{j},{c}]", (m, "S (per chunk)"))
                res = np.max(np.abs((I + it["S"]) @ T[b, j, c].astype(np.float64) - I))
                worst = max(worst, res)
                assert res <= RES_TOL, f"ladder residual {res:.2e} at {(b, j, c)}"
                assert_rel(w[b, j, c], it["w"], 1e-2, "w", (m, "w (per chunk)"))
                assert_rel(u[b, j, c], it["u"], 1e-2, "u", (m, "u (per chunk)"))
    record_margin(f"{name} (chunk 64)", "ladder residual max|(I+S)T - I|", worst, RES_TOL)


@pytest.mark.parametrize("S", [1, 2, 5, 11])
def test_chunk64_segment_fold(gdn_lib, S):
    """gdn_segment_fold with 64-token chunks: each segment's composed chunk
    maps against the oracle's pass-1 fold with C = 64, and for one segment
    A h0 + B against the per-token rule's final state."""
    wl = WORKLOADS["tiny_t1024"].replace(T=11 * C + 21, Hk=1, Hv=2, gate_shift=-4.0,
                                         h0_std=0.5, seed=215)
    inp = make_host(wl)
    d = inp.to("cuda")
    A, Bm = gdn_lib.segment_fold(d.k, d.v, d.g, d.beta, S, chunk=C)
    torch.cuda.synchronize()
    A, Bm = A.cpu().numpy(), Bm.cpu().numpy()
    for j in range(wl.Hv):
        pairs = chunked.head_fwd_segmented(*head(inp, 0, j), C, S)[2]
        for s, (rA, rB) in enumerate(pairs):
            assert_rel(A[0, j, s], rA, H_TOL, f"A[{j},{s}]", ("segment fold (chunk 64)", "A_s"))
            assert_rel(Bm[0, j, s], rB, H_TOL, f"B[{j},{s}]", ("segment fold (chunk 64)", "B_s"))
    if S == 1:
        _, rh = oracle.fwd(inp)
        h0 = as64(inp, "h0")[0]
        for j in range(wl.Hv):
            assert_rel(A[0, j, 0].astype(np.float64) @ h0[j] + Bm[0, j, 0], rh[j], H_TOL,
                       f"A h0 + B vs per-token hT[{j}]")
    if S == 11:  # 12 chunks: segment boundaries at multiples of 64 tokens, not of 128
        A2, B2 = gdn_lib.segment_fold(d.k, d.v, d.g, d.beta, 1, chunk=C)
        A1, B1 = gdn_lib.segment_fold(d.k, d.v, d.g, d.beta, 1)
        assert_rel(B2.cpu().numpy(), B1.cpu().numpy(), H_TOL, "one segment: chunk 64 vs 128")
        assert_rel(A2.cpu().numpy(), A1.cpu().numpy(), H_TOL, "one segment: chunk 64 vs 128 (A)")


def test_chunk64_layer_forward(gdn_lib):
    """gdn_layer_fwd with 64-token chunks: the rule on raw q, k normalised in
    the kernels, gate logits and the output gate, against the oracle."""
    wl = WORKLOADS["tiny_t1024"].replace(T=700, Hk=2, Hv=4, h0_std=0.2, seed=217)
    raw = make_layer_host(wl)
    d = raw.to("cuda")
    y, o, hT = gdn_lib.layer_fwd(d.q, d.k, d.v, d.a, d.b, d.z, d.h0, chunk=C)
    torch.cuda.synchronize()
    f64 = lambda t: t.detach().cpu().to(torch.float64).numpy()
    qn, kn = ol.l2norm(f64(raw.q)), ol.l2norm(f64(raw.k))
    g, beta = ol.gates(f64(raw.a), f64(raw.b))
    grp = wl.Hv // wl.Hk
    for j in range(wl.Hv):
        ro, rh = chunked.head_fwd(qn[0, :, j // grp], kn[0, :, j // grp], f64(raw.v)[0, :, j],
                                  g[0, :, j], beta[0, :, j], f64(raw.h0)[0, j], 128)
        ry = ol.out_gate(ro, f64(raw.z)[0, :, j])
        assert_rel(f64(o)[0, :, j], ro, O_TOL, f"o[{j}] (layer, chunk 64)")
        assert_rel(f64(y)[0, :, j], ry, O_TOL, f"y[{j}] (layer, chunk 64)")
        assert_rel(f64(hT)[0, j], rh, H_TOL, f"hT[{j}] (layer, chunk 64)")


def test_chunk64_backward_is_refused(gdn_lib):
    """The backward takes 128-token chunks; chunk = 64 there, or a forward
    keeping tiles for the backward with chunk = 64, is refused before any
    work, and the 128-token backward serves a forward run with 64."""
    wl = WORKLOADS["tiny_t1024"].replace(T=256, Hk=1, Hv=2, backward=True, seed=219)
    d = make_host(wl).to("cuda")
    with pytest.raises(gdn_lib.GDNError) as e:
        gdn_lib.chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.dO, d.dhT, chunk=C)
    assert e.value.code == -2
    sv = torch.empty(gdn_lib.saved_bytes(wl.B, wl.T, wl.Hk, wl.Hv), dtype=torch.uint8, device="cuda")
    with pytest.raises(gdn_lib.GDNError) as e:
        gdn_lib.chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, chunk=C, saved=sv)
    assert e.value.code == -2
