"""C-ABI library: builds, loads, exports every declared symbol, and rejects bad
arguments on the host (before any CUDA call) -- no GPU needed."""
import ctypes

import pytest

import linear_attention_rnn_gb300 as gdn


@pytest.fixture(scope="module")
def L():
    gdn.build()
    return gdn.lib()


def test_exports_every_declared_function(L):
    names = gdn.header_functions()
    assert {"gdn_chunk_fwd", "gdn_chunk_bwd", "gdn_affine_compose", "gdn_debug_ut",
            "gdn_strerror", "gdn_fwd_workspace_bytes", "gdn_bwd_workspace_bytes",
            "gdn_default_segments"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_strerror_covers_codes(L):
    for code in range(-6, 1):
        assert L.gdn_strerror(code)
    assert L.gdn_strerror(-99) == b"unknown status"


P = ctypes.c_void_p
FAKE = P(1 << 20)          # aligned, never dereferenced (validation fails first)
MISAL = P((1 << 20) + 2)


def _fwd(L, q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, h0=None, o=FAKE, hT=None,
         B=1, T=256, Hk=2, Hv=4, dk=128, dv=128, chunk=128, S=0, ws=FAKE, ws_bytes=0):
    return L.gdn_chunk_fwd(q, k, v, g, beta, h0, o, hT, B, T, Hk, Hv, dk, dv, chunk, S, ws,
                           ws_bytes, None)


def test_fwd_argument_errors(L):
    assert _fwd(L, dk=64) == -2
    assert _fwd(L, dv=96) == -2
    assert _fwd(L, chunk=32) == -2
    assert _fwd(L, chunk=64) == -3             # 64-token chunks accepted; workspace of 0 bytes
    assert _fwd(L, Hk=3, Hv=4) == -1
    assert _fwd(L, T=-1) == -1
    assert _fwd(L, S=-2) == -1
    assert _fwd(L, q=None) == -1
    assert _fwd(L, o=None) == -1
    assert _fwd(L, k=MISAL) == -1
    assert _fwd(L, ws_bytes=10) == -3          # too small
    assert _fwd(L, ws=None, ws_bytes=1 << 40) == -3
    assert _fwd(L, B=0) == 0                   # nothing to do
    assert _fwd(L, q=None, k=None, v=None, g=None, beta=None, o=None, T=0) == 0  # T=0, no hT


def test_bwd_argument_errors(L):
    args = [FAKE] * 5 + [None, FAKE, None] + [FAKE] * 5 + [None]
    ok = dict(B=1, T=256, Hk=2, Hv=4, dk=128, dv=128, chunk=128, S=0)

    def call(a, **kw):
        d = dict(ok, **kw)
        return L.gdn_chunk_bwd(*a, d["B"], d["T"], d["Hk"], d["Hv"], d["dk"], d["dv"],
                               d["chunk"], d["S"], FAKE, 16, None)
    assert call(args, dk=256) == -2
    assert call(args, chunk=64) == -2  # the backward takes 128-token chunks
    assert call(args, Hv=5) == -1
    bad = list(args)
    bad[6] = None  # dO
    assert call(bad) == -1
    assert call(args) == -3  # workspace of 16 bytes


def test_compose_argument_errors(L):
    assert L.gdn_affine_compose(FAKE, FAKE, FAKE, FAKE, 1, 4, 64, 128, None) == -2
    assert L.gdn_affine_compose(FAKE, FAKE, FAKE, FAKE, 1, 4, 128, 20, None) == -2
    assert L.gdn_affine_compose(None, FAKE, FAKE, FAKE, 1, 4, 128, 128, None) == -1
    assert L.gdn_affine_compose(FAKE, MISAL, FAKE, FAKE, 1, 4, 128, 128, None) == -1
    assert L.gdn_affine_compose(None, None, None, None, 0, 4, 128, 128, None) == 0


def test_segment_fold_argument_errors(L):
    def call(S=1, T=256, A=FAKE, Bo=FAKE, dk=128, ws=FAKE, ws_bytes=0, chunk=128):
        return L.gdn_segment_fold(FAKE, FAKE, FAKE, FAKE, A, Bo, 1, T, 2, 4, dk, 128, chunk, S, ws,
                                  ws_bytes, None)
    assert call(dk=64) == -2
    assert call(chunk=32) == -2
    assert call(S=0) == -1
    assert call(S=3) == -1          # 2 chunks
    assert call(S=3, chunk=64) == -3  # 4 chunks of 64 tokens; workspace of 0 bytes
    assert call(S=5, chunk=64) == -1
    assert call(Bo=None) == -1
    assert call(A=MISAL) == -1
    assert call() == -3             # workspace of 0 bytes
    assert call(S=2, A=None, ws=None) == -3


def test_saved_buffer_argument_errors(L):
    import linear_attention_rnn_gb300 as g
    need = g.saved_bytes(1, 256, 2, 4, n_segments=1)
    assert need == 6 * 4 * 2 * 128 * 128 * 2  # w, u, P, T, h, Delta: bf16 tiles per (chunk, value head)
    assert g.saved_bytes(1, 256, 2, 4, chunk=64) == 0
    # with 2 segments also the fp32 state entering each segment of each value head
    assert g.saved_bytes(1, 256, 2, 4, n_segments=2) == need + 4 * 2 * 128 * 128 * 4
    fwd = lambda saved, nbytes: L.gdn_chunk_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None,
                                                   1, 256, 2, 4, 128, 128, 128, 1, saved, nbytes,
                                                   FAKE, 1 << 30, None, None, 0)
    assert fwd(FAKE, need - 1) == -3
    assert fwd(MISAL, need) == -1
    fwd64 = L.gdn_chunk_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, 1, 256, 2, 4, 128, 128,
                               64, 1, FAKE, need, FAKE, 1 << 30, None, None, 0)
    assert fwd64 == -2  # tiles for the backward: 128-token chunks only
    args = [FAKE] * 5 + [None, FAKE, None] + [FAKE] * 5 + [None]
    bwd = lambda saved, nbytes: L.gdn_chunk_bwd_ex(*args, 1, 256, 2, 4, 128, 128, 128, 1, saved,
                                                   nbytes, FAKE, 1 << 30, None, None, 0)
    assert bwd(FAKE, 16) == -3


def test_layer_argument_errors(L):
    import linear_attention_rnn_gb300 as g
    need_f = g.layer_workspace_bytes(0, 1, 256, 2, 4)
    need_b = g.layer_workspace_bytes(1, 1, 256, 2, 4)
    # forward: the rule's workspace, the rows' 1/||k|| and 1/||q|| (fp32 [Hk, chunks, 2, 128]) and a
    # v-shaped bf16 buffer; backward: normalised q, k (bf16 [T, Hk, 128]), their cotangents and
    # the v-shaped buffer
    qk, vv = 256 * 2 * 128 * 2, 256 * 4 * 128 * 2
    assert need_f == g.fwd_workspace_bytes(1, 256, 2, 4) + 2 * 2 * 2 * 128 * 4 + vv
    assert need_b == g.bwd_workspace_bytes(1, 256, 2, 4) + 4 * qk + vv
    assert g.layer_workspace_bytes(0, 1, 256, 2, 4, dk=64) == 0
    # 64-token chunks: the forward only; the same tiles (two chunks to a 128-row tile)
    assert g.layer_workspace_bytes(0, 1, 256, 2, 4, chunk=64) == (
        g.fwd_workspace_bytes(1, 256, 2, 4, chunk=64) + 2 * 2 * 2 * 128 * 4 + vv)
    assert g.layer_workspace_bytes(1, 1, 256, 2, 4, chunk=64) == 0

    def fwd(z=FAKE, y=FAKE, a=FAKE, ws=FAKE, nbytes=1 << 30, T=256, dk=128):
        return L.gdn_layer_fwd(FAKE, FAKE, FAKE, a, FAKE, z, None, y, None, None, 1, T, 2, 4, dk, 128,
                               128, 1, ws, nbytes, None)
    assert fwd(dk=64) == -2
    assert fwd(a=None) == -1
    assert fwd(y=None) == -1
    assert fwd(z=MISAL) == -1
    assert fwd(nbytes=need_f - 1) == -3
    assert fwd(T=0, ws=None, nbytes=0) == 0  # no tokens, no h0, no hT: nothing to do

    def bwd(z=FAKE, o=FAKE, dz=FAKE, nbytes=1 << 30):
        return L.gdn_layer_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, z, None, o, FAKE, None, FAKE, FAKE,
                               FAKE, FAKE, FAKE, dz, None, 1, 256, 2, 4, 128, 128, 128, 1, FAKE,
                               nbytes, None)
    assert bwd(o=None) == -1          # the gate's backward needs the ungated output
    assert bwd(dz=None) == -1
    assert bwd(nbytes=need_b - 1) == -3
    assert bwd(z=None, o=None, dz=None, nbytes=16) == -3  # without a gate o and dz are not needed


def test_workspace_sizes(L):
    f = gdn.fwd_workspace_bytes
    b = gdn.bwd_workspace_bytes
    assert f(1, 4096, 16, 32, 64) == 0  # unsupported d_k
    w1 = f(1, 4096, 16, 32, n_segments=1)
    # w, u and P: three bf16 128x128 tiles per (chunk, value head)
    assert w1 >= 3 * 32 * 32 * 128 * 128 * 2
    assert f(1, 4096, 16, 32, n_segments=4) > w1  # per-segment (A, B) and entering states
    assert b(1, 4096, 16, 32, n_segments=1) > w1
    assert f(2, 1000, 2, 4) > 0
    # 64-token chunks keep the 128-row tiles: the same workspace with one segment
    assert f(1, 4096, 16, 32, chunk=64, n_segments=1) == w1
    assert f(1, 4096 + 64, 16, 32, chunk=64, n_segments=1) == f(1, 4096 + 64, 16, 32, n_segments=1)
    assert f(1, 4096, 16, 32, chunk=32) == 0
    assert b(1, 4096, 16, 32, chunk=64) == 0


def test_default_segments(L):
    assert gdn.default_segments(1, 4096, 32) == 1
    assert gdn.default_segments(1, 0, 32) == 1
    # 32 value heads: the one-segment walk keeps 128 CTAs busy, so no segments
    assert gdn.default_segments(1, 262144, 32) == 1
    assert gdn.default_segments(1, 1 << 20, 32) == 1
    # one or two heads: enough segments to fill the SMs, at least 8 chunks each
    s1 = gdn.default_segments(1, 262144, 1)
    assert 2 <= s1 <= 2048 // 8
    assert s1 >= gdn.default_segments(1, 262144, 2) >= 2
    assert gdn.default_segments(1, 64 * 128 + 1, 1) == 8  # 65 chunks, 8 per segment
    assert gdn.default_segments(1, 64 * 64 + 1, 1, 64) == 8  # 65 chunks of 64 tokens
    assert gdn.default_segments(1, 4096, 32, 64) == 1


def test_binding_validates_before_calling():
    import torch
    q = torch.zeros(1, 8, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        gdn.chunk_fwd(q, q, q, torch.zeros(1, 8, 1), torch.zeros(1, 8, 1))  # CPU tensors
