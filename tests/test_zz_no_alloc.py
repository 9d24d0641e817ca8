"""The forward that allocates nothing (gdn_chunk_fwd_noalloc).

It serves callers that may not allocate device memory when they call the
forward and have no scratch buffer to lend -- a service that planned and
locked its device memory at start-up, or a plug-in whose host framework owns
all device memory.  Its scratch is a fixed array inside the library, shared by
every call and never cleared, so these tests call it twice in a row with
different inputs and sizes and compare each result with the ordinary
gdn_chunk_fwd (which uses a caller workspace), through the C ABI: the two run
the same deterministic kernels, so their outputs must be equal bit for bit;
each result is also checked against the fp64 oracle.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import oracle
from linear_attention_rnn_gb300.inputs import WORKLOADS, make_host
from conftest import assert_rel

pytestmark = pytest.mark.gpu

O_TOL, H_TOL = 2e-2, 1e-2  # the forward parity tolerances used throughout the tests


def _noalloc(gdn):
    f = gdn.lib().gdn_chunk_fwd_noalloc
    f.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_int] * 7 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f


def _call(gdn, f, d):
    wl = d.wl
    o = torch.empty((wl.B, wl.T, wl.Hv, wl.dv), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty((wl.B, wl.Hv, wl.dk, wl.dv), dtype=torch.float32, device="cuda")
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = f(p(d.q), p(d.k), p(d.v), p(d.g), p(d.beta), p(d.h0), p(o), p(hT), wl.B, wl.T, wl.Hk,
           wl.Hv, wl.dk, wl.dv, wl.chunk,
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, gdn.lib().gdn_strerror(rc)
    return o, hT


def test_noalloc_forward_matches_workspace_forward_twice(gdn_lib):
    f = _noalloc(gdn_lib)
    cases = [
        WORKLOADS["tiny_t1024"].replace(T=1000, Hk=2, Hv=4, h0_std=0.1, seed=41),
        WORKLOADS["tiny_t1024"].replace(B=2, T=640, Hk=1, Hv=2, gate_shift=-3.0, h0_std=0.5,
                                        seed=42),
    ]
    for wl in cases:  # two calls in a row; the second finds the first one's scratch
        host = make_host(wl)
        d = host.to("cuda")
        o1, h1 = _call(gdn_lib, f, d)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        assert gdn_lib.lib().gdn_noalloc_status(stream) == 0  # no bounded wait gave up
        o2, h2 = gdn_lib.chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, n_segments=1)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2), "o (no-alloc) differs from the workspace forward"
        assert torch.equal(h1, h2), "hT (no-alloc) differs from the workspace forward"
        ro, rh = oracle.fwd(host)
        o1, h1 = o1.float().cpu().numpy(), h1.cpu().numpy()
        for b in range(wl.B):
            for j in range(wl.Hv):
                i = b * wl.Hv + j
                assert_rel(o1[b, :, j], ro[i], O_TOL, f"o[{b},{j}] (no-alloc)")
                assert_rel(h1[b, j], rh[i], H_TOL, f"hT[{b},{j}] (no-alloc)")


def test_noalloc_refuses_sizes_beyond_its_scratch(gdn_lib):
    f = _noalloc(gdn_lib)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    # 1 x 32 value heads x 9 chunks = 288 units > 256
    rc = f(fake, fake, fake, fake, fake, None, fake, None, 1, 9 * 128, 16, 32, 128, 128, 128,
           None)
    assert rc == -3
    assert b"workspace" in gdn_lib.lib().gdn_strerror(rc)
