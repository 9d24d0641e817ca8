"""Failure detection on the GPU without a GPU fault.

Every wait inside the kernels (for a TMA copy, a tensor-core product or a
hand-off between warps of one block) is bounded in wall-clock time.  Here a
wait on a barrier that nothing ever signals has to give up, report
GDN_ERR_TIMEOUT through the status word, and leave the context usable: a
forward call afterwards still matches the oracle and reports a clean status.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from linear_attention_rnn_gb300.inputs import WORKLOADS, make_host
from conftest import assert_rel

pytestmark = pytest.mark.gpu

GDN_OK, GDN_ERR_ARG, GDN_ERR_TIMEOUT = 0, -1, -5


def test_wait_that_never_completes_gives_up(gdn_lib):
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    limit_ns = 20_000_000  # 20 ms
    t0 = time.perf_counter()
    rc = gdn_lib.selftest_wait_timeout(limit_ns, status)
    dt = time.perf_counter() - t0
    assert rc == GDN_ERR_TIMEOUT
    assert int(status.item()) == 1  # cleared, then bit 0 set; bit 1 (completed) never
    assert 0.015 < dt < 5.0
    assert gdn_lib.selftest_wait_timeout(10, status) == GDN_ERR_ARG  # limit below 1 us


def test_context_usable_after_timeout(gdn_lib):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert gdn_lib.selftest_wait_timeout(1_000_000, status) == GDN_ERR_TIMEOUT
    inp = make_host(WORKLOADS["tiny_t1024"])
    d = inp.to("cuda")
    wl = inp.wl
    nbytes = gdn_lib.fwd_workspace_bytes(wl.B, wl.T, wl.Hk, wl.Hv)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")  # status word starts set
    o, hT = gdn_lib.chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, workspace=ws)
    assert gdn_lib.workspace_status(ws) == GDN_OK  # the call cleared it; no wait gave up
    heads = [(b, j) for b in range(wl.B) for j in range(wl.Hv)]
    ro, rh = oracle.fwd(inp, heads=heads)
    o = o.float().cpu().numpy()
    for i, (b, j) in enumerate(heads):
        assert_rel(o[b, :, j], ro[i], 2e-2, f"o[{b},{j}]")
