import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from linear_attention_rnn_gb300.inputs import Inputs, Workload  # noqa: E402


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running (full-size workloads)")


def from_arrays(q, k, v, g, beta, h0=None, dO=None, dhT=None, chunk=128, name="adhoc"):
    """Build an Inputs from arrays shaped [B,T,H,D] / [B,T,H] / [B,H,dk,dv].

    q, k, v, dO are rounded to bf16 (RNE); callers that need exact values pass
    values representable in bf16.
    """
    q = np.asarray(q, np.float32)
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    B, T, Hk, dk = k.shape
    Hv, dv = v.shape[2], v.shape[3]
    wl = Workload(name, B=B, T=T, Hk=Hk, Hv=Hv, dk=dk, dv=dv, chunk=chunk,
                  h0_std=1.0 if h0 is not None else 0.0, backward=dO is not None)
    bf = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    f32 = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x, np.float32))
    return Inputs(wl, bf(q), bf(k), bf(v), f32(g), f32(beta), f32(h0),
                  None if dO is None else bf(dO), f32(dhT))


def as64(inp, name):
    """Exact fp64 copy of an input tensor (bf16 and fp32 widen exactly)."""
    x = getattr(inp, name)
    return None if x is None else x.detach().cpu().to(torch.float64).numpy()


def head(inp, b, j):
    """fp64 per-head slices (q, k, v, g, beta, h0) of value head j."""
    grp = inp.wl.Hv // inp.wl.Hk
    kh = j // grp
    q, k, v = as64(inp, "q"), as64(inp, "k"), as64(inp, "v")
    g, beta, h0 = as64(inp, "g"), as64(inp, "beta"), as64(inp, "h0")
    return (q[b, :, kh], k[b, :, kh], v[b, :, j], g[b, :, j], beta[b, :, j],
            None if h0 is None else h0[b, j])


def relmax(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(x - ref)) / (den if den > 0 else 1.0))


def random_small(B=1, T=40, Hk=1, Hv=1, dk=8, dv=8, seed=0, gate_shift=0.0, h0=True,
                 bwd=False, unit=True):
    """Small random inputs with the workload distributions (host numpy)."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hk, dk))
    k = rng.standard_normal((B, T, Hk, dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hv, dv))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, T, Hv))))
    x = rng.standard_normal((B, T, Hv)) + gate_shift
    g = -(np.maximum(x, 0) + np.log1p(np.exp(-np.abs(x))))
    h0a = rng.standard_normal((B, Hv, dk, dv)) * 0.5 if h0 else None
    dO = rng.standard_normal((B, T, Hv, dv)) if bwd else None
    dhT = rng.standard_normal((B, Hv, dk, dv)) * 0.3 if bwd else None
    return from_arrays(q, k, v, g, beta, h0a, dO, dhT)


# --------------------------------------------------------------------- GPU side
@pytest.fixture(scope="session")
def gdn_lib():
    """The built C-ABI library (GPU tests only)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_rnn_gb300 as gdn
    gdn.build()
    gdn.lib()
    return gdn


def key_head_slice(inp, b, kh):
    """Inputs restricted to batch row b, key head kh and its value heads
    (host tensors) -- what the oracle needs to check those heads exactly."""
    wl = inp.wl
    grp = wl.Hv // wl.Hk
    j0 = kh * grp
    cut = lambda x, lo, n: None if x is None else x[b:b + 1, :, lo:lo + n].contiguous().cpu()
    cut_s = lambda x: None if x is None else x[b:b + 1, j0:j0 + grp].contiguous().cpu()
    sub = Inputs(wl.replace(B=1, Hk=1, Hv=grp), cut(inp.q, kh, 1), cut(inp.k, kh, 1),
                 cut(inp.v, j0, grp), cut(inp.g, j0, grp), cut(inp.beta, j0, grp),
                 cut_s(inp.h0), cut(inp.dO, j0, grp) if inp.dO is not None else None,
                 cut_s(inp.dhT))
    return sub, j0, grp


# Error margins of the parity tests, per (workload, tensor): the largest
# max|x - ref| / max|ref| seen and its tolerance.  Written as JSON at the end of
# the session when GDN_MARGINS_OUT names a file.
MARGINS = {}


def record_margin(workload, tensor, err, tol):
    key = f"{workload}|{tensor}"
    prev = MARGINS.get(key)
    if prev is None or err > prev["err"]:
        MARGINS[key] = {"workload": workload, "tensor": tensor, "err": float(err),
                        "tol": float(tol)}


def pytest_sessionfinish(session, exitstatus):
    out = os.environ.get("GDN_MARGINS_OUT")
    if out and MARGINS:
        import json
        os.makedirs(os.path.dirname(os.path.abspath(out)), exist_ok=True)
        with open(out, "w") as f:
            json.dump(sorted(MARGINS.values(), key=lambda m: (m["workload"], m["tensor"])), f,
                      indent=1)


def assert_rel(x, ref, tol, what, margin=None):
    """max|x - ref| <= tol * max|ref|; margin = (workload, tensor) records the
    error in the session's margin table."""
    err = relmax(x, ref)
    if margin is not None:
        record_margin(margin[0], margin[1], err, tol)
    assert err <= tol, f"{what}: max|x - ref| / max|ref| = {err:.3e} > {tol:.1e}"
    return err
