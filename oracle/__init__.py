"""fp64 CPU oracle of the chunked gated delta rule.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package's smoke
check and by the bench's CPU-baseline leg, never by the product path.

* ``gdn_oracle.c`` -- the per-token rule and its exact adjoint (plain C,
  fp64, OpenMP over independent heads / state columns), reached here through
  ctypes.
* ``chunked.py``   -- the chunked WY/UT form, the doubling-ladder and
  forward-substitution inverses, affine maps, their composition and the
  two-pass segment scan, in fp64 numpy.

Inputs come from ``linear_attention_rnn_gb300.inputs`` (the seeded generator,
which holds none of the method's arithmetic).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import chunked  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into oracle/_build/libgdn_oracle.so (gcc, OpenMP)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i = ctypes.c_int
        L.orc_fwd.argtypes = [i] * 6 + [P] * 6 + [i, P, P, P, P, i]
        L.orc_fwd.restype = i
        L.orc_bwd.argtypes = [i] * 6 + [P] * 8 + [i, P, P] + [P] * 6 + [i]
        L.orc_bwd.restype = i
        L.orc_num_threads.argtypes = []
        L.orc_num_threads.restype = i
        _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().orc_num_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _heads(wl, heads):
    if heads is None:
        heads = [(b, j) for b in range(wl.B) for j in range(wl.Hv)]
    sb = np.ascontiguousarray([h[0] for h in heads], dtype=np.int32)
    sj = np.ascontiguousarray([h[1] for h in heads], dtype=np.int32)
    return heads, sb, sj


def fwd(inp, heads=None, want_o: bool = True, col_block: int = 16):
    """Per-token forward for the selected (b, j) heads (default: all).

    Returns (o, hT): o [n_sel, T, dv] fp64 (None if want_o is False) and
    hT [n_sel, dk, dv] fp64.
    """
    wl = inp.wl
    heads, sb, sj = _heads(wl, heads)
    n = len(heads)
    q, k, v = inp.bits("q"), inp.bits("k"), inp.bits("v")
    g, beta, h0 = inp.f32("g"), inp.f32("beta"), inp.f32("h0")
    o = np.zeros((n, wl.T, wl.dv)) if want_o else None
    hT = np.zeros((n, wl.dk, wl.dv))
    cb = col_block if wl.dv % col_block == 0 else wl.dv
    rc = lib().orc_fwd(wl.B, wl.T, wl.Hk, wl.Hv, wl.dk, wl.dv, _ptr(q), _ptr(k), _ptr(v),
                       _ptr(g), _ptr(beta), _ptr(h0), n, _ptr(sb), _ptr(sj), _ptr(o),
                       _ptr(hT), cb)
    if rc != 0:
        raise RuntimeError(f"orc_fwd failed ({rc})")
    return o, hT


def bwd(inp, heads=None, ckpt: int = 64):
    """Per-token adjoint for the selected (b, j) heads (default: all).

    Returns a dict of fp64 arrays: dq_v, dk_v [n_sel, T, dk] (each value
    head's contribution), dv [n_sel, T, dv], dg, dbeta [n_sel, T],
    dh0 [n_sel, dk, dv], and 'heads'.
    """
    wl = inp.wl
    heads, sb, sj = _heads(wl, heads)
    n = len(heads)
    q, k, v, dO = inp.bits("q"), inp.bits("k"), inp.bits("v"), inp.bits("dO")
    g, beta, h0, dhT = inp.f32("g"), inp.f32("beta"), inp.f32("h0"), inp.f32("dhT")
    T, dk, dv = wl.T, wl.dk, wl.dv
    out = dict(dq_v=np.zeros((n, T, dk)), dk_v=np.zeros((n, T, dk)), dv=np.zeros((n, T, dv)),
               dg=np.zeros((n, T)), dbeta=np.zeros((n, T)), dh0=np.zeros((n, dk, dv)))
    rc = lib().orc_bwd(wl.B, T, wl.Hk, wl.Hv, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                       _ptr(beta), _ptr(h0), _ptr(dO), _ptr(dhT), n, _ptr(sb), _ptr(sj),
                       _ptr(out["dq_v"]), _ptr(out["dk_v"]), _ptr(out["dv"]), _ptr(out["dg"]),
                       _ptr(out["dbeta"]), _ptr(out["dh0"]), ckpt)
    if rc != 0:
        raise RuntimeError(f"orc_bwd failed ({rc})")
    out["heads"] = heads
    return out


def key_head_grads(wl, res):
    """Sum the per-value-head dq/dk contributions of `res` (from bwd over
    every value head of some batch rows) into key heads.  Returns
    {(b, kh): (dq [T, dk], dk [T, dk])} for each key head whose value heads
    are all present."""
    grp = wl.Hv // wl.Hk
    idx = {h: i for i, h in enumerate(res["heads"])}
    out = {}
    for b in sorted({h[0] for h in res["heads"]}):
        for kh in range(wl.Hk):
            members = [(b, kh * grp + r) for r in range(grp)]
            if all(m in idx for m in members):
                dq = sum(res["dq_v"][idx[m]] for m in members)
                dk = sum(res["dk_v"][idx[m]] for m in members)
                out[(b, kh)] = (dq, dk)
    return out
