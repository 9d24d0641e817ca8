"""GB300 (sm_103a) chunked Gated DeltaNet -- Python binding of libgdn.

Thin marshalling over the C ABI in include/gdn.h: shape/dtype checks,
allocation of outputs and workspace with torch, and the ctypes call on the
current CUDA stream.  Every step of the computation runs in the library's
kernels; there is no fallback path.  If libgdn.so has not been built, the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

import torch

from . import inputs  # noqa: F401  (seeded input generator)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libgdn.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "gdn.h")

GDN_OK = 0
STATUS = {0: "GDN_OK", -1: "GDN_ERR_ARG", -2: "GDN_ERR_SHAPE", -3: "GDN_ERR_WORKSPACE",
          -4: "GDN_ERR_CUDA", -5: "GDN_ERR_TIMEOUT", -6: "GDN_ERR_UNSUPPORTED"}

_lib = None


class GDNError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = lib().gdn_strerror(code).decode() if _lib is not None else str(code)
        super().__init__(f"{where}: {STATUS.get(code, code)} ({msg})")
        self.code = code


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libgdn.so in-tree (nvcc, sm_103a)."""
    from .build import build as _build
    return _build(force=force, verbose=verbose)


def header_functions():
    """Names of the functions include/gdn.h declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", txt)))


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libgdn.so is not built ({LIB_PATH}); run linear_attention_rnn_gb300.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.gdn_strerror.argtypes = [I]
        L.gdn_strerror.restype = ctypes.c_char_p
        L.gdn_default_segments.argtypes = [I, I, I, I]
        L.gdn_default_segments.restype = I
        for name in ("gdn_fwd_workspace_bytes", "gdn_bwd_workspace_bytes"):
            f = getattr(L, name)
            f.argtypes = [I] * 8
            f.restype = Z
        L.gdn_chunk_fwd.argtypes = [P] * 8 + [I] * 8 + [P, Z, P]
        L.gdn_chunk_fwd.restype = I
        L.gdn_chunk_bwd.argtypes = [P] * 14 + [I] * 8 + [P, Z, P]
        L.gdn_chunk_bwd.restype = I
        L.gdn_chunk_fwd_timed.argtypes = [P] * 8 + [I] * 8 + [P, Z, P, P, I]
        L.gdn_chunk_fwd_timed.restype = I
        L.gdn_chunk_bwd_timed.argtypes = [P] * 14 + [I] * 8 + [P, Z, P, P, I]
        L.gdn_chunk_bwd_timed.restype = I
        L.gdn_saved_bytes.argtypes = [I] * 8
        L.gdn_saved_bytes.restype = Z
        L.gdn_chunk_fwd_ex.argtypes = [P] * 8 + [I] * 8 + [P, Z, P, Z, P, P, I]
        L.gdn_chunk_fwd_ex.restype = I
        L.gdn_chunk_bwd_ex.argtypes = [P] * 14 + [I] * 8 + [P, Z, P, Z, P, P, I]
        L.gdn_chunk_bwd_ex.restype = I
        L.gdn_affine_compose.argtypes = [P] * 4 + [I] * 4 + [P]
        L.gdn_affine_compose.restype = I
        L.gdn_debug_ut.argtypes = [P] * 8 + [I] * 7 + [P]
        L.gdn_debug_ut.restype = I
        L.gdn_workspace_status.argtypes = [P, P]
        L.gdn_workspace_status.restype = I
        L.gdn_layer_workspace_bytes.argtypes = [I] * 9
        L.gdn_layer_workspace_bytes.restype = Z
        L.gdn_layer_fwd.argtypes = [P] * 10 + [I] * 8 + [P, Z, P]
        L.gdn_layer_fwd.restype = I
        L.gdn_layer_bwd.argtypes = [P] * 17 + [I] * 8 + [P, Z, P]
        L.gdn_layer_bwd.restype = I
        L.gdn_segment_fold.argtypes = [P] * 6 + [I] * 8 + [P, Z, P]
        L.gdn_segment_fold.restype = I
        L.gdn_chunk_fwd_noalloc.argtypes = [P] * 8 + [I] * 7 + [P]
        L.gdn_chunk_fwd_noalloc.restype = I
        L.gdn_noalloc_status.argtypes = [P]
        L.gdn_noalloc_status.restype = I
        L.gdn_selftest_wait_timeout.argtypes = [ctypes.c_longlong, P, P]
        L.gdn_selftest_wait_timeout.restype = I
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(t, name, dtype, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _dims(q, k, v, g, beta):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, T, H, D]")
    B, T, Hk, dk = k.shape
    Hv, dv = v.shape[2], v.shape[3]
    _check(q, "q", torch.bfloat16, (B, T, Hk, dk))
    _check(k, "k", torch.bfloat16)
    _check(v, "v", torch.bfloat16, (B, T, Hv, dv))
    _check(g, "g", torch.float32, (B, T, Hv))
    _check(beta, "beta", torch.float32, (B, T, Hv))
    return B, T, Hk, Hv, dk, dv


def default_segments(B: int, T: int, Hv: int, chunk: int = 128) -> int:
    return int(lib().gdn_default_segments(B, T, Hv, chunk))


def fwd_workspace_bytes(B, T, Hk, Hv, dk=128, dv=128, chunk=128, n_segments=0) -> int:
    return int(lib().gdn_fwd_workspace_bytes(B, T, Hk, Hv, dk, dv, chunk, n_segments))


def bwd_workspace_bytes(B, T, Hk, Hv, dk=128, dv=128, chunk=128, n_segments=0) -> int:
    return int(lib().gdn_bwd_workspace_bytes(B, T, Hk, Hv, dk, dv, chunk, n_segments))


def saved_bytes(B, T, Hk, Hv, dk=128, dv=128, chunk=128, n_segments=0) -> int:
    """Bytes of the buffer in which a forward keeps w, u, P and T (and, with
    segments, the segments' entering states) for its backward."""
    return int(lib().gdn_saved_bytes(B, T, Hk, Hv, dk, dv, chunk, n_segments))


def _events(events):
    """ctypes array of raw cudaEvent_t handles of torch.cuda.Event objects
    (each must have been recorded once, so that it exists)."""
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    return arr, len(events)


def _workspace(nbytes, device, ws):
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError("workspace too small")
        return ws
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)


def chunk_fwd(q, k, v, g, beta, h0=None, *, chunk: int = 128, n_segments: int = 0,
              want_hT: bool = True, o=None, hT=None, workspace=None, events=None, saved=None
              ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Forward of the chunked gated delta rule.  Returns (o, hT).
    events: optional torch.cuda.Event list recorded after each kernel launch.
    saved: optional uint8 CUDA buffer of saved_bytes(...) bytes in which the
    forward keeps w, u, P and T for chunk_bwd(..., saved=the same buffer)."""
    B, T, Hk, Hv, dk, dv = _dims(q, k, v, g, beta)
    dev = q.device
    _check(h0, "h0", torch.float32, (B, Hv, dk, dv))
    if o is None:
        o = torch.empty((B, T, Hv, dv), dtype=torch.bfloat16, device=dev)
    _check(o, "o", torch.bfloat16, (B, T, Hv, dv))
    if want_hT and hT is None:
        hT = torch.empty((B, Hv, dk, dv), dtype=torch.float32, device=dev)
    nbytes = fwd_workspace_bytes(B, T, Hk, Hv, dk, dv, chunk, n_segments)
    ws = _workspace(nbytes, dev, workspace)
    if saved is not None:
        ev = _events(events) if events else (None, 0)
        rc = lib().gdn_chunk_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                    _ptr(o), _ptr(hT), B, T, Hk, Hv, dk, dv, chunk, n_segments,
                                    _ptr(saved), saved.numel() * saved.element_size(), _ptr(ws),
                                    ws.numel(), _stream(dev), *ev)
        if rc != GDN_OK:
            raise GDNError(rc, "gdn_chunk_fwd_ex")
        return o, hT
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(hT), B, T,
            Hk, Hv, dk, dv, chunk, n_segments, _ptr(ws), ws.numel(), _stream(dev)]
    if events:
        rc = lib().gdn_chunk_fwd_timed(*args, *_events(events))
    else:
        rc = lib().gdn_chunk_fwd(*args)
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_chunk_fwd")
    return o, hT


def chunk_bwd(q, k, v, g, beta, h0, dO, dhT=None, *, chunk: int = 128, n_segments: int = 0,
              want_dh0: bool = True, out=None, workspace=None, events=None, saved=None):
    """Backward of the chunked gated delta rule.
    Returns (dq, dk, dv, dg, dbeta, dh0).
    out: optional (dq, dk, dv, dg, dbeta, dh0) tensors to write (dh0 may be
    None), e.g. views of one buffer that leaves the device in one copy.
    events: optional torch.cuda.Event list recorded after each kernel launch."""
    B, T, Hk, Hv, dk, dv = _dims(q, k, v, g, beta)
    dev = q.device
    _check(h0, "h0", torch.float32, (B, Hv, dk, dv))
    _check(dO, "dO", torch.bfloat16, (B, T, Hv, dv))
    _check(dhT, "dhT", torch.float32, (B, Hv, dk, dv))
    if out is not None:
        dq, dk_, dv_, dg, db, dh0 = out
        _check(dq, "dq", torch.bfloat16, tuple(q.shape))
        _check(dk_, "dk", torch.bfloat16, tuple(k.shape))
        _check(dv_, "dv", torch.bfloat16, tuple(v.shape))
        _check(dg, "dg", torch.float32, tuple(g.shape))
        _check(db, "dbeta", torch.float32, tuple(beta.shape))
        _check(dh0, "dh0", torch.float32, (B, Hv, dk, dv))
    else:
        dq = torch.empty_like(q)
        dk_ = torch.empty_like(k)
        dv_ = torch.empty_like(v)
        dg = torch.empty_like(g)
        db = torch.empty_like(beta)
        dh0 = torch.empty((B, Hv, dk, dv), dtype=torch.float32, device=dev) if want_dh0 else None
    nbytes = bwd_workspace_bytes(B, T, Hk, Hv, dk, dv, chunk, n_segments)
    ws = _workspace(nbytes, dev, workspace)
    if saved is not None:  # w, u, P, T kept by chunk_fwd(..., saved=saved) on these inputs
        ev = _events(events) if events else (None, 0)
        rc = lib().gdn_chunk_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                    _ptr(dO), _ptr(dhT), _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg),
                                    _ptr(db), _ptr(dh0), B, T, Hk, Hv, dk, dv, chunk, n_segments,
                                    _ptr(saved), saved.numel() * saved.element_size(), _ptr(ws),
                                    ws.numel(), _stream(dev), *ev)
        if rc != GDN_OK:
            raise GDNError(rc, "gdn_chunk_bwd_ex")
        return dq, dk_, dv_, dg, db, dh0
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(dO), _ptr(dhT),
            _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg), _ptr(db), _ptr(dh0), B, T, Hk, Hv, dk, dv,
            chunk, n_segments, _ptr(ws), ws.numel(), _stream(dev)]
    if events:
        rc = lib().gdn_chunk_bwd_timed(*args, *_events(events))
    else:
        rc = lib().gdn_chunk_bwd(*args)
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_chunk_bwd")
    return dq, dk_, dv_, dg, db, dh0


def layer_workspace_bytes(backward, B, T, Hk, Hv, dk=128, dv=128, chunk=128, n_segments=0) -> int:
    return int(lib().gdn_layer_workspace_bytes(int(backward), B, T, Hk, Hv, dk, dv, chunk,
                                               n_segments))


def layer_fwd(q, k, v, a, b, z=None, h0=None, *, chunk: int = 128, n_segments: int = 0,
              keep_o: bool = True, want_hT: bool = True, workspace=None):
    """Layer forward: q, k raw (normalised inside), a, b gate logits
    (g = -softplus(a), beta = sigmoid(b)), optional output gate z.
    Returns (y, o, hT): o is the ungated output (None unless keep_o and z)."""
    B, T, Hk, Hv, dk, dv = _dims(q, k, v, a, b)
    dev = q.device
    _check(z, "z", torch.bfloat16, (B, T, Hv, dv))
    _check(h0, "h0", torch.float32, (B, Hv, dk, dv))
    y = torch.empty((B, T, Hv, dv), dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(y) if (keep_o and z is not None) else None
    hT = torch.empty((B, Hv, dk, dv), dtype=torch.float32, device=dev) if want_hT else None
    ws = _workspace(layer_workspace_bytes(0, B, T, Hk, Hv, dk, dv, chunk, n_segments), dev,
                    workspace)
    rc = lib().gdn_layer_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(z), _ptr(h0),
                             _ptr(y), _ptr(o), _ptr(hT), B, T, Hk, Hv, dk, dv, chunk, n_segments,
                             _ptr(ws), ws.numel(), _stream(dev))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_layer_fwd")
    return y, o, hT


def layer_bwd(q, k, v, a, b, z, h0, o, dy, dhT=None, *, chunk: int = 128, n_segments: int = 0,
              want_dh0: bool = True, workspace=None):
    """Layer backward.  Returns (dq, dk, dv, da, db, dz, dh0) for the raw q, k
    and the gate logits; dz is None without a gate."""
    B, T, Hk, Hv, dk, dv = _dims(q, k, v, a, b)
    dev = q.device
    _check(z, "z", torch.bfloat16, (B, T, Hv, dv))
    _check(o, "o", torch.bfloat16, (B, T, Hv, dv))
    _check(dy, "dy", torch.bfloat16, (B, T, Hv, dv))
    _check(h0, "h0", torch.float32, (B, Hv, dk, dv))
    _check(dhT, "dhT", torch.float32, (B, Hv, dk, dv))
    dq, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    da, db = torch.empty_like(a), torch.empty_like(b)
    dz = torch.empty_like(z) if z is not None else None
    dh0 = torch.empty((B, Hv, dk, dv), dtype=torch.float32, device=dev) if want_dh0 else None
    ws = _workspace(layer_workspace_bytes(1, B, T, Hk, Hv, dk, dv, chunk, n_segments), dev,
                    workspace)
    rc = lib().gdn_layer_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(z), _ptr(h0),
                             _ptr(o), _ptr(dy), _ptr(dhT), _ptr(dq), _ptr(dk_), _ptr(dv_),
                             _ptr(da), _ptr(db), _ptr(dz), _ptr(dh0), B, T, Hk, Hv, dk, dv, chunk,
                             n_segments, _ptr(ws), ws.numel(), _stream(dev))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_layer_bwd")
    return dq, dk_, dv_, da, db, dz, dh0


def affine_compose(A: torch.Tensor, Bm: torch.Tensor):
    """Inclusive prefix of affine maps along dim 1: A [batch, n, dk, dk],
    B [batch, n, dk, dv] (fp32)."""
    batch, n, dk, _ = A.shape
    dv = Bm.shape[3]
    _check(A, "A", torch.float32, (batch, n, dk, dk))
    _check(Bm, "B", torch.float32, (batch, n, dk, dv))
    Ao = torch.empty_like(A)
    Bo = torch.empty_like(Bm)
    rc = lib().gdn_affine_compose(_ptr(A), _ptr(Bm), _ptr(Ao), _ptr(Bo), batch, n, dk, dv,
                                  _stream(A.device))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_affine_compose")
    return Ao, Bo


def segment_fold(k, v, g, beta, n_segments: int = 1, *, chunk: int = 128, want_A: bool = True,
                 workspace=None):
    """Per-segment affine maps (A_s, B_s) of the inter-chunk recurrence:
    A [B, Hv, S, dk, dk] (None if want_A is False) and B [B, Hv, S, dk, dv],
    fp32, with the state leaving segment s equal to A_s h_in + B_s."""
    B, T, Hk, dk = k.shape
    Hv, dv = v.shape[2], v.shape[3]
    _check(k, "k", torch.bfloat16)
    _check(v, "v", torch.bfloat16, (B, T, Hv, dv))
    _check(g, "g", torch.float32, (B, T, Hv))
    _check(beta, "beta", torch.float32, (B, T, Hv))
    dev = k.device
    A = (torch.empty((B, Hv, n_segments, dk, dk), dtype=torch.float32, device=dev)
         if want_A else None)
    Bm = torch.empty((B, Hv, n_segments, dk, dv), dtype=torch.float32, device=dev)
    nbytes = fwd_workspace_bytes(B, T, Hk, Hv, dk, dv, chunk, 1)
    ws = _workspace(nbytes, dev, workspace)
    rc = lib().gdn_segment_fold(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A), _ptr(Bm), B, T,
                                Hk, Hv, dk, dv, chunk, n_segments, _ptr(ws), ws.numel(),
                                _stream(dev))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_segment_fold")
    return A, Bm


def debug_ut(k, v, g, beta, chunk: int = 128, tiles: bool = False):
    """Per-chunk S, T (fp32) and w, u (bf16), each [B, Hv, N, chunk, .].

    The library exports 128-row tiles; with chunk = 64 each holds two chunks
    (S and T block diagonal).  tiles=True returns those tiles as exported,
    [B, Hv, ceil(T / 128), 128, .]."""
    B, T, Hk, dk = k.shape
    Hv, dv = v.shape[2], v.shape[3]
    _check(k, "k", torch.bfloat16)
    _check(v, "v", torch.bfloat16, (B, T, Hv, dv))
    _check(g, "g", torch.float32, (B, T, Hv))
    _check(beta, "beta", torch.float32, (B, T, Hv))
    NT = (T + 127) // 128
    dev = k.device
    S = torch.empty((B, Hv, NT, 128, 128), dtype=torch.float32, device=dev)
    Tm = torch.empty_like(S)
    w = torch.empty((B, Hv, NT, 128, dk), dtype=torch.bfloat16, device=dev)
    u = torch.empty((B, Hv, NT, 128, dv), dtype=torch.bfloat16, device=dev)
    rc = lib().gdn_debug_ut(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S), _ptr(Tm), _ptr(w),
                            _ptr(u), B, T, Hk, Hv, dk, dv, chunk, _stream(dev))
    if rc != GDN_OK:
        raise GDNError(rc, "gdn_debug_ut")
    if tiles or chunk == 128:
        return S, Tm, w, u
    N = (T + chunk - 1) // chunk  # chunk 64: the diagonal blocks and row halves of the tiles

    def diag(x):
        x6 = x.view(B, Hv, NT, 2, 64, 2, 64)
        return torch.stack([x6[:, :, :, 0, :, 0, :], x6[:, :, :, 1, :, 1, :]], 3).reshape(
            B, Hv, 2 * NT, 64, 64)[:, :, :N]

    def rows(x):
        return x.reshape(B, Hv, 2 * NT, 64, x.shape[-1])[:, :, :N]

    return diag(S), diag(Tm), rows(w), rows(u)


def workspace_status(ws: torch.Tensor) -> int:
    """Status code (GDN_OK or GDN_ERR_TIMEOUT) of the bounded in-kernel waits of
    the last forward/backward call that used workspace `ws`.  Synchronises the
    current stream."""
    return lib().gdn_workspace_status(_ptr(ws), _stream(ws.device))


def selftest_wait_timeout(limit_ns: int, status: torch.Tensor) -> int:
    """Runs one block whose bounded wait can never complete and must give up
    after limit_ns; returns the library's status code (GDN_ERR_TIMEOUT = -5 is
    the expected outcome).  status: a one-element int32 CUDA tensor."""
    _check(status, "status", torch.int32, (1,))
    return lib().gdn_selftest_wait_timeout(int(limit_ns), _ptr(status), _stream(status.device))


__all__ = ["build", "lib", "chunk_fwd", "chunk_bwd", "layer_fwd", "layer_bwd",
           "layer_workspace_bytes", "saved_bytes", "affine_compose", "segment_fold", "debug_ut",
           "fwd_workspace_bytes", "bwd_workspace_bytes", "default_segments", "GDNError",
           "header_functions", "workspace_status", "selftest_wait_timeout"]
