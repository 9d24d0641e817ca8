"""Where the final state's rounding error comes from, on a rounding model of
the forward's bf16 operands (CPU).

The device keeps the state in fp32 but hands it to the tensor cores as bf16
(the w h and Q h products), stores w and u as bf16 tiles, and rounds Delta to
bf16 for the state update.  A split-precision (hi + lo) state operand would
remove the first rounding only.  This model replays the chunked forward with
those roundings, in fp64 otherwise, and shows on the slow-decay inputs of the
million-token workload that the state operand's rounding is not what the hT
error is made of (splitting it changes the error by well under 1%), and that
the error does not grow with the sequence length: with g ~ -softplus(N(-3, 1))
a 128-token chunk still scales the state by about exp(-9), so the rounding of
one chunk does not survive many chunks.  The fp64 chunked route is the
reference (pinned to the per-token rule elsewhere).
"""
import numpy as np
import torch

from oracle import chunked
from linear_attention_rnn_gb300.inputs import WORKLOADS, make_host

C = 128


def _bf(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()


def _model_states(q, k, v, g, beta, h0, split_state=False):
    """States after every chunk, (model, fp64 reference), with the forward's
    bf16 operand roundings in the model: T' = T diag(beta) and T'' = T
    diag(beta gamma) as bf16 operands, w and u stored as bf16, the state as a
    bf16 operand (or hi + lo), ef Delta as a bf16 operand."""
    h = np.zeros((k.shape[1], v.shape[1])) if h0 is None else h0.copy()
    href = h.copy()
    out = []
    for c0 in range(0, k.shape[0], C):
        sl = slice(c0, min(c0 + C, k.shape[0]))
        K, V, b = k[sl], v[sl], beta[sl]
        it = chunked.chunk_intermediates(q[sl], K, V, g[sl], b)
        G = np.cumsum(g[sl])
        w = _bf(_bf(it["T"] * (b * np.exp(G))[None, :]) @ K)
        u = _bf(_bf(it["T"] * b[None, :]) @ V)
        hb = _bf(h) + _bf(h - _bf(h)) if split_state else _bf(h)
        delta = u - w @ hb
        h = np.exp(G[-1]) * h + K.T @ _bf(np.exp(G[-1] - G)[:, None] * delta)
        href = np.exp(G[-1]) * href + it["kg"].T @ (it["u"] - it["w"] @ href)
        out.append((h.copy(), href.copy()))
    return out


def _rel(x, ref):
    return float(np.max(np.abs(x - ref)) / np.max(np.abs(ref)))


def test_state_operand_rounding_is_not_the_final_state_error():
    wl = WORKLOADS["million_t1048576_slow"].replace(T=64 * C, Hk=1, Hv=2, seed=7)
    x = make_host(wl, backward=False)
    f = lambda t: t.to(torch.float64).numpy()
    for j in range(2):
        args = (f(x.q)[0, :, 0], f(x.k)[0, :, 0], f(x.v)[0, :, j], f(x.g)[0, :, j],
                f(x.beta)[0, :, j], f(x.h0)[0, j])
        base = [_rel(h, r) for h, r in _model_states(*args)]
        split = [_rel(h, r) for h, r in _model_states(*args, split_state=True)]
        # the reference walk is the oracle's chunked forward
        assert np.array_equal(_model_states(*args)[-1][1], chunked.head_fwd(*args, C)[1])
        assert max(base) <= 1e-2  # every chunk's state within the final state's tolerance
        for c, (e0, e1) in enumerate(zip(base, split)):
            assert abs(e1 - e0) <= 0.01 * e0, (j, c, e0, e1)
        # no drift along the sequence: the last 16 chunks' mean error is no
        # larger than the first 16 chunks' (after 8 chunks of warm-up), up to noise
        assert np.mean(base[48:]) <= 1.5 * np.mean(base[8:24]), (np.mean(base[8:24]), np.mean(base[48:]))
