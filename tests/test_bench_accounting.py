"""The bench's algorithmic accounting, on CPU.

The roofline fractions the bench reports divide algorithmic work by measured
time, so the work figures are checked here against independent counts: the
bytes against the tensors the input recipe actually builds, the FLOP constants
by explicit loops over the products they stand for, and the roofline arithmetic
on known timings.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from linear_attention_rnn_gb300.inputs import WORKLOADS, make_host  # noqa: E402

C = D = 128


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def test_bytes_match_the_tensors_of_a_step():
    wl = WORKLOADS["tiny_t1024"].replace(B=2, T=384, Hk=2, Hv=4, h0_std=0.1, backward=True)
    x = make_host(wl)
    ins = sum(_nbytes(t) for t in (x.q, x.k, x.v, x.g, x.beta, x.h0))
    # outputs: o like v, hT like h0; gradients like their inputs
    fwd = ins + _nbytes(x.v) + _nbytes(x.h0)
    bwd = ins + _nbytes(x.dO) + _nbytes(x.dhT) + ins
    alg = bench.algorithmic(wl)
    assert alg["fwd_bytes"] == fwd
    assert alg["bwd_bytes"] == bwd


def test_layer_bytes_are_the_documented_figures():
    alg = bench.algorithmic(WORKLOADS["layer_t4096"])
    assert alg["fwd_bytes"] == 105_906_176
    assert alg["bwd_bytes"] == 176_160_768


def test_triangular_product_flops_by_counting():
    # lower-triangular 128 x 128 times 128 x 128: one multiply-add per nonzero
    # of the triangle per output column
    flops = sum(2 * D for r in range(C) for s in range(r + 1))
    assert bench.FLOP_TRI == flops
    assert bench.FLOP_FULL == sum(2 * D for r in range(C) for s in range(C))


def test_ladder_flops_by_walking_its_levels():
    # doubling levels b = 1, 2, ..., 64; at each, for every pair of b x b
    # diagonal blocks: Y = S_l X_A and then -X_D Y, two b x b x b products
    flops, b = 0, 1
    while b < C:
        for _pair in range(C // (2 * b)):
            flops += 2 * b * b * b  # S_l X_A
            flops += 2 * b * b * b  # X_D Y
        b *= 2
    assert bench.FLOP_LADDER == flops


def test_kernel_table_and_roofline_arithmetic():
    wl = WORKLOADS["layer_t4096"]
    alg = bench.algorithmic(wl)
    pk = {"hbm": 6789.6, "bf16": 1886.0, "source": "test"}
    kern = {"prep": 0.085, "walk": 0.070, "prep_b": 0.087, "walks": 0.113, "grads": 0.152}
    step = sum(kern.values())
    kernels, roof = bench.kernel_table(kern, alg, pk, step)
    assert set(kernels) == set(kern)
    assert sum(k["share"] for k in kernels.values()) == pytest.approx(1.0, abs=1e-3)
    # backward launches of a kernel carry its symbol and its work
    assert kernels["prep_b"]["symbol"] == kernels["prep"]["symbol"] == "k_prep"
    prep_flops = alg["units"] * bench.FLOPS["prep"] + alg["kunits"] * bench.FLOP_PER_CHUNK_KHEAD
    assert kernels["prep_b"]["tflops"] == pytest.approx(prep_flops / 0.087e-3 / 1e12, abs=0.01)
    # the dominant kernel is the slowest, and its fraction is work / time / peak
    assert roof["kernel"] == "k_grads"
    achieved = alg["units"] * bench.FLOPS["grads"] / 0.152e-3 / 1e12
    assert roof["achieved"] == pytest.approx(achieved, abs=0.01)
    assert roof["frac"] == pytest.approx(achieved / 1886.0, abs=1e-4)
    assert roof["traffic"] == bench.NCU_TRAFFIC.get("grads")


def test_chunk64_flops_by_counting():
    # 64-token chunks: the same products on 64 rows; the ladder's levels stop at b = 32
    C64 = 64
    f = bench.chunk_flops(C64, D)
    assert f["tri"] == sum(2 * D for r in range(C64) for s in range(r + 1))
    assert f["full"] == sum(2 * D for r in range(C64) for s in range(D))
    flops, b = 0, 1
    while b < C64:
        flops += (C64 // (2 * b)) * 2 * (2 * b * b * b)
        b *= 2
    assert f["ladder"] == flops
    # K K^T and Q K^T: each a C x C triangle of D-long dot products, counted at half the square
    assert f["khead"] == 2 * (2 * C64 * C64 * D) // 2
    assert bench.chunk_flops(C, D) == dict(khead=bench.FLOP_PER_CHUNK_KHEAD, ladder=bench.FLOP_LADDER,
                                           tri=bench.FLOP_TRI, full=bench.FLOP_FULL)
    # per token the D x D products are unchanged and the intra-chunk ones halve
    a128 = bench.algorithmic(WORKLOADS["layer_t4096"])
    a64 = bench.algorithmic(WORKLOADS["layer_t4096"].replace(chunk=64))
    assert a64["fwd_bytes"] == a128["fwd_bytes"]
    assert a64["fwd_flops"] < a128["fwd_flops"]
