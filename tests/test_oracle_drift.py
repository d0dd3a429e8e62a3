"""The oracle against itself on the full 16-layer decoder: the spread of valid summation orders.

Two evaluations of the same network by the oracle, one with the hidden and MLP features
relabelled (exactly the same function in real arithmetic, see tests/_drift.py), drift apart
by about 1.4e-2 relative Frobenius after 16 bf16 decode layers and 1.7e-2 after 16 prefill
layers on the causal prefix. An end-to-end bound of 5e-3 is therefore out of reach for any
implementation that sums in another order; the GPU end-to-end checks hold the megakernel to
MARGIN (2) times the drift measured on their own inputs, while every node is also checked
against the oracle applied to the GPU's own inputs of that node at 5e-3.

The figures asserted below are measured on the decode workload's own inputs (seed 0, the
inputs the GPU test and the benchmark use).
"""
import numpy as np
import pytest

import _drift
from oracle import models
from tensor_core_gemm_gb300 import synth, workloads


@pytest.fixture(scope="module")
def decode_wl():
    return workloads.decode(device="cpu", seed=0)


def test_decode_drift_of_two_summation_orders_at_16_layers(decode_wl):
    wl = decode_wl
    sh, cap = wl.info["shape"], wl.info["cap"]
    wts = _drift.decoder_weights(wl)
    f32 = synth.to_numpy_f32
    kc = list(f32(wl.data[wl.info["kc"]]).reshape(sh.layers, cap, -1))
    vc = list(f32(wl.data[wl.info["vc"]]).reshape(sh.layers, cap, -1))
    (fro, mx), ref = _drift.decode_drift(f32(wl.data[0]), wts, kc, vc, wl.info["pos"])
    # measured 1.42e-2 (seeds 1-3 of the relabelling: 1.39e-2 .. 1.42e-2)
    assert 1.0e-2 < fro < 2.0e-2, fro
    assert mx > 0.0
    # after one layer the two orders still agree within the parity tolerance
    one = models.DecoderWeights(wts.wqkv[:1], wts.wo[:1], wts.wg[:1], wts.wu[:1], wts.wd[:1],
                                wts.g_attn[:1], wts.g_mlp[:1], sh.hq, sh.hkv, sh.hd, sh.eps,
                                sh.theta)
    (fro1, _), _ = _drift.decode_drift(f32(wl.data[0]), one, kc[:1], vc[:1], wl.info["pos"])
    assert fro1 < 5e-3, fro1


def test_prefill_drift_of_two_summation_orders_at_16_layers(decode_wl):
    # the prefill workload has the same weights as the decode one (same seeds per tensor)
    wts = _drift.decoder_weights(decode_wl)
    sh = decode_wl.info["shape"]
    x = synth.to_numpy_f32(synth.normal((64, sh.hidden), 1.0, "bf16", 0, "cpu"))
    (fro, _), _ = _drift.prefill_drift(x, wts)
    # measured 1.75e-2 on a 64-token prefix (1.69e-2 on 256 tokens)
    assert 1.0e-2 < fro < 2.5e-2, fro
