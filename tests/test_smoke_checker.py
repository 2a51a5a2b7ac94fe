"""The checker behind ``__graft_entry__.smoke()``, run on the CPU: buffers
that the oracle itself produces for the tiny MLP step pass it, and a planted
mistake in a scale layout, a GEMM output or a weight transpose fails it.
(The oracle here only builds the buffers; the GPU run feeds the checker the
library's buffers instead.)"""
import numpy as np
import pytest
import torch

import __graft_entry__ as ge
import oracle
import synth


def bf16_bits(a):
    t = torch.from_numpy(np.asarray(a, np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module")
def buffers():
    x, wgu, wd, dy = synth.mlp_step(1, 256, 256, 384)
    h = {"X": x, "dY": dy, "Wgu": wgu, "Wd": wd}
    for src in ("X", "dY"):
        h["q" + src], h["s" + src], _ = oracle.quant_1x128(h[src])
        h["q" + src + "T"], h["s" + src + "T"], _ = oracle.quant_128x1_transposed(h[src])
    for w in ("Wgu", "Wd"):
        h["q" + w], h["s" + w], _ = oracle.quant_128x128(h[w])
        h["q" + w + "T"] = np.ascontiguousarray(h["q" + w].T)
        h["s" + w + "T"] = np.ascontiguousarray(h["s" + w].T)

    def gemm(a, sa, ga, b, sb, gb):
        return oracle.gemm_full(h[a], oracle.E4M3, h[sa], ga, h[b], oracle.E4M3, h[sb], gb)

    h["GU"] = bf16_bits(gemm("qX", "sX", 0, "qWgu", "sWgu", 1))
    hv = oracle.swiglu_fwd(h["GU"])
    h["qH"], h["sH"], _ = oracle.quant_1x128(hv)
    h["qHT"], h["sHT"], _ = oracle.quant_128x1_transposed(hv)
    h["Y"] = bf16_bits(gemm("qH", "sH", 0, "qWd", "sWd", 1))
    h["dH"] = bf16_bits(gemm("qdY", "sdY", 0, "qWdT", "sWdT", 1))
    dgu = oracle.swiglu_bwd(h["GU"], h["dH"])
    h["qdGU"], h["sdGU"], _ = oracle.quant_1x128(dgu)
    h["qdGUT"], h["sdGUT"], _ = oracle.quant_128x1_transposed(dgu)
    h["dX"] = bf16_bits(gemm("qdGU", "sdGU", 0, "qWguT", "sWguT", 1))
    h["dWd"] = gemm("qdYT", "sdYT", 0, "qHT", "sHT", 0).astype(np.float32)
    h["dWgu"] = gemm("qdGUT", "sdGUT", 0, "qXT", "sXT", 0).astype(np.float32)
    return h


def test_oracle_made_step_passes(buffers):
    ge._check_step(buffers)


def test_swapped_scale_rows_fail(buffers):
    bad = dict(buffers, sXT=buffers["sXT"][::-1].copy())
    with pytest.raises(AssertionError):
        ge._check_step(bad)


def test_one_wrong_output_fails(buffers):
    dX = buffers["dX"].copy()
    dX[5, 7] ^= 0x0040                      # one BF16 mantissa bit of one dgrad output
    with pytest.raises(AssertionError):
        ge._check_step(dict(buffers, dX=dX))


def test_wrong_weight_transpose_fails(buffers):
    qT = buffers["qWdT"].copy()
    qT[[0, 1]] = qT[[1, 0]]                 # two rows of W_down^T swapped
    with pytest.raises(AssertionError):
        ge._check_step(dict(buffers, qWdT=qT))
