"""Exhaustive check of the quantizers' per-element division.

The fine-grained scale is s = RN(amax / fmax) with amax the magnitude of a
BF16 value, so each format has exactly one scale per positive finite BF16
pattern (32639 of them), and a group quantized with that scale only ever
divides BF16 values of magnitude <= amax.  These tests run every such pair
(amax, x) -- both signs of x, every finite positive amax, E4M3 and E5M2 --
through the GPU quantizers and compare codes and scales bit for bit with the
oracle's IEEE division x / s followed by the round-to-nearest-even encoder
("FP8-LM" review, tensor scaling x_fp8 = Cast(x / s); the division, not a
multiplication by a reciprocal, is the page's convention):

* 1x128 tiles (the rows-only kernel): one tile per 127 test values, its
  first element the amax;
* the transposed 128x1 copy of the fused kernel: the same tiles laid out
  as columns, so every column's quantization is one of those tiles';
* 128x128 blocks: 128 tiles of one amax per block.

Each format is about 1.07e9 (amax, x) pairs, processed in chunks."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
from gpu_helpers import assert_status_ok, dev_bf16

FMTS = [oracle.E4M3, oracle.E5M2]
AMAX_ALL = np.arange(0x0001, 0x7F80, dtype=np.int64)        # every positive finite BF16 pattern
CHUNK_TILES = 1 << 20                                        # 128 Mi elements per chunk


def tiles_for(amax_bits, per_amax_multiple=1):
    """[T, 128] BF16 tiles: for each amax a, tiles [a, x_1 .. x_127] whose x run
    over every pattern of magnitude <= a (0 .. a and 0x8000 .. 0x8000 + a),
    the last tile filled up with zeros; the tile count of each amax is padded
    (with [a, 0, ...] tiles) to a multiple of ``per_amax_multiple``."""
    parts = []
    for a in amax_bits:
        a = int(a)
        vals = np.concatenate([np.arange(0, a + 1, dtype=np.int64), np.arange(0x8000, 0x8000 + a + 1, dtype=np.int64)])
        n_t = -(-len(vals) // 127)
        n_t = -(-n_t // per_amax_multiple) * per_amax_multiple
        body = np.zeros(n_t * 127, np.uint16)
        body[:len(vals)] = vals
        t = np.empty((n_t, 128), np.uint16)
        t[:, 0] = a
        t[:, 1:] = body.reshape(n_t, 127)
        parts.append(t)
    return np.concatenate(parts)


def amax_chunks(per_amax_multiple=1):
    """Consecutive amax ranges whose tiles add up to about CHUNK_TILES."""
    tiles = -(-(2 * (AMAX_ALL + 1)) // 127)
    tiles = -(-tiles // per_amax_multiple) * per_amax_multiple
    csum = np.cumsum(tiles)
    start = 0
    while start < len(AMAX_ALL):
        base = csum[start - 1] if start else 0
        stop = int(np.searchsorted(csum, base + CHUNK_TILES, side="right"))
        stop = max(stop, start + 1)
        yield AMAX_ALL[start:stop]
        start = stop


def test_tile_generator_covers_every_pair():
    """The generator itself: amax 3 gives the 8 patterns +-0..3 once each."""
    t = tiles_for([3])
    assert t.shape == (1, 128) and t[0, 0] == 3
    assert sorted(t[0, 1:9].tolist()) == [0, 1, 2, 3, 0x8000, 0x8001, 0x8002, 0x8003]
    assert np.all(t[0, 9:] == 0)
    assert sum(len(c) for c in amax_chunks()) == 0x7F7F


def same_bits(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint32), np.ascontiguousarray(b).view(np.uint32))


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", FMTS, ids=["e4m3", "e5m2"])
def test_every_scale_every_value_1x128_and_128x1(fmt):
    for amaxes in amax_chunks():
        x = tiles_for(amaxes)
        T = x.shape[0]
        Tp = -(-T // 128) * 128
        if Tp != T:                                       # zero tiles up to a multiple of 128 columns
            x = np.concatenate([x, np.zeros((Tp - T, 128), np.uint16)])
        q_ref, s_ref, st = oracle.quant_1x128(x, fmt)
        assert st == oracle.OK
        # rows-only kernel on the tiles
        xd = dev_bf16(x)
        q = torch.empty((Tp, 128), dtype=torch.uint8, device="cuda")
        s = torch.empty((1, Tp), dtype=torch.float32, device="cuda")
        fg.quant_1x128(xd, fmt, q, s)
        assert_status_ok()
        bad = int((q.cpu().numpy() != q_ref).sum())
        assert bad == 0, f"1x128: {bad} codes differ for amax in [{amaxes[0]:#x}, {amaxes[-1]:#x}]"
        assert same_bits(s.cpu().numpy(), s_ref)
        # the fused kernel's 128x1 copy of the transposed layout: column j is tile j
        y = xd.t().contiguous()                           # [128, Tp]
        del xd, q, s
        q1, s1 = torch.empty((128, Tp), dtype=torch.uint8, device="cuda"), torch.empty((Tp // 128, 128), device="cuda")
        qT, sT = torch.empty((Tp, 128), dtype=torch.uint8, device="cuda"), torch.empty((1, Tp), device="cuda")
        fg.quant_1x128(y, fmt, q1, s1, qT, sT)
        assert_status_ok()
        bad = int((qT.cpu().numpy() != q_ref).sum())
        assert bad == 0, f"128x1: {bad} codes differ for amax in [{amaxes[0]:#x}, {amaxes[-1]:#x}]"
        assert same_bits(sT.cpu().numpy(), s_ref)
        del y, q1, s1, qT, sT


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", FMTS, ids=["e4m3", "e5m2"])
def test_every_scale_every_value_128x128(fmt):
    for amaxes in amax_chunks(per_amax_multiple=128):
        t = tiles_for(amaxes, per_amax_multiple=128)          # [NB * 128, 128], 128 tiles of one amax per block
        nb = t.shape[0] // 128
        w = np.ascontiguousarray(t.reshape(nb, 128, 128).transpose(1, 0, 2).reshape(128, nb * 128))
        q_ref, s_ref, st = oracle.quant_128x128(w, fmt)
        assert st == oracle.OK
        q = torch.empty((128, nb * 128), dtype=torch.uint8, device="cuda")
        s = torch.empty((1, nb), dtype=torch.float32, device="cuda")
        fg.quant_128x128(dev_bf16(w), fmt, q, s)
        assert_status_ok()
        bad = int((q.cpu().numpy() != q_ref).sum())
        assert bad == 0, f"128x128: {bad} codes differ for amax in [{amaxes[0]:#x}, {amaxes[-1]:#x}]"
        assert same_bits(s.cpu().numpy(), s_ref)
