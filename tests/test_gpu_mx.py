"""GPU parity of the MXFP8 quantizer (1x32 blocks, power-of-two scales):
codes and scale exponents bit-exact against the oracle (oracle/mx.py) on
ragged and strided shapes, blocks at the edges of the exponent rule (amax
exactly fmax * 2^j and just above, subnormal BF16 amax, all-zero blocks,
values near the BF16 maximum, signed zeros), a tensor holding Inf/NaN
(reported) and the 8192 x 4096 activation of the MLP step."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
import synth
from gpu_helpers import assert_status_ok, dev_bf16
from oracle import mx

pytestmark = pytest.mark.gpu


def run(xb, fmt, ldx=None):
    R, C = xb.shape
    if ldx is None:
        x = dev_bf16(xb)
    else:
        full = np.zeros((R, ldx), np.uint16)
        full[:, :C] = xb
        x = dev_bf16(full)[:, :C]
    q = torch.full((R, C), 0x55, dtype=torch.uint8, device="cuda")
    e8 = torch.full((R, C // 32), 0x55, dtype=torch.uint8, device="cuda")
    fg.quant_mx(x, fmt, q, e8)
    return q.cpu().numpy(), e8.cpu().numpy()


def edge_cases(fmt):
    """Rows of 32-blocks built to sit on the exponent rule's edges."""
    rng = np.random.default_rng(7)
    fm = oracle.fmax(fmt)
    blocks, bump = [], []
    for j in (-30, -3, 0, 5, 100):
        peak = fm * 2.0 ** j
        for above in (False, True):
            b = rng.normal(0, peak / 4, 32).clip(-peak / 2, peak / 2)
            b[3] = -peak if above else peak           # amax exactly fmax * 2^j: X = 2^j
            if above:                                 # ... and one BF16 step above it: X = 2^(j+1)
                bump.append(len(blocks) * 32 + 3)
            blocks.append(b)
    blocks.append(np.zeros(32))                       # all zero: X = 1
    blocks.append(np.full(32, -0.0))                  # signed zeros
    blocks.append(rng.normal(0, 1, 32) * 2.0 ** -130)  # subnormal BF16 amax
    blocks.append(rng.normal(0, 1, 32) * 5e37)        # near the BF16 maximum
    x = np.concatenate(blocks).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    bits[bump] += 1
    return np.tile(bits, (3, 1))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("shape,ldx", [((256, 1024), None), ((37, 96), None), ((5, 160), 200), ((1, 32), None)])
def test_mx_quant_bit_exact(fmt, shape, ldx):
    xb = synth.bf16_normal(shape, 41, 1.0, 1e-3, 50.0)
    q, e8 = run(xb, fmt, ldx)
    assert_status_ok()
    rq, re8, st = mx.quant_mx(xb, fmt)
    assert st == oracle.OK
    assert np.array_equal(e8, re8) and np.array_equal(q, rq)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_mx_quant_exponent_edges(fmt):
    xb = edge_cases(fmt)
    q, e8 = run(xb, fmt)
    assert_status_ok()
    rq, re8, _ = mx.quant_mx(xb, fmt)
    assert np.array_equal(e8, re8) and np.array_equal(q, rq)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("shape,ldx", [((256, 1024), None), ((128, 128), None), ((384, 512), 640)])
def test_mx_quant_tiled_bit_exact(fmt, shape, ldx):
    """quant_mx_tiled: the same codes as the oracle, the scale codes at the
    positions of the oracle's GEMM-ready tiling (mx_tile_scales)."""
    R, C = shape
    xb = synth.bf16_normal(shape, 44, 1.0, 1e-3, 50.0)
    if ldx is None:
        x = dev_bf16(xb)
    else:
        full = np.zeros((R, ldx), np.uint16)
        full[:, :C] = xb
        x = dev_bf16(full)[:, :C]
    q = torch.full((R, C), 0x55, dtype=torch.uint8, device="cuda")
    e8t = torch.full((R * C // 32,), 0x55, dtype=torch.uint8, device="cuda")
    fg.quant_mx_tiled(x, fmt, q, e8t)
    assert_status_ok()
    rq, re8, st = mx.quant_mx(xb, fmt)
    assert st == oracle.OK
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(e8t.cpu().numpy(), mx.mx_tile_scales(re8))


def test_mx_quant_tiled_nonfinite_is_reported_and_empty_is_a_no_op():
    xb = synth.bf16_normal((128, 256), 45)
    xb[77, 200] = 0xFF80                           # -Inf
    q = torch.empty((128, 256), dtype=torch.uint8, device="cuda")
    e8t = torch.empty(128 * 256 // 32, dtype=torch.uint8, device="cuda")
    fg.quant_mx_tiled(dev_bf16(xb), fg.E4M3, q, e8t)
    assert fg.device_status() == fg.ERR_NONFINITE
    fg.quant_mx_tiled(torch.empty((0, 128), dtype=torch.bfloat16, device="cuda"), fg.E4M3,
                      torch.empty((0, 128), dtype=torch.uint8, device="cuda"),
                      torch.empty(0, dtype=torch.uint8, device="cuda"))
    assert_status_ok()


def test_mx_quant_tiled_needs_whole_tiles():
    x = torch.zeros((100, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((100, 128), dtype=torch.uint8, device="cuda")
    e8t = torch.empty(400, dtype=torch.uint8, device="cuda")
    with pytest.raises(fg.Fp8Error) as e:
        fg.quant_mx_tiled(x, fg.E4M3, q, e8t)
    assert e.value.code == fg.ERR_SHAPE


def test_mx_quant_nonfinite_is_reported_and_empty_is_a_no_op():
    xb = synth.bf16_normal((4, 64), 42)
    xb[1, 33] = 0x7FC0
    run(xb, oracle.E4M3)
    assert fg.device_status() == fg.ERR_NONFINITE
    fg.quant_mx(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"), fg.E4M3,
                torch.empty((0, 64), dtype=torch.uint8, device="cuda"), torch.empty((0, 2), dtype=torch.uint8, device="cuda"))
    assert_status_ok()


def test_mx_quant_mlp_activation_full_size():
    """X of the MLP step, 8192 tokens x 4096, E4M3, every code and exponent."""
    xb = synth.bf16_normal((8192, 4096), 43, 1.0, 1e-3, 50.0)
    q, e8 = run(xb, oracle.E4M3)
    assert_status_ok()
    rq, re8, _ = mx.quant_mx(xb, oracle.E4M3)
    assert np.array_equal(e8, re8) and np.array_equal(q, rq)


# ---------------------------------------------------------------- MXFP8 GEMM

def mx_operand(rows, K, seed, fmt, std=1.0):
    xb = synth.bf16_normal((rows, K), seed, std, 1e-3, 50.0)
    q, e8, st = mx.quant_mx(xb, fmt)
    assert st == oracle.OK
    return q, e8


def run_mx_gemm(qa, ea, fa, qb, eb, fb, out_dtype):
    from gpu_helpers import dev_u8, guarded
    M, N = qa.shape[0], qb.shape[0]
    D = guarded((M, N), out_dtype)
    fg.mx_gemm(dev_u8(qa), fa, dev_u8(ea), dev_u8(qb), fb, dev_u8(eb), D)
    assert_status_ok()
    return D


MX_CASES = [
    # name, M, N, K, fmtA, fmtB: BN = 256 and BN = 128 tiles, several waves of tiles, E5M2 operands
    ("bn256", 256, 512, 512, oracle.E4M3, oracle.E4M3),
    ("bn128_tail", 384, 384, 640, oracle.E4M3, oracle.E4M3),
    ("waves", 1024, 1536, 1024, oracle.E4M3, oracle.E4M3),
    ("e5m2_a", 256, 256, 384, oracle.E5M2, oracle.E4M3),
    ("one_chunk", 128, 256, 128, oracle.E4M3, oracle.E5M2),      # K = 128: a one-chunk group
    ("smallest", 128, 128, 128, oracle.E5M2, oracle.E5M2),       # one tile, BN = 128
]


@pytest.mark.parametrize("case", MX_CASES, ids=[c[0] for c in MX_CASES])
def test_mx_gemm_full_compare(case):
    """Every output against the oracle's exact per-32-block sum (R16), FP32
    and BF16 outputs; the BF16 output is the RNE rounding of the FP32 one."""
    from gpu_helpers import bf16_to_f64, gemm_tolerance_check, host_u16
    name, M, N, K, fa, fb = case
    qa, ea = mx_operand(M, K, 51, fa)
    qb, eb = mx_operand(N, K, 52, fb, std=0.5)
    ref = mx.mx_gemm_full(qa, ea, fa, qb, eb, fb)
    d32 = run_mx_gemm(qa, ea, fa, qb, eb, fb, torch.float32)
    gemm_tolerance_check(d32.cpu().numpy().astype(np.float64), ref, bf16_out=False)
    d16 = run_mx_gemm(qa, ea, fa, qb, eb, fb, torch.bfloat16)
    gemm_tolerance_check(bf16_to_f64(host_u16(d16)), ref, bf16_out=True)
    assert torch.equal(d16, d32.to(torch.bfloat16))


@pytest.mark.parametrize("case", MX_CASES, ids=[c[0] for c in MX_CASES])
def test_mx_gemm_tiled_bit_identical_to_row_major(case):
    """mx_gemm_tiled on the oracle's tiling of the scale codes: bit for bit the
    output of mx_gemm (whose scale words are reordered by a warp of the GEMM
    instead of fetched in tile order), FP32 and BF16, and within the oracle's
    tolerance."""
    from gpu_helpers import dev_u8, gemm_tolerance_check, guarded
    name, M, N, K, fa, fb = case
    qa, ea = mx_operand(M, K, 51, fa)
    qb, eb = mx_operand(N, K, 52, fb, std=0.5)
    ref = mx.mx_gemm_full(qa, ea, fa, qb, eb, fb)
    for dt in (torch.float32, torch.bfloat16):
        d_rm = run_mx_gemm(qa, ea, fa, qb, eb, fb, dt)
        D = guarded((M, N), dt)
        fg.mx_gemm_tiled(dev_u8(qa), fa, dev_u8(mx.mx_tile_scales(ea)), dev_u8(qb), fb,
                         dev_u8(mx.mx_tile_scales(eb)), D)
        assert_status_ok()
        assert torch.equal(D, d_rm)
    gemm_tolerance_check(D.float().cpu().numpy().astype(np.float64), ref, bf16_out=True)


def test_mx_gemm_tiled_empty_shapes():
    """K == 0 writes zeros (FP32 and BF16, ldD > N leaves the padding alone);
    M == 0 or N == 0 is a no-op."""
    from gpu_helpers import CANARY_BYTE, guarded
    for dt in (torch.float32, torch.bfloat16):
        full = guarded((256, 384 + 64), dt)
        D = full[:, :384]
        z = torch.empty((256, 0), dtype=torch.uint8, device="cuda")
        fg.mx_gemm_tiled(z, fg.E4M3, torch.empty(0, dtype=torch.uint8, device="cuda"),
                         torch.empty((384, 0), dtype=torch.uint8, device="cuda"), fg.E4M3,
                         torch.empty(0, dtype=torch.uint8, device="cuda"), D)
        assert_status_ok()
        assert bool((D == 0).all())
        assert bool((full[:, 384:].contiguous().view(torch.uint8) == CANARY_BYTE).all())
    D0 = torch.empty((0, 128), dtype=torch.float32, device="cuda")
    fg.mx_gemm_tiled(torch.empty((0, 128), dtype=torch.uint8, device="cuda"), fg.E4M3,
                     torch.empty(0, dtype=torch.uint8, device="cuda"),
                     torch.empty((128, 128), dtype=torch.uint8, device="cuda"), fg.E4M3,
                     torch.zeros(512, dtype=torch.uint8, device="cuda"), D0)
    assert_status_ok()


def test_mx_gemm_tiled_needs_16_byte_aligned_tiles():
    from gpu_helpers import dev_u8
    M, N, K = 128, 128, 128
    qa, ea = mx_operand(M, K, 53, oracle.E4M3)
    buf = torch.zeros(M * K // 32 + 16, dtype=torch.uint8, device="cuda")
    off = buf[4:4 + M * K // 32]
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    with pytest.raises(fg.Fp8Error) as e:
        fg.mx_gemm_tiled(dev_u8(qa), fg.E4M3, off, dev_u8(qa), fg.E4M3, dev_u8(mx.mx_tile_scales(ea)), D)
    assert e.value.code == fg.ERR_ALIGNMENT


def test_mx_gemm_exponents_at_4_byte_offsets():
    """K a multiple of 512 with the exponent arrays 4-byte but not 16-byte
    aligned (views at a 4-byte offset): the kernel reads the words one chunk at
    a time instead of four at once, with the same result as aligned arrays."""
    from gpu_helpers import dev_u8
    M, N, K = 256, 512, 1024
    qa, ea = mx_operand(M, K, 61, oracle.E4M3)
    qb, eb = mx_operand(N, K, 62, oracle.E4M3, std=0.5)
    aligned = run_mx_gemm(qa, ea, oracle.E4M3, qb, eb, oracle.E4M3, torch.float32)

    def offset_view(e):
        buf = torch.zeros(e.size + 16, dtype=torch.uint8, device="cuda")
        v = buf[4:4 + e.size].view(e.shape)
        v.copy_(dev_u8(e))
        assert v.data_ptr() % 16 == 4
        return v
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fg.mx_gemm(dev_u8(qa), fg.E4M3, offset_view(ea), dev_u8(qb), fg.E4M3, offset_view(eb), D)
    assert_status_ok()
    assert torch.equal(D, aligned)


def test_mx_gemm_block_scales_are_applied_per_32_block():
    """Operands whose 32-blocks carry very different exponents (2^-20 .. 2^20
    within one row): a scale applied per 128-chunk or per row instead of per
    32-block would be far off."""
    from gpu_helpers import gemm_tolerance_check
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 256
    qa = rng.integers(0, 0x7E, (M, K), dtype=np.uint8) | (rng.integers(0, 2, (M, K), dtype=np.uint8) << 7)
    qb = rng.integers(0, 0x7E, (N, K), dtype=np.uint8) | (rng.integers(0, 2, (N, K), dtype=np.uint8) << 7)
    ea = rng.integers(127 - 20, 127 + 20, (M, K // 32), dtype=np.uint8)
    eb = rng.integers(127 - 20, 127 + 20, (N, K // 32), dtype=np.uint8)
    ref = mx.mx_gemm_full(qa, ea, oracle.E4M3, qb, eb, oracle.E4M3)
    d32 = run_mx_gemm(qa, ea, oracle.E4M3, qb, eb, oracle.E4M3, torch.float32)
    gemm_tolerance_check(d32.cpu().numpy().astype(np.float64), ref, bf16_out=False)


@pytest.mark.parametrize("layout", ["row_major", "tiled"])
@pytest.mark.parametrize("case", ["complementary", "tiny"])
def test_mx_gemm_extreme_scale_codes(layout, case):
    """Scale codes at the ends of the UE8M0 range, on positive codes (no
    cancellation, so a relative bound of 1e-5 holds for FP32 accumulation
    and shows any scale applied wrongly).  complementary: per 32-block eA in
    {0, 1, 2, 252, 253, 254} and eB = 254 - eA, so X_A alone is 2^-127 or
    2^127 while every scale product is 1 (a product formed after applying the
    two factors one at a time in binary32 would overflow or flush).  tiny: eA
    in {0, ..., 4} with eB = 127, so single products fall into binary32's
    subnormal range (a flush to zero would show)."""
    from gpu_helpers import dev_u8, gemm_tolerance_check
    rng = np.random.default_rng(17)
    M, N, K = 256, 256, 512
    qa = rng.integers(0x08, 0x7E, (M, K), dtype=np.uint8)
    qb = rng.integers(0x08, 0x7E, (N, K), dtype=np.uint8)
    if case == "complementary":
        codes = np.array([0, 1, 2, 252, 253, 254], np.uint8)
        ea = np.broadcast_to(codes[rng.integers(0, codes.size, (1, K // 32))], (M, K // 32)).copy()
        eb = np.broadcast_to((254 - ea[:1].astype(np.int64)).astype(np.uint8), (N, K // 32)).copy()
    else:
        ea = rng.integers(0, 5, (M, K // 32)).astype(np.uint8)
        eb = np.full((N, K // 32), 127, np.uint8)
    ref = mx.mx_gemm_full(qa, ea, oracle.E4M3, qb, eb, oracle.E4M3)
    assert np.all(np.isfinite(ref)) and np.all(ref > 0)
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    if layout == "tiled":
        fg.mx_gemm_tiled(dev_u8(qa), fg.E4M3, dev_u8(mx.mx_tile_scales(ea)), dev_u8(qb), fg.E4M3,
                         dev_u8(mx.mx_tile_scales(eb)), D)
    else:
        fg.mx_gemm(dev_u8(qa), fg.E4M3, dev_u8(ea), dev_u8(qb), fg.E4M3, dev_u8(eb), D)
    assert_status_ok()
    got = D.cpu().numpy().astype(np.float64)
    rel = np.abs(got - ref) / ref
    assert float(rel.max()) <= 1e-5, float(rel.max())
    gemm_tolerance_check(got, ref, bf16_out=False)


def test_mx_gemm_headline_shape_sampled():
    """The block-scaled GEMM's headline shape, 8192 x 28672 x 4096: X and W_gu
    of the MLP step quantized to MXFP8 by the oracle; the GPU quantizer gives
    the same codes in both scale layouts; the GEMM from the row-major and from
    the tiled scales gives one bit-identical D, checked against the oracle's
    exact per-block sum on >= 2^20 stratified outputs (every 128 x 128 tile
    hit >= 16 times)."""
    from gpu_helpers import bf16_to_f64, dev_u8, gemm_tolerance_check, host_u16, sample_points_dense
    M, N, K = 8192, 28672, 4096
    xb = synth.bf16_normal((M, K), 0, 1.0, 1e-3, 50.0)
    wb = synth.bf16_normal((N, K), 1000, 0.02)
    ops = []
    for bits in (xb, wb):
        R = bits.shape[0]
        rq, re8, st = mx.quant_mx(bits, oracle.E4M3)
        assert st == oracle.OK
        x = dev_bf16(bits)
        q = torch.empty((R, K), dtype=torch.uint8, device="cuda")
        e8 = torch.empty((R, K // 32), dtype=torch.uint8, device="cuda")
        e8t = torch.empty(R * K // 32, dtype=torch.uint8, device="cuda")
        fg.quant_mx(x, fg.E4M3, q, e8)
        assert_status_ok()
        assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(e8.cpu().numpy(), re8)
        fg.quant_mx_tiled(x, fg.E4M3, q, e8t)
        assert_status_ok()
        assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(e8t.cpu().numpy(), mx.mx_tile_scales(re8))
        del x
        ops.append((rq, re8, dev_u8(rq), dev_u8(re8), e8t))
    (rqa, rea, qa, ea, eat), (rqb, reb, qb, eb, ebt) = ops
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fg.mx_gemm(qa, fg.E4M3, ea, qb, fg.E4M3, eb, D)
    assert_status_ok()
    Dt = torch.empty_like(D)
    fg.mx_gemm_tiled(qa, fg.E4M3, eat, qb, fg.E4M3, ebt, Dt)
    assert_status_ok()
    assert torch.equal(D, Dt)
    del Dt
    pm, pn = sample_points_dense(M, N, seed=9)
    ref = mx.mx_gemm_points(rqa, rea, oracle.E4M3, rqb, reb, oracle.E4M3, pm, pn)
    got = D[torch.from_numpy(pm).cuda(), torch.from_numpy(pn).cuda()]
    gemm_tolerance_check(bf16_to_f64(host_u16(got)), ref, bf16_out=True)
