"""GPU parity of the MoE backward pieces: the batched on-demand FP8 transpose of
the expert weights (bit-exact) and the grouped weight gradient over each
expert's dispatch rows (GEMM tolerance), from hand-made offsets with an empty
expert and from a real routing map whose dispatch-ordered gradients and
activations go through the fused 1x128 + 128x1 quantizer."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
import synth
from gpu_helpers import assert_status_ok, bf16_to_f64, dev_bf16, dev_f32, dev_u8, gemm_tolerance_check, host_u16

pytestmark = pytest.mark.gpu


def rand_codes(shape, seed, fmt):
    """Random finite FP8 codes (NaN / Inf codes replaced)."""
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    mag = c & 0x7F
    bad = (mag == 0x7F) if fmt == oracle.E4M3 else (mag >= 0x7C)
    c[bad] = 0x38
    return c


def rand_scales(shape, seed):
    rng = np.random.default_rng(seed)
    return np.exp(rng.uniform(-6, 1, size=shape)).astype(np.float32)


def test_batched_transpose_bit_exact():
    B, R, C = 3, 256, 384
    q = np.random.default_rng(1).integers(0, 256, size=(B, R, C), dtype=np.uint8)
    s = rand_scales((B, R // 128, C // 128), 2)
    qT = torch.empty((B, C, R), dtype=torch.uint8, device="cuda")
    sT = torch.empty((B, C // 128, R // 128), dtype=torch.float32, device="cuda")
    fg.transpose_128x128_batched(dev_u8(q), dev_f32(s), qT, sT)
    assert_status_ok()
    for b in range(B):
        assert np.array_equal(qT[b].cpu().numpy(), oracle.fp8_transpose(q[b]))
        assert np.array_equal(sT[b].cpu().numpy(), s[b].T)


def run_wgrad(offs, AT, fa, sA, BT, fb, sB, dtype):
    G, N, K = len(offs) - 1, AT.shape[0], BT.shape[0]
    D = torch.full((G * N, K), float("nan"), dtype=dtype, device="cuda")
    fg.grouped_gemm_wgrad(torch.from_numpy(np.asarray(offs, np.int32)).cuda(), dev_u8(AT), fa, dev_f32(sA),
                          dev_u8(BT), fb, dev_f32(sB), D)
    assert_status_ok()
    if dtype == torch.float32:
        return D.cpu().numpy().astype(np.float64).reshape(G, N, K)
    return bf16_to_f64(host_u16(D)).reshape(G, N, K)


def transposed_operand(rows, ldt, seed, fmt, std, outliers, mult):
    """A transposed copy [rows][ldt] as the quantizer writes it: 1x128 tiles along
    the dispatch rows, scales S[ldt/128][rows]."""
    q, s, _ = oracle.quant_1x128(synth.bf16_normal((rows, ldt), seed, std, outliers, mult), fmt)
    return q, s


@pytest.mark.parametrize("K", [384, 512])   # 128- and 256-column tiles
def test_grouped_wgrad_with_empty_expert(K):
    offs = np.array([0, 256, 256, 640, 768], np.int32)   # expert 1 has no rows
    ldt, N = 896, 256                                    # capacity past the last expert
    fa, fb = oracle.E5M2, oracle.E4M3
    AT, sA = transposed_operand(N, ldt, 11, fa, 1e-3, 0.0, 1.0)
    BT, sB = transposed_operand(K, ldt, 12, fb, 1.0, 1e-3, 50.0)
    ref = oracle.grouped_wgrad_full(offs, AT, fa, sA, BT, fb, sB)
    for dtype in (torch.float32, torch.bfloat16):
        got = run_wgrad(offs, AT, fa, sA, BT, fb, sB, dtype)
        assert np.all(got[1] == 0.0)
        gemm_tolerance_check(got.reshape(-1, K), ref.reshape(-1, K), bf16_out=dtype == torch.bfloat16)


def test_grouped_wgrad_all_experts_empty_gives_zeros():
    offs = np.zeros(5, np.int32)
    N, K, ldt = 128, 256, 256
    AT, BT = rand_codes((N, ldt), 21, oracle.E4M3), rand_codes((K, ldt), 22, oracle.E4M3)
    got = run_wgrad(offs, AT, oracle.E4M3, rand_scales((ldt // 128, N), 23), BT, oracle.E4M3,
                    rand_scales((ldt // 128, K), 24), torch.float32)
    assert np.all(got == 0.0)


def test_grouped_wgrad_rejects_bad_offsets():
    N, K, ldt = 128, 128, 256
    offs = torch.tensor([0, 64, 256], dtype=torch.int32, device="cuda")   # not a multiple of 128
    D = torch.zeros((2 * N, K), dtype=torch.float32, device="cuda")
    fg.grouped_gemm_wgrad(offs, dev_u8(rand_codes((N, ldt), 31, 0)), fg.E4M3, dev_f32(np.ones((2, N))),
                          dev_u8(rand_codes((K, ldt), 32, 0)), fg.E4M3, dev_f32(np.ones((2, K))), D)
    assert fg.device_status() == fg.ERR_INVALID_ARG


def test_moe_wgrad_from_routing_map():
    """dW_e = dY_e^T . X_e over the rows the routing map dispatches to expert e:
    gradients (E5M2) and activations (E4M3) in dispatch order go through the fused
    quantizer's transposed copies, which must match the oracle's 128x1 quantization
    bit for bit, then the grouped wgrad is checked against the oracle."""
    T, E, topk, N, K = 512, 8, 2, 256, 384
    z = synth.f32_normal((T, E), 41)
    ref = oracle.moe_route(z, topk=topk, align=128)
    offs, rows, tot = ref["offsets"], ref["row_token"], ref["total"]
    cap = (ref["cap"] + 127) // 128 * 128   # the transposed copies need whole 128-row groups
    dy_tok = synth.bf16_normal((T, N), 42, 1e-3, 0.0, 1.0)
    x_tok = synth.bf16_normal((T, K), 43, 1.0, 1e-3, 50.0)
    # dispatch order: real rows copy their token; rows past the total are zero
    dy_d = np.zeros((cap, N), np.uint16)
    x_d = np.zeros((cap, K), np.uint16)
    dy_d[:tot] = dy_tok[rows[:tot]]
    x_d[:tot] = x_tok[rows[:tot]]
    dy_d[:tot][ref["row_is_pad"][:tot] == 1] = 0     # padding rows carry no gradient
    ops = []
    for bits, fmt in ((dy_d, oracle.E5M2), (x_d, oracle.E4M3)):
        R, C = bits.shape
        q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
        s = torch.empty((C // 128, R), dtype=torch.float32, device="cuda")
        qT = torch.empty((C, R), dtype=torch.uint8, device="cuda")
        sT = torch.empty((R // 128, C), dtype=torch.float32, device="cuda")
        fg.quant_1x128(dev_bf16(bits), fmt, q, s, qT, sT)
        assert_status_ok()
        rqT, rsT, _ = oracle.quant_128x1_transposed(bits, fmt)
        assert np.array_equal(qT.cpu().numpy(), rqT)
        assert np.array_equal(sT.cpu().numpy().view(np.uint32), rsT.view(np.uint32))
        ops.append((rqT, rsT))
    (AT, sA), (BT, sB) = ops
    want = oracle.grouped_wgrad_full(offs, AT, oracle.E5M2, sA, BT, oracle.E4M3, sB)
    got = run_wgrad(offs, AT, oracle.E5M2, sA, BT, oracle.E4M3, sB, torch.float32)
    gemm_tolerance_check(got.reshape(-1, K), want.reshape(-1, K), bf16_out=False)


def test_moe_dgrad_through_batched_transpose():
    """dH_e = dY_e . W_e for the down projection: the expert weights W_e [H][F]
    are quantized 128x128, transposed on the GPU into W_e^T [F][H] (codes and
    scale grid), and the grouped GEMM contracts the dispatch rows of dY (1x128
    along H) with them; checked against the oracle's grouped GEMM over the
    oracle's own transposes, with an empty expert and a 3-tile expert."""
    E, H, F = 4, 256, 384
    offs = np.array([0, 128, 128, 512, 640], np.int32)
    cap = 768                                            # rows past the last expert stay untouched
    w = synth.bf16_normal((E, H, F), 81, 0.02)
    qw = np.empty((E, H, F), np.uint8)
    sw = np.empty((E, H // 128, F // 128), np.float32)
    for e in range(E):
        qw[e], sw[e], _ = oracle.quant_128x128(w[e])
    qwT = torch.empty((E, F, H), dtype=torch.uint8, device="cuda")
    swT = torch.empty((E, F // 128, H // 128), dtype=torch.float32, device="cuda")
    fg.transpose_128x128_batched(dev_u8(qw), dev_f32(sw), qwT, swT)
    dy = synth.bf16_normal((cap, H), 82, 1e-3, 1e-3, 20.0)
    qa, sa, _ = oracle.quant_1x128(dy)
    D = torch.full((cap, F), 7.0, dtype=torch.float32, device="cuda")
    fg.grouped_gemm(torch.from_numpy(offs).cuda(), dev_u8(qa), dev_f32(sa), qwT, swT, D)
    assert_status_ok()
    refT = np.stack([oracle.fp8_transpose(qw[e]) for e in range(E)])
    assert np.array_equal(qwT.cpu().numpy(), refT)
    srefT = np.ascontiguousarray(sw.transpose(0, 2, 1))
    pm, pn = np.meshgrid(np.arange(offs[-1]), np.arange(F), indexing="ij")
    pm, pn = pm.reshape(-1), pn.reshape(-1)
    want = oracle.grouped_gemm_points(offs, qa, sa, cap, refT, srefT, pm, pn).reshape(offs[-1], F)
    got = D.cpu().numpy().astype(np.float64)
    gemm_tolerance_check(got[: offs[-1]], want, bf16_out=False)
    assert np.all(got[offs[-1]:] == 7.0)


def test_moe_down_wgrad_full_size():
    """The MoE block's shapes (8192 tokens, 128 experts, top-8, hidden 2048,
    FFN 768): dW_down_e = dY_e^T . H_e over each expert's dispatch rows, from a
    real routing map.  The fused quantizer's transposed copies of the dispatch
    buffers must equal the oracle's 128x1 quantization bit for bit; the grouped
    wgrad is checked on sampled outputs of every expert."""
    T, E, topk, Hd, F = 8192, 128, 8, 2048, 768
    _, logits, _, _ = synth.moe_inputs()
    ref = oracle.moe_route(logits, topk=topk, align=128)
    offs, rows, tot = ref["offsets"], ref["row_token"], ref["total"]
    cap = (ref["cap"] + 127) // 128 * 128
    dy_tok = synth.bf16_normal((T, Hd), 91, 1e-3, 1e-3, 20.0)
    h_tok = synth.bf16_normal((T, F), 92, 1.0, 1e-3, 20.0)
    dy_d = np.zeros((cap, Hd), np.uint16)
    h_d = np.zeros((cap, F), np.uint16)
    dy_d[:tot] = dy_tok[rows[:tot]]
    h_d[:tot] = h_tok[rows[:tot]]
    dy_d[:tot][ref["row_is_pad"][:tot] == 1] = 0          # padding rows carry no gradient
    ops = []
    for bits, fmt in ((dy_d, oracle.E5M2), (h_d, oracle.E4M3)):
        R, C = bits.shape
        q, s = torch.empty((R, C), dtype=torch.uint8, device="cuda"), torch.empty((C // 128, R), device="cuda")
        qT, sT = torch.empty((C, R), dtype=torch.uint8, device="cuda"), torch.empty((R // 128, C), device="cuda")
        fg.quant_1x128(dev_bf16(bits), fmt, q, s, qT, sT)
        assert_status_ok()
        rqT, rsT, _ = oracle.quant_128x1_transposed(bits, fmt)
        assert np.array_equal(qT.cpu().numpy(), rqT)
        assert np.array_equal(sT.cpu().numpy().view(np.uint32), rsT.view(np.uint32))
        ops.append((qT, sT, rqT, rsT))
        del q, s
    (AT, sA, rAT, rsA), (BT, sB, rBT, rsB) = ops
    D = torch.empty((E * Hd, F), dtype=torch.float32, device="cuda")
    fg.grouped_gemm_wgrad(torch.from_numpy(offs.astype(np.int32)).cuda(), AT, fg.E5M2, sA, BT, fg.E4M3, sB, D)
    assert_status_ok()
    rng = np.random.default_rng(93)
    pg = np.repeat(np.arange(E), 256)                     # 256 samples from every expert
    pn = rng.integers(0, Hd, pg.size)
    pk = rng.integers(0, F, pg.size)
    want = oracle.grouped_wgrad_points(offs, rAT, oracle.E5M2, rsA, rBT, oracle.E4M3, rsB, pg, pn, pk)
    got = D.view(E, Hd, F)[torch.from_numpy(pg).cuda(), torch.from_numpy(pn).cuda(), torch.from_numpy(pk).cuda()]
    gemm_tolerance_check(got.cpu().numpy().astype(np.float64), want, bf16_out=False)


def test_batched_transpose_full_size():
    """The benchmarked size: the 128 experts' gate/up weights [1536][2048] as
    FP8 codes with 128x128 scale grids; the GPU transposes equal the byte and
    scale-grid transposes bit for bit."""
    E, R, C = 128, 1536, 2048
    g = torch.Generator(device="cuda").manual_seed(13)
    q = torch.randint(0, 256, (E, R, C), generator=g, device="cuda", dtype=torch.uint8)
    s = torch.rand((E, R // 128, C // 128), generator=g, device="cuda") + 0.5
    qT = torch.empty((E, C, R), dtype=torch.uint8, device="cuda")
    sT = torch.empty((E, C // 128, R // 128), device="cuda")
    fg.transpose_128x128_batched(q, s, qT, sT)
    assert_status_ok()
    assert torch.equal(qT, q.transpose(1, 2))
    assert torch.equal(sT.view(torch.int32), s.transpose(1, 2).contiguous().view(torch.int32))
