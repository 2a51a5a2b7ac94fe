"""GPU parity of the MoE path: router top-k, the padded routing map and its
dispatch rows (bit-exact integers), the FP8 row gather (bit-exact), the
grouped expert GEMM (GEMM tolerance), and the SwiGLU glue (within one BF16
ulp of the FP64 oracle); small cases with empty experts and the full
128-expert top-8 workload."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
import synth
from gpu_helpers import (assert_status_ok, bf16_to_f64, dev_bf16, dev_f32, dev_u8, empty_f32, empty_u8,
                         gemm_tolerance_check, host_u16, sample_points_dense)

pytestmark = pytest.mark.gpu


def gpu_route(z, topk, align, cap):
    T, E = z.shape
    logits = dev_f32(z)
    ti = torch.empty((T, topk), dtype=torch.int32, device="cuda")
    tp = torch.empty((T, topk), dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    rt = torch.empty(cap, dtype=torch.int32, device="cuda")
    rp = torch.empty(cap, dtype=torch.float32, device="cuda")
    pad = torch.empty(cap, dtype=torch.uint8, device="cuda")
    fg.moe_route_pad(logits, topk, align, cap, ti, tp, counts, offs, rt, rp, pad)
    assert_status_ok()
    return dict(topk_idx=ti, topk_prob=tp, counts=counts, offsets=offs, row_token=rt, row_prob=rp, row_is_pad=pad)


def check_route(z, topk, align):
    T, E = z.shape
    ref = oracle.moe_route(z, topk=topk, align=align)
    cap = ref["cap"]
    g = gpu_route(z, topk, align, cap)
    assert np.array_equal(g["topk_idx"].cpu().numpy(), ref["topk_idx"])
    assert np.allclose(g["topk_prob"].cpu().numpy(), ref["topk_prob"], rtol=2e-6, atol=1e-12)
    assert np.array_equal(g["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(g["offsets"].cpu().numpy(), ref["offsets"])
    tot = ref["total"]
    assert np.array_equal(g["row_token"].cpu().numpy()[:tot], ref["row_token"][:tot])
    assert np.all(g["row_token"].cpu().numpy()[tot:] == -1)
    assert np.array_equal(g["row_is_pad"].cpu().numpy()[:tot], ref["row_is_pad"][:tot])
    rp = g["row_prob"].cpu().numpy()
    assert np.allclose(rp[:tot], ref["row_prob"][:tot], rtol=2e-6, atol=1e-12)
    assert np.all(rp[:tot][ref["row_is_pad"][:tot] == 1] == 0.0)
    return g, ref


@pytest.mark.parametrize("T,E,topk,align", [(512, 16, 4, 128), (1000, 40, 3, 8), (256, 8, 8, 128), (256, 1, 1, 128), (96, 2, 1, 32)])
def test_route_pad_small(T, E, topk, align):
    z = synth.f32_normal((T, E), 5)
    z[3, :] = 0.25
    z[4, 0] = z[4, E - 1]
    check_route(z, topk, align)


def test_route_pad_full_size():
    _, logits, _, _ = synth.moe_inputs()
    check_route(logits, 8, 128)


def test_route_pad_impossible_padding_is_reported():
    # 96 tokens all routed to the single expert cannot be padded to 128 distinct tokens
    z = synth.f32_normal((96, 1), 5)
    cap = 256
    logits = dev_f32(z)
    ti = torch.empty((96, 1), dtype=torch.int32, device="cuda")
    tp = torch.empty((96, 1), dtype=torch.float32, device="cuda")
    counts = torch.empty(1, dtype=torch.int32, device="cuda")
    offs = torch.empty(2, dtype=torch.int32, device="cuda")
    rt = torch.empty(cap, dtype=torch.int32, device="cuda")
    rp = torch.empty(cap, dtype=torch.float32, device="cuda")
    fg.moe_route_pad(logits, 1, 128, cap, ti, tp, counts, offs, rt, rp)
    assert fg.device_status() == fg.ERR_INVALID_ARG


def test_gather_bit_exact():
    T, K, E = 512, 256, 16
    xb = synth.bf16_normal((T, K), 2, 1.0, 1e-3, 50.0)
    z = synth.f32_normal((T, E), 6)
    g, ref = check_route(z, 4, 128)
    q, s, _ = oracle.quant_1x128(xb)
    cap = ref["cap"]
    qg, sg = empty_u8(cap, K), torch.zeros((K // 128, cap), dtype=torch.float32, device="cuda")
    fg.moe_gather(dev_u8(q), dev_f32(s), g["row_token"], g["offsets"], E, cap, qg, sg)
    assert_status_ok()
    qg_ref, sg_ref = oracle.moe_gather(q, s, ref["row_token"], ref["total"], cap)
    tot = ref["total"]
    assert np.array_equal(qg.cpu().numpy()[:tot], qg_ref[:tot])
    assert np.array_equal(sg.cpu().numpy()[:, :tot], sg_ref[:, :tot])


def expert_weights(E, N, K, seed):
    wb = synth.bf16_normal((E * N, K), seed, 0.02).reshape(E, N, K)
    q = np.empty((E, N, K), np.uint8)
    s = np.empty((E, N // 128, K // 128), np.float32)
    for e in range(E):
        q[e], s[e], _ = oracle.quant_128x128(wb[e])
    return q, s


@pytest.mark.parametrize("N", [256, 384])
def test_grouped_gemm_small_with_empty_groups(N):
    G, K = 6, 512
    offs = np.array([0, 128, 128, 384, 384, 640, 768], np.int32)   # groups 1 and 3 empty
    cap = 1024
    xb = synth.bf16_normal((cap, K), 8, 1.0, 1e-3, 50.0)
    qa, sa, _ = oracle.quant_1x128(xb)
    qb, sb = expert_weights(G, N, K, 9)
    D = torch.full((cap, N), -1.0, dtype=torch.float32, device="cuda")
    fg.grouped_gemm(dev_u8(offs.view(np.uint8)).view(torch.int32), dev_u8(qa), dev_f32(sa), dev_u8(qb), dev_f32(sb), D)
    assert_status_ok()
    pm, pn = np.meshgrid(np.arange(offs[-1]), np.arange(N), indexing="ij")
    ref = oracle.grouped_gemm_points(offs, qa, sa, cap, qb, sb, pm.ravel(), pn.ravel()).reshape(-1, N)
    got = D.cpu().numpy().astype(np.float64)
    gemm_tolerance_check(got[: offs[-1]], ref, bf16_out=False)
    assert np.all(got[offs[-1]:] == -1.0)          # rows past the last group untouched


def test_grouped_gemm_rejects_bad_offsets():
    G, N, K, cap = 2, 256, 256, 256
    offs = torch.tensor([0, 100, 256], dtype=torch.int32, device="cuda")   # not a multiple of 128
    A = empty_u8(cap, K)
    D = torch.full((cap, N), 3.0, dtype=torch.float32, device="cuda")
    fg.grouped_gemm(offs, A, empty_f32(K // 128, cap), empty_u8(G, N, K), empty_f32(G, N // 128, K // 128), D)
    assert fg.device_status() == fg.ERR_INVALID_ARG
    assert torch.all(D == 3.0)


def test_swiglu_fwd_bwd_within_one_ulp():
    R, F = 256, 768
    gu = synth.bf16_normal((R, 2 * F), 9, 2.0)
    dh = synth.bf16_normal((R, F), 10, 1.0)
    h = torch.empty((R, F), dtype=torch.bfloat16, device="cuda")
    dgu = torch.empty((R, 2 * F), dtype=torch.bfloat16, device="cuda")
    fg.swiglu_fwd(dev_bf16(gu), h)
    fg.swiglu_bwd(dev_bf16(gu), dev_bf16(dh), dgu)
    assert_status_ok()
    for got, ref in ((host_u16(h), oracle.swiglu_fwd(gu)), (host_u16(dgu), oracle.swiglu_bwd(gu, dh))):
        # as sign-magnitude integers, adjacent BF16 values differ by 1
        gi = np.where(got & 0x8000, -(got & 0x7FFF).astype(np.int64), (got & 0x7FFF).astype(np.int64))
        ri = np.where(ref & 0x8000, -(ref & 0x7FFF).astype(np.int64), (ref & 0x7FFF).astype(np.int64))
        assert np.max(np.abs(gi - ri)) <= 1


def test_swiglu_extreme_gates_within_one_ulp():
    """Gates over [-100, 100] (the fast sigmoid's range ends near -87; below -64
    the correctly rounded form takes over) and the zero of the gate gradient's
    factor 1 + g(1 - sig(g)) near g = -1.28."""
    R, F = 128, 1024
    rng = np.random.default_rng(12)
    g = np.concatenate([np.linspace(-100.0, 100.0, R * F // 2), rng.uniform(-1.4, -1.15, R * F // 2)])
    gate = synth.f32_to_bf16_bits(rng.permutation(g).astype(np.float32)).reshape(R, F)
    up = synth.bf16_normal((R, F), 13, 1.0)
    gu = np.concatenate([gate, up], axis=1)
    dh = synth.bf16_normal((R, F), 14, 1.0)
    h = torch.empty((R, F), dtype=torch.bfloat16, device="cuda")
    dgu = torch.empty((R, 2 * F), dtype=torch.bfloat16, device="cuda")
    fg.swiglu_fwd(dev_bf16(gu), h)
    fg.swiglu_bwd(dev_bf16(gu), dev_bf16(dh), dgu)
    assert_status_ok()
    si = lambda b: np.where(b & 0x8000, -(b & 0x7FFF).astype(np.int64), (b & 0x7FFF).astype(np.int64))
    for got, ref in ((host_u16(h), oracle.swiglu_fwd(gu)), (host_u16(dgu), oracle.swiglu_bwd(gu, dh))):
        assert np.max(np.abs(si(got) - si(ref))) <= 1


def test_moe_fprop_full_size():
    """128 experts, hidden 2048, FFN 768, top-8 over 8192 tokens: route+pad,
    quantize once, gather, gate/up grouped GEMM, SwiGLU, 1x128 quantize,
    down grouped GEMM; each stage checked against the oracle fed the GPU's
    own inputs to that stage (per-stage parity), GEMMs on sampled outputs."""
    T, Hd, E, F, topk = 8192, 2048, 128, 768, 8
    xb, logits, w_gu, w_dn = synth.moe_inputs()
    g, ref = check_route(logits, topk, 128)
    cap = ((ref["cap"] + 127) // 128) * 128
    offs = g["offsets"]
    tot = ref["total"]
    # quantize X once, gather
    qx, sx = empty_u8(T, Hd), empty_f32(Hd // 128, T)
    fg.quant_1x128(dev_bf16(xb), fg.E4M3, qx, sx)
    rt = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    rt[: g["row_token"].shape[0]] = g["row_token"]
    qg, sg = torch.zeros((cap, Hd), dtype=torch.uint8, device="cuda"), torch.zeros((Hd // 128, cap), dtype=torch.float32, device="cuda")
    fg.moe_gather(qx, sx, rt, offs, E, cap, qg, sg)
    # expert weights
    qgu = np.empty((E, 2 * F, Hd), np.uint8); sgu = np.empty((E, 2 * F // 128, Hd // 128), np.float32)
    qdn = np.empty((E, Hd, F), np.uint8); sdn = np.empty((E, Hd // 128, F // 128), np.float32)
    for e in range(E):
        qgu[e], sgu[e], _ = oracle.quant_128x128(w_gu[e])
        qdn[e], sdn[e], _ = oracle.quant_128x128(w_dn[e])
    GU = torch.zeros((cap, 2 * F), dtype=torch.bfloat16, device="cuda")
    fg.grouped_gemm(offs, qg, sg, dev_u8(qgu), dev_f32(sgu), GU)
    H = torch.zeros((cap, F), dtype=torch.bfloat16, device="cuda")
    fg.swiglu_fwd(GU, H)
    qh, sh = empty_u8(cap, F), empty_f32(F // 128, cap)
    fg.quant_1x128(H, fg.E4M3, qh, sh)
    Y = torch.zeros((cap, Hd), dtype=torch.bfloat16, device="cuda")
    fg.grouped_gemm(offs, qh, sh, dev_u8(qdn), dev_f32(sdn), Y)
    assert_status_ok()
    offs_np = offs.cpu().numpy()
    # stage: gather == quantize-then-gather in the oracle
    q_ref, s_ref, _ = oracle.quant_1x128(xb)
    qg_ref, sg_ref = oracle.moe_gather(q_ref, s_ref, ref["row_token"], tot, cap)
    assert np.array_equal(qg.cpu().numpy()[:tot], qg_ref[:tot])
    assert np.array_equal(sg.cpu().numpy()[:, :tot], sg_ref[:, :tot])
    # stage: gate/up grouped GEMM
    pm, pn = sample_points_dense(tot, 2 * F, seed=2)
    ref_gu = oracle.grouped_gemm_points(offs_np, qg_ref, sg_ref, cap, qgu, sgu, pm, pn)
    gemm_tolerance_check(bf16_to_f64(host_u16(GU))[pm, pn], ref_gu, bf16_out=True)
    # stage: SwiGLU on the GPU's GU, then 1x128 quantization of the GPU's H (bit-exact)
    gu_host = host_u16(GU)[:tot]
    h_host = host_u16(H)[:tot]
    h_ref = oracle.swiglu_fwd(gu_host)
    hi = lambda b: np.where(b & 0x8000, -(b & 0x7FFF).astype(np.int64), (b & 0x7FFF).astype(np.int64))
    assert np.max(np.abs(hi(h_host) - hi(h_ref))) <= 1
    qh_ref, sh_ref, _ = oracle.quant_1x128(h_host)
    assert np.array_equal(qh.cpu().numpy()[:tot], qh_ref)
    assert np.array_equal(sh.cpu().numpy()[:, :tot].view(np.uint32), sh_ref.view(np.uint32))
    # stage: down grouped GEMM
    qh_full = np.zeros((cap, F), np.uint8); qh_full[:tot] = qh_ref
    sh_full = np.zeros((F // 128, cap), np.float32); sh_full[:, :tot] = sh_ref
    pm, pn = sample_points_dense(tot, Hd, seed=3)
    ref_y = oracle.grouped_gemm_points(offs_np, qh_full, sh_full, cap, qdn, sdn, pm, pn)
    gemm_tolerance_check(bf16_to_f64(host_u16(Y))[pm, pn], ref_y, bf16_out=True)
