"""Shared helpers for the GPU parity tests: host<->device marshalling of the
seeded inputs and the GEMM tolerance check (the same numbers the oracle sees
go to the CUDA library)."""
import numpy as np
import torch

import fp8_fine_grained_x128_gb300 as fg


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint8)).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def empty_u8(*shape):
    return torch.empty(shape, dtype=torch.uint8, device="cuda")


def empty_f32(*shape):
    return torch.empty(shape, dtype=torch.float32, device="cuda")


def assert_status_ok():
    st = fg.device_status()
    assert st == fg.OK, fg.status_string(st)


def half_ulp_bf16(ref: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(ref), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 8)


def gemm_tolerance_check(got: np.ndarray, ref: np.ndarray, bf16_out: bool, rel: float = 1e-3):
    """The parity bar for FP32-accumulated GEMM outputs.

    got: GPU values (float64 view of BF16 or FP32 results); ref: the oracle's
    unrounded FP64 values.  Passing needs both
      |got - ref| <= rel * max(|ref|, 1)          (+ half a BF16 ulp of ref for BF16 output)
      |got - ref| <= rel * max(|ref|, rms(ref))   (+ same)  -- a gate that still bites
                                                    when every |ref| << 1 (dgrad / wgrad)
    Returns (max error / bound) for reporting.
    """
    err = np.abs(got - ref)
    extra = half_ulp_bf16(ref) if bf16_out else 0.0
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    b1 = rel * np.maximum(np.abs(ref), 1.0) + extra
    b2 = rel * np.maximum(np.abs(ref), rms) + extra
    bad1 = err > b1
    bad2 = err > b2
    assert not bad1.any(), f"{int(bad1.sum())} outputs beyond 1e-3*max(|ref|,1): worst {float((err / b1).max())}"
    assert not bad2.any(), f"{int(bad2.sum())} outputs beyond 1e-3*max(|ref|,rms): worst {float((err / b2).max())}"
    return float((err / b2).max()) if err.size else 0.0


def sample_points(M: int, N: int, n: int, seed: int = 0, tile_m: int = 128, tile_n: int = 128):
    """A seeded sample of output coordinates that hits every 128x128 output tile
    at its four corners plus ``n`` uniformly drawn points."""
    rng = np.random.default_rng(seed)
    mt, nt = np.meshgrid(np.arange(0, M, tile_m), np.arange(0, N, tile_n), indexing="ij")
    mt, nt = mt.ravel(), nt.ravel()
    corners_m = np.concatenate([mt, mt, mt + tile_m - 1, mt + tile_m - 1])
    corners_n = np.concatenate([nt, nt + tile_n - 1, nt, nt + tile_n - 1])
    pm = np.concatenate([corners_m, rng.integers(0, M, n)])
    pn = np.concatenate([corners_n, rng.integers(0, N, n)])
    return pm.astype(np.int64), pn.astype(np.int64)
