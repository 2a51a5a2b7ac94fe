"""Shared helpers for the GPU parity tests: host<->device marshalling of the
seeded inputs, guard-banded output buffers, the stratified GEMM sample and
the GEMM tolerance check (the same numbers the oracle sees go to the CUDA
library).

Guard bands stand in for a memory checker (compute-sanitizer is not
available on the test machines): every output buffer made by ``empty_u8`` /
``empty_f32`` / ``guarded`` lives inside a larger allocation whose bytes
before and after it are filled with a sentinel, and the buffer itself starts
out holding the sentinel too (so an element a kernel forgets to write shows
up in the parity comparison).  ``check_canaries`` -- run by the test suite
after every GPU test -- asserts that no kernel wrote into a band."""
import numpy as np
import torch

import fp8_fine_grained_x128_gb300 as fg

CANARY_BYTE = 0xA5
CANARY_BAND = 1 << 14          # bytes on each side (keeps the 16-byte alignment of the buffer)
_bands = []                    # (raw allocation, buffer bytes, label) of every live guarded buffer


def guarded(shape, dtype, label=""):
    """An uninitialised-looking output buffer with sentinel bands around it."""
    esz = torch.empty((), dtype=dtype).element_size()
    n = int(np.prod(shape)) if len(shape) else 1
    nbytes = n * esz
    raw = torch.full((2 * CANARY_BAND + nbytes,), CANARY_BYTE, dtype=torch.uint8, device="cuda")
    t = raw[CANARY_BAND:CANARY_BAND + nbytes].view(dtype).view(shape)
    _bands.append((raw, nbytes, label or f"{tuple(shape)} {dtype}"))
    return t


def check_canaries():
    """Assert that every guard band registered since the last call is intact."""
    global _bands
    bands, _bands = _bands, []
    if not bands:
        return
    torch.cuda.synchronize()
    for raw, nbytes, label in bands:
        lo = raw[:CANARY_BAND]
        hi = raw[CANARY_BAND + nbytes:]
        bad_lo = int((lo != CANARY_BYTE).sum().item())
        bad_hi = int((hi != CANARY_BYTE).sum().item())
        assert bad_lo == 0 and bad_hi == 0, (
            f"guard band of the buffer {label} overwritten: {bad_lo} bytes before it, {bad_hi} after it")


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
    return guarded(shape, torch.uint8)


def empty_f32(*shape):
    return guarded(shape, torch.float32)


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


def sample_points_dense(M: int, N: int, per_tile: int = 16, total: int = 1 << 20, seed: int = 0,
                        tile_m: int = 128, tile_n: int = 128):
    """A seeded, stratified sample of output coordinates: every tile_m x tile_n
    output tile is hit k = max(per_tile, ceil(total / tiles)) times -- its four
    corners plus k - 4 points drawn uniformly inside it -- so the sample holds
    at least ``total`` points and no tile is hit fewer than ``per_tile`` times."""
    rng = np.random.default_rng(seed)
    tm, tn = M // tile_m, N // tile_n
    ntiles = tm * tn
    k = max(per_tile, -(-total // ntiles))
    mt, nt = np.meshgrid(np.arange(tm, dtype=np.int64) * tile_m, np.arange(tn, dtype=np.int64) * tile_n,
                         indexing="ij")
    mt, nt = mt.ravel(), nt.ravel()
    cm = np.array([0, 0, tile_m - 1, tile_m - 1], np.int64)
    cn = np.array([0, tile_n - 1, 0, tile_n - 1], np.int64)
    pm = [mt[:, None] + cm[None, :], mt[:, None] + rng.integers(0, tile_m, (ntiles, k - 4))]
    pn = [nt[:, None] + cn[None, :], nt[:, None] + rng.integers(0, tile_n, (ntiles, k - 4))]
    return np.concatenate(pm, axis=1).ravel(), np.concatenate(pn, axis=1).ravel()
