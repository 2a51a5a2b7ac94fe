"""The binding's argument checks on the GPU: element types, layouts and
buffer sizes the C ABI cannot see behind a pointer are refused before a
launch, and a 2-D input given as a row-strided view (leading dimension >
columns) is quantized exactly like its contiguous copy."""
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
from gpu_helpers import assert_status_ok, empty_f32, empty_u8

pytestmark = pytest.mark.gpu


def bf(*shape, seed=3):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)


def test_wrong_element_type_is_refused():
    x = bf(128, 256)
    with pytest.raises(TypeError, match="dtype"):
        fg.quant_1x128(x.float(), fg.E4M3, empty_u8(128, 256), empty_f32(2, 128))
    with pytest.raises(TypeError, match="dtype"):
        fg.quant_1x128(x, fg.E4M3, empty_u8(128, 256), torch.empty((2, 128), dtype=torch.float16, device="cuda"))
    D16 = torch.empty((128, 128), dtype=torch.float16, device="cuda")
    A, sA = empty_u8(128, 128), empty_f32(1, 128)
    with pytest.raises(TypeError, match="dtype"):
        fg.blockscaled_gemm(A, fg.E4M3, sA, fg.GRAN_1x128, A, fg.E4M3, sA, fg.GRAN_1x128, D16)


def test_bad_layouts_and_short_buffers_are_refused():
    x = bf(256, 256)
    q, s = empty_u8(256, 256), empty_f32(2, 256)
    with pytest.raises(ValueError, match="columns must be contiguous"):
        fg.quant_1x128(x.t(), fg.E4M3, q, s)
    with pytest.raises(ValueError, match="contiguous"):
        fg.quant_1x128(x, fg.E4M3, empty_u8(256, 512)[:, :256], s)
    with pytest.raises(ValueError, match="needs"):
        fg.quant_1x128(x, fg.E4M3, q, empty_f32(1, 256))
    with pytest.raises(ValueError, match="needs"):
        fg.quant_1x128(x, fg.E4M3, q, s, empty_u8(256, 128), empty_f32(2, 256))
    A, sA = empty_u8(256, 256), empty_f32(2, 256)
    with pytest.raises(ValueError, match="writes"):
        fg.blockscaled_gemm(A, fg.E4M3, sA, fg.GRAN_1x128, A, fg.E4M3, sA, fg.GRAN_1x128, empty_f32(128, 256))
    with pytest.raises(ValueError, match="expected"):
        fg.blockscaled_gemm(A, fg.E4M3, sA, fg.GRAN_1x128, empty_u8(256, 128), fg.E4M3, sA, fg.GRAN_1x128,
                            empty_f32(256, 256))
    with pytest.raises(ValueError, match="needs"):
        fg.swiglu_bwd(bf(128, 256), bf(128, 64), torch.empty((128, 256), dtype=torch.bfloat16, device="cuda"))
    assert_status_ok()


def test_row_strided_input_equals_contiguous_copy():
    wide = bf(256, 640, seed=5)
    view = wide[:, 128:512]                     # leading dimension 640, columns 384
    assert view.stride() == (640, 1)
    got = (empty_u8(256, 384), empty_f32(3, 256), empty_u8(384, 256), empty_f32(2, 384))
    ref = (empty_u8(256, 384), empty_f32(3, 256), empty_u8(384, 256), empty_f32(2, 384))
    fg.quant_1x128(view, fg.E4M3, *got)
    fg.quant_1x128(view.contiguous(), fg.E4M3, *ref)
    assert_status_ok()
    for a, b in zip(got, ref):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_output_with_leading_dimension_is_accepted():
    """D may be a row-strided view: the GEMM writes [M][N] with ldD = D.stride(0)
    and leaves the columns beyond N alone."""
    A, sA = empty_u8(128, 128).fill_(0x38), empty_f32(1, 128).fill_(1.0)   # 0x38 = 1.0 in E4M3
    big = torch.full((128, 384), -5.0, dtype=torch.float32, device="cuda")
    fg.blockscaled_gemm(A, fg.E4M3, sA, fg.GRAN_1x128, A, fg.E4M3, sA, fg.GRAN_1x128, big[:, :128])
    assert_status_ok()
    assert torch.all(big[:, :128] == 128.0) and torch.all(big[:, 128:] == -5.0)
