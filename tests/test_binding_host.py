"""Host-side pieces of the Python binding that need no GPU."""

import pytest


def test_int8_weight_quantize_rule():
    """Int8Weight.quantize: symmetric per row, scale = max|W[n]| / 127, every
    element within half a step of its dequantized value; rejects wrong types."""
    import torch
    from adapter_gemm_linear_gb300 import Int8Weight
    g = torch.Generator().manual_seed(0)
    W = torch.randn(37, 96, generator=g) * torch.linspace(0.01, 3.0, 37)[:, None]
    W[5] = 0.0  # an all-zero row keeps a positive scale and zero codes
    qw = Int8Weight.quantize(W)
    assert qw.q.dtype == torch.int8 and qw.q.shape == (37, 96)
    assert qw.scale.dtype == torch.float32 and qw.scale.shape == (37,)
    assert int(qw.q.abs().max()) <= 127 and bool((qw.scale > 0).all())
    amax = W.abs().amax(dim=1)
    nz = amax > 0
    assert torch.allclose(qw.scale[nz], amax[nz] / 127.0)
    assert bool((qw.q[5] == 0).all())
    deq = qw.q.float() * qw.scale[:, None]
    assert bool(((deq - W).abs() <= qw.scale[:, None] * 0.5 + 1e-7).all())
    with pytest.raises(ValueError):
        Int8Weight(qw.q.to(torch.int16), qw.scale)
    with pytest.raises(ValueError):
        Int8Weight(qw.q, qw.scale[:-1])
