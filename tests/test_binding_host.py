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


def test_int4_weight_pack_and_quantize_rule():
    """Int4Weight.pack puts element 2j in the low nibble of byte j (two's
    complement); quantize is symmetric per row with scale = max|W[n]| / 7."""
    import torch
    from adapter_gemm_linear_gb300 import Int4Weight
    q = torch.tensor([[-8, 7, 0, -1, 3, -5]], dtype=torch.int8)
    packed = Int4Weight.pack(q)
    assert packed.dtype == torch.uint8 and packed.tolist() == [[0x78, 0xF0, 0xB3]]
    # unpacking by hand gives the values back
    lo = (packed & 0xF).to(torch.int16)
    hi = (packed >> 4).to(torch.int16)
    back = torch.stack([lo, hi], dim=2).reshape(1, 6)
    back = torch.where(back >= 8, back - 16, back)
    assert back.tolist() == q.tolist()
    g = torch.Generator().manual_seed(1)
    W = torch.randn(9, 64, generator=g)
    qw = Int4Weight.quantize(W)
    assert qw.q.shape == (9, 32) and qw.scale.shape == (9,)
    assert torch.allclose(qw.scale, W.abs().amax(dim=1) / 7.0)
    lo = (qw.q & 0xF).to(torch.int16)
    hi = (qw.q >> 4).to(torch.int16)
    v = torch.stack([lo, hi], dim=2).reshape(9, 64)
    v = torch.where(v >= 8, v - 16, v)
    assert int(v.abs().max()) <= 7
    assert bool(((v.float() * qw.scale[:, None] - W).abs() <= qw.scale[:, None] * 0.5 + 1e-6).all())
    with pytest.raises(ValueError):
        Int4Weight.pack(torch.tensor([[9, 0]]))
