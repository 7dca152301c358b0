"""The seeded input generators: determinism and the stated recipes."""

import numpy as np
import pytest

from workloads import CONFIG_NAMES, bf16_bits, bf16_round, make_config, synth


def test_bf16_round_ties_to_even_and_exactness():
    v = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 3.14159], np.float32)
    r = bf16_round(v)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0
    assert r[1] == 1.0
    # 1 + 3*2^-8 is halfway between 1+2^-7 and 1+2^-6: ties to even -> 1 + 2^-6
    assert r[2] == np.float32(1.0 + 2**-6)
    assert r[3] == 1.0
    assert r[4] == -2.5
    bits = bf16_bits(r)
    assert bits.dtype == np.uint16
    with pytest.raises(ValueError):
        bf16_bits(np.array([1.0 + 2**-10], np.float32))


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_deterministic(idx):
    a, b = make_config(idx), make_config(idx)
    assert np.array_equal(a.x, b.x)
    assert np.array_equal(a.row_adapter, b.row_adapter)
    assert np.array_equal(a.projections[0].W, b.projections[0].W)
    s = int(a.used_slots[0])
    for u, v in zip(a.adapter(0, s), b.adapter(0, s)):
        assert np.array_equal(u, v)


def test_recipes():
    c1 = make_config("tiny_fp32")
    assert c1.x.shape == (16, 256) and c1.projections[0].W.shape == (256, 256)
    assert set(c1.row_adapter.tolist()) <= {-1, 0, 1, 2, 3}
    assert (c1.ranks == 8).all() and (c1.alphas == 16).all()

    c2 = make_config("decode_bgmv")
    assert (c2.row_adapter == -1).sum() == 6
    assert (c2.ranks == 16).all() and (c2.alphas == 32).all()
    assert bf16_bits(c2.x).shape == (64, 4096)
    # Zipf(1.2): the most popular adapter carries many rows
    counts = np.bincount(c2.row_adapter[c2.row_adapter >= 0])
    assert counts.max() >= 8

    c3 = make_config("prefill_sgmv")
    lengths = np.diff(c3.seg_offsets)
    assert lengths.sum() == 8192 and (lengths >= 1).all() and lengths.size == 16
    assert np.array_equal(c3.seg_adapter, np.arange(16))
    assert set(c3.ranks.tolist()) <= {8, 16, 32, 64}
    assert np.array_equal(c3.alphas, 2.0 * c3.ranks)
    assert np.array_equal(np.repeat(c3.seg_adapter, lengths), c3.row_adapter)

    c4 = make_config("decode_70b_qv")
    assert [p.N for p in c4.projections] == [8192, 1024]
    assert (c4.row_adapter >= 0).all()

    c5 = make_config("slora_mixed")
    assert (c5.row_adapter == -1).sum() == 26
    assert c5.num_slots == 2048 and set(c5.ranks.tolist()) <= {8, 16, 32, 64, 128}
    assert c5.used_slots.size <= 200


def test_adapter_shapes_and_std():
    c2 = make_config("decode_bgmv")
    A, B = c2.adapter(0, 3)
    assert A.shape == (16, 4096) and B.shape == (4096, 16)
    assert abs(A.std() - 0.02) < 0.002 and abs(B.std() - 0.02) < 0.002
    bf16_bits(A), bf16_bits(B)


def test_synth_integer_and_sgmv():
    wl = synth(M=50, K=64, Ns=[32, 16], num_slots=5, integer=True, mode="sgmv")
    assert set(np.unique(wl.x).tolist()) <= {-2, -1, 0, 1, 2}
    offs, adp = wl.seg_offsets, wl.seg_adapter
    assert offs[0] == 0 and offs[-1] == 50
    assert np.array_equal(np.repeat(adp, np.diff(offs)), wl.row_adapter)
    assert (np.diff(wl.row_adapter) >= 0).all()
    A, B = wl.adapter(1, 2)
    assert B.shape == (16, int(wl.ranks[2]))


def test_config_names():
    assert len(CONFIG_NAMES) == 5


def test_widening_workloads():
    """The other target modules: q, k, v of a 70B layer in one call (GQA: k
    and v 1024 wide) and a down projection with K > N, reachable by name and
    by index after the five."""
    from workloads import WIDENING_NAMES
    assert WIDENING_NAMES == ("decode_70b_qkv", "prefill_down_proj")
    q = make_config("decode_70b_qkv")
    assert [p.N for p in q.projections] == [8192, 1024, 1024] and q.K == 8192 and q.M == 256
    assert set(q.ranks.tolist()) == {64} and float(q.alphas[0]) == 128.0
    assert (q.row_adapter == -1).sum() == 13
    assert make_config(5).row_adapter.tolist() == q.row_adapter.tolist()
    d = make_config("prefill_down_proj")
    assert d.K == 13824 and d.projections[0].N == 5120 and d.K > d.projections[0].N
    assert d.seg_offsets[0] == 0 and d.seg_offsets[-1] == 4096 and d.mode == "sgmv"
    assert np.array_equal(np.repeat(d.seg_adapter, np.diff(d.seg_offsets)), d.row_adapter)

