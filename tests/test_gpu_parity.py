"""GPU parity: lora_linear_forward (through the C ABI) against the float64
oracle on the same seeded inputs.

Small cases span several output tiles with ragged tails in M, N and K; the
five named workloads and the two of other target modules run at full size
with the oracle evaluated on every row (small ones) or on sampled rows
(large ones).  Integer-valued cases must be
bit-exact; mutation cases check that the tolerance is not vacuous.
"""

import numpy as np
import pytest
import torch

import lora_harness as H
from workloads import make_config, synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _sample_rows(wl, n=48, seed=0, per_tile=0, tile=128):
    """Rows to check at full size: both ends, segment boundaries, base-only
    rows, a seeded random sample, and ``per_tile`` seeded rows of every
    ``tile``-row token tile (the large-M GEMM's unit along M)."""
    rng = np.random.default_rng(seed)
    rows = {0, wl.M - 1}
    for t0 in range(0, wl.M, tile) if per_tile else ():
        rows.update(int(r) for r in rng.choice(np.arange(t0, min(wl.M, t0 + tile)),
                                                size=min(per_tile, min(wl.M, t0 + tile) - t0), replace=False))
    if wl.seg_offsets is not None:
        for o in wl.seg_offsets[1:-1]:
            rows.update({int(o) - 1, int(o)})
    base = np.nonzero(wl.row_adapter < 0)[0]
    rows.update(int(r) for r in base[:4])
    rows.update(int(r) for r in rng.choice(wl.M, size=min(n, wl.M), replace=False))
    return np.array(sorted(r for r in rows if 0 <= r < wl.M), dtype=np.int64)


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
@pytest.mark.parametrize("shape", [(300, 520, 392), (130, 1024, 264), (1, 64, 8), (257, 136, 1000),
                                   (64, 2048, 520), (17, 4096, 136), (600, 256, 200), (520, 1024, 2056),
                                   (480, 1024, 2056), (400, 512, 6152), (700, 1000, 520), (600, 64, 264)])
def test_small_mixed_ranks(shape, mode):
    """(700, 1000, 520): the two-SM GEMM with a ragged last k-block (the V
    items' K-slices of 8 and 8 k-blocks, the last one partly past K); (600,
    64, 264): one k-block, so one of a tile's two V slices is empty."""
    M, K, N = shape
    wl = synth(M=M, K=K, Ns=[N], num_slots=7, rank_choices=(1, 7, 16, 33, 64), seed=M + K + N)
    pools = H.make_pools(wl, DEV)
    out = H.forward(wl, pools, mode)[0]
    H.assert_close("bf16", out, H.oracle_rows(wl, 0), f"{shape} {mode}")


def test_presorted_segments_without_perm():
    wl = synth(M=333, K=256, Ns=[200], num_slots=9, rank_choices=(8, 16, 48), mode="sgmv", seed=5)
    pools = H.make_pools(wl, DEV)
    out = H.forward(wl, pools, "sorted")[0]
    H.assert_close("bf16", out, H.oracle_rows(wl, 0), "sorted")


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
def test_integer_exact_bitwise(mode):
    """Small-integer inputs with scale 2: every partial sum is an exact
    integer, so the bf16 output bits must equal the oracle's rounded bits.
    Mixed ranks up to 128 in shuffled pool blocks pin the block-table gather
    and the row->adapter indexing exactly."""
    wl = synth(M=200, K=256, Ns=[136, 64], num_slots=11, rank_choices=(1, 8, 16, 17, 64, 128),
               integer=True, seed=21, none_frac=0.15)
    pools = H.make_pools(wl, DEV, extra_blocks=13)
    outs = H.forward(wl, pools, mode)
    for p in range(2):
        want = H.oracle_bf16_bits(H.oracle_rows(wl, p))
        got = torch.from_numpy(outs[p]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, want), f"projection {p}: {np.sum(got != want)} outputs differ"


@pytest.mark.parametrize("mode", ["sorted", "sgmv", "bgmv"])
def test_integer_exact_prefill_geometry(mode):
    """The prefill workload's geometry at a size the oracle finishes in
    seconds: 2048 tokens in 16 sorted segments that straddle the 128-token
    tiles, 16 slots with ranks {8, 16, 32, 64} (alpha = 2r) in scattered pool
    blocks, 5% base-only rows.  Integer inputs, so the large-M path (the LoRA
    term on the tensor cores) must be bit-exact for every row."""
    wl = synth(M=2048, K=1024, Ns=[1032], num_slots=16, rank_choices=(8, 16, 32, 64), integer=True,
               seed=2048, none_frac=0.05, mode="sgmv")
    assert sorted(set(int(r) for r in wl.ranks)) == [8, 16, 32, 64]
    straddle = [int(o) for o in wl.seg_offsets[1:-1] if int(o) % 128]
    assert len(straddle) >= 8
    pools = H.make_pools(wl, DEV, extra_blocks=29)
    out = H.forward(wl, pools, mode)[0]
    want = H.oracle_bf16_bits(H.oracle_rows(wl, 0))
    got = torch.from_numpy(out).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want), f"{mode}: {np.sum(got != want)} outputs differ"


def test_integer_exact_many_units():
    """More 256 x 256 units (8 token tiles x 20 column tiles = 160) than two
    rounds of the pairs, so most are handed out on demand, with LoRA steps
    on every tile; integer inputs, every output bit-exact."""
    wl = synth(M=2048, K=192, Ns=[5120], num_slots=16, rank_choices=(8, 16, 32, 64), integer=True,
               seed=5120, none_frac=0.05, mode="sgmv")
    pools = H.make_pools(wl, DEV, extra_blocks=11)
    out = H.forward(wl, pools, "sorted")[0]
    want = H.oracle_bf16_bits(H.oracle_rows(wl, 0))
    got = torch.from_numpy(out).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want), f"{np.sum(got != want)} outputs differ"


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
def test_integer_exact_large_m_tile_fallback(mode):
    """Large M where some 128-token tiles name adapters spanning more than 16
    pool blocks (rows in no order: up to 12 slots of rank 48-64 per tile) and
    take the CUDA-core fallback, while the tiles of the sorted first half take
    the tensor-core LoRA steps; one call, every row bit-exact."""
    wl = synth(M=900, K=256, Ns=[264, 136], num_slots=12, rank_choices=(48, 64), integer=True, seed=900,
               none_frac=0.1)
    ids = wl.row_adapter.copy()
    half = ids[:450]
    ids[:450] = np.sort(half)  # the first half sorted: few slots per tile
    pools = H.make_pools(wl, DEV, extra_blocks=7)
    outs = H.forward(wl, pools, mode, ids=ids)
    for p in range(2):
        want = H.oracle_bf16_bits(H.oracle_rows(wl, p, ids=ids))
        got = torch.from_numpy(outs[p]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, want), f"{mode} projection {p}: {np.sum(got != want)} outputs differ"


@pytest.mark.parametrize("shape", [(64, 2048, (264, 520)), (37, 1024, (1032,)), (700, 192, (136,)),
                                   (448, 320, (2064,)), (200, 2048, (1032,)), (256, 4096, (520, 264))])
def test_integer_exact_split_k_and_orientations(shape):
    """Bit-exact through the split-K reduction (few tokens, long K: several
    CTAs share each output tile), the swapped orientation near its row
    limit (448 tokens) and the non-swapped orientation (many tokens); 200
    and 256 tokens take one 256-token tile (a ragged token tail, and two
    projections in one launch)."""
    M, K, Ns = shape
    wl = synth(M=M, K=K, Ns=list(Ns), num_slots=6, rank_choices=(4, 16, 32), integer=True,
               seed=M + K, none_frac=0.2)
    pools = H.make_pools(wl, DEV)
    outs = H.forward(wl, pools, "bgmv")
    for p in range(len(Ns)):
        want = H.oracle_bf16_bits(H.oracle_rows(wl, p))
        got = torch.from_numpy(outs[p]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, want), f"{shape} projection {p}: {np.sum(got != want)} outputs differ"


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
@pytest.mark.parametrize("shape", [(500, 1032, 392), (480, 1032, 136)])
def test_grouped_path_small(shape, mode):
    """Rows few enough for the swapped GEMM but ranks large enough that the
    library groups rows by adapter (device group table, grouped shrink and
    expand) instead of reading each row's A and B per row; a popular adapter
    spans several row chunks, the column tail is ragged."""
    M, K, N = shape
    wl = synth(M=M, K=K, Ns=[N], num_slots=9, rank_choices=(1, 40, 129, 256), seed=M + N,
               zipf_s=1.5, mode=mode)
    pools = H.make_pools(wl, DEV)
    out = H.forward(wl, pools, mode)[0]
    H.assert_close("bf16", out, H.oracle_rows(wl, 0), f"grouped {shape} {mode}")


def test_grouped_path_integer_exact():
    wl = synth(M=450, K=1024, Ns=[264, 72], num_slots=7, rank_choices=(3, 64, 200, 256), integer=True,
               seed=33, none_frac=0.2, zipf_s=1.3)
    pools = H.make_pools(wl, DEV)
    outs = H.forward(wl, pools, "bgmv")
    for p in range(2):
        want = H.oracle_bf16_bits(H.oracle_rows(wl, p))
        got = torch.from_numpy(outs[p]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, want), f"projection {p}: {np.sum(got != want)} outputs differ"


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
@pytest.mark.parametrize("shape", [(500, 2056, 1032), (480, 4104, 264), (200, 8200, 3080)])
def test_pipelined_grouped_path(shape, mode):
    """Pools of max_rank <= 128 take the pipelined grouped kernels (rows
    sorted in every CTA, adapter pieces streamed by bulk copies, 16 x 16 x 16
    warp MMAs).  K is ragged against the 512-wide stages and the K slices, N
    against the 1024-column ranges; a popular adapter spans several 16-row
    chunks; ranks 1 and 100 leave partial rank blocks."""
    M, K, N = shape
    wl = synth(M=M, K=K, Ns=[N], num_slots=9, rank_choices=(1, 40, 100, 128), seed=M + K + N,
               zipf_s=1.5, mode=mode, none_frac=0.12)
    assert H.pool_max_rank(wl) <= 128
    pools = H.make_pools(wl, DEV)
    out = H.forward(wl, pools, mode)[0]
    H.assert_close("bf16", out, H.oracle_rows(wl, 0), f"pipelined {shape} {mode}")


def test_pipelined_grouped_integer_exact():
    """Integer inputs through the pipelined grouped kernels: V's bf16 hi/lo
    parts carry the integer partial sums exactly, so the output bits must
    equal the oracle's."""
    wl = synth(M=450, K=2048, Ns=[1032, 264], num_slots=13, rank_choices=(3, 16, 64, 120, 128), integer=True,
               seed=35, none_frac=0.2, zipf_s=1.3)
    pools = H.make_pools(wl, DEV, extra_blocks=5)
    outs = H.forward(wl, pools, "bgmv")
    for p in range(2):
        want = H.oracle_bf16_bits(H.oracle_rows(wl, p))
        got = torch.from_numpy(outs[p]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, want), f"projection {p}: {np.sum(got != want)} outputs differ"


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
@pytest.mark.parametrize("shape, launches", [
    ((300, 4096, (1032, 264)), 4),          # the grouping, one shrink, one expand, one GEMM for the pair
    ((256, 4096, (2048, 512, 520)), 5),     # ... and a second GEMM for the third projection
])
def test_pipelined_projection_pairs(shape, launches, mode):
    """Several projections whose LoRA terms go through the pipelined kernels:
    the rows grouped once, one shrink and one expand launch for all of them
    (the SMs split between the projections, each its own correction array),
    then one GEMM launch per two projections (SGMV adds the segments-to-rows
    kernel).  Integer inputs: every projection bit-exact."""
    from adapter_gemm_linear_gb300 import kernel_launches
    M, K, Ns = shape
    wl = synth(M=M, K=K, Ns=list(Ns), num_slots=11, rank_choices=(16, 64, 128), integer=True, seed=M + K,
               none_frac=0.1, zipf_s=1.2)
    pools = H.make_pools(wl, DEV)
    H.forward(wl, pools, mode)
    torch.cuda.synchronize()
    before = kernel_launches()
    outs = H.forward(wl, pools, mode)
    assert kernel_launches() - before == launches + (1 if mode == "sgmv" else 0)
    for p in range(len(Ns)):
        want = H.oracle_bf16_bits(H.oracle_rows(wl, p))
        got = torch.from_numpy(outs[p]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, want), f"{shape} projection {p}: {np.sum(got != want)} outputs differ"


@pytest.mark.parametrize("shape", [(300, 1024, 9856), (400, 2056, 9992)])
def test_integer_exact_many_tiles(shape):
    """Swapped GEMM with 256-token tiles and more tiles than SMs (a short last
    wave).  Integer inputs: bit-exact."""
    M, K, N = shape
    wl = synth(M=M, K=K, Ns=[N], num_slots=5, rank_choices=(8, 16, 32), integer=True, seed=M + N,
               none_frac=0.1)
    pools = H.make_pools(wl, DEV)
    out = H.forward(wl, pools, "bgmv")[0]
    want = H.oracle_bf16_bits(H.oracle_rows(wl, 0))
    got = torch.from_numpy(out).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want), f"{shape}: {np.sum(got != want)} outputs differ"


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
@pytest.mark.parametrize("shape, launches", [
    ((128, 1024, (256, 512, 264)), 3),         # a pair and a single GEMM launch, both split-K (own tile counters)
    ((256, 2048, (1024, 1040, 512, 520)), 3),  # two pairs
    ((448, 512, (4096, 1024)), 2),             # a pair with 256-token tiles
    ((300, 1024, (8192, 2048)), 2),            # a pair with more tiles than SMs: the last round split along K
])
def test_fused_projection_launches(shape, launches, mode):
    """Several projections whose LoRA terms go through the per-row kernel:
    one launch of it for all of them, then the GEMMs two projections per
    launch (SGMV adds the segments-to-rows kernel).  Integer inputs: every
    projection bit-exact."""
    from adapter_gemm_linear_gb300 import kernel_launches
    M, K, Ns = shape
    wl = synth(M=M, K=K, Ns=list(Ns), num_slots=7, rank_choices=(8, 16), integer=True, seed=M + K + len(Ns),
               none_frac=0.1)
    pools = H.make_pools(wl, DEV)
    H.forward(wl, pools, mode)
    torch.cuda.synchronize()
    before = kernel_launches()
    outs = H.forward(wl, pools, mode)
    assert kernel_launches() - before == launches + (1 if mode == "sgmv" else 0)
    for p in range(len(Ns)):
        want = H.oracle_bf16_bits(H.oracle_rows(wl, p))
        got = torch.from_numpy(outs[p]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, want), f"{shape} projection {p}: {np.sum(got != want)} outputs differ"


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
@pytest.mark.parametrize("shape", [
    (64, 2048, (2048, 256, 256)),         # q, k, v with grouped-query k/v, sharing x
    (200, 1024, (2752, 2752)),            # gate and up sharing x
    (96, 5504, (1024,)),                  # down: K > N
    (520, 2752, (1024, 1032, 264, 8)),    # four projections, large M (the other GEMM orientation)
    (300, 8192, (1024, 8192)),            # 70B-shaped k/v and o widths at a prefill-ish M
])
def test_more_target_modules(shape, mode):
    """Several target modules of one layer in one call (shared x and row ids,
    one pool per projection), including K > N and widths down to 8."""
    M, K, Ns = shape
    wl = synth(M=M, K=K, Ns=list(Ns), num_slots=9, rank_choices=(8, 16, 64), seed=M + K + len(Ns), mode=mode)
    pools = H.make_pools(wl, DEV)
    outs = H.forward(wl, pools, mode)
    rows = _sample_rows(wl, n=64) if M * K > 2_000_000 else np.arange(M)
    for p in range(len(Ns)):
        H.assert_close("bf16", outs[p][rows], H.oracle_rows(wl, p, rows), f"{shape} {mode} projection {p}")


@pytest.mark.parametrize("case", ["all_base", "one_adapter", "all_max_rank"])
def test_pipelined_grouped_edges(case):
    """Edges of the pipelined grouped path (pools of max_rank <= 128, rows
    too many for the per-row kernel): every row without an adapter (only
    zero items); one adapter owning all 512 rows (32 chunks of one group);
    every slot at rank 128 (eight rank blocks per item)."""
    M, K, N = 512, 2056, 1032
    if case == "all_base":
        wl = synth(M=M, K=K, Ns=[N], num_slots=4, rank_choices=(128,), seed=71, none_frac=1.0)
    elif case == "one_adapter":
        wl = synth(M=M, K=K, Ns=[N], num_slots=1, rank_choices=(128,), seed=72, none_frac=0.0)
    else:
        wl = synth(M=M, K=K, Ns=[N], num_slots=12, rank_choices=(128,), seed=73, none_frac=0.05, zipf_s=1.2)
    assert H.pool_max_rank(wl) == 128
    pools = H.make_pools(wl, DEV, slots=list(range(wl.num_slots)))
    out = H.forward(wl, pools, "bgmv")[0]
    rows = _sample_rows(wl, n=96)
    H.assert_close("bf16", out[rows], H.oracle_rows(wl, 0, rows), f"pipelined edge {case}")
    assert not np.isnan(out).any()


def test_tiny_fp32_full():
    wl = make_config("tiny_fp32")
    pools = H.make_pools(wl, DEV)
    out = H.forward(wl, pools, "bgmv")[0]
    H.assert_close("fp32", out, H.oracle_rows(wl, 0), "tiny_fp32")


def test_decode_bgmv_full():
    wl = make_config("decode_bgmv")
    pools = H.make_pools(wl, DEV)
    out = H.forward(wl, pools, "bgmv")[0]
    H.assert_close("bf16", out, H.oracle_rows(wl, 0), "decode_bgmv")


def test_prefill_sgmv_sampled():
    """The full prefill workload: two rows of every 128-token tile (each
    tile has its own slot range on the large-M path), the segment
    boundaries and a random sample, against the oracle."""
    wl = make_config("prefill_sgmv")
    pools = H.make_pools(wl, DEV)
    out = H.forward(wl, pools, "sorted")[0]
    rows = _sample_rows(wl, per_tile=2)
    assert len(set(int(r) // 128 for r in rows)) == wl.M // 128
    H.assert_close("bf16", out[rows], H.oracle_rows(wl, 0, rows), "prefill_sgmv")
    assert not np.isnan(out).any()


def test_decode_70b_qv_sampled():
    wl = make_config("decode_70b_qv")
    pools = H.make_pools(wl, DEV)
    outs = H.forward(wl, pools, "bgmv")
    rows = _sample_rows(wl, n=64)
    for p in range(2):
        H.assert_close("bf16", outs[p][rows], H.oracle_rows(wl, p, rows), f"decode_70b_qv p{p}")
        assert not np.isnan(outs[p]).any()


def test_slora_mixed_sampled():
    wl = make_config("slora_mixed")
    pools = H.make_pools(wl, DEV)
    out = H.forward(wl, pools, "bgmv")[0]
    rows = _sample_rows(wl, n=64)
    H.assert_close("bf16", out[rows], H.oracle_rows(wl, 0, rows), "slora_mixed")
    assert not np.isnan(out).any()


def test_decode_70b_qkv_sampled():
    """q, k and v of a 70B layer in one call (k and v 1024 wide, GQA), rank-64
    adapters on all three."""
    wl = make_config("decode_70b_qkv")
    pools = H.make_pools(wl, DEV)
    outs = H.forward(wl, pools, "bgmv")
    rows = _sample_rows(wl, n=64)
    for p in range(3):
        H.assert_close("bf16", outs[p][rows], H.oracle_rows(wl, p, rows), f"decode_70b_qkv p{p}")
        assert not np.isnan(outs[p]).any()


def test_prefill_down_proj_sampled():
    """A down projection (K = 13824 > N = 5120) at prefill size: two rows of
    every 256-token tile, the segment boundaries and a random sample."""
    wl = make_config("prefill_down_proj")
    pools = H.make_pools(wl, DEV)
    out = H.forward(wl, pools, "sorted")[0]
    rows = _sample_rows(wl, per_tile=2, tile=256)
    assert len(set(int(r) // 256 for r in rows)) == wl.M // 256
    H.assert_close("bf16", out[rows], H.oracle_rows(wl, 0, rows), "prefill_down_proj")
    assert not np.isnan(out).any()


@pytest.mark.parametrize("cfg", ["tiny_fp32", "decode_bgmv", "prefill_sgmv", "decode_70b_qv", "slora_mixed",
                                 "decode_70b_qkv", "prefill_down_proj"])
def test_mutations_fail_tolerance(cfg):
    """Outputs computed with a wrong assignment or scale must fail the
    tolerance against the true oracle, on every workload and every
    projection: (i) every id forced to -1, (ii) ids rotated to another slot,
    (iii) every scale halved.  The unmutated forward passes on the same rows,
    so the tolerance separates the two."""
    wl = make_config(cfg)
    rows = _sample_rows(wl, n=32) if wl.M > 64 else np.arange(wl.M)
    ids = wl.row_adapter
    none = np.full_like(ids, -1)
    used = wl.used_slots
    rot = ids.copy()
    for k, s in enumerate(used):
        rot[ids == s] = used[(k + 1) % used.size]
    pools = H.make_pools(wl, DEV)
    outs_ok = H.forward(wl, pools, "bgmv")
    outs_none = H.forward(wl, pools, "bgmv", ids=none)
    outs_rot = H.forward(wl, pools, "bgmv", ids=rot)
    del pools
    half = H.make_pools(wl, DEV, alpha_scale=0.5)
    outs_half = H.forward(wl, half, "bgmv")
    for p in range(len(wl.projections)):
        ref = H.oracle_rows(wl, p, rows)
        H.assert_close(wl.dtype, outs_ok[p][rows], ref, f"{cfg} p{p} unmutated")
        for name, outs in (("none", outs_none), ("rotated", outs_rot), ("half scale", outs_half)):
            assert H.fails_tolerance(wl.dtype, outs[p][rows], ref), f"{cfg} p{p}: mutation '{name}' passed"


def test_base_only_and_empty():
    wl = synth(M=96, K=128, Ns=[72], num_slots=3, seed=9)
    pools = H.make_pools(wl, DEV)
    none = np.full(wl.M, -1, np.int32)
    out = H.forward(wl, pools, "bgmv", ids=none)[0]
    H.assert_close("bf16", out, H.oracle_rows(wl, 0, ids=none), "all base-only")
    # M = 0 is a no-op
    wl0 = synth(M=0, K=128, Ns=[72], num_slots=3, seed=9)
    assert H.forward(wl0, pools, "bgmv")[0].shape == (0, 72)


def test_device_source_load_matches_host_load():
    wl = synth(M=64, K=192, Ns=[96], num_slots=5, rank_choices=(3, 16, 40), seed=13)
    ph = H.make_pools(wl, DEV, src="host")[0]
    pd = H.make_pools(wl, DEV, src="device")[0]
    torch.cuda.synchronize()
    for s in wl.used_slots:
        rh, sh, bh = ph.slot_info(int(s))
        rd, sd, bd = pd.slot_info(int(s))
        assert (rh, sh, bh) == (rd, sd, bd)
        A, B = wl.adapter(0, int(s))
        r = int(wl.ranks[s])
        for t in range(-(-r // 16)):
            rows = min(16, r - 16 * t)
            for pool in (ph, pd):
                blk = pool.a_arena[bh[t]].float().cpu().numpy()
                assert np.array_equal(blk[:rows], A[16 * t:16 * t + rows])
                assert not blk[rows:].any()
                blb = pool.b_arena[bh[t]].float().cpu().numpy()  # [N, 16]
                assert np.array_equal(blb[:, :rows], B[:, 16 * t:16 * t + rows])
                assert not blb[:, rows:].any()


def test_unload_reload_and_errors():
    from adapter_gemm_linear_gb300 import LoraError, device_status
    wl = synth(M=40, K=64, Ns=[48], num_slots=4, rank_choices=(16, 32), seed=17, none_frac=0.0)
    pool = H.make_pools(wl, DEV, slots=range(4))[0]
    free0 = pool.free_blocks
    r2 = pool.slot_info(2)[0]
    pool.unload(2)
    assert pool.free_blocks == free0 + -(-r2 // 16)
    with pytest.raises(LoraError):
        pool.unload(2)
    # a row that names the empty slot gets no correction and is reported
    device_status()
    ids = wl.row_adapter.copy()
    out = H.forward(wl, [pool], "bgmv", ids=ids)[0]
    st, detail = device_status()
    assert (st != 0) == bool((ids == 2).any())
    ids_ref = np.where(ids == 2, -1, ids)
    H.assert_close("bf16", out, H.oracle_rows(wl, 0, ids=ids_ref), "empty slot rows -> base")
    # out-of-range id
    bad = ids_ref.copy()
    bad[5] = 99
    out = H.forward(wl, [pool], "bgmv", ids=bad)[0]
    st, detail = device_status()
    assert st == 7 and detail == 5
    H.assert_close("bf16", out, H.oracle_rows(wl, 0, ids=np.where(bad == 99, -1, bad)), "bad id")
    # reload
    A, B = wl.adapter(0, 2)
    pool.load(2, torch.from_numpy(A).to(torch.bfloat16), torch.from_numpy(B).to(torch.bfloat16),
              float(wl.alphas[2]))
    assert pool.free_blocks == free0
    out = H.forward(wl, [pool], "bgmv")[0]
    H.assert_close("bf16", out, H.oracle_rows(wl, 0), "after reload")
    assert device_status()[0] == 0
