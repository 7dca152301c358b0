"""Failure paths and per-call options of lora_linear_forward on the GPU.

- A bounded wait that runs out: the test hook makes the split-K tile-counter
  waits (small M) or the waits for a token tile's LoRA intermediate (the
  large-M two-SM GEMM) of the next forward expect an arrival that never
  comes, with a 20 ms limit.  The GEMM must report LORA_ERR_DEVICE_TIMEOUT through the status
  word, leave the tiles it could not finish unwritten, release its tensor
  memory and end; the next forward on the same context must be right.  No
  GPU fault is involved: every wait is bounded and the kernel returns.
- Per-call scales (lora_forward_args_t.scales) replace the pools' alpha/r for
  one call, on each kernel path.
- A forward never writes to the adapter pool.
"""

import numpy as np
import pytest
import torch

import lora_harness as H
from adapter_gemm_linear_gb300 import LinearCall, device_status, arm_test_wait_timeout
from workloads import make_config, synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
LORA_ERR_DEVICE_TIMEOUT = 10
SPLITK_COUNTER_SITE = 5  # detail the GEMM records for its split-K counter wait


def test_wait_timeout_reports_and_recovers():
    # 64 tokens x 4096 -> 1024: 8 W tiles, so the GEMM splits K over many CTAs
    wl = synth(M=64, K=4096, Ns=[1024], num_slots=5, rank_choices=(16,), seed=91)
    pools = H.make_pools(wl, DEV)
    assert device_status() == (0, 0)
    arm_test_wait_timeout(20_000_000)
    out = H.forward(wl, pools, "bgmv")[0]
    st, detail = device_status()
    assert st == LORA_ERR_DEVICE_TIMEOUT and detail == SPLITK_COUNTER_SITE, (st, detail)
    # no split finished a tile: the NaN fill of the output is still there
    assert np.isnan(out).all()
    # the context is usable and the hook is spent: a normal forward is right
    out = H.forward(wl, pools, "bgmv")[0]
    assert device_status() == (0, 0)
    H.assert_close("bf16", out, H.oracle_rows(wl, 0), "after the timed-out forward")


VT_READY_SITE = 16  # detail the two-SM GEMM records for its wait on a tile's LoRA intermediate


def test_wait_timeout_two_sm_gemm():
    """The large-M two-SM GEMM armed the same way: its producers' waits for a
    token tile's Vt expect one count more than the V items give.  The first
    one runs out after 20 ms; the kernel records the timeout, its other
    roles give up within their own bounded waits, and it ends; a normal
    forward right after on the same context is right."""
    wl = synth(M=1100, K=512, Ns=[264], num_slots=6, rank_choices=(8, 16, 32), seed=93, mode="sgmv")
    pools = H.make_pools(wl, DEV)
    assert device_status() == (0, 0)
    arm_test_wait_timeout(20_000_000)
    H.forward(wl, pools, "sorted")
    st, detail = device_status()
    assert st == LORA_ERR_DEVICE_TIMEOUT and detail == VT_READY_SITE, (st, detail)
    out = H.forward(wl, pools, "sorted")[0]
    assert device_status() == (0, 0)
    H.assert_close("bf16", out, H.oracle_rows(wl, 0), "after the timed-out two-SM forward")


def _scaled_oracle(wl, p, factors, rows=None):
    """The oracle with every slot's alpha multiplied by its factor."""
    import copy
    w2 = copy.copy(wl)
    w2.alphas = (wl.alphas * factors).astype(np.float32)
    return H.oracle_rows(w2, p, rows)


@pytest.mark.parametrize("case", [
    ("rows", dict(M=64, K=1024, Ns=[520], rank_choices=(8, 16))),                   # per-row kernel
    ("pipelined", dict(M=480, K=2056, Ns=[1032], rank_choices=(16, 64, 128))),      # pipelined grouped kernels
    ("large_m", dict(M=1100, K=512, Ns=[264, 136], rank_choices=(8, 16, 32, 64))),  # LoRA term on the tensor cores
    ("fp32", dict(M=40, K=256, Ns=[256], rank_choices=(8,), dtype="fp32")),         # CUDA-core path
])
@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
def test_per_call_scales(case, mode):
    name, kw = case
    wl = synth(num_slots=9, seed=7 + len(name), zipf_s=1.2, **kw)
    pools = H.make_pools(wl, DEV)
    rng = np.random.default_rng(3)
    factors = rng.choice(np.array([0.5, 2.0, -1.0, 0.0], np.float32), size=wl.num_slots)
    scales = torch.from_numpy((wl.alphas / wl.ranks * factors).astype(np.float32)).to(DEV)
    outs = H.forward(wl, pools, mode, scales=scales)
    rows = np.arange(wl.M)
    for p in range(len(wl.projections)):
        want = _scaled_oracle(wl, p, factors, rows)
        H.assert_close(wl.dtype, outs[p], want, f"{name} {mode} p{p} with per-call scales")
        # and the pools' own scales give a different, also correct, result
        assert H.fails_tolerance(wl.dtype, outs[p], H.oracle_rows(wl, p))
    outs = H.forward(wl, pools, mode)
    for p in range(len(wl.projections)):
        H.assert_close(wl.dtype, outs[p], H.oracle_rows(wl, p), f"{name} {mode} p{p} pool scales")


@pytest.mark.parametrize("cfg", ["decode_bgmv", "prefill_sgmv"])
def test_forward_leaves_pool_unchanged(cfg):
    wl = make_config(cfg)
    pools = H.make_pools(wl, DEV)
    before = [(p.a_arena.clone(), p.b_arena.clone(), p.block_table.clone(), p.ranks.clone(), p.scales.clone())
              for p in pools]
    H.forward(wl, pools, "bgmv")
    H.forward(wl, pools, "sgmv")
    for p, b in zip(pools, before):
        after = (p.a_arena, p.b_arena, p.block_table, p.ranks, p.scales)
        for name, x, y in zip(("A arena", "B arena", "block table", "ranks", "scales"), b, after):
            assert torch.equal(x, y), f"{cfg}: the forward changed the pool's {name}"


def test_scales_must_be_float32():
    wl = synth(M=8, K=64, Ns=[64], num_slots=2, seed=1)
    pools = H.make_pools(wl, DEV)
    x, Ws = H.device_inputs(wl)
    out = torch.empty((8, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        LinearCall(x, [(Ws[0], pools[0], out)], row_adapter=torch.zeros(8, dtype=torch.int32, device=DEV),
                   scales=torch.ones(2, dtype=torch.float64, device=DEV))


@pytest.mark.parametrize("M", [300, 1100])
def test_bad_segment_offsets_reported(M):
    """Decreasing segment offsets are reported as LORA_ERR_SEGMENTS with the
    offending index, by the segments-to-rows kernel (300 rows) and by the
    large-M plan kernel that reads pre-sorted segments itself (1100 rows)."""
    wl = synth(M=M, K=256, Ns=[264], num_slots=3, rank_choices=(16,), seed=5, none_frac=0.0)
    pools = H.make_pools(wl, DEV, slots=range(3))
    x, Ws = H.device_inputs(wl)
    out = torch.empty((M, 264), dtype=torch.bfloat16, device=DEV)
    offs = torch.tensor([0, M // 2, M // 4, M], dtype=torch.int32, device=DEV)  # decreasing at index 2
    adp = torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV)
    device_status()
    LinearCall(x, [(Ws[0], pools[0], out)], seg_offsets=offs, seg_adapter=adp)()
    torch.cuda.synchronize()
    assert device_status() == (8, 2)
    # valid offsets afterwards: no error, and the oracle's result
    offs = torch.tensor([0, M // 4, M // 2, M], dtype=torch.int32, device=DEV)
    LinearCall(x, [(Ws[0], pools[0], out)], seg_offsets=offs, seg_adapter=adp)()
    torch.cuda.synchronize()
    assert device_status() == (0, 0)
    ids = np.repeat(np.arange(3, dtype=np.int32), [M // 4, M // 2 - M // 4, M - M // 2])
    H.assert_close("bf16", out.float().cpu().numpy(), H.oracle_rows(wl, 0, ids=ids), f"segments M={M}")
