"""Shared helpers for the GPU tests: pools from workloads, the forward call
through the C ABI, and the parity tolerance.

Tolerances (per output row m, over its N columns):
  bf16 inputs, fp32 accumulation:  max |y - y_ref| <= 2e-2 * (max |y_ref| + 1)
  fp32 inputs:                     max |y - y_ref| <= 1e-4 * max(max |y_ref|, 1)
"""

from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np
import torch

import oracle
from adapter_gemm_linear_gb300 import LinearCall, LoraPool, segment_rows
from workloads import bf16_round

BF16_TOL = 2e-2
FP32_TOL = 1e-4


def row_tolerance(dtype: str, ref: np.ndarray) -> np.ndarray:
    amax = np.max(np.abs(ref), axis=1)
    if dtype == "bf16":
        return BF16_TOL * (amax + 1.0)
    return FP32_TOL * np.maximum(amax, 1.0)


def row_errors(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    return np.max(np.abs(got.astype(np.float64) - ref), axis=1)


def assert_close(dtype: str, got: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    err = row_errors(got, ref)
    tol = row_tolerance(dtype, ref)
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, (f"{what}: {bad.size} rows over tolerance; worst row {int(bad[0])} "
                           f"err {err[bad[0]]:.4g} tol {tol[bad[0]]:.4g}")


def fails_tolerance(dtype: str, got: np.ndarray, ref: np.ndarray) -> bool:
    return bool(np.any(row_errors(got, ref) > row_tolerance(dtype, ref)))


def torch_dtype(dtype: str) -> torch.dtype:
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def pool_max_rank(wl) -> int:
    return max(16, -(-int(wl.ranks.max()) // 16) * 16)


def make_pools(wl, device="cuda", slots: Optional[Sequence[int]] = None, src: str = "host",
               extra_blocks: int = 0, alpha_scale: float = 1.0) -> List[LoraPool]:
    """One pool per projection, loaded with ``slots`` (default: the slots the
    rows use) from the workload's seeded adapters."""
    td = torch_dtype(wl.dtype)
    slots = wl.used_slots if slots is None else np.asarray(slots, dtype=np.int32)
    need = sum(-(-int(wl.ranks[s]) // 16) for s in slots) + extra_blocks
    pools = []
    for p, proj in enumerate(wl.projections):
        pool = LoraPool(wl.K, proj.N, wl.num_slots, pool_max_rank(wl), max(need, 1), dtype=td,
                        device=device, free_list_seed=wl.free_list_seed + p)
        for s in slots:
            A, B = wl.adapter(p, int(s))
            At, Bt = torch.from_numpy(A).to(td), torch.from_numpy(B).to(td)
            if src == "device":
                At, Bt = At.to(device), Bt.to(device)
            pool.load(int(s), At, Bt, float(wl.alphas[s]) * alpha_scale)
        pools.append(pool)
    return pools


def device_inputs(wl, device="cuda"):
    td = torch_dtype(wl.dtype)
    x = torch.from_numpy(wl.x).to(td).to(device)
    Ws = [torch.from_numpy(p.W).to(td).to(device) for p in wl.projections]
    return x, Ws


def forward(wl, pools, mode: str = "bgmv", device="cuda", ids: Optional[np.ndarray] = None,
            x=None, Ws=None, outs=None) -> List[np.ndarray]:
    """Run lora_linear_forward through the C ABI; returns float32 outputs.

    mode "bgmv": per-row ids; "sgmv": host segmenter + permutation;
    "sorted": the workload's own pre-sorted segments (no permutation).
    """
    td = torch_dtype(wl.dtype)
    if x is None or Ws is None:
        x, Ws = device_inputs(wl, device)
    ids = wl.row_adapter if ids is None else ids
    if outs is None:
        outs = [torch.full((wl.M, p.N), float("nan"), dtype=td, device=device) for p in wl.projections]
    projs = [(W, pool, out) for W, pool, out in zip(Ws, pools, outs)]
    if mode == "bgmv":
        call = LinearCall(x, projs, row_adapter=torch.from_numpy(np.ascontiguousarray(ids, np.int32)).to(device))
    elif mode == "sgmv":
        perm, offs, adp = segment_rows(ids, wl.num_slots)
        call = LinearCall(x, projs, seg_offsets=torch.from_numpy(offs).to(device),
                          seg_adapter=torch.from_numpy(adp).to(device),
                          perm=torch.from_numpy(perm).to(device))
    elif mode == "sorted":
        call = LinearCall(x, projs, seg_offsets=torch.from_numpy(wl.seg_offsets).to(device),
                          seg_adapter=torch.from_numpy(wl.seg_adapter).to(device))
    else:
        raise ValueError(mode)
    call()
    torch.cuda.synchronize()
    return [o.float().cpu().numpy() for o in outs]


def oracle_rows(wl, p: int, rows=None, ids: Optional[np.ndarray] = None) -> np.ndarray:
    """Float64 oracle for projection p (optionally on a row subset)."""
    ids = wl.row_adapter if ids is None else ids
    sel = ids if rows is None else ids[np.asarray(rows)]
    used = sorted(set(int(i) for i in sel if i >= 0))
    adapters = {i: wl.adapter(p, i) for i in used}
    return oracle.forward(wl.x, wl.projections[p].W, ids, wl.ranks, wl.alphas, adapters, rows=rows)


def oracle_bf16_bits(y: np.ndarray) -> np.ndarray:
    """Round float64 oracle values to bf16 (nearest-even) and return the bits.
    Values here are integers below 2^24, so float32 holds them exactly and
    one rounding to bf16 gives the bits a correct kernel produces."""
    y32 = y.astype(np.float32)
    assert np.array_equal(y32.astype(np.float64), y), "not exact in fp32"
    return (bf16_round(y32).view(np.uint32) >> 16).astype(np.uint16)
