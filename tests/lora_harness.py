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

# Guard regions around every output and the workspace of a forward: rows
# above and below each output, columns past N in each row (ldo = N + 16),
# and bytes on both sides of the workspace, all filled with a sentinel and
# checked unchanged afterwards, so that a stray store past a tile edge fails
# the test even where the output itself is right.
GUARD_ROWS = 2
GUARD_COLS = 16
GUARD_BYTES = 4096
SENTINEL = -7.75  # exact in bf16 and fp32
WS_SENTINEL = 0xA5


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


def guarded_output(M: int, N: int, dtype: torch.dtype, device):
    """An [M, N] output view (row stride N + GUARD_COLS) inside a buffer whose
    other elements hold SENTINEL; the view itself is NaN-filled, so a missing
    store shows too.  Returns (view, buffer)."""
    buf = torch.full((M + 2 * GUARD_ROWS, N + GUARD_COLS), SENTINEL, dtype=dtype, device=device)
    out = buf[GUARD_ROWS:GUARD_ROWS + M, :N]
    out.fill_(float("nan"))
    return out, buf


def check_output_guard(buf: torch.Tensor, M: int, N: int, what: str) -> None:
    g = buf.clone()
    g[GUARD_ROWS:GUARD_ROWS + M, :N] = SENTINEL
    bad = int((g != SENTINEL).sum())
    assert bad == 0, f"{what}: {bad} guard elements around the output were overwritten"


def guarded_workspace(nbytes: int, device):
    """A workspace of nbytes inside a buffer with GUARD_BYTES of WS_SENTINEL
    on both sides.  Returns (view, buffer)."""
    buf = torch.full((nbytes + 2 * GUARD_BYTES,), WS_SENTINEL, dtype=torch.uint8, device=device)
    return buf[GUARD_BYTES:GUARD_BYTES + nbytes], buf


def check_workspace_guard(buf: torch.Tensor, what: str) -> None:
    head, tail = buf[:GUARD_BYTES], buf[buf.numel() - GUARD_BYTES:]
    bad = int((head != WS_SENTINEL).sum()) + int((tail != WS_SENTINEL).sum())
    assert bad == 0, f"{what}: {bad} guard bytes around the workspace were overwritten"


def index_args(wl, mode: str, ids: np.ndarray, device) -> dict:
    """The row map of a forward in one of the three forms.

    mode "bgmv": per-row ids; "sgmv": host segmenter + permutation;
    "sorted": the workload's own pre-sorted segments (no permutation)."""
    if mode == "bgmv":
        return dict(row_adapter=torch.from_numpy(np.ascontiguousarray(ids, np.int32)).to(device))
    if mode == "sgmv":
        perm, offs, adp = segment_rows(ids, wl.num_slots)
        return dict(seg_offsets=torch.from_numpy(offs).to(device), seg_adapter=torch.from_numpy(adp).to(device),
                    perm=torch.from_numpy(perm).to(device))
    if mode == "sorted":
        return dict(seg_offsets=torch.from_numpy(wl.seg_offsets).to(device),
                    seg_adapter=torch.from_numpy(wl.seg_adapter).to(device))
    raise ValueError(mode)


def forward(wl, pools, mode: str = "bgmv", device="cuda", ids: Optional[np.ndarray] = None,
            x=None, Ws=None, outs=None, scales: Optional[torch.Tensor] = None) -> List[np.ndarray]:
    """Run lora_linear_forward through the C ABI; returns float32 outputs.

    mode: see index_args.  Unless ``outs`` is given, every output and the
    workspace sit between guard regions that are checked after the call.
    ``scales``: the call's own per-slot scales (device float32), or None.
    """
    td = torch_dtype(wl.dtype)
    if x is None or Ws is None:
        x, Ws = device_inputs(wl, device)
    ids = wl.row_adapter if ids is None else ids
    bufs = None
    if outs is None:
        made = [guarded_output(wl.M, p.N, td, device) for p in wl.projections]
        outs, bufs = [o for o, _ in made], [b for _, b in made]
    projs = [(W, pool, out) for W, pool, out in zip(Ws, pools, outs)]
    index = index_args(wl, mode, ids, device)
    need = LinearCall(x, projs, scales=scales, **index).workspace_bytes
    ws, ws_buf = guarded_workspace(need, device)
    call = LinearCall(x, projs, workspace=ws, scales=scales, **index)
    call()
    torch.cuda.synchronize()
    check_workspace_guard(ws_buf, f"{wl.name} {mode}")
    if bufs is not None:
        for p, (b, proj) in enumerate(zip(bufs, wl.projections)):
            check_output_guard(b, wl.M, proj.N, f"{wl.name} {mode} projection {p}")
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
