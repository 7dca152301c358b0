"""Float64 CPU oracle of the multi-adapter LoRA linear layer.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
baseline are the only callers.  Nothing in the product package imports this
package, and this package imports nothing from the product package.

Contents
--------
``forward``            y = W x + (alpha_i/r_i) B_i (A_i x) per row, float64
                       (C code in ``lora_oracle.c``, loaded through ctypes).
``rows_from_segments`` expands sorted segments (+ permutation) to per-row ids.
``segment_rows``       stable sort of rows by adapter id (pure Python).
``lora_params`` etc.   parameter / byte counts the pages work out.

Each function cites the passage it follows.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Iterable, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblora_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Load a compiled oracle library and declare its entry point."""
    lib = ctypes.CDLL(path)
    f = lib.lora_oracle_forward
    f.restype = ctypes.c_int
    f.argtypes = [
        ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_int,
    ]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def usable_cores() -> int:
    """Host cores this process may run on (affinity / cgroup limited)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def forward(
    x: np.ndarray,
    W: np.ndarray,
    row_adapter: np.ndarray,
    ranks: np.ndarray,
    alphas: np.ndarray,
    adapters: Dict[int, Tuple[np.ndarray, np.ndarray]],
    rows: Optional[Sequence[int]] = None,
    threads: Optional[int] = None,
    lib=None,
) -> np.ndarray:
    """Float64 y[rows, :] of the multi-adapter LoRA linear layer.

    Follows "Your LoRA Adapters Are Thrashing Your GPUs" §02 (scaled form
    W' = W + (alpha/r) B A, applied additively as W x + (alpha/r) B (A x)) and
    the adapted_linear sketch of "Adapter Residency When One Replica Serves
    Many Fine-Tunes" §"What the forward pass has to do differently", with the
    scale stored and applied per adapter (same section: the scale is a
    property of the trained adapter, not of the request) and each row picking
    its own adapter slot or no adapter at all ("LoRA Adapters: Many Models in
    One", §"A picture").

    x [M, K], W [N, K] float32 (bf16- or fp32-exact values); row_adapter [M]
    int, -1 = base only; ranks/alphas per slot; ``adapters[slot] = (A [r, K],
    B [N, r])`` for at least every slot a computed row uses.  ``lib`` selects
    another build of the C code (the mutation tests use it).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    W = np.ascontiguousarray(W, dtype=np.float32)
    ids = np.ascontiguousarray(row_adapter, dtype=np.int32)
    ranks = np.ascontiguousarray(ranks, dtype=np.int32)
    alphas = np.ascontiguousarray(alphas, dtype=np.float64)
    M, K = x.shape
    N = W.shape[0]
    if W.shape[1] != K or ids.shape != (M,):
        raise ValueError("shape mismatch")
    S = int(ranks.shape[0])
    if rows is None:
        rows_arr = np.arange(M, dtype=np.int32)
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        if rows_arr.size and (rows_arr.min() < 0 or rows_arr.max() >= M):
            raise ValueError("row index out of range")
    need = set(int(i) for i in ids[rows_arr] if i >= 0)
    for i in need:
        if not (0 <= i < S):
            raise ValueError(f"adapter id {i} out of range")
        if i not in adapters:
            raise ValueError(f"adapter {i} used by a row but not supplied")
    keep = []
    a_ptrs = (ctypes.c_void_p * max(S, 1))()
    b_ptrs = (ctypes.c_void_p * max(S, 1))()
    for i, (A, B) in adapters.items():
        A = np.ascontiguousarray(A, dtype=np.float32)
        B = np.ascontiguousarray(B, dtype=np.float32)
        r = int(ranks[i])
        if A.shape != (r, K) or B.shape != (N, r):
            raise ValueError(f"adapter {i}: A {A.shape} B {B.shape} vs r={r} K={K} N={N}")
        keep += [A, B]
        a_ptrs[i] = _ptr(A)
        b_ptrs[i] = _ptr(B)
    y = np.empty((rows_arr.size, N), dtype=np.float64)
    nt = threads if threads is not None else usable_cores()
    st = (lib if lib is not None else _load()).lora_oracle_forward(
        int(rows_arr.size), _ptr(rows_arr), K, N, _ptr(x), _ptr(W), _ptr(ids), S,
        _ptr(ranks), _ptr(alphas), ctypes.addressof(a_ptrs), ctypes.addressof(b_ptrs),
        _ptr(y), int(nt))
    del keep
    if st != 0:
        raise RuntimeError(f"oracle failed with status {st}")
    return y


def workload_forward(wl, p: int = 0, rows: Optional[Sequence[int]] = None,
                     threads: Optional[int] = None) -> np.ndarray:
    """``forward`` on projection ``p`` of a ``workloads.Workload``."""
    ids = wl.row_adapter
    sel = ids if rows is None else ids[np.asarray(rows, dtype=np.int64)]
    used = sorted(set(int(i) for i in sel if i >= 0))
    adapters = {i: wl.adapter(p, i) for i in used}
    return forward(wl.x, wl.projections[p].W, ids, wl.ranks, wl.alphas, adapters,
                   rows=rows, threads=threads)


def rows_from_segments(M: int, seg_offsets: Sequence[int], seg_adapter: Sequence[int],
                       perm: Optional[Sequence[int]] = None) -> np.ndarray:
    """Per-row adapter ids from SGMV segments.

    Rows sorted by adapter ("Adapter Residency…", §"Batch composition under
    many adapters": the batch is reordered so rows sharing an adapter sit next
    to each other) are described by segments: sorted position
    p in [seg_offsets[s], seg_offsets[s+1]) is input row perm[p] (p itself
    when perm is None) and uses slot seg_adapter[s].  Positions outside every
    segment are base-only (-1).
    """
    ids = np.full(M, -1, dtype=np.int32)
    offs = [int(o) for o in seg_offsets]
    for s, a in enumerate(seg_adapter):
        for p in range(offs[s], offs[s + 1]):
            row = p if perm is None else int(perm[p])
            ids[row] = int(a)
    return ids


def segment_rows(ids: Iterable[int], num_slots: int):
    """Stable sort of rows by adapter id -> (perm, seg_offsets, seg_adapter).

    Follows "Adapter Residency…", §"Batch composition under many adapters"
    (before the forward pass the batch is reordered so that the rows of one
    adapter are adjacent) and "S-LoRA: what the paper actually says…",
    §"Batched LoRA computation" (requests ordered by adapter index).  Readings: ascending id with base-only rows (-1) first, ties in
    input order, one segment per id present (the base-only rows form their
    own segment with adapter -1), empty segments omitted.  Raises ValueError
    for ids outside [-1, num_slots).
    """
    ids = [int(i) for i in ids]
    buckets: Dict[int, list] = {}
    for m, i in enumerate(ids):
        if i < -1 or i >= num_slots:
            raise ValueError(f"row {m}: adapter id {i} outside [-1, {num_slots})")
        buckets.setdefault(i, []).append(m)
    perm, offs, adp = [], [0], []
    for i in sorted(buckets):
        perm.extend(buckets[i])
        offs.append(len(perm))
        adp.append(i)
    return (np.asarray(perm, dtype=np.int32), np.asarray(offs, dtype=np.int32),
            np.asarray(adp, dtype=np.int32))


# ---------------------------------------------------------------------------
# Counts the pages work out.
# ---------------------------------------------------------------------------

def lora_params(d: int, k: int, r: int) -> int:
    """Parameters of one adapted d x k projection: B is d x r, A is r x k,
    so r(d + k) ("Adapter Residency…", second paragraph)."""
    return r * d + r * k


def adapter_bytes(d_in: int, d_out: int, rank: int, bytes_per_param: int) -> int:
    """Bytes of one adapted projection, (d_in + d_out) x rank x bytes per
    parameter ("Multi-LoRA Adapter Caching in Production…", §"Adapter
    Capacity Planning Can't Be Based on 'Count' Alone")."""
    return (d_in + d_out) * rank * bytes_per_param


def slot_memory_numbers(max_loras: int, layers: int, modules: int, d: int,
                        max_lora_rank: int) -> int:
    """Numbers held by the GPU adapter slots: max_loras x layers x modules x 2
    x d x max_lora_rank ("LoRA Adapters: Many Models in One", §"What it
    costs"), every slot padded to the maximum rank."""
    return max_loras * layers * modules * 2 * d * max_lora_rank


def blocks_for(nbytes: int, block_bytes: int) -> int:
    """Fixed-size pool blocks covering ``nbytes`` ("S-LoRA: what the paper
    actually says…", §"Unified paging": an 80MB adapter in 256KB blocks)."""
    return -(-nbytes // block_bytes)
