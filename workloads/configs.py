"""The five synthetic workloads of the multi-adapter LoRA linear layer, two
more for other target modules, and a parametric generator for small parity
cases.

Shapes and distributions follow the workloads described on the pages (see
"S-LoRA: what the paper actually says…", §"Batched LoRA computation"; "LoRA
Adapters: Many Models in One", §"The model runner's part"; "Your LoRA Adapters
Are Thrashing Your GPUs", §02 "Concrete parameter counts for a 70B model"):

==============  ======  ======================================================
name            dtype   shape
==============  ======  ======================================================
tiny_fp32       fp32    x 16x256, W 256x256, 4 slots rank 8, alpha 16
decode_bgmv     bf16    x 64x4096, W 4096x4096, 32 slots rank 16, alpha 32
prefill_sgmv    bf16    x 8192x4096, W 4096x4096, 16 slots rank {8..64}, a=2r
decode_70b_qv   bf16    x 256x8192, W_q 8192x8192 + W_v 1024x8192, 128 slots
slora_mixed     bf16    x 512x5120, W 13824x5120, 2048 slots rank {8..128}
==============  ======  ======================================================

Other target modules (WIDENING_NAMES; "Your LoRA Adapters Are Thrashing Your
GPUs", §02 "Which layers to adapt" and "Concrete parameter counts for a 70B
model"):

=================  ======  ===================================================
decode_70b_qkv     bf16    x 256x8192, W_q 8192x8192, W_k and W_v 1024x8192
                           (GQA) in one call, 64 slots rank 64, alpha 128
prefill_down_proj  bf16    x 4096x13824, W 5120x13824 (K > N: the down
                           projection of the slora_mixed model's FFN), 16
                           slots rank {8..64}, SGMV segments
=================  ======  ===================================================

Value recipe: x ~ N(0, 1); W ~ N(0, variance 1/K); A and B ~ N(0, std 0.02);
bf16 configurations round every drawn value once, to nearest-even, to bf16,
so that every array below holds values that are exact in its dtype.  Arrays
are returned as float32 (exact for both dtypes); ``bf16_bits`` gives the raw
16-bit patterns for upload.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np

CONFIG_NAMES = (
    "tiny_fp32",
    "decode_bgmv",
    "prefill_sgmv",
    "decode_70b_qv",
    "slora_mixed",
)

WIDENING_NAMES = (
    "decode_70b_qkv",
    "prefill_down_proj",
)

_ROOT_SEED = 0


def _rng(*key: int) -> np.random.Generator:
    """A PCG64 stream of its own for every (config, tensor, ...) key."""
    ss = np.random.SeedSequence(_ROOT_SEED, spawn_key=tuple(int(k) for k in key))
    return np.random.Generator(np.random.PCG64(ss))


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even).

    Returns float32 holding bf16-exact values.  Inputs are finite and far from
    the float32 range limits (they are synthetic normals), so no NaN/overflow
    handling is needed.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (u.astype(np.uint32) << 16).view(np.float32).reshape(a.shape)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """The bf16 bit patterns of float32 values that are already bf16-exact."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("array holds values that are not exact in bf16")
    return (u >> 16).astype(np.uint16).reshape(a.shape)


def _quant(a: np.ndarray, dtype: str) -> np.ndarray:
    a = np.asarray(a, dtype=np.float32)
    return bf16_round(a) if dtype == "bf16" else np.ascontiguousarray(a)


def _zipf_rank(rng: np.random.Generator, n: int, s: float, size: int) -> np.ndarray:
    """Popularity ranks 0..n-1 with P(rank k) proportional to (k+1)^-s."""
    k = np.arange(1, n + 1, dtype=np.float64)
    p = k ** (-float(s))
    p /= p.sum()
    return rng.choice(n, size=size, p=p)


def _largest_remainder(raw: Sequence[float], total: int) -> np.ndarray:
    """Scale positive weights to integers summing to ``total``, each >= 1."""
    raw = np.asarray(raw, dtype=np.float64)
    f = raw * (total / raw.sum())
    base = np.floor(f).astype(np.int64)
    rem = int(total - base.sum())
    order = np.argsort(-(f - base), kind="stable")
    base[order[:rem]] += 1
    while (base < 1).any():
        base[int(np.argmin(base))] += 1
        base[int(np.argmax(base))] -= 1
    return base


@dataclasses.dataclass
class Projection:
    """One adapted projection: base weight W [N, K] and its adapters' seeds."""

    name: str
    N: int
    W: np.ndarray  # float32 [N, K], exact in the workload dtype
    key: Tuple[int, ...]  # seed key prefix of this projection's adapters


@dataclasses.dataclass
class Workload:
    """Inputs of one multi-adapter LoRA linear call (one or more projections).

    ``row_adapter[m]`` is the slot of row m, or -1 for base-only rows.  SGMV
    workloads also carry ``seg_offsets``/``seg_adapter`` describing rows that
    are already sorted by adapter (segment s covers rows
    ``seg_offsets[s]:seg_offsets[s+1]`` and uses slot ``seg_adapter[s]``).
    """

    name: str
    dtype: str  # "bf16" | "fp32"
    M: int
    K: int
    x: np.ndarray  # float32 [M, K]
    projections: List[Projection]
    num_slots: int
    ranks: np.ndarray  # int32 [num_slots]
    alphas: np.ndarray  # float32 [num_slots]
    row_adapter: np.ndarray  # int32 [M]
    mode: str  # "bgmv" | "sgmv"
    seg_offsets: Optional[np.ndarray] = None  # int32 [S+1]
    seg_adapter: Optional[np.ndarray] = None  # int32 [S]
    integer: bool = False
    a_std: float = 0.02
    b_std: float = 0.02
    free_list_seed: int = 0
    description: str = ""

    @property
    def used_slots(self) -> np.ndarray:
        ids = self.row_adapter
        return np.unique(ids[ids >= 0]).astype(np.int32)

    def adapter(self, p: int, slot: int) -> Tuple[np.ndarray, np.ndarray]:
        """(A [r, K], B [N, r]) of ``slot`` in projection ``p``, float32.

        Each (projection, slot) pair draws from its own stream, so any subset
        of slots can be produced without producing the rest.
        """
        proj = self.projections[p]
        r = int(self.ranks[slot])
        rng = _rng(*proj.key, int(slot))
        if self.integer:
            A = rng.integers(-2, 3, size=(r, self.K)).astype(np.float32)
            B = rng.integers(-2, 3, size=(proj.N, r)).astype(np.float32)
        else:
            A = rng.standard_normal((r, self.K), dtype=np.float32) * np.float32(self.a_std)
            B = rng.standard_normal((proj.N, r), dtype=np.float32) * np.float32(self.b_std)
        return _quant(A, self.dtype), _quant(B, self.dtype)

    def blocks_needed(self, block_rows: int = 16) -> int:
        """Pool blocks for every slot at its own rank (no padding to max)."""
        return int(sum(-(-int(r) // block_rows) for r in self.ranks))

    @property
    def max_rank(self) -> int:
        return int(self.ranks.max())


def _normal(rng, shape, std, dtype):
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return _quant(a, dtype)


def make_config(name_or_index) -> Workload:
    """Build one of the named workloads (deterministic, seed 0): the five of
    CONFIG_NAMES (by name or index 0-4) or one of WIDENING_NAMES (by name, or
    index 5 on)."""
    names = CONFIG_NAMES + WIDENING_NAMES
    idx = name_or_index if isinstance(name_or_index, int) else names.index(name_or_index)
    builder = [_tiny_fp32, _decode_bgmv, _prefill_sgmv, _decode_70b_qv, _slora_mixed,
               _decode_70b_qkv, _prefill_down_proj][idx]
    return builder(idx)


def _tiny_fp32(c: int) -> Workload:
    M, K, N, S = 16, 256, 256, 4
    x = _normal(_rng(c, 0), (M, K), 1.0, "fp32")
    W = _normal(_rng(c, 1), (N, K), 1.0 / np.sqrt(K), "fp32")
    ids = _rng(c, 2).integers(-1, S, size=M).astype(np.int32)
    return Workload(
        name="tiny_fp32", dtype="fp32", M=M, K=K, x=x,
        projections=[Projection("proj", N, W, (c, 100))],
        num_slots=S, ranks=np.full(S, 8, np.int32), alphas=np.full(S, 16.0, np.float32),
        row_adapter=ids, mode="bgmv", free_list_seed=0x5EED0 + c,
        description="tiny fp32: x 16x256, W 256x256, 4 slots rank 8, alpha 16, ids uniform over {-1..3}",
    )


def _decode_bgmv(c: int) -> Workload:
    M, K, N, S = 64, 4096, 4096, 32
    x = _normal(_rng(c, 0), (M, K), 1.0, "bf16")
    W = _normal(_rng(c, 1), (N, K), 1.0 / np.sqrt(K), "bf16")
    rid = _rng(c, 2)
    none_rows = rid.choice(M, size=int(round(0.1 * M)), replace=False)
    slot_of_rank = rid.permutation(S)
    ids = slot_of_rank[_zipf_rank(rid, S, 1.2, M)].astype(np.int32)
    ids[none_rows] = -1
    return Workload(
        name="decode_bgmv", dtype="bf16", M=M, K=K, x=x,
        projections=[Projection("q_proj", N, W, (c, 100))],
        num_slots=S, ranks=np.full(S, 16, np.int32), alphas=np.full(S, 32.0, np.float32),
        row_adapter=ids, mode="bgmv", free_list_seed=0x5EED0 + c,
        description="decode BGMV: bf16 4096->4096, 64 rows, 32 slots rank 16 alpha 32, "
                    "ids Zipf(1.2), 6 rows base-only",
    )


def _prefill_sgmv(c: int) -> Workload:
    M, K, N, S = 8192, 4096, 4096, 16
    x = _normal(_rng(c, 0), (M, K), 1.0, "bf16")
    W = _normal(_rng(c, 1), (N, K), 1.0 / np.sqrt(K), "bf16")
    rr = _rng(c, 2)
    ranks = rr.choice(np.array([8, 16, 32, 64]), size=S).astype(np.int32)
    lengths = _largest_remainder(rr.geometric(1.0 / 512.0, size=S), M)
    seg_offsets = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    seg_adapter = np.arange(S, dtype=np.int32)
    ids = np.repeat(seg_adapter, lengths).astype(np.int32)
    return Workload(
        name="prefill_sgmv", dtype="bf16", M=M, K=K, x=x,
        projections=[Projection("proj", N, W, (c, 100))],
        num_slots=S, ranks=ranks, alphas=(2.0 * ranks).astype(np.float32),
        row_adapter=ids, mode="sgmv", seg_offsets=seg_offsets, seg_adapter=seg_adapter,
        free_list_seed=0x5EED0 + c,
        description="prefill SGMV: bf16 4096->4096, 8192 tokens in 16 sorted segments "
                    "(geometric lengths, mean 512), ranks {8,16,32,64}, alpha 2r",
    )


def _decode_70b_qv(c: int) -> Workload:
    M, K, S = 256, 8192, 128
    x = _normal(_rng(c, 0), (M, K), 1.0, "bf16")
    Wq = _normal(_rng(c, 1), (8192, K), 1.0 / np.sqrt(K), "bf16")
    Wv = _normal(_rng(c, 3), (1024, K), 1.0 / np.sqrt(K), "bf16")
    rid = _rng(c, 2)
    slot_of_rank = rid.permutation(S)
    ids = slot_of_rank[_zipf_rank(rid, S, 1.1, M)].astype(np.int32)
    return Workload(
        name="decode_70b_qv", dtype="bf16", M=M, K=K, x=x,
        projections=[Projection("q_proj", 8192, Wq, (c, 100)),
                     Projection("v_proj", 1024, Wv, (c, 101))],
        num_slots=S, ranks=np.full(S, 16, np.int32), alphas=np.full(S, 32.0, np.float32),
        row_adapter=ids, mode="bgmv", free_list_seed=0x5EED0 + c,
        description="70B-shaped decode: bf16 hidden 8192, q 8192->8192 and v 8192->1024 in "
                    "one call, 256 rows, 128 slots rank 16 alpha 32, ids Zipf(1.1)",
    )


def _slora_mixed(c: int) -> Workload:
    M, K, N, S = 512, 5120, 13824, 2048
    x = _normal(_rng(c, 0), (M, K), 1.0, "bf16")
    W = _normal(_rng(c, 1), (N, K), 1.0 / np.sqrt(K), "bf16")
    rr = _rng(c, 2)
    ranks = rr.choice(np.array([8, 16, 32, 64, 128]), size=S).astype(np.int32)
    declared = rr.choice(S, size=200, replace=False).astype(np.int32)
    none_rows = rr.choice(M, size=int(round(0.05 * M)), replace=False)
    ids = declared[_zipf_rank(rr, 200, 1.0, M)].astype(np.int32)
    ids[none_rows] = -1
    return Workload(
        name="slora_mixed", dtype="bf16", M=M, K=K, x=x,
        projections=[Projection("up_proj", N, W, (c, 100))],
        num_slots=S, ranks=ranks, alphas=(2.0 * ranks).astype(np.float32),
        row_adapter=ids, mode="bgmv", free_list_seed=0x5EED0 + c,
        description="S-LoRA-scale mixed batch: bf16 5120->13824, 2048 slots ranks "
                    "{8..128} alpha 2r, 512 rows over 200 adapters (power law s=1.0), "
                    "26 rows base-only",
    )


def _decode_70b_qkv(c: int) -> Workload:
    M, K, S = 256, 8192, 64
    x = _normal(_rng(c, 0), (M, K), 1.0, "bf16")
    Wq = _normal(_rng(c, 1), (8192, K), 1.0 / np.sqrt(K), "bf16")
    Wk = _normal(_rng(c, 3), (1024, K), 1.0 / np.sqrt(K), "bf16")
    Wv = _normal(_rng(c, 4), (1024, K), 1.0 / np.sqrt(K), "bf16")
    rid = _rng(c, 2)
    none_rows = rid.choice(M, size=int(round(0.05 * M)), replace=False)
    slot_of_rank = rid.permutation(S)
    ids = slot_of_rank[_zipf_rank(rid, S, 1.1, M)].astype(np.int32)
    ids[none_rows] = -1
    return Workload(
        name="decode_70b_qkv", dtype="bf16", M=M, K=K, x=x,
        projections=[Projection("q_proj", 8192, Wq, (c, 100)),
                     Projection("k_proj", 1024, Wk, (c, 101)),
                     Projection("v_proj", 1024, Wv, (c, 102))],
        num_slots=S, ranks=np.full(S, 64, np.int32), alphas=np.full(S, 128.0, np.float32),
        row_adapter=ids, mode="bgmv", free_list_seed=0x5EED0 + c,
        description="70B-shaped decode, rank-64 Q+K+V adapters: bf16 hidden 8192, q 8192->8192, "
                    "k and v 8192->1024 (GQA) in one call, 256 rows, 64 slots alpha 128, "
                    "ids Zipf(1.1), 13 rows base-only",
    )


def _prefill_down_proj(c: int) -> Workload:
    M, K, N, S = 4096, 13824, 5120, 16
    x = _normal(_rng(c, 0), (M, K), 1.0, "bf16")
    W = _normal(_rng(c, 1), (N, K), 1.0 / np.sqrt(K), "bf16")
    rr = _rng(c, 2)
    ranks = rr.choice(np.array([8, 16, 32, 64]), size=S).astype(np.int32)
    lengths = _largest_remainder(rr.geometric(1.0 / 256.0, size=S), M)
    seg_offsets = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    seg_adapter = np.arange(S, dtype=np.int32)
    ids = np.repeat(seg_adapter, lengths).astype(np.int32)
    return Workload(
        name="prefill_down_proj", dtype="bf16", M=M, K=K, x=x,
        projections=[Projection("down_proj", N, W, (c, 100))],
        num_slots=S, ranks=ranks, alphas=(2.0 * ranks).astype(np.float32),
        row_adapter=ids, mode="sgmv", seg_offsets=seg_offsets, seg_adapter=seg_adapter,
        free_list_seed=0x5EED0 + c,
        description="prefill SGMV of a down projection (K > N): bf16 13824->5120, 4096 tokens "
                    "in 16 sorted segments (geometric lengths, mean 256), ranks {8,16,32,64}, alpha 2r",
    )


def synth(
    name: str = "synth",
    *,
    M: int,
    K: int,
    Ns: Sequence[int],
    num_slots: int,
    rank_choices: Sequence[int] = (16,),
    dtype: str = "bf16",
    integer: bool = False,
    seed: int = 1,
    none_frac: float = 0.1,
    mode: str = "bgmv",
    zipf_s: Optional[float] = None,
    alpha_mode: str = "2r",
) -> Workload:
    """A small parametric workload for parity and edge-case tests.

    ``integer=True`` draws x, W, A, B from {-2..2} with alpha = 2r (scale 2),
    so every product and partial sum is an integer far below 2^24: any
    correct evaluation order in fp32 or float64 gives the same exact value.
    ``mode="sgmv"`` sorts rows by adapter (stable, base-only rows first) and
    emits one segment per run of equal ids, the base-only run included (its
    ``seg_adapter`` entry is -1).
    """
    key = (1000 + int(seed),)
    rx, rw, rid = _rng(*key, 0), _rng(*key, 1), _rng(*key, 2)
    if integer:
        x = rx.integers(-2, 3, size=(M, K)).astype(np.float32)
        Ws = [_rng(*key, 10 + i).integers(-2, 3, size=(n, K)).astype(np.float32)
              for i, n in enumerate(Ns)]
    else:
        x = _normal(rx, (M, K), 1.0, dtype)
        Ws = [_normal(_rng(*key, 10 + i), (n, K), 1.0 / np.sqrt(K), dtype)
              for i, n in enumerate(Ns)]
    ranks = rid.choice(np.asarray(rank_choices), size=num_slots).astype(np.int32)
    if alpha_mode == "2r":
        alphas = (2.0 * ranks).astype(np.float32)
    elif alpha_mode == "16":
        alphas = np.full(num_slots, 16.0, np.float32)
    else:
        raise ValueError(alpha_mode)
    if num_slots > 0:
        if zipf_s is None:
            ids = rid.integers(0, num_slots, size=M).astype(np.int32)
        else:
            ids = rid.permutation(num_slots)[_zipf_rank(rid, num_slots, zipf_s, M)].astype(np.int32)
        n_none = int(round(none_frac * M))
        if n_none:
            ids[rid.choice(M, size=n_none, replace=False)] = -1
    else:
        ids = np.full(M, -1, np.int32)
    seg_offsets = seg_adapter = None
    if mode == "sgmv":
        order = np.argsort(ids, kind="stable")
        x = np.ascontiguousarray(x[order])
        ids = np.ascontiguousarray(ids[order])
        bounds = [0] + [m for m in range(1, M) if ids[m] != ids[m - 1]] + [M]
        segs = [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)] if M > 0 else []
        seg_offsets = np.array([a for a, _ in segs] + ([segs[-1][1]] if segs else [0]), np.int32)
        seg_adapter = np.array([ids[a] for a, _ in segs], np.int32)
    return Workload(
        name=name, dtype=dtype, M=M, K=K, x=x,
        projections=[Projection(f"p{i}", n, W, key + (100 + i,)) for i, (n, W) in enumerate(zip(Ns, Ws))],
        num_slots=num_slots, ranks=ranks, alphas=alphas, row_adapter=ids, mode=mode,
        seg_offsets=seg_offsets, seg_adapter=seg_adapter, integer=integer,
        free_list_seed=0xB10C + int(seed),
        description=f"synthetic M={M} K={K} N={list(Ns)} slots={num_slots} ranks={list(rank_choices)}",
    )
