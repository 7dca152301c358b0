"""GPU parity of the quantized base: int8 or packed int4 W with one fp32
scale per output row, dequantized inside the GEMM, adapters in bf16 ("Your LoRA Adapters Are
Thrashing Your GPUs", §02 "Numerical precision: FP16 adapters on INT4 base
models").  The oracle takes the dequantized weight q[n][k] * scale[n]."""

import numpy as np
import pytest
import torch

import lora_harness as H
import oracle
from adapter_gemm_linear_gb300 import Int4Weight, Int8Weight, LoraError
from workloads import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _quantize(W: np.ndarray, pow2: bool = False):
    """Symmetric per-row int8 (numpy, on the workload's own W): scale =
    max|W[n]| / 127, or the power of two at or above it."""
    amax = np.maximum(np.abs(W).max(axis=1), 1e-30).astype(np.float64)
    s = amax / 127.0
    if pow2:
        s = 2.0 ** np.ceil(np.log2(s))
    s = s.astype(np.float32)
    q = np.clip(np.rint(W / s[:, None]), -127, 127).astype(np.int8)
    return q, s


def _oracle(wl, p, deq, rows=None):
    ids = wl.row_adapter
    sel = ids if rows is None else ids[np.asarray(rows)]
    used = sorted(set(int(i) for i in sel if i >= 0))
    adapters = {i: wl.adapter(p, i) for i in used}
    return oracle.forward(wl.x, deq, ids, wl.ranks, wl.alphas, adapters, rows=rows)


def _int8_weights(qs):
    return [Int8Weight(torch.from_numpy(q).to(DEV), torch.from_numpy(s).to(DEV)) for q, s in qs]


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
@pytest.mark.parametrize("shape", [(64, 4096, 4096), (16, 1024, 520), (48, 2048, 1032), (64, 512, 8)])
def test_int8_base_matches_oracle(shape, mode):
    M, K, N = shape
    wl = synth(M=M, K=K, Ns=[N], num_slots=9, rank_choices=(8, 16, 64), seed=M + K + N, none_frac=0.1, mode=mode)
    qs = [_quantize(p.W) for p in wl.projections]
    pools = H.make_pools(wl, DEV)
    x, _ = H.device_inputs(wl, DEV)
    out = H.forward(wl, pools, mode, x=x, Ws=_int8_weights(qs))[0]
    q, s = qs[0]
    deq = (q.astype(np.float64) * s.astype(np.float64)[:, None]).astype(np.float32)
    H.assert_close("bf16", out, _oracle(wl, 0, deq), f"int8 W {shape} {mode}")


@pytest.mark.parametrize("shape", [(64, 1024, 1032), (30, 768, 264)])
def test_int8_base_integer_exact(shape):
    """Integer x, A, B, int8 q in [-100, 100] and power-of-two scales: every
    sum is exact, so the output equals the oracle's bit for bit."""
    M, K, N = shape
    wl = synth(M=M, K=K, Ns=[N], num_slots=5, rank_choices=(8, 16, 32), integer=True, seed=M + N, none_frac=0.1)
    rng = np.random.default_rng(M * K + N)
    q = rng.integers(-100, 101, size=(N, K)).astype(np.int8)
    s = (2.0 ** rng.integers(-3, 2, size=N)).astype(np.float32)
    pools = H.make_pools(wl, DEV)
    x, _ = H.device_inputs(wl, DEV)
    out = H.forward(wl, pools, "bgmv", x=x, Ws=_int8_weights([(q, s)]))[0]
    deq = (q.astype(np.float64) * s.astype(np.float64)[:, None]).astype(np.float32)
    want = H.oracle_bf16_bits(_oracle(wl, 0, deq))
    got = torch.from_numpy(out).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want), f"{shape}: {np.sum(got != want)} outputs differ"


def test_int8_and_bf16_projections_in_one_call():
    """q in int8, v in bf16, sharing x and the row ids."""
    wl = synth(M=64, K=2048, Ns=[2048, 520], num_slots=7, rank_choices=(16,), seed=3, none_frac=0.1)
    q, s = _quantize(wl.projections[0].W)
    pools = H.make_pools(wl, DEV)
    x, Ws = H.device_inputs(wl, DEV)
    outs = H.forward(wl, pools, "bgmv", x=x, Ws=[_int8_weights([(q, s)])[0], Ws[1]])
    deq = (q.astype(np.float64) * s.astype(np.float64)[:, None]).astype(np.float32)
    H.assert_close("bf16", outs[0], _oracle(wl, 0, deq), "int8 q")
    H.assert_close("bf16", outs[1], H.oracle_rows(wl, 1), "bf16 v")


def test_int8_base_unsupported_shapes():
    """Rows beyond the decode orientation, or K not a multiple of 16: the call
    is refused before any launch."""
    wl = synth(M=96, K=512, Ns=[256], num_slots=3, rank_choices=(16,), seed=9, none_frac=0.0)
    pools = H.make_pools(wl, DEV)
    x, _ = H.device_inputs(wl, DEV)
    with pytest.raises(LoraError) as e:
        H.forward(wl, pools, "bgmv", x=x, Ws=_int8_weights([_quantize(wl.projections[0].W)]))
    assert e.value.status == 13  # LORA_ERR_UNSUPPORTED
    wl2 = synth(M=32, K=520, Ns=[256], num_slots=3, rank_choices=(16,), seed=10, none_frac=0.0)
    pools2 = H.make_pools(wl2, DEV)
    x2, _ = H.device_inputs(wl2, DEV)
    with pytest.raises(LoraError) as e:
        H.forward(wl2, pools2, "bgmv", x=x2, Ws=_int8_weights([_quantize(wl2.projections[0].W)]))
    assert e.value.status == 2  # LORA_ERR_ALIGNMENT


def _pack4(q: np.ndarray) -> np.ndarray:
    """int [N][K] in [-8, 7] to bytes [N][K/2], element 2j in the low nibble."""
    u = (q.astype(np.int16) & 0xF).astype(np.uint8)
    return np.ascontiguousarray(u[:, 0::2] | (u[:, 1::2] << 4))


def _int4_weights(qs):
    return [Int4Weight(torch.from_numpy(_pack4(q)).to(DEV), torch.from_numpy(s).to(DEV)) for q, s in qs]


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
@pytest.mark.parametrize("shape", [(64, 4096, 4096), (16, 1024, 520), (48, 2080, 1032)])
def test_int4_base_matches_oracle(shape, mode):
    M, K, N = shape
    wl = synth(M=M, K=K, Ns=[N], num_slots=9, rank_choices=(8, 16, 64), seed=M + K + N + 4, none_frac=0.1,
               mode=mode)
    W = wl.projections[0].W
    s = (np.maximum(np.abs(W).max(axis=1), 1e-30) / 7.0).astype(np.float32)
    q = np.clip(np.rint(W / s[:, None]), -7, 7).astype(np.int8)
    pools = H.make_pools(wl, DEV)
    x, _ = H.device_inputs(wl, DEV)
    out = H.forward(wl, pools, mode, x=x, Ws=_int4_weights([(q, s)]))[0]
    deq = (q.astype(np.float64) * s.astype(np.float64)[:, None]).astype(np.float32)
    H.assert_close("bf16", out, _oracle(wl, 0, deq), f"int4 W {shape} {mode}")


@pytest.mark.parametrize("shape", [(64, 1024, 1032), (30, 96, 264)])
def test_int4_base_integer_exact(shape):
    """Integer x, A, B, int4 q over all of [-8, 7] (K = 96 leaves a ragged last
    k-block) and power-of-two scales: the output equals the oracle's bit for
    bit."""
    M, K, N = shape
    wl = synth(M=M, K=K, Ns=[N], num_slots=5, rank_choices=(8, 16, 32), integer=True, seed=M + N + 4,
               none_frac=0.1)
    rng = np.random.default_rng(M * K + N + 4)
    q = rng.integers(-8, 8, size=(N, K)).astype(np.int8)
    s = (2.0 ** rng.integers(-3, 2, size=N)).astype(np.float32)
    pools = H.make_pools(wl, DEV)
    x, _ = H.device_inputs(wl, DEV)
    out = H.forward(wl, pools, "bgmv", x=x, Ws=_int4_weights([(q, s)]))[0]
    deq = (q.astype(np.float64) * s.astype(np.float64)[:, None]).astype(np.float32)
    want = H.oracle_bf16_bits(_oracle(wl, 0, deq))
    got = torch.from_numpy(out).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want), f"{shape}: {np.sum(got != want)} outputs differ"


def test_int4_base_needs_k_multiple_of_32():
    wl = synth(M=32, K=528, Ns=[256], num_slots=3, rank_choices=(16,), seed=12, none_frac=0.0)
    pools = H.make_pools(wl, DEV)
    x, _ = H.device_inputs(wl, DEV)
    q = np.zeros((256, 528), np.int8)
    s = np.ones(256, np.float32)
    with pytest.raises(LoraError) as e:
        H.forward(wl, pools, "bgmv", x=x, Ws=_int4_weights([(q, s)]))
    assert e.value.status == 2  # LORA_ERR_ALIGNMENT
