"""lora_linear_forward_noalloc, the forward for callers that cannot allocate
device memory (a framework plugin given no workspace, a process with all of
its memory reserved up front, a loop that must not risk a cudaMalloc).

It must give the same outputs as lora_linear_forward with a caller-provided
workspace, call after call, while using only the library's own fixed scratch
array; and it must refuse a call that needs more scratch than that array.
This file is collected last so that a failure here stops a run only after
every other test has run.
"""

import ctypes

import numpy as np
import pytest
import torch

import lora_harness as H
from adapter_gemm_linear_gb300 import LinearCall, LoraPool, _lib, segment_rows
from workloads import synth

pytestmark = pytest.mark.gpu

NOALLOC_MAX = 16 * 1024 * 1024


def _call_noalloc(call):
    """Issue the prepared arguments through lora_linear_forward_noalloc with
    no workspace at all (the entry point ignores the workspace fields)."""
    args = _lib.ForwardArgs()
    ctypes.pointer(args)[0] = call.args
    args.workspace = None
    args.workspace_bytes = 0
    return _lib.lib().lora_linear_forward_noalloc(ctypes.byref(args),
                                                  torch.cuda.current_stream().cuda_stream)


def _index(wl, mode):
    if mode == "bgmv":
        return dict(row_adapter=torch.from_numpy(wl.row_adapter).cuda())
    perm, offs, adp = segment_rows(wl.row_adapter, wl.num_slots)
    return dict(seg_offsets=torch.from_numpy(offs).cuda(), seg_adapter=torch.from_numpy(adp).cuda(),
                perm=torch.from_numpy(perm).cuda())


# Each case takes a different layout of the scratch memory: the per-row
# LoRA kernel with one correction array per projection (two projections in
# one call); the pipelined grouped kernels (V planes, correction array, split-K
# partial tiles and counters); the large-M path (tile plans, V slices and Vt
# for the two-SM GEMM, the shrink's accumulator for the one-SM GEMM); int8
# and int4 base weights.
CASES = {
    "per_row_two_proj": dict(M=128, K=1024, Ns=[256, 520], rank_choices=(8, 16)),
    "grouped": dict(M=300, K=520, Ns=[392, 136], rank_choices=(1, 7, 16, 33, 64)),
    "pipelined": dict(M=480, K=1600, Ns=[520], rank_choices=(16, 64, 128)),
    "large_m": dict(M=1100, K=512, Ns=[264, 136], rank_choices=(8, 16, 32, 64)),
    "int8_base": dict(M=64, K=1024, Ns=[520], rank_choices=(8, 16), wq=8),
    "int4_base": dict(M=48, K=1024, Ns=[264], rank_choices=(16,), wq=4),
}


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_workspace_entry_point(case, mode):
    """Two calls in a row through the no-alloc entry point give the outputs
    of the workspace entry point (same kernels, so within the parity
    tolerance; in practice the same bits), and both match the oracle."""
    from adapter_gemm_linear_gb300 import Int4Weight, Int8Weight
    kw = dict(CASES[case])
    wq = kw.pop("wq", 0)
    wl = synth(num_slots=7, seed=77 + len(case), zipf_s=1.2, **kw)
    pools = H.make_pools(wl, "cuda")
    x, Ws = H.device_inputs(wl)
    if wq:
        Ws = [(Int8Weight if wq == 8 else Int4Weight).quantize(W) for W in Ws]
        # the oracle takes the dequantized weights as its W
        for p, W in enumerate(Ws):
            q = W.q if wq == 8 else _unpack_int4(W.q)
            wl.projections[p].W = (q.float() * W.scale[:, None]).cpu().numpy().astype(np.float64)
    index = _index(wl, mode)
    ref_outs = [torch.empty((wl.M, p.N), dtype=torch.bfloat16, device="cuda") for p in wl.projections]
    LinearCall(x, list(zip(Ws, pools, ref_outs)), **index)()
    torch.cuda.synchronize()
    refs = [o.double().cpu().numpy() for o in ref_outs]
    for p in range(len(wl.projections)):
        H.assert_close("bf16", refs[p], H.oracle_rows(wl, p), f"workspace entry point {case} {mode} p{p}")

    outs = [torch.empty((wl.M, p.N), dtype=torch.bfloat16, device="cuda") for p in wl.projections]
    call = LinearCall(x, list(zip(Ws, pools, outs)), **index)
    assert call.workspace_bytes <= NOALLOC_MAX
    for _ in range(2):  # two calls in a row share (and reuse) the same scratch
        for o in outs:
            o.fill_(float("nan"))
        assert _call_noalloc(call) == 0
        torch.cuda.synchronize()
        for p, (o, ref) in enumerate(zip(outs, refs)):
            H.assert_close("bf16", o.float().cpu().numpy(), ref, f"noalloc {case} {mode} p{p}")


def _unpack_int4(packed):
    lo = (packed & 0xF).to(torch.int16)
    hi = (packed >> 4).to(torch.int16)
    lo = torch.where(lo >= 8, lo - 16, lo)
    hi = torch.where(hi >= 8, hi - 16, hi)
    return torch.stack([lo, hi], dim=2).reshape(packed.shape[0], -1)


def test_noalloc_refuses_oversized_call():
    M, K = 8192, 64
    pool = LoraPool(K, 64, 1, 1024, 1, device="cuda")  # V alone needs M*1024*4 = 32 MiB
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((64, K), dtype=torch.bfloat16, device="cuda")
    out = torch.full((M, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    ids = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    call = LinearCall(x, [(W, pool, out)], row_adapter=ids)
    assert call.workspace_bytes > NOALLOC_MAX
    assert _call_noalloc(call) == 12  # LORA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
