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


@pytest.mark.parametrize("mode", ["bgmv", "sgmv"])
def test_noalloc_matches_workspace_entry_point(mode):
    wl = synth(M=300, K=520, Ns=[392, 136], num_slots=7, rank_choices=(1, 7, 16, 33, 64), seed=77)
    pools = H.make_pools(wl, "cuda")
    x, Ws = H.device_inputs(wl)
    if mode == "bgmv":
        index = dict(row_adapter=torch.from_numpy(wl.row_adapter).cuda())
    else:
        perm, offs, adp = segment_rows(wl.row_adapter, wl.num_slots)
        index = dict(seg_offsets=torch.from_numpy(offs).cuda(), seg_adapter=torch.from_numpy(adp).cuda(),
                     perm=torch.from_numpy(perm).cuda())
    ref_outs = [torch.empty((wl.M, p.N), dtype=torch.bfloat16, device="cuda") for p in wl.projections]
    LinearCall(x, list(zip(Ws, pools, ref_outs)), **index)()
    torch.cuda.synchronize()
    refs = [o.double().cpu().numpy() for o in ref_outs]

    outs = [torch.empty((wl.M, p.N), dtype=torch.bfloat16, device="cuda") for p in wl.projections]
    call = LinearCall(x, list(zip(Ws, pools, outs)), **index)
    assert call.workspace_bytes <= NOALLOC_MAX
    for _ in range(2):  # two calls in a row share (and reuse) the same scratch
        for o in outs:
            o.fill_(float("nan"))
        assert _call_noalloc(call) == 0
        torch.cuda.synchronize()
        for p, (o, ref) in enumerate(zip(outs, refs)):
            H.assert_close("bf16", o.float().cpu().numpy(), ref, f"noalloc {mode} p{p}")


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
