"""GPU tests of the pool residency path: adapters loaded straight from
page-locked host memory (the scatter kernel reads it over the host link,
asynchronously on the stream), and the LRU bookkeeping that never evicts a
pinned (in-flight) slot.

The forward after a mapped load must equal the forward after a staged host
load bit for bit (same pool layout, same values), and match the oracle.
"""

import ctypes

import numpy as np
import pytest
import torch

import lora_harness as H
from adapter_gemm_linear_gb300 import LoraError, LoraPool, _lib
from workloads import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _pool_like(wl, p, src, stream=None):
    td = H.torch_dtype(wl.dtype)
    pool = LoraPool(wl.K, wl.projections[p].N, wl.num_slots, H.pool_max_rank(wl), wl.blocks_needed(), dtype=td,
                    device=DEV, free_list_seed=wl.free_list_seed + p)
    for s in wl.used_slots:
        A, B = wl.adapter(p, int(s))
        At, Bt = torch.from_numpy(A).to(td), torch.from_numpy(B).to(td)
        if src == "mapped":
            At, Bt = At.pin_memory(), Bt.pin_memory()
        pool.load(int(s), At, Bt, float(wl.alphas[s]), stream=stream, src=src)
    return pool


@pytest.mark.parametrize("shape", [(96, 520, 392), (300, 2056, 1032)])
def test_mapped_host_load_matches_host_load(shape):
    M, K, N = shape
    wl = synth(M=M, K=K, Ns=[N], num_slots=7, rank_choices=(1, 16, 33, 64), seed=M + K, none_frac=0.1)
    host = [_pool_like(wl, 0, "host")]
    torch.cuda.synchronize()
    mapped = [_pool_like(wl, 0, "mapped")]
    torch.cuda.synchronize()
    out_h = H.forward(wl, host, "bgmv")[0]
    out_m = H.forward(wl, mapped, "bgmv")[0]
    assert np.array_equal(out_h, out_m)
    H.assert_close("bf16", out_m, H.oracle_rows(wl, 0), f"mapped {shape}")


def test_mapped_load_is_stream_ordered():
    """Loads issued on a side stream without a host wait; a forward queued
    after them on the same stream sees the adapters."""
    wl = synth(M=128, K=1024, Ns=[520], num_slots=9, rank_choices=(8, 40, 128), seed=5, none_frac=0.05)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        pool = _pool_like(wl, 0, "mapped", stream=side)
        x, Ws = H.device_inputs(wl)
        out = torch.empty((wl.M, 520), dtype=torch.bfloat16, device=DEV)
        from adapter_gemm_linear_gb300 import LinearCall
        ids = torch.from_numpy(np.ascontiguousarray(wl.row_adapter, np.int32)).to(DEV)
        LinearCall(x, [(Ws[0], pool, out)], row_adapter=ids)(side)
    side.synchronize()
    H.assert_close("bf16", out.float().cpu().numpy(), H.oracle_rows(wl, 0), "stream-ordered mapped load")


def test_mapped_load_of_unregistered_host_memory():
    """Host memory that is not page-locked: where the GPU cannot address it
    the C ABI refuses the load (INVALID_ARG) before any access and leaves no
    CUDA error behind; where it can (pageable memory access over NVLink-C2C on
    Grace), the adapter loads like any other.  Either way the pool stays
    consistent and the forward matches the oracle."""
    wl = synth(M=48, K=256, Ns=[136], num_slots=3, rank_choices=(16,), seed=2, none_frac=0.0)
    td = H.torch_dtype(wl.dtype)
    pool = LoraPool(wl.K, 136, wl.num_slots, 16, wl.blocks_needed(), dtype=td, device=DEV)
    refused = []
    for s in wl.used_slots:
        A, B = wl.adapter(0, int(s))
        # pageable numpy copies of the bf16 bits
        An = torch.from_numpy(A).to(td).view(torch.int16).numpy().copy()
        Bn = torch.from_numpy(B).to(td).view(torch.int16).numpy().copy()
        st = _lib.lib().lora_pool_load_slot(pool.handle, int(s), 16, float(wl.alphas[s]),
                                            An.ctypes.data_as(ctypes.c_void_p), Bn.ctypes.data_as(ctypes.c_void_p),
                                            2, int(torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()  # the numpy buffers die with this iteration
        assert st in (0, 1), st
        if st == 1:
            refused.append(int(s))
            assert pool.slot_info(int(s))[0] == 0
            pool.load(int(s), torch.from_numpy(A).to(td), torch.from_numpy(B).to(td), float(wl.alphas[s]))
    assert len(refused) in (0, len(wl.used_slots))  # one behaviour per system
    with pytest.raises(ValueError):  # the Python wrapper asks for page-locked tensors
        pool.load(0, torch.zeros(16, wl.K, dtype=td), torch.zeros(136, 16, dtype=td), 32.0, src="mapped")
    out = H.forward(wl, [pool], "bgmv")[0]
    H.assert_close("bf16", out, H.oracle_rows(wl, 0), f"unregistered host memory (refused: {bool(refused)})")


def test_lru_eviction_respects_pins():
    wl = synth(M=64, K=512, Ns=[264], num_slots=6, rank_choices=(16, 32), seed=11, none_frac=0.0)
    td = H.torch_dtype(wl.dtype)
    pool = LoraPool(wl.K, 264, wl.num_slots, H.pool_max_rank(wl), wl.blocks_needed(), dtype=td, device=DEV)
    for s in range(wl.num_slots):
        A, B = wl.adapter(0, s)
        pool.load(s, torch.from_numpy(A).to(td), torch.from_numpy(B).to(td), float(wl.alphas[s]))
    # use order: 0..5 by load; touch 0 and 1, so 2 is the least recent
    pool.touch(0)
    pool.touch(1)
    pool.pin(2)                       # in flight: protected, and counts as a use
    assert pool.slot_use(2)[1] == 1
    with pytest.raises(LoraError):
        pool.unload(2)                # an in-flight slot is not torn out
    order = [pool.evict_lru() for _ in range(5)]
    assert order == [3, 4, 5, 0, 1]
    with pytest.raises(LoraError):
        pool.evict_lru()              # only the pinned slot is left
    pool.unpin(2)
    with pytest.raises(LoraError):
        pool.unpin(2)                 # no pins left
    assert pool.evict_lru() == 2
    assert pool.free_blocks == wl.blocks_needed()
    assert all(pool.slot_use(s) == (0, 0) for s in range(wl.num_slots))
    # the emptied pool takes the adapters again and serves them correctly
    for s in wl.used_slots:
        A, B = wl.adapter(0, int(s))
        pool.load(int(s), torch.from_numpy(A).to(td), torch.from_numpy(B).to(td), float(wl.alphas[s]))
    out = H.forward(wl, [pool], "bgmv")[0]
    H.assert_close("bf16", out, H.oracle_rows(wl, 0), "after eviction and reload")
