"""The C-ABI library on the host (no GPU needed): it builds, loads, exports
every entry point include/lora.h declares, and its host-only logic (row
segmenter, byte counts, argument validation) is right."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from adapter_gemm_linear_gb300 import build
    from adapter_gemm_linear_gb300 import _lib
    build()
    return _lib.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "lora.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    from adapter_gemm_linear_gb300 import _lib
    declared = _declared_functions()
    assert len(declared) >= 15
    for name in declared:
        assert hasattr(L, name), f"{name} not exported"
    assert sorted(n for n, _, _ in _lib.SIGNATURES) == declared


def test_abi_version_and_status_strings(L):
    assert L.lora_abi_version() == 5
    from adapter_gemm_linear_gb300._lib import STATUS_NAMES
    texts = {L.lora_status_string(c).decode() for c in STATUS_NAMES}
    assert len(texts) == len(STATUS_NAMES) and all(texts)


def test_slot_bytes_matches_oracle_counts(L):
    for K, N, r in [(4096, 4096, 16), (8192, 1024, 16), (5120, 13824, 128), (256, 256, 8)]:
        assert L.lora_pool_slot_bytes(K, N, r, 0) == oracle.adapter_bytes(K, N, r, 2)
        assert L.lora_pool_slot_bytes(K, N, r, 1) == oracle.adapter_bytes(K, N, r, 4)
    assert L.lora_pool_slot_bytes(0, 8, 8, 0) == 0
    # 16 rank-rows of a K = 8192 bf16 arena: the 256 KiB block of the pages
    assert L.lora_pool_arena_bytes(8192, 8, 1, 0) == 16 * (8192 + 8) * 2


@pytest.mark.parametrize("seed,M,S", [(0, 0, 3), (1, 1, 1), (2, 64, 32), (3, 8192, 16), (4, 512, 2048)])
def test_segmenter_bit_exact_vs_oracle(L, seed, M, S):
    from adapter_gemm_linear_gb300 import segment_rows
    rng = np.random.default_rng(seed)
    ids = rng.integers(-1, S, size=M).astype(np.int32)
    got = segment_rows(ids, S)
    want = oracle.segment_rows(ids, S)
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


def test_segmenter_rejects_bad_ids(L):
    from adapter_gemm_linear_gb300 import LoraError, segment_rows
    for bad in ([0, 3], [-2, 0], [7]):
        with pytest.raises(LoraError) as e:
            segment_rows(np.array(bad, np.int32), 3)
        assert e.value.status == 7


def test_pool_create_validation_without_device(L):
    from adapter_gemm_linear_gb300._lib import PoolDesc
    out = ctypes.c_void_p()
    assert L.lora_pool_create(None, None, ctypes.byref(out)) == 1

    def desc(**kw):
        d = dict(dtype=0, K=64, N=64, max_slots=4, max_rank=16, num_blocks=8,
                 a_arena=0x10000, b_arena=0x20000, block_table=0x30000, ranks=0x40000,
                 scales=0x50000, free_list_seed=0)
        d.update(kw)
        return PoolDesc(**d)

    assert L.lora_pool_create(ctypes.byref(desc(a_arena=None)), None, ctypes.byref(out)) == 1
    assert L.lora_pool_create(ctypes.byref(desc(b_arena=0x20008)), None, ctypes.byref(out)) == 2
    assert L.lora_pool_create(ctypes.byref(desc(K=60)), None, ctypes.byref(out)) == 2
    assert L.lora_pool_create(ctypes.byref(desc(max_rank=20)), None, ctypes.byref(out)) == 4
    assert L.lora_pool_create(ctypes.byref(desc(max_rank=2048)), None, ctypes.byref(out)) == 4
    assert L.lora_pool_create(ctypes.byref(desc(dtype=5)), None, ctypes.byref(out)) == 3
    assert L.lora_pool_create(ctypes.byref(desc(num_blocks=0)), None, ctypes.byref(out)) == 1
    assert out.value is None


def test_forward_validation_without_device(L):
    from adapter_gemm_linear_gb300._lib import ForwardArgs, Proj
    projs = (Proj * 1)(Proj(0x1000, None, 0x2000, 64, None, 0))

    def args(**kw):
        d = dict(dtype=0, M=4, K=64, x=0x3000, ldx=64, n_proj=1,
                 proj=ctypes.cast(projs, ctypes.POINTER(Proj)), row_adapter=0x4000,
                 seg_offsets=None, seg_adapter=None, perm=None, num_segs=0,
                 workspace=None, workspace_bytes=0, stage_events=None, num_stage_events=0)
        d.update(kw)
        return ForwardArgs(**d)

    fwd = L.lora_linear_forward
    assert fwd(None, None) == 1
    assert fwd(ctypes.byref(args(n_proj=0)), None) == 1
    assert fwd(ctypes.byref(args(n_proj=5)), None) == 1
    assert fwd(ctypes.byref(args(dtype=9)), None) == 3
    assert fwd(ctypes.byref(args(K=60, ldx=60)), None) == 2
    assert fwd(ctypes.byref(args(ldx=32)), None) == 1
    assert fwd(ctypes.byref(args(x=0x3004)), None) == 2
    assert fwd(ctypes.byref(args(M=-1)), None) == 1
    # pool missing in the projection
    assert fwd(ctypes.byref(args()), None) == 1
    # both index forms at once
    assert fwd(ctypes.byref(args(seg_offsets=0x5000, num_segs=1)), None) == 1
    assert L.lora_forward_workspace_bytes(ctypes.byref(args())) == 0
    # stage events: count must be 1 + 2*n_proj
    assert fwd(ctypes.byref(args(num_stage_events=2)), None) == 1
    # per-call scales must be 16-byte aligned like every device pointer
    assert fwd(ctypes.byref(args(scales=0x6004)), None) == 2
    assert L.lora_kernel_launches() == 0


def test_wait_timeout_hook_range(L):
    """The test hook accepts limits of 1 ms to 2 s, and 0 to disarm (left
    disarmed here, so that no later forward in this process is affected)."""
    assert L.lora_test_arm_wait_timeout(999_999) == 1
    assert L.lora_test_arm_wait_timeout(2_000_000_001) == 1
    assert L.lora_test_arm_wait_timeout(50_000_000) == 0
    assert L.lora_test_arm_wait_timeout(0) == 0
