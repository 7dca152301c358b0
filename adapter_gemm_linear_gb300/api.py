"""PyTorch-facing binding of the C ABI: tensors in, pointers out.

Every function here only marshals arguments: torch allocates device memory
and provides the stream, the C library (liblora.so) does all the work.
Names follow include/lora.h without the ``lora_`` prefix.
"""

from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

from . import _lib
from ._lib import LORA_BLOCK_ROWS, LORA_BF16, LORA_FP32, STATUS_NAMES

_TORCH_DTYPE = {LORA_BF16: torch.bfloat16, LORA_FP32: torch.float32}
_LORA_DTYPE = {torch.bfloat16: LORA_BF16, torch.float32: LORA_FP32}


class LoraError(RuntimeError):
    """A C-ABI call returned a status other than LORA_OK."""

    def __init__(self, status: int, what: str):
        self.status = int(status)
        self.name = STATUS_NAMES.get(self.status, str(status))
        msg = _lib.lib().lora_status_string(self.status).decode()
        self.cuda_error = 0
        if self.name == "LORA_ERR_CUDA":
            self.cuda_error = int(_lib.lib().lora_last_cuda_error())
            if self.cuda_error:
                msg += ": " + _lib.lib().lora_cuda_error_name(self.cuda_error).decode()
        super().__init__(f"{what}: {self.name} ({msg})")


def _check(status: int, what: str) -> None:
    if status != 0:
        raise LoraError(status, what)


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def lora_dtype(dtype: torch.dtype) -> int:
    if dtype not in _LORA_DTYPE:
        raise TypeError(f"unsupported dtype {dtype}; use torch.bfloat16 or torch.float32")
    return _LORA_DTYPE[dtype]


def status_string(status: int) -> str:
    return _lib.lib().lora_status_string(int(status)).decode()


def abi_version() -> int:
    return int(_lib.lib().lora_abi_version())


def pool_slot_bytes(K: int, N: int, rank: int, dtype: torch.dtype = torch.bfloat16) -> int:
    return int(_lib.lib().lora_pool_slot_bytes(K, N, rank, lora_dtype(dtype)))


def pool_arena_bytes(K: int, N: int, num_blocks: int, dtype: torch.dtype = torch.bfloat16) -> int:
    return int(_lib.lib().lora_pool_arena_bytes(K, N, num_blocks, lora_dtype(dtype)))


class LoraPool:
    """One projection's paged adapter pool (lora_pool_create & co.).

    Device memory (A-arena [num_blocks, 16, K] and B-arena [num_blocks, N, 16],
    the block table, ranks and scales) is allocated here with torch and handed to the
    library, which keeps only host metadata.
    """

    def __init__(self, K: int, N: int, max_slots: int, max_rank: int, num_blocks: int,
                 dtype: torch.dtype = torch.bfloat16, device=None, free_list_seed: int = 0,
                 stream: Optional[torch.cuda.Stream] = None):
        self.device = torch.device(device if device is not None else "cuda")
        self.dtype = dtype
        self.K, self.N = int(K), int(N)
        self.max_slots, self.max_rank, self.num_blocks = int(max_slots), int(max_rank), int(num_blocks)
        bps = max(1, self.max_rank // LORA_BLOCK_ROWS)
        self.a_arena = torch.empty((num_blocks, LORA_BLOCK_ROWS, K), dtype=dtype, device=self.device)
        self.b_arena = torch.empty((num_blocks, N, LORA_BLOCK_ROWS), dtype=dtype, device=self.device)
        self.block_table = torch.empty((max_slots, bps), dtype=torch.int32, device=self.device)
        self.ranks = torch.empty((max_slots,), dtype=torch.int32, device=self.device)
        self.scales = torch.empty((max_slots,), dtype=torch.float32, device=self.device)
        desc = _lib.PoolDesc(
            lora_dtype(dtype), self.K, self.N, self.max_slots, self.max_rank, self.num_blocks,
            _ptr(self.a_arena), _ptr(self.b_arena), _ptr(self.block_table), _ptr(self.ranks),
            _ptr(self.scales), int(free_list_seed))
        handle = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(_lib.lib().lora_pool_create(ctypes.byref(desc), _stream_handle(stream),
                                               ctypes.byref(handle)), "lora_pool_create")
        self._handle = handle

    @property
    def handle(self) -> int:
        if self._handle is None:
            raise RuntimeError("pool is closed")
        return self._handle.value

    def load(self, slot: int, A: torch.Tensor, B: torch.Tensor, alpha: float,
             stream: Optional[torch.cuda.Stream] = None, src: str = "auto") -> None:
        """lora_pool_load_slot: A [r, K], B [N, r] in the pool dtype.

        src "auto": this pool's device if A is on the GPU, else "host".
        "host": staged copies, synchronous.  "device": a kernel on `stream`.
        "mapped": A and B are page-locked host tensors (pin_memory=True) read
        by that kernel over the host link, asynchronously on `stream`; this
        object keeps them alive until the stream has passed the load.  (The C
        ABI also takes pageable memory where the GPU can address it.)"""
        r = int(A.shape[0])
        if A.shape != (r, self.K) or B.shape != (self.N, r):
            raise ValueError(f"A {tuple(A.shape)} / B {tuple(B.shape)} do not match K={self.K}, N={self.N}")
        if src == "auto":
            src = "device" if A.is_cuda else "host"
        mode = {"host": 0, "device": 1, "mapped": 2}.get(src)
        if mode is None:
            raise ValueError(f"unknown src {src!r}")
        if (mode == 1) != A.is_cuda or A.is_cuda != B.is_cuda:
            raise ValueError("A and B must both be on this pool's device for src='device', else on the host")
        if mode == 2:
            if not (A.dtype == self.dtype and B.dtype == self.dtype and A.is_contiguous() and B.is_contiguous()
                    and A.is_pinned() and B.is_pinned()):
                raise ValueError("src='mapped' needs contiguous page-locked tensors in the pool dtype")
        else:
            A = A.to(self.dtype).contiguous()
            B = B.to(self.dtype).contiguous()
        with torch.cuda.device(self.device):
            st = stream if stream is not None else torch.cuda.current_stream()
            _check(_lib.lib().lora_pool_load_slot(self.handle, int(slot), r, float(alpha), _ptr(A), _ptr(B),
                                                  mode, int(st.cuda_stream)),
                   f"lora_pool_load_slot(slot={slot}, rank={r})")
            if mode == 1:
                A.record_stream(st)
                B.record_stream(st)
            elif mode == 2:
                done = torch.cuda.Event()
                done.record(st)
                self._inflight = [(e, a, b) for e, a, b in getattr(self, "_inflight", []) if not e.query()]
                self._inflight.append((done, A, B))

    # residency bookkeeping (host side): LRU with in-flight pins
    def touch(self, slot: int) -> None:
        _check(_lib.lib().lora_pool_touch(self.handle, int(slot)), f"lora_pool_touch(slot={slot})")

    def pin(self, slot: int) -> None:
        _check(_lib.lib().lora_pool_pin(self.handle, int(slot)), f"lora_pool_pin(slot={slot})")

    def unpin(self, slot: int) -> None:
        _check(_lib.lib().lora_pool_unpin(self.handle, int(slot)), f"lora_pool_unpin(slot={slot})")

    def evict_lru(self, stream: Optional[torch.cuda.Stream] = None) -> int:
        """Unloads the least recently used unpinned slot; returns it."""
        out = ctypes.c_int32(-1)
        with torch.cuda.device(self.device):
            _check(_lib.lib().lora_pool_evict_lru(self.handle, _stream_handle(stream), ctypes.byref(out)),
                   "lora_pool_evict_lru")
        return int(out.value)

    def slot_use(self, slot: int) -> Tuple[int, int]:
        """(last use on the pool's use clock, 0 if empty; in-flight pins)."""
        last, pins = ctypes.c_int64(0), ctypes.c_int32(0)
        _check(_lib.lib().lora_pool_slot_use(self.handle, int(slot), ctypes.byref(last), ctypes.byref(pins)),
               f"lora_pool_slot_use(slot={slot})")
        return int(last.value), int(pins.value)

    def unload(self, slot: int, stream: Optional[torch.cuda.Stream] = None) -> None:
        with torch.cuda.device(self.device):
            _check(_lib.lib().lora_pool_unload_slot(self.handle, int(slot), _stream_handle(stream)),
                   f"lora_pool_unload_slot(slot={slot})")

    def slot_info(self, slot: int) -> Tuple[int, float, List[int]]:
        r = ctypes.c_int32()
        s = ctypes.c_float()
        blocks = (ctypes.c_int32 * self.block_table.shape[1])()
        _check(_lib.lib().lora_pool_slot_info(self.handle, int(slot), ctypes.byref(r), ctypes.byref(s),
                                              blocks), "lora_pool_slot_info")
        return int(r.value), float(s.value), list(blocks)

    @property
    def free_blocks(self) -> int:
        return int(_lib.lib().lora_pool_free_blocks(self.handle))

    def close(self) -> None:
        if getattr(self, "_handle", None) is not None:
            _lib.lib().lora_pool_destroy(self._handle.value)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def segment_rows(ids, num_slots: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """lora_segment_rows on host ids -> (perm, seg_offsets, seg_adapter)."""
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    M = int(ids.size)
    perm = np.empty(max(M, 1), np.int32)
    offs = np.empty(M + 1, np.int32)
    adp = np.empty(max(M, 1), np.int32)
    n = ctypes.c_int32()
    _check(_lib.lib().lora_segment_rows(ids.ctypes.data if M else None, M, int(num_slots),
                                        perm.ctypes.data, offs.ctypes.data, adp.ctypes.data,
                                        ctypes.byref(n)), "lora_segment_rows")
    S = int(n.value)
    return perm[:M].copy(), offs[:S + 1].copy(), adp[:S].copy()


class Int8Weight:
    """A quantized base weight: W[n][k] = q[n][k] * scale[n] (int8 q [N][K]
    row-major, fp32 scale [N]), dequantized inside the GEMM; the adapters
    stay 16-bit ("Your LoRA Adapters Are Thrashing Your GPUs", §02
    "Numerical precision: FP16 adapters on INT4 base models")."""

    def __init__(self, q: torch.Tensor, scale: torch.Tensor):
        if q.dtype != torch.int8 or q.dim() != 2 or not q.is_contiguous():
            raise ValueError("q must be a contiguous int8 [N][K] tensor")
        if scale.dtype != torch.float32 or scale.shape != (q.shape[0],) or not scale.is_contiguous():
            raise ValueError("scale must be a contiguous float32 [N] tensor")
        self.q, self.scale = q, scale

    @staticmethod
    def quantize(W: torch.Tensor) -> "Int8Weight":
        """Symmetric per-row int8 of a float weight: scale = max|W[n]| / 127."""
        Wf = W.float()
        scale = (Wf.abs().amax(dim=1) / 127.0).clamp_min(torch.finfo(torch.float32).tiny)
        q = torch.round(Wf / scale[:, None]).clamp_(-127, 127).to(torch.int8)
        return Int8Weight(q.contiguous(), scale.contiguous())


class Int4Weight:
    """A 4-bit quantized base weight: W[n][k] = q[n][k] * scale[n] with q in
    [-8, 7] packed two per byte (uint8 [N][K/2], element 2j in the low nibble
    of byte j), fp32 scale [N]; dequantized inside the GEMM like Int8Weight."""

    def __init__(self, packed: torch.Tensor, scale: torch.Tensor):
        if packed.dtype != torch.uint8 or packed.dim() != 2 or not packed.is_contiguous():
            raise ValueError("packed must be a contiguous uint8 [N][K/2] tensor")
        if scale.dtype != torch.float32 or scale.shape != (packed.shape[0],) or not scale.is_contiguous():
            raise ValueError("scale must be a contiguous float32 [N] tensor")
        self.q, self.scale = packed, scale

    @staticmethod
    def pack(q: torch.Tensor) -> torch.Tensor:
        """int [N][K] values in [-8, 7] (K even) to the packed uint8 [N][K/2]."""
        if q.shape[1] % 2 or int(q.min()) < -8 or int(q.max()) > 7:
            raise ValueError("need an even K and values in [-8, 7]")
        u = (q.to(torch.int16) & 0xF).to(torch.uint8)
        return (u[:, 0::2] | (u[:, 1::2] << 4)).contiguous()

    @staticmethod
    def quantize(W: torch.Tensor) -> "Int4Weight":
        """Symmetric per-row int4 of a float weight: scale = max|W[n]| / 7."""
        Wf = W.float()
        scale = (Wf.abs().amax(dim=1) / 7.0).clamp_min(torch.finfo(torch.float32).tiny)
        q = torch.round(Wf / scale[:, None]).clamp_(-7, 7).to(torch.int8)
        return Int4Weight(Int4Weight.pack(q), scale.contiguous())


class LinearCall:
    """Prepared arguments of one lora_linear_forward call.

    Building the ctypes argument block once and re-issuing it keeps the
    per-call host cost to one foreign call; the tensors passed in must stay
    alive (this object holds references to them).
    """

    def __init__(self, x: torch.Tensor, projections: Sequence[Tuple[torch.Tensor, LoraPool, torch.Tensor]],
                 row_adapter: Optional[torch.Tensor] = None,
                 seg_offsets: Optional[torch.Tensor] = None, seg_adapter: Optional[torch.Tensor] = None,
                 perm: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 scales: Optional[torch.Tensor] = None):
        if x.dim() != 2 or (x.numel() > 0 and x.stride(1) != 1):
            raise ValueError("x must be a row-major 2-D tensor")
        if (row_adapter is None) == (seg_offsets is None and seg_adapter is None):
            if row_adapter is not None or x.shape[0] > 0:
                raise ValueError("give either row_adapter or (seg_offsets, seg_adapter)")
        dt = lora_dtype(x.dtype)
        if scales is not None and (scales.dtype != torch.float32 or not scales.is_contiguous()):
            raise ValueError("scales must be a contiguous float32 [max_slots] tensor")
        self._keep = [x, row_adapter, seg_offsets, seg_adapter, perm, scales]
        projs = (_lib.Proj * len(projections))()
        for i, (W, pool, out) in enumerate(projections):
            if out.dim() != 2 or (out.numel() > 0 and out.stride(1) != 1):
                raise ValueError("out must be a row-major 2-D tensor")
            ldo = int(out.stride(0)) if out.numel() > 0 else int(out.shape[1])
            if isinstance(W, (Int8Weight, Int4Weight)):
                bits = 4 if isinstance(W, Int4Weight) else 8
                projs[i] = _lib.Proj(_ptr(W.q), pool.handle, _ptr(out), ldo, _ptr(W.scale), bits)
                self._keep += [W.q, W.scale, pool, out]
            else:
                projs[i] = _lib.Proj(_ptr(W), pool.handle, _ptr(out), ldo, None, 0)
                self._keep += [W, pool, out]
        self._projs = projs
        for t in (row_adapter, seg_offsets, seg_adapter, perm):
            if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
                raise ValueError("index tensors must be contiguous int32")
        num_segs = 0 if seg_adapter is None else int(seg_adapter.numel())
        ldx = int(x.stride(0)) if x.numel() > 0 else int(x.shape[1])
        self.args = _lib.ForwardArgs(
            dt, int(x.shape[0]), int(x.shape[1]), _ptr(x), ldx, len(projections),
            ctypes.cast(projs, ctypes.POINTER(_lib.Proj)), _ptr(row_adapter), _ptr(seg_offsets),
            _ptr(seg_adapter), _ptr(perm), num_segs, None, 0, None, 0, _ptr(scales))
        self.n_proj = len(projections)
        need = int(_lib.lib().lora_forward_workspace_bytes(ctypes.byref(self.args)))
        if need == 0:
            # the arguments failed validation: the forward reports why (it
            # validates before touching the device, so nothing is launched)
            st = _lib.lib().lora_linear_forward(ctypes.byref(self.args), None)
            raise LoraError(st if st else 1, "lora_linear_forward")
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
        if workspace.numel() * workspace.element_size() < need:
            raise LoraError(12, f"workspace has {workspace.numel()} bytes, needs {need}")
        self.workspace = workspace
        self.workspace_bytes = need
        self.args.workspace = _ptr(workspace)
        self.args.workspace_bytes = workspace.numel() * workspace.element_size()
        self.device = x.device
        self._fn = _lib.lib().lora_linear_forward
        self._argref = ctypes.byref(self.args)

    def set_stage_events(self, events: Optional[Sequence[torch.cuda.Event]]) -> None:
        """Have the next calls record ``events`` (1 + 2*n_proj timing events)
        at the stage boundaries on the launching stream; None turns it off."""
        if events is None:
            self._events = None
            self.args.stage_events = None
            self.args.num_stage_events = 0
            return
        if len(events) != 1 + 2 * self.n_proj:
            raise ValueError(f"need {1 + 2 * self.n_proj} events")
        handles = []
        for ev in events:
            if not ev.cuda_event:
                ev.record()  # torch creates the event lazily on first record
            handles.append(ev.cuda_event)
        self._events = (events, (ctypes.c_void_p * len(handles))(*handles))
        self.args.stage_events = ctypes.cast(self._events[1], ctypes.POINTER(ctypes.c_void_p))
        self.args.num_stage_events = len(handles)

    def __call__(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        st = self._fn(self._argref, _stream_handle(stream))
        if st != 0:
            raise LoraError(st, "lora_linear_forward")


def kernel_launches() -> int:
    """lora_kernel_launches: kernels the library launched in this process."""
    return int(_lib.lib().lora_kernel_launches())


def linear_forward(x: torch.Tensor, projections, row_adapter=None, seg_offsets=None,
                   seg_adapter=None, perm=None, workspace=None,
                   stream: Optional[torch.cuda.Stream] = None, scales=None) -> None:
    """lora_linear_forward: out_p = x W_p^T + per-row (alpha_i/r_i) B_i (A_i x).

    ``projections`` is a sequence of (W [N, K], LoraPool, out [M, >=N]).
    Rows reach adapters through ``row_adapter`` (device int32 [M], -1 = none)
    or through sorted segments (``seg_offsets``, ``seg_adapter``, optional
    ``perm``; device int32).  ``scales`` (device float32 [max_slots]) replaces
    the pools' own alpha/r for this call.
    """
    LinearCall(x, projections, row_adapter, seg_offsets, seg_adapter, perm, workspace, scales)(stream)


def arm_test_wait_timeout(limit_ns: int) -> None:
    """lora_test_arm_wait_timeout: the next forward's split-K counter waits
    expect an arrival that never comes and give up after ``limit_ns``."""
    _check(_lib.lib().lora_test_arm_wait_timeout(int(limit_ns)), "lora_test_arm_wait_timeout")


def device_status(stream: Optional[torch.cuda.Stream] = None) -> Tuple[int, int]:
    """lora_get_device_status -> (status, detail); clears the word."""
    d = ctypes.c_int32(0)
    st = _lib.lib().lora_get_device_status(_stream_handle(stream), ctypes.byref(d))
    return int(st), int(d.value)
