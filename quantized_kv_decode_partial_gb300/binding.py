"""Thin Python binding of libpkvdecode.so (include/pkv_decode.h).

Argument marshalling only: shapes are read off the tensors, pointers and the
current CUDA stream are passed through, and PyTorch allocates the output and
the workspace. Every step of the computation runs in the library's kernels;
there is no fallback, and a missing library raises ``LibraryNotBuilt``.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB_PATH

EXPORTS = (
    "pkv_make_plan",
    "pkv_plan_for_current_device",
    "pkv_paged_decode_attention",
    "pkv_paged_decode_partial",
    "pkv_merge_partitions",
    "pkv_paged_decode_attention_no_alloc",
    "pkv_paged_decode_attention_host",
    "pkv_step_create",
    "pkv_step_run",
    "pkv_step_destroy",
    "pkv_paged_decode_append_attention",
    "pkv_paged_append",
    "pkv_paged_gather",
    "pkv_strerror",
    "pkv_last_cuda_error",
    "pkv_set_wait_limit_ns",
    "pkv_version",
)

PKV_OK = 0
PKV_ERR_NULL_POINTER = -1
PKV_ERR_MISALIGNED = -2
PKV_ERR_BAD_LAYOUT = -3
PKV_ERR_BAD_PARAMS = -4
PKV_ERR_UNSUPPORTED_SHAPE = -5
PKV_ERR_WORKSPACE_TOO_SMALL = -6
PKV_ERR_CUDA = -7
PKV_ERR_SCRATCH_TOO_SMALL = -8
PKV_STATIC_SCRATCH_BYTES = 16 << 20

PKV_CONTRACTION_AUTO = 0
PKV_CONTRACTION_TENSOR = 1
PKV_CONTRACTION_CUDA_CORE = 2

PKV_SCHEDULE_AUTO = 0
PKV_SCHEDULE_PARTITIONS = 1
PKV_SCHEDULE_BALANCED = 2

PKV_DEVERR_BAD_BLOCK = 1
PKV_DEVERR_BAD_SEQ_LEN = 2
PKV_DEVERR_TIMEOUT = 4


class LibraryNotBuilt(RuntimeError):
    pass


class PkvError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"pkv error {code}: {message}")
        self.code = code


class PoolLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("num_blocks", "num_kv_heads", "block_size", "head_dim", "bits", "group_size", "v_head_dim")]


class DecodeParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("num_seqs", "num_q_heads", "n_query", "max_blocks_per_seq", "partition_tokens", "window",
                 "contraction", "schedule")]


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("partition_tokens", "max_partitions", "chunk_rows", "sm_count", "threads_per_cta",
                 "smem_bytes", "merge_in_cluster", "contraction")] + [("workspace_bytes", ctypes.c_size_t),
                                                                      ("balanced", ctypes.c_int32)]


_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads (once) and returns the library with its prototypes declared."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise LibraryNotBuilt(f"{path} is missing: run __graft_entry__.build() or "
                              "python -m quantized_kv_decode_partial_gb300.build")
    lib = ctypes.CDLL(path)
    P, I32, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    lib.pkv_make_plan.argtypes = [ctypes.POINTER(PoolLayout), ctypes.POINTER(DecodeParams), I32, ctypes.POINTER(Plan)]
    lib.pkv_make_plan.restype = ctypes.c_int
    lib.pkv_plan_for_current_device.argtypes = [ctypes.POINTER(PoolLayout), ctypes.POINTER(DecodeParams),
                                                ctypes.POINTER(Plan)]
    lib.pkv_plan_for_current_device.restype = ctypes.c_int
    lib.pkv_paged_decode_attention.argtypes = [ctypes.POINTER(PoolLayout), ctypes.POINTER(DecodeParams),
                                               P, P, P, P, P, P, P, P, P, F, P, P, SZ, P, P]
    lib.pkv_paged_decode_attention.restype = ctypes.c_int
    lib.pkv_paged_decode_partial.argtypes = lib.pkv_paged_decode_attention.argtypes
    lib.pkv_paged_decode_partial.restype = ctypes.c_int
    lib.pkv_merge_partitions.argtypes = [ctypes.POINTER(PoolLayout), ctypes.POINTER(DecodeParams), P, P, SZ, P,
                                         P, P]
    lib.pkv_merge_partitions.restype = ctypes.c_int
    lib.pkv_paged_decode_attention_no_alloc.argtypes = [ctypes.POINTER(PoolLayout), ctypes.POINTER(DecodeParams),
                                                        P, P, P, P, P, P, P, P, P, F, P, P, P]
    lib.pkv_paged_decode_attention_no_alloc.restype = ctypes.c_int
    lib.pkv_paged_decode_attention_host.argtypes = [ctypes.POINTER(PoolLayout), ctypes.POINTER(DecodeParams),
                                                    P, P, SZ, P, P, P, P, P, P, P, P, P, P, P, P, F, P, P, SZ, P, P]
    lib.pkv_paged_decode_attention_host.restype = ctypes.c_int
    lib.pkv_step_create.argtypes = [ctypes.POINTER(PoolLayout), ctypes.POINTER(DecodeParams),
                                    P, P, SZ, P, P, P, P, P, P, P, P, P, P, P, P, F, P, P, SZ, P, P,
                                    ctypes.POINTER(ctypes.c_void_p)]
    lib.pkv_step_create.restype = ctypes.c_int
    lib.pkv_step_run.argtypes = [P]
    lib.pkv_step_run.restype = ctypes.c_int
    lib.pkv_step_destroy.argtypes = [P]
    lib.pkv_step_destroy.restype = None
    lib.pkv_paged_decode_append_attention.argtypes = [ctypes.POINTER(PoolLayout), ctypes.POINTER(DecodeParams),
                                                      P, P, P, P, P, P, P, P, P, P, P, F, P, P, SZ, P, P]
    lib.pkv_paged_decode_append_attention.restype = ctypes.c_int
    lib.pkv_paged_append.argtypes = [ctypes.POINTER(PoolLayout), I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.pkv_paged_append.restype = ctypes.c_int
    lib.pkv_paged_gather.argtypes = [P, I32, I32, I32, I32, P, P, I32, I32, I32, P, P, P]
    lib.pkv_paged_gather.restype = ctypes.c_int
    lib.pkv_strerror.argtypes = [ctypes.c_int]
    lib.pkv_strerror.restype = ctypes.c_char_p
    lib.pkv_last_cuda_error.argtypes = []
    lib.pkv_last_cuda_error.restype = ctypes.c_char_p
    lib.pkv_version.argtypes = []
    lib.pkv_version.restype = ctypes.c_int
    lib.pkv_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.pkv_set_wait_limit_ns.restype = ctypes.c_uint64
    if path == LIB_PATH:
        _lib = lib
    return lib


def _check(rc: int, lib) -> None:
    if rc != PKV_OK:
        msg = lib.pkv_strerror(rc).decode()
        if rc == PKV_ERR_CUDA:
            msg += ": " + lib.pkv_last_cuda_error().decode()
        raise PkvError(rc, msg)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def v_head_dim_of(v_pool: torch.Tensor, bits: int) -> int:
    """Value head dim of a V pool: its row width, in values (bf16) or codes (affine words)."""
    w = v_pool.shape[-1]
    return w if bits == 16 else w * 32 // bits


def layout_for(k_pool: torch.Tensor, head_dim: int, bits: int, group_size: int = 64,
               v_pool: Optional[torch.Tensor] = None) -> PoolLayout:
    nb, hk, bs, _ = k_pool.shape
    dv = 0 if v_pool is None else v_head_dim_of(v_pool, bits)
    return PoolLayout(nb, hk, bs, head_dim, bits, group_size, 0 if dv == head_dim else dv)


def _out_like(q: torch.Tensor, layout: PoolLayout) -> torch.Tensor:
    dv = layout.v_head_dim or layout.head_dim
    return torch.empty(q.shape[:-1] + (dv,), dtype=q.dtype, device=q.device)


_plan_cache = {}


def _plan_key(layout: PoolLayout, params: DecodeParams):
    return (torch.cuda.current_device(),) + tuple(getattr(layout, f) for f, _ in PoolLayout._fields_) + \
        tuple(getattr(params, f) for f, _ in DecodeParams._fields_)


def _cached_plan(layout: PoolLayout, params: DecodeParams) -> Plan:
    key = _plan_key(layout, params)
    plan = _plan_cache.get(key)
    if plan is None:
        plan = make_plan(layout, params)
        if len(_plan_cache) > 1024:
            _plan_cache.clear()
        _plan_cache[key] = plan
    return plan


def set_wait_limit_ns(ns: int) -> int:
    """Bound of one main-loop pipeline wait for decode calls made from now on
    (pkv_set_wait_limit_ns; 0 restores the default of one second). Returns the
    previous bound."""
    return int(load_library().pkv_set_wait_limit_ns(int(ns)))


def make_plan(layout: PoolLayout, params: DecodeParams, sm_count: Optional[int] = None) -> Plan:
    """The library's plan (partition size, workspace bytes) for these shapes."""
    lib = load_library()
    plan = Plan()
    if sm_count is None:
        rc = lib.pkv_plan_for_current_device(ctypes.byref(layout), ctypes.byref(params), ctypes.byref(plan))
    else:
        rc = lib.pkv_make_plan(ctypes.byref(layout), ctypes.byref(params), sm_count, ctypes.byref(plan))
    _check(rc, lib)
    return plan


def paged_decode_attention(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float, *,
                           bits: int = 16, group_size: int = 64,
                           k_scales: Optional[torch.Tensor] = None, k_biases: Optional[torch.Tensor] = None,
                           v_scales: Optional[torch.Tensor] = None, v_biases: Optional[torch.Tensor] = None,
                           partition_tokens: int = 0, window: int = 0, out: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None,
                           error_flag: Optional[torch.Tensor] = None, contraction: int = 0,
                           schedule: int = 0) -> torch.Tensor:
    """Decode attention over a paged cache (see include/pkv_decode.h).

    q bf16 [B, HQ, N, D]; pools bf16 [NB, HK, BS, D] (bits=16) or int32 code
    words [NB, HK, BS, D*bits/32] with bf16 scale/bias planes [NB, HK, BS, D/64];
    block_tables int32 [B, max_blocks]; seq_lens int32 [B]. Runs on the current
    CUDA stream of q's device and returns bf16 [B, HQ, N, D].
    """
    lib = load_library()
    B, HQ, N, D = q.shape
    layout = layout_for(k_pool, D, bits, group_size, v_pool)
    params = DecodeParams(B, HQ, N, block_tables.shape[1], partition_tokens, window, contraction, schedule)
    with _on_device(q.device):
        plan = _cached_plan(layout, params)
        if out is None:
            out = _out_like(q, layout)
        if workspace is None and plan.workspace_bytes:
            workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=q.device)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        stream = torch.cuda.current_stream(q.device).cuda_stream
        rc = lib.pkv_paged_decode_attention(
            ctypes.byref(layout), ctypes.byref(params), _ptr(q), _ptr(k_pool), _ptr(v_pool),
            _ptr(k_scales), _ptr(k_biases), _ptr(v_scales), _ptr(v_biases), _ptr(block_tables),
            _ptr(seq_lens), float(scale), _ptr(out), _ptr(workspace), ws_bytes, _ptr(error_flag), stream)
    _check(rc, lib)
    return out


def paged_decode_append_attention(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                  k_pool: torch.Tensor, v_pool: torch.Tensor, block_tables: torch.Tensor,
                                  seq_lens: torch.Tensor, scale: float, *, bits: int = 16, group_size: int = 64,
                                  k_scales: Optional[torch.Tensor] = None, k_biases: Optional[torch.Tensor] = None,
                                  v_scales: Optional[torch.Tensor] = None, v_biases: Optional[torch.Tensor] = None,
                                  partition_tokens: int = 0, window: int = 0, out: Optional[torch.Tensor] = None,
                                  workspace: Optional[torch.Tensor] = None,
                                  error_flag: Optional[torch.Tensor] = None, contraction: int = 0,
                                  schedule: int = 0) -> torch.Tensor:
    """One decode step with its write (pkv_paged_decode_append_attention): writes
    k_new/v_new bf16 [B, HK, N, D] at cache positions seq_lens[b]-N .. seq_lens[b]-1
    (seq_lens counts the new rows), then attends as ``paged_decode_attention``."""
    lib = load_library()
    B, HQ, N, D = q.shape
    layout = layout_for(k_pool, D, bits, group_size, v_pool)
    params = DecodeParams(B, HQ, N, block_tables.shape[1], partition_tokens, window, contraction, schedule)
    with _on_device(q.device):
        plan = _cached_plan(layout, params)
        if out is None:
            out = _out_like(q, layout)
        if workspace is None and plan.workspace_bytes:
            workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=q.device)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        stream = torch.cuda.current_stream(q.device).cuda_stream
        rc = lib.pkv_paged_decode_append_attention(
            ctypes.byref(layout), ctypes.byref(params), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool),
            _ptr(v_pool), _ptr(k_scales), _ptr(k_biases), _ptr(v_scales), _ptr(v_biases), _ptr(block_tables),
            _ptr(seq_lens), float(scale), _ptr(out), _ptr(workspace), ws_bytes, _ptr(error_flag), stream)
    _check(rc, lib)
    return out


class HostDecodeStep:
    """One decode step driven from host memory (a pkv_step: pkv_paged_decode_attention_host
    prepared once).

    The step's host inputs (q, lengths, the new K/V rows for the fused step, block
    tables) live in one pinned block with a device twin. Each call enqueues the decode
    (fused with the append when ``k_new``/``v_new`` are given); the kernels read the
    inputs from the pinned block and write the output into pinned ``out_host`` over
    NVLink-C2C (the library falls back to copies where the memory is not mapped).
    Write the next step's values into ``host[name]`` (views of the pinned block)
    before calling again; ``copy_tables=False`` keeps the block tables out of the
    per-step data (the device copy made at construction is used, until
    ``refresh_tables()``). Pools, scale/bias planes and the workspace are device
    tensors, as for ``paged_decode_attention``.
    """

    def __init__(self, q: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor, k_pool: torch.Tensor,
                 v_pool: torch.Tensor, scale: float, *, k_new: Optional[torch.Tensor] = None,
                 v_new: Optional[torch.Tensor] = None, bits: int = 16, group_size: int = 64, k_scales=None,
                 k_biases=None, v_scales=None, v_biases=None, partition_tokens: int = 0, window: int = 0,
                 workspace: Optional[torch.Tensor] = None, error_flag: Optional[torch.Tensor] = None, stream=None,
                 copy_tables: bool = True, contraction: int = 0, schedule: int = 0):
        self.lib = lib = load_library()
        dev = k_pool.device
        B, HQ, N, D = q.shape
        self.layout = layout_for(k_pool, D, bits, group_size, v_pool)
        self.params = DecodeParams(B, HQ, N, block_tables.shape[1], partition_tokens, window, contraction,
                                   schedule)
        named = [("q", q), ("seq_lens", seq_lens)]
        if k_new is not None:
            named += [("k_new", k_new), ("v_new", v_new)]
        named.append(("block_tables", block_tables))  # last: a per-step copy can stop before it
        offs, total = {}, 0
        for name, t in named:  # 256-byte aligned slots
            offs[name] = total
            total += -(-(t.numel() * t.element_size()) // 256) * 256
        self.block_host = torch.empty(total, dtype=torch.uint8, pin_memory=True)
        self.block_dev = torch.empty(total, dtype=torch.uint8, device=dev)
        self.host, self.dev = {}, {}
        for name, t in named:
            n = t.numel() * t.element_size()
            self.host[name] = self.block_host[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)
            self.dev[name] = self.block_dev[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)
            self.host[name].copy_(t.cpu())
        self.dev["block_tables"].copy_(self.host["block_tables"])
        # bytes copied per step: everything up to the tables' slot, or the whole block
        self.in_bytes = total if copy_tables else offs["block_tables"]
        with _on_device(dev):
            plan = _cached_plan(self.layout, self.params)
            self.out = _out_like(self.dev["q"], self.layout)
            if workspace is None and plan.workspace_bytes:
                workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
            st = (stream or torch.cuda.current_stream(dev)).cuda_stream
        self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        self.h2d_bytes, self.d2h_bytes = self.in_bytes, self.out_host.numel() * self.out_host.element_size()
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        self._keep = (k_pool, v_pool, k_scales, k_biases, v_scales, v_biases, workspace, error_flag)
        d = self.dev
        handle = ctypes.c_void_p()
        with _on_device(dev):
            rc = lib.pkv_step_create(
                ctypes.byref(self.layout), ctypes.byref(self.params), _ptr(self.block_host), _ptr(self.block_dev),
                self.in_bytes, _ptr(self.out_host), _ptr(d["q"]), _ptr(d.get("k_new")), _ptr(d.get("v_new")),
                _ptr(k_pool), _ptr(v_pool), _ptr(k_scales), _ptr(k_biases), _ptr(v_scales), _ptr(v_biases),
                _ptr(d["block_tables"]), _ptr(d["seq_lens"]), float(scale), _ptr(self.out), _ptr(workspace),
                ws_bytes, _ptr(error_flag), st, ctypes.byref(handle))
        _check(rc, lib)
        self._handle = handle
        self._run = lib.pkv_step_run
        self._destroy = lib.pkv_step_destroy
        self._device = dev

    def refresh_tables(self):
        """Copies the host block tables to the device now (synchronously)."""
        self.dev["block_tables"].copy_(self.host["block_tables"])

    def __call__(self) -> torch.Tensor:
        """Enqueues the step (pkv_step_run) and returns the pinned output tensor,
        which holds the result once the stream reaches this point."""
        rc = self._run(self._handle)
        if rc != PKV_OK:
            _check(rc, self.lib)
        return self.out_host

    def __del__(self):
        # the handle is host memory only; work in flight keeps using the tensors, which
        # the caller keeps alive as long as it needs the results
        handle = getattr(self, "_handle", None)
        if handle is not None and handle.value:
            self._destroy(handle)
            self._handle = None


class _on_device:
    """Makes `device` current for the call (a no-op when it already is)."""

    def __init__(self, device: torch.device):
        self.index = device.index if device.index is not None else torch.cuda.current_device()
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.index:
            self.prev = cur
            torch.cuda.set_device(self.index)
        return self

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
        return False


def paged_decode_passes(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                        block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float, *, passes: str,
                        bits: int = 16, group_size: int = 64, k_scales=None, k_biases=None, v_scales=None,
                        v_biases=None, partition_tokens: int = 0, window: int = 0,
                        out: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None,
                        error_flag: Optional[torch.Tensor] = None, contraction: int = 0,
                        schedule: int = 0) -> torch.Tensor:
    """One pass of the decode: ``passes="partial"`` (pkv_paged_decode_partial) or
    ``"merge"`` (pkv_merge_partitions). ``out`` and, with more than one
    partition, ``workspace`` must be given so the two calls share them."""
    lib = load_library()
    B, HQ, N, D = q.shape
    layout = layout_for(k_pool, D, bits, group_size, v_pool)
    params = DecodeParams(B, HQ, N, block_tables.shape[1], partition_tokens, window, contraction, schedule)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on_device(q.device):
        stream = torch.cuda.current_stream(q.device).cuda_stream
        if passes == "partial":
            rc = lib.pkv_paged_decode_partial(
                ctypes.byref(layout), ctypes.byref(params), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                _ptr(k_scales), _ptr(k_biases), _ptr(v_scales), _ptr(v_biases), _ptr(block_tables),
                _ptr(seq_lens), float(scale), _ptr(out), _ptr(workspace), ws_bytes, _ptr(error_flag), stream)
        elif passes == "merge":
            rc = lib.pkv_merge_partitions(ctypes.byref(layout), ctypes.byref(params), _ptr(seq_lens),
                                          _ptr(workspace), ws_bytes, _ptr(out), _ptr(error_flag), stream)
        else:
            raise ValueError(passes)
    _check(rc, lib)
    return out


def paged_append(k_new: torch.Tensor, v_new: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                 k_pool: torch.Tensor, v_pool: torch.Tensor, *, bits: int = 16, group_size: int = 64,
                 k_scales=None, k_biases=None, v_scales=None, v_biases=None,
                 error_flag: Optional[torch.Tensor] = None) -> None:
    """Writes k_new/v_new bf16 [B, HK, n_new, D] at positions seq_lens[b].. of each
    sequence (quantising affine pages); see include/pkv_decode.h."""
    lib = load_library()
    B, HK, n_new, D = k_new.shape
    layout = layout_for(k_pool, D, bits, group_size, v_pool)
    with _on_device(k_new.device):
        stream = torch.cuda.current_stream(k_new.device).cuda_stream
        rc = lib.pkv_paged_append(ctypes.byref(layout), B, block_tables.shape[1], n_new, _ptr(k_new), _ptr(v_new),
                                  _ptr(block_tables), _ptr(seq_lens), _ptr(k_pool), _ptr(v_pool), _ptr(k_scales),
                                  _ptr(k_biases), _ptr(v_scales), _ptr(v_biases), _ptr(error_flag), stream)
    _check(rc, lib)


def paged_gather(pool: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor, max_len: int,
                 out: Optional[torch.Tensor] = None, error_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Bit-exact gather of one pool plane [NB, HK, BS, W] into [B, HK, max_len, W]."""
    lib = load_library()
    nb, hk, bs = pool.shape[:3]
    row_bytes = pool[0, 0, 0].numel() * pool.element_size()
    B = block_tables.shape[0]
    if out is None:
        out = torch.zeros((B, hk, max_len) + tuple(pool.shape[3:]), dtype=pool.dtype, device=pool.device)
    with _on_device(pool.device):
        stream = torch.cuda.current_stream(pool.device).cuda_stream
        rc = lib.pkv_paged_gather(_ptr(pool), nb, hk, bs, row_bytes, _ptr(block_tables), _ptr(seq_lens), B,
                                  block_tables.shape[1], max_len, _ptr(out), _ptr(error_flag), stream)
    _check(rc, lib)
    return out
