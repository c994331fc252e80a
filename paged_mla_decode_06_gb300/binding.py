"""Thin ctypes binding over the C ABI of ``include/mla_decode.h``.

Argument marshalling only: tensors become raw device pointers, the current
PyTorch stream becomes the ``cudaStream_t``, and a non-OK status raises
``MLAError``. Every step of the decode runs in the library's kernels; there
is no fallback. Names match the C entry points.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MLA_OK = 0
MLA_ERR_INVALID_ARG = 1
MLA_ERR_UNSUPPORTED = 2
MLA_ERR_WORKSPACE = 3
MLA_ERR_CUDA = 4
MLA_ERR_DEVICE_STATUS = 5

MLA_DTYPE_BF16 = 0
MLA_DTYPE_FP8_E4M3 = 1

MLA_KERNEL_AUTO = 0
MLA_KERNEL_WARP_MMA = 1
MLA_KERNEL_TCGEN05 = 2
MLA_KERNEL_TCGEN05_ROWS_N = 3

HEAD_DIM = 576
KV_LORA_RANK = 512


class MLAError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        name = _status_name(status)
        msg = f"{fn} failed: {name}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_tokens", "num_reqs", "num_heads", "head_dim", "kv_lora_rank", "block_size",
        "max_blocks_per_req", "num_blocks", "max_seq_len", "max_qlen", "topk", "q_dtype",
        "kv_dtype", "has_sinks", "num_segments", "num_sms", "kernel")]


class Plan(ctypes.Structure):
    _fields_ = [("prob", Problem)] + [(n, ctypes.c_int32) for n in (
        "num_segments", "tile_size", "kernel", "rows_per_cta", "row_tiles", "grid_x", "grid_y",
        "grid_z", "num_sms", "schedule", "max_items", "split_items", "wait_limit_us", "tile_rows")] + [
        ("workspace_bytes", ctypes.c_size_t), ("status_offset", ctypes.c_size_t),
        ("segm_output_offset", ctypes.c_size_t), ("segm_max_offset", ctypes.c_size_t),
        ("segm_expsum_offset", ctypes.c_size_t)]


_lib = None
_lock = threading.Lock()
_vp = ctypes.c_void_p


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the compiled library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library not found at {p}; build it with "
                "`python -m paged_mla_decode_06_gb300.build`")
        lib = ctypes.CDLL(p)
        st = ctypes.c_int32
        lib.mla_decode_plan.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(Plan)]
        lib.mla_decode_plan.restype = st
        common = [ctypes.POINTER(Plan), _vp, _vp, _vp, ctypes.c_int64, _vp, _vp, _vp, _vp,
                  ctypes.c_float, ctypes.c_float, ctypes.c_float]
        lib.mla_decode_fwd.argtypes = common + [_vp, _vp, ctypes.c_size_t, _vp, _vp, _vp]
        lib.mla_decode_fwd.restype = st
        lib.mla_decode_fwd_static.argtypes = common + [_vp, _vp, _vp, _vp, _vp]
        lib.mla_decode_fwd_static.restype = st
        lib.mla_decode_segments.argtypes = common + [_vp, _vp, _vp, _vp]
        lib.mla_decode_segments.restype = st
        lib.mla_decode_schedule.argtypes = [ctypes.POINTER(Plan), _vp, _vp, _vp, _vp,
                                            ctypes.c_size_t, _vp]
        lib.mla_decode_schedule.restype = st
        lib.mla_decode_items.argtypes = common + [_vp, _vp, ctypes.c_size_t, _vp, _vp, _vp]
        lib.mla_decode_items.restype = st
        lib.mla_merge_items.argtypes = [ctypes.POINTER(Plan), _vp, _vp, _vp, ctypes.c_size_t,
                                        _vp, _vp, _vp]
        lib.mla_merge_items.restype = st

        lib.mla_merge_segments.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp,
                                           ctypes.c_int32, _vp, _vp, _vp]
        lib.mla_merge_segments.restype = st
        lib.mla_sparse_index_convert.argtypes = [_vp, _vp, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_int64, _vp, ctypes.c_int64,
                                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                 _vp, _vp, _vp]
        lib.mla_sparse_index_convert.restype = st
        lib.mla_sparse_seqlen.argtypes = [_vp, _vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          _vp, _vp, _vp]
        lib.mla_sparse_seqlen.restype = st
        lib.mla_fit_kpool_indices.argtypes = [_vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, _vp, ctypes.c_int64, _vp]
        lib.mla_fit_kpool_indices.restype = st
        lib.mla_merge_lse.argtypes = [_vp, _vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, _vp, _vp, _vp, _vp]
        lib.mla_merge_lse.restype = st
        lib.mla_concat_quant_q.argtypes = [_vp, ctypes.c_int64, ctypes.c_int64, _vp,
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _vp,
                                           _vp]
        lib.mla_concat_quant_q.restype = st
        lib.mla_workspace_status.argtypes = [ctypes.POINTER(Plan), _vp, ctypes.POINTER(ctypes.c_int32),
                                             ctypes.c_int32, _vp]
        lib.mla_workspace_status.restype = st
        lib.mla_status_string.argtypes = [ctypes.c_int32]
        lib.mla_status_string.restype = ctypes.c_char_p
        lib.mla_last_cuda_error.argtypes = []
        lib.mla_last_cuda_error.restype = ctypes.c_char_p
        lib.mla_version.argtypes = []
        lib.mla_version.restype = ctypes.c_int32
        _lib = lib
        return lib


def _status_name(status: int) -> str:
    names = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED",
             3: "MLA_ERR_WORKSPACE", 4: "MLA_ERR_CUDA", 5: "MLA_ERR_DEVICE_STATUS"}
    return names.get(int(status), f"status {status}")


def _check(fn: str, status: int):
    if status != MLA_OK:
        detail = ""
        if status == MLA_ERR_CUDA and _lib is not None:
            detail = _lib.mla_last_cuda_error().decode()
        raise MLAError(fn, status, detail)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(name: str) -> int:
    return {"bf16": MLA_DTYPE_BF16, "fp8": MLA_DTYPE_FP8_E4M3}[name]


def make_problem(*, num_tokens: int, num_heads: int, block_size: int, num_blocks: int,
                 num_reqs: int = 0, max_blocks_per_req: int = 0, max_seq_len: int = 0,
                 max_qlen: int = 1, topk: int = 0, dtype: str = "bf16",
                 has_sinks: bool = False, num_segments: int = 0, num_sms: int = 0,
                 kernel: int = MLA_KERNEL_AUTO) -> Problem:
    return Problem(num_tokens=num_tokens, num_reqs=num_reqs, num_heads=num_heads,
                   head_dim=HEAD_DIM, kv_lora_rank=KV_LORA_RANK, block_size=block_size,
                   max_blocks_per_req=max_blocks_per_req, num_blocks=num_blocks,
                   max_seq_len=max_seq_len, max_qlen=max_qlen, topk=topk,
                   q_dtype=_dtype_code(dtype), kv_dtype=_dtype_code(dtype),
                   has_sinks=int(bool(has_sinks)), num_segments=num_segments, num_sms=num_sms,
                   kernel=kernel)


def mla_decode_plan(problem: Problem) -> Plan:
    lib = load_library()
    plan = Plan()
    _check("mla_decode_plan", lib.mla_decode_plan(ctypes.byref(problem), ctypes.byref(plan)))
    return plan


def mla_decode_fwd(plan: Plan, q, kv_cache, *, block_table=None, block_table_stride=None,
                   seq_lens=None, qo_indptr=None, sparse_slots=None, sparse_indptr=None,
                   softmax_scale: float, q_scale: float = 1.0, kv_scale: float = 1.0,
                   sinks=None, workspace=None, out, lse, stream=None) -> None:
    lib = load_library()
    if block_table_stride is None:
        block_table_stride = block_table.stride(0) if block_table is not None else 0
    ws_bytes = 0
    if workspace is not None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("mla_decode_fwd", lib.mla_decode_fwd(
        ctypes.byref(plan), _ptr(q), _ptr(kv_cache), _ptr(block_table), int(block_table_stride),
        _ptr(seq_lens), _ptr(qo_indptr), _ptr(sparse_slots), _ptr(sparse_indptr),
        float(softmax_scale), float(q_scale), float(kv_scale), _ptr(sinks), _ptr(workspace),
        ws_bytes, _ptr(out), _ptr(lse), _stream(stream)))


def mla_decode_fwd_static(plan: Plan, q, kv_cache, *, block_table=None,
                          block_table_stride=None, seq_lens=None, qo_indptr=None,
                          sparse_slots=None, sparse_indptr=None, softmax_scale: float,
                          q_scale: float = 1.0, kv_scale: float = 1.0, sinks=None, out, lse,
                          status_out=None, stream=None) -> None:
    """mla_decode_fwd on the library's own static device scratch (no workspace)."""
    lib = load_library()
    if block_table_stride is None:
        block_table_stride = block_table.stride(0) if block_table is not None else 0
    _check("mla_decode_fwd_static", lib.mla_decode_fwd_static(
        ctypes.byref(plan), _ptr(q), _ptr(kv_cache), _ptr(block_table), int(block_table_stride),
        _ptr(seq_lens), _ptr(qo_indptr), _ptr(sparse_slots), _ptr(sparse_indptr),
        float(softmax_scale), float(q_scale), float(kv_scale), _ptr(sinks), _ptr(out), _ptr(lse),
        _ptr(status_out), _stream(stream)))


def mla_workspace_status(plan: Plan, workspace, *, clear: bool = False, stream=None) -> int:
    """The workspace's device status word after the stream's work so far
    (0: no kernel reported a timed-out wait); with ``clear`` a nonzero word
    is reset. Returns the word instead of raising on MLA_ERR_DEVICE_STATUS."""
    lib = load_library()
    code = ctypes.c_int32(0)
    st = lib.mla_workspace_status(ctypes.byref(plan), _ptr(workspace), ctypes.byref(code),
                                  1 if clear else 0, _stream(stream))
    if st not in (MLA_OK, MLA_ERR_DEVICE_STATUS):
        _check("mla_workspace_status", st)
    return int(code.value)


def _ws_bytes(workspace) -> int:
    return 0 if workspace is None else workspace.numel() * workspace.element_size()


def mla_decode_schedule(plan: Plan, *, seq_lens=None, qo_indptr=None, sparse_indptr=None,
                        workspace, stream=None) -> None:
    """Balanced plans: the work list into ``workspace``."""
    lib = load_library()
    _check("mla_decode_schedule", lib.mla_decode_schedule(
        ctypes.byref(plan), _ptr(seq_lens), _ptr(qo_indptr), _ptr(sparse_indptr),
        _ptr(workspace), _ws_bytes(workspace), _stream(stream)))


def mla_decode_items(plan: Plan, q, kv_cache, *, block_table=None, block_table_stride=None,
                     seq_lens=None, qo_indptr=None, sparse_slots=None, sparse_indptr=None,
                     softmax_scale: float, q_scale: float = 1.0, kv_scale: float = 1.0,
                     sinks=None, workspace, out, lse, stream=None) -> None:
    """Balanced plans: the decode kernel over the work list in ``workspace``."""
    lib = load_library()
    if block_table_stride is None:
        block_table_stride = block_table.stride(0) if block_table is not None else 0
    _check("mla_decode_items", lib.mla_decode_items(
        ctypes.byref(plan), _ptr(q), _ptr(kv_cache), _ptr(block_table), int(block_table_stride),
        _ptr(seq_lens), _ptr(qo_indptr), _ptr(sparse_slots), _ptr(sparse_indptr),
        float(softmax_scale), float(q_scale), float(kv_scale), _ptr(sinks), _ptr(workspace),
        _ws_bytes(workspace), _ptr(out), _ptr(lse), _stream(stream)))


def mla_merge_items(plan: Plan, *, qo_indptr=None, sinks=None, workspace, out, lse,
                    stream=None) -> None:
    """Balanced plans: out and lse of the split rows from their partials."""
    lib = load_library()
    _check("mla_merge_items", lib.mla_merge_items(
        ctypes.byref(plan), _ptr(qo_indptr), _ptr(sinks), _ptr(workspace), _ws_bytes(workspace),
        _ptr(out), _ptr(lse), _stream(stream)))


def mla_decode_segments(plan: Plan, q, kv_cache, *, block_table=None, block_table_stride=None,
                        seq_lens=None, qo_indptr=None, sparse_slots=None, sparse_indptr=None,
                        softmax_scale: float, q_scale: float = 1.0, kv_scale: float = 1.0,
                        segm_output, segm_max, segm_expsum, stream=None) -> None:
    lib = load_library()
    if block_table_stride is None:
        block_table_stride = block_table.stride(0) if block_table is not None else 0
    _check("mla_decode_segments", lib.mla_decode_segments(
        ctypes.byref(plan), _ptr(q), _ptr(kv_cache), _ptr(block_table), int(block_table_stride),
        _ptr(seq_lens), _ptr(qo_indptr), _ptr(sparse_slots), _ptr(sparse_indptr),
        float(softmax_scale), float(q_scale), float(kv_scale), _ptr(segm_output),
        _ptr(segm_max), _ptr(segm_expsum), _stream(stream)))


def mla_merge_segments(segm_output, segm_max, segm_expsum, part_lens, *, tile_size: int,
                       sinks=None, out, lse, stream=None) -> None:
    lib = load_library()
    T, H, NS, rank = segm_output.shape
    _check("mla_merge_segments", lib.mla_merge_segments(
        _ptr(segm_output), _ptr(segm_max), _ptr(segm_expsum), _ptr(part_lens), T, H, NS, rank,
        int(tile_size), _ptr(sinks), MLA_DTYPE_BF16, _ptr(out), _ptr(lse), _stream(stream)))


def mla_merge_lse(shard_out, shard_lse, *, sinks=None, out, lse, stream=None) -> None:
    lib = load_library()
    W, T, H, rank = shard_out.shape
    _check("mla_merge_lse", lib.mla_merge_lse(
        _ptr(shard_out), _ptr(shard_lse), W, T, H, rank, _ptr(sinks), _ptr(out), _ptr(lse),
        _stream(stream)))


def mla_concat_quant_q(ql_nope, q_pe, *, out, q_scale: float | None = None, stream=None) -> None:
    """q = ql_nope || q_pe into ``out`` (bf16), or e4m3 codes of q / q_scale
    when ``q_scale`` is given (``out`` then holds uint8 codes)."""
    lib = load_library()
    T, H, _ = ql_nope.shape
    fp8 = q_scale is not None
    _check("mla_concat_quant_q", lib.mla_concat_quant_q(
        _ptr(ql_nope), ql_nope.stride(0), ql_nope.stride(1), _ptr(q_pe), q_pe.stride(0),
        q_pe.stride(1), T, H, MLA_DTYPE_FP8_E4M3 if fp8 else MLA_DTYPE_BF16,
        float(q_scale) if fp8 else 1.0, _ptr(out), _stream(stream)))


def mla_sparse_seqlen(query_start_loc, seq_lens, *, topk: int, indptr, lens=None,
                      stream=None) -> None:
    """Per-token sparse list lengths (``lens``, optional) and their exclusive
    prefix sum (``indptr``, ``[T + 1]``)."""
    lib = load_library()
    num_reqs = query_start_loc.numel() - 1
    num_tokens = indptr.numel() - 1
    _check("mla_sparse_seqlen", lib.mla_sparse_seqlen(
        _ptr(query_start_loc), _ptr(seq_lens), num_reqs, num_tokens, int(topk), _ptr(lens),
        _ptr(indptr), _stream(stream)))


def mla_fit_kpool_indices(token_indices, *, topk: int, out, stream=None) -> None:
    """``[T, W]`` top-k rows fitted to width ``topk`` into ``out [T, topk]``."""
    lib = load_library()
    T, W = token_indices.shape
    _check("mla_fit_kpool_indices", lib.mla_fit_kpool_indices(
        _ptr(token_indices), token_indices.stride(0), T, W, int(topk), _ptr(out), out.stride(0),
        _stream(stream)))


def mla_sparse_index_convert(req_id, block_table, token_indices, *, block_size: int,
                             cu_seqlens=None, out, stream=None) -> None:
    lib = load_library()
    bt_rows, bt_cols = block_table.shape
    T, topk = token_indices.shape
    _check("mla_sparse_index_convert", lib.mla_sparse_index_convert(
        _ptr(req_id), _ptr(block_table), bt_rows, bt_cols, block_table.stride(0),
        _ptr(token_indices), token_indices.stride(0), T, topk, int(block_size),
        _ptr(cu_seqlens), _ptr(out), _stream(stream)))


# ---------------------------------------------------------------------------
# convenience: one decode call on a Workload whose tensors live on a device
# ---------------------------------------------------------------------------

class DeviceWorkload:
    """Device copies of an ``inputs.Workload`` plus a plan and output buffers."""

    def __init__(self, w, device="cuda", num_segments=None, num_sms=0, plan=True,
                 kernel=MLA_KERNEL_AUTO):
        import torch

        self.w = w
        dev = torch.device(device)
        self.device = dev
        self.q = torch.from_numpy(w.q.view(_np_view(w.q_dtype))).to(dev)
        self.cache = torch.from_numpy(w.cache.view(_np_view(w.kv_dtype))).to(dev)
        self.block_table = torch.from_numpy(w.block_table).to(dev)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(dev)
        self.qo_indptr = None if w.qo_indptr is None else torch.from_numpy(w.qo_indptr).to(dev)
        self.sinks = None if w.sinks is None else torch.from_numpy(w.sinks).to(dev)
        self.slots = None
        if w.sparse:
            self.req_id = torch.from_numpy(w.req_id_per_token).to(dev)
            self.topk_indices = torch.from_numpy(w.topk_indices).to(dev)
            self.slots = torch.empty_like(self.topk_indices)
        T, H = w.num_tokens, w.num_heads
        self.out = torch.empty((T, H, KV_LORA_RANK), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        ns = w.num_segments if num_segments is None else num_segments
        self.problem = make_problem(
            num_tokens=T, num_heads=H, block_size=w.block_size, num_blocks=w.num_blocks,
            num_reqs=w.num_reqs if not w.sparse else 0,
            max_blocks_per_req=w.max_blocks_per_req,
            max_seq_len=int(w.seq_lens.max()) if w.num_reqs else 0,
            max_qlen=w.max_qlen, topk=w.topk, dtype=w.kv_dtype, has_sinks=w.sinks is not None,
            num_segments=ns, num_sms=num_sms, kernel=kernel)
        self.plan = mla_decode_plan(self.problem) if plan else None
        self.workspace = None
        if self.plan is not None and self.plan.workspace_bytes:
            # zeroed once: its first int32 is the device status word
            self.workspace = torch.zeros(self.plan.workspace_bytes, dtype=torch.uint8, device=dev)

    def status(self) -> int:
        """Device status word of the workspace (0 = no kernel reported a timeout)."""
        import torch

        if self.workspace is None:
            return 0
        return int(self.workspace[:4].view(torch.int32).item())

    def convert(self, stream=None):
        """Top-k positions -> global slots (sparse workloads)."""
        mla_sparse_index_convert(self.req_id, self.block_table, self.topk_indices,
                                 block_size=self.w.block_size, out=self.slots, stream=stream)

    def forward(self, stream=None, convert=True):
        w = self.w
        if w.sparse and convert:
            self.convert(stream)
        mla_decode_fwd(self.plan, self.q, self.cache,
                       block_table=None if w.sparse else self.block_table,
                       seq_lens=None if w.sparse else self.seq_lens, qo_indptr=self.qo_indptr,
                       sparse_slots=self.slots, softmax_scale=w.softmax_scale,
                       q_scale=w.q_scale, kv_scale=w.kv_scale, sinks=self.sinks,
                       workspace=self.workspace, out=self.out, lse=self.lse, stream=stream)
        return self.out, self.lse


def _np_view(dtype_name: str):
    import numpy as np
    return np.int16 if dtype_name == "bf16" else np.uint8
