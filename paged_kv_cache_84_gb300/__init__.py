"""Paged KV write and ragged paged attention on GB300 (sm_103a).

A thin ctypes binding over ``libpkv.so`` (C ABI in ``include/pkv.h``).  The
functions here only marshal torch tensors into pointers, sizes and the
current CUDA stream; every step of the computation runs in the library's
CUDA kernels.  There is no CPU or PyTorch fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

__all__ = [
    "PkvError", "load", "paged_kv_write", "ragged_paged_attention", "attention_workspace_bytes",
    "make_workspace", "read_device_error", "clear_device_error", "launch_count", "LIB_PATH",
    "DEVERR_SLOT", "DEVERR_BLOCK", "DEVERR_TIMEOUT", "DEVERR_META", "DEVERR_COUNTER", "WORKSPACE_MIN_BYTES", "profile_start", "profile_stop", "profile_records",
    "plan_request_kernels", "CLASS_NAMES", "paged_kv_write_fp8", "ragged_paged_attention_fp8", "copy_blocks", "gather_blocks", "scatter_blocks", "MAX_POOLS", "copy_async", "paged_kv_write_attention", "fp8_prefill_scratch_bytes", "paged_kv_write_attention_fp8", "plan_attention",
    "AttentionOptions", "set_options", "reset_options", "options", "current_options",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkv.so")
DEVERR_SLOT = 1
DEVERR_BLOCK = 2
DEVERR_TIMEOUT = 4
DEVERR_META = 8
DEVERR_COUNTER = 16
WORKSPACE_MIN_BYTES = 256

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape or alignment",
          3: "workspace missing or too small", 4: "CUDA error", 5: "device bounds violation recorded"}

_c_i32, _c_i64, _c_p, _c_f, _c_sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
_lib = None


class _Plan(ctypes.Structure):
    """pkv_attention_plan (include/pkv.h)."""
    _fields_ = [("decode_requests", _c_i32), ("prefill_tensor_requests", _c_i32),
                ("prefill_mma_requests", _c_i32), ("decode_split_tokens", _c_i32),
                ("max_decode_splits", _c_i32), ("decode_cluster", _c_i32), ("decode_streaming", _c_i32),
                ("split_counters", _c_i32), ("overlap", _c_i32), ("decode_on_caller_stream", _c_i32),
                ("prefill_key_splits", _c_i32), ("prefill_tensor_pieces", _c_i32),
                ("quantized_prefill_scratch", _c_sz), ("partial_bytes", _c_sz), ("mixed_launch", _c_i32),
                ("mixed_decode_items", _c_i32), ("mixed_decode_ctas", _c_i32),
                ("mixed_predicted_us", _c_i32), ("prefill_tensor_own_rows", _c_i32)]


class AttentionOptions(ctypes.Structure):
    """pkv_attention_options (include/pkv.h): each field overrides one choice
    of the planner; all zero leaves every choice to it."""
    _fields_ = [("disable_tcgen05", _c_i32), ("tc_min_rows", _c_i32), ("fp8_prefill_on_mma", _c_i32),
                ("split_tokens", _c_i32), ("cluster", _c_i32), ("decode_main", _c_i32), ("no_overlap", _c_i32),
                ("prefill_key_splits", _c_i32), ("separate_write", _c_i32), ("decode_row_tiles", _c_i32),
                ("no_pdl", _c_i32), ("tc_key_pieces", _c_i32), ("mixed_launch", _c_i32), ("mixed_decode_ctas", _c_i32),
                ("device_lengths", _c_i32), ("reserved", _c_i32)]


# The options the attention wrappers pass to the library's _ex calls (None:
# a NULL pointer, the planner's choices).  Set by tests and comparisons only.
_options = None


def set_options(**fields):
    """Override planner choices for the following attention calls (fields of
    AttentionOptions; merged into the options already set)."""
    global _options
    o = AttentionOptions() if _options is None else _options
    names = {f for f, _ in AttentionOptions._fields_ if f != "reserved"}
    for k, v in fields.items():
        if k not in names:
            raise TypeError(f"unknown attention option {k!r}")
        setattr(o, k, int(v))
    _options = o


def reset_options():
    """Back to the planner's choices."""
    global _options
    _options = None


def current_options():
    """The options passed to the library now (a dict of the non-zero fields)."""
    if _options is None:
        return {}
    return {f: getattr(_options, f) for f, _ in AttentionOptions._fields_
            if f != "reserved" and getattr(_options, f)}


@contextlib.contextmanager
def options(**fields):
    """Attention calls inside the block use these options, then the previous ones again."""
    global _options
    saved = None if _options is None else AttentionOptions.from_buffer_copy(_options)
    try:
        set_options(**fields)
        yield
    finally:
        _options = saved


def _opts():
    return ctypes.byref(_options) if _options is not None else None


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        msg = f"{what}: {STATUS.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


def load():
    """Load libpkv.so (built by ``build.py``); raise if it is not there."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with paged_kv_cache_84_gb300/build.py "
                          "(nvcc, sm_103a); there is no fallback path")
    L = ctypes.CDLL(LIB_PATH)
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_status_string.argtypes = [ctypes.c_int]
    L.pkv_last_cuda_error.restype = ctypes.c_char_p
    L.pkv_last_cuda_error.argtypes = []
    L.pkv_launch_count.restype = _c_i64
    L.pkv_launch_count.argtypes = []
    L.pkv_paged_kv_write.restype = ctypes.c_int
    L.pkv_paged_kv_write.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                     _c_p, _c_p]
    L.pkv_attention_workspace_bytes.restype = _c_sz
    L.pkv_attention_workspace_bytes.argtypes = [_c_i32] * 5
    L.pkv_ragged_paged_attention.restype = ctypes.c_int
    L.pkv_ragged_paged_attention.argtypes = [_c_p] * 7 + [_c_i32, _c_p, _c_p] + [_c_i32] * 9 + \
        [_c_f, _c_i32, _c_p, _c_sz, _c_p]
    L.pkv_clear_device_error.restype = ctypes.c_int
    L.pkv_clear_device_error.argtypes = [_c_p, _c_p]
    L.pkv_read_device_error.restype = ctypes.c_int
    L.pkv_read_device_error.argtypes = [_c_p, ctypes.POINTER(ctypes.c_uint32), _c_p]
    L.pkv_profile_start.restype = ctypes.c_int
    L.pkv_profile_start.argtypes = [_c_i32]
    L.pkv_profile_stop.restype = _c_i32
    L.pkv_profile_stop.argtypes = []
    L.pkv_profile_read.restype = ctypes.c_int
    L.pkv_profile_read.argtypes = [_c_i32, ctypes.POINTER(_c_i32), ctypes.POINTER(ctypes.c_float)]
    L.pkv_kernel_name.restype = ctypes.c_char_p
    L.pkv_kernel_name.argtypes = [_c_i32]
    L.pkv_plan_request_kernels.restype = ctypes.c_int
    L.pkv_plan_request_kernels.argtypes = [_c_p, _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_p]
    L.pkv_paged_kv_write_fp8.restype = ctypes.c_int
    L.pkv_paged_kv_write_fp8.argtypes = [_c_p] * 7 + [_c_i32] * 5 + [_c_p, _c_p]
    L.pkv_ragged_paged_attention_fp8.restype = ctypes.c_int
    L.pkv_ragged_paged_attention_fp8.argtypes = [_c_p] * 9 + [_c_i32, _c_p, _c_p] + [_c_i32] * 9 + \
        [_c_f, _c_i32, _c_p, _c_sz, _c_p]
    L.pkv_copy_blocks.restype = ctypes.c_int
    L.pkv_copy_blocks.argtypes = [_c_p, _c_i32, _c_p, _c_p, _c_i32, _c_i32, _c_sz, _c_p, _c_p]
    L.pkv_gather_blocks.restype = ctypes.c_int
    L.pkv_gather_blocks.argtypes = [_c_p, _c_i32, _c_p, _c_i32, _c_i32, _c_sz, _c_p, _c_p, _c_p]
    L.pkv_scatter_blocks.restype = ctypes.c_int
    L.pkv_scatter_blocks.argtypes = [_c_p, _c_i32, _c_p, _c_i32, _c_i32, _c_sz, _c_p, _c_p, _c_p]
    L.pkv_paged_kv_write_attention_fp8.restype = ctypes.c_int
    L.pkv_paged_kv_write_attention_fp8.argtypes = [_c_p] * 12 + [_c_i32, _c_p, _c_p] + [_c_i32] * 9 + \
        [_c_f, _c_i32, _c_p, _c_sz, _c_p]
    L.pkv_fp8_prefill_scratch_bytes.restype = _c_sz
    L.pkv_fp8_prefill_scratch_bytes.argtypes = [_c_p, _c_p, _c_i32, _c_i32, _c_i32, _c_i32]
    L.pkv_copy_async.restype = ctypes.c_int
    L.pkv_copy_async.argtypes = [_c_p, _c_p, _c_sz, _c_p]
    L.pkv_plan_attention.restype = ctypes.c_int
    L.pkv_plan_attention.argtypes = [_c_p, _c_p] + [_c_i32] * 8 + [_c_sz, _c_i32, _c_p, ctypes.POINTER(_Plan)]
    L.pkv_paged_kv_write_attention.restype = ctypes.c_int
    L.pkv_paged_kv_write_attention.argtypes = [_c_p] * 10 + [_c_i32, _c_p, _c_p] + [_c_i32] * 9 + \
        [_c_f, _c_i32, _c_p, _c_sz, _c_p]
    for name, n_ptr in (("pkv_ragged_paged_attention_ex", 7), ("pkv_ragged_paged_attention_fp8_ex", 9),
                        ("pkv_paged_kv_write_attention_ex", 10), ("pkv_paged_kv_write_attention_fp8_ex", 12)):
        f = getattr(L, name)
        f.restype = ctypes.c_int
        f.argtypes = [_c_p] * n_ptr + [_c_i32, _c_p, _c_p] + [_c_i32] * 9 + [_c_f, _c_i32, _c_p, _c_sz, _c_p, _c_p]
    _lib = L
    return L


def _check(status: int, what: str):
    if status != 0:
        detail = load().pkv_last_cuda_error().decode() if status == 4 else ""
        raise PkvError(status, what, detail)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return _c_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return _c_p(s.cuda_stream)


def _host_i32(x, name):
    t = torch.as_tensor(x, dtype=torch.int32)
    if t.device.type != "cpu":
        raise TypeError(f"{name} must be host data")
    return t.contiguous()


def _check_meta(query_start_loc, seq_lens, block_table, num_reqs):
    """Device metadata with room for every request (the kernels index it by
    request; the library sees only pointers)."""
    if block_table.dim() != 2 or block_table.shape[0] < num_reqs:
        raise ValueError("block_table must be [num_reqs, width]")
    if query_start_loc.numel() < num_reqs + 1 or seq_lens.numel() < num_reqs:
        raise ValueError("query_start_loc and seq_lens need num_reqs + 1 and num_reqs entries")


def profile_start(capacity: int = 4096):
    """Time each library kernel launch with CUDA events on its stream (diagnostics)."""
    _check(load().pkv_profile_start(capacity), "profile_start")


def profile_stop(read: bool = True):
    """Stop recording; return [(kernel name, ms), ...] in launch order (waits
    for them).  read=False returns only the number of records, for launches
    captured into a CUDA graph: read them with profile_records(n) after the
    graph has run."""
    n = load().pkv_profile_stop()
    return profile_records(n) if read else n


def profile_records(n: int):
    """[(kernel name, ms), ...] of the first n records (waits for them)."""
    L = load()
    out = []
    kid, ms = _c_i32(0), ctypes.c_float(0)
    for i in range(n):
        _check(L.pkv_profile_read(i, ctypes.byref(kid), ctypes.byref(ms)), "profile_read")
        out.append((L.pkv_kernel_name(kid.value).decode(), float(ms.value)))
    return out


CLASS_NAMES = {0: "none", 1: "padding", 2: "decode", 3: "prefill_mma", 4: "prefill_tensor"}


def plan_request_kernels(query_start_loc_host, seq_lens_host, num_q_heads, num_kv_heads, head_dim):
    """Kernel class of every request, as the attention planner assigns it (host only)."""
    qsl = _host_i32(query_start_loc_host, "query_start_loc_host")
    sl = _host_i32(seq_lens_host, "seq_lens_host")
    out = torch.zeros(sl.numel(), dtype=torch.int32)
    _check(load().pkv_plan_request_kernels(_c_p(qsl.data_ptr()), _c_p(sl.data_ptr()), sl.numel(), num_q_heads,
                                           num_kv_heads, head_dim, _c_p(out.data_ptr())), "plan_request_kernels")
    return [CLASS_NAMES[int(c)] for c in out]


def plan_attention(query_start_loc_host, seq_lens_host, num_q_heads, num_kv_heads, head_dim, block_size=16,
                   window=0, quantized=False, combined=False, workspace_bytes=None, num_sms=0) -> dict:
    """The launch plan of an attention call with these host metadata (host
    only when num_sms > 0): request classes, decode split length and split
    count, cluster and streaming choice, stream overlap, workspace use.
    workspace_bytes defaults to attention_workspace_bytes for the batch."""
    qsl = _host_i32(query_start_loc_host, "query_start_loc_host")
    sl = _host_i32(seq_lens_host, "seq_lens_host")
    if workspace_bytes is None:
        n = sl.numel()
        workspace_bytes = attention_workspace_bytes(max(1, n), max(1, int(qsl[-1]) if qsl.numel() else 1),
                                                    num_q_heads, head_dim, max(1, int(sl.max()) if n else 1))
    out = _Plan()
    _check(load().pkv_plan_attention(_c_p(qsl.data_ptr()), _c_p(sl.data_ptr()), sl.numel(), num_q_heads,
                                     num_kv_heads, head_dim, block_size, window, int(bool(quantized)),
                                     int(bool(combined)), workspace_bytes, num_sms, _opts(), ctypes.byref(out)),
           "plan_attention")
    return {name: int(getattr(out, name)) for name, _ in _Plan._fields_ if name != "reserved"}


def launch_count() -> int:
    """Kernels launched by the library since it was loaded."""
    return int(load().pkv_launch_count())


def paged_kv_write(k, v, k_cache, v_cache, slot_mapping, device_error=None, stream=None):
    """Scatter k, v [N, Hkv, d] into the pools [nbt, bs, Hkv, d] at ``slot_mapping`` (int64 [N])."""
    L = load()
    n, hkv, d = k.shape
    nbt, bs, hkv2, d2 = k_cache.shape
    if (hkv2, d2) != (hkv, d) or v.shape != k.shape or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between k/v and the pools")
    err = _dev(device_error, "device_error", torch.int32) if device_error is not None else None
    st = L.pkv_paged_kv_write(_dev(k, "k", torch.bfloat16), _dev(v, "v", torch.bfloat16),
                              _dev(k_cache, "k_cache", torch.bfloat16), _dev(v_cache, "v_cache", torch.bfloat16),
                              _dev(slot_mapping, "slot_mapping", torch.int64), n, hkv, d, bs, nbt, err,
                              _stream(stream))
    _check(st, "paged_kv_write")


def attention_workspace_bytes(max_num_reqs, max_num_tokens, num_q_heads, head_dim, max_seq_len) -> int:
    return int(load().pkv_attention_workspace_bytes(max_num_reqs, max_num_tokens, num_q_heads, head_dim,
                                                    max_seq_len))


def make_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zeroed uint8 CUDA buffer of ``nbytes`` (torch allocations are 256-byte aligned)."""
    return torch.zeros(max(int(nbytes), WORKSPACE_MIN_BYTES), dtype=torch.uint8, device=device or "cuda")


def ragged_paged_attention(out, q, k_cache, v_cache, query_start_loc, seq_lens, block_table,
                           query_start_loc_host, seq_lens_host, max_query_len, max_seq_len, scale,
                           workspace, stream=None, window: int = 0):
    """Causal GQA attention of a flattened ragged batch over the paged pool; writes ``out``.
    ``window`` > 0 restricts the query at position p to the keys above p - window."""
    L = load()
    n, hq, d = q.shape
    nbt, bs, hkv, d2 = k_cache.shape
    if out.shape != q.shape or d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    qsl_h = _host_i32(query_start_loc_host, "query_start_loc_host")
    sl_h = _host_i32(seq_lens_host, "seq_lens_host")
    if qsl_h.numel() != sl_h.numel() + 1:
        raise ValueError("query_start_loc needs num_reqs + 1 entries")
    _check_meta(query_start_loc, seq_lens, block_table, sl_h.numel())
    st = L.pkv_ragged_paged_attention_ex(
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16),
        _dev(k_cache, "k_cache", torch.bfloat16), _dev(v_cache, "v_cache", torch.bfloat16),
        _dev(query_start_loc, "query_start_loc", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        _dev(block_table, "block_table", torch.int32), block_table.shape[1],
        _c_p(qsl_h.data_ptr()), _c_p(sl_h.data_ptr()), sl_h.numel(), n, int(max_query_len), int(max_seq_len),
        hq, hkv, d, bs, nbt, float(scale), int(window), _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _opts(), _stream(stream))
    _check(st, "ragged_paged_attention")


def paged_kv_write_attention(k, v, k_cache, v_cache, slot_mapping, out, q, query_start_loc, seq_lens, block_table,
                             query_start_loc_host, seq_lens_host, max_query_len, max_seq_len, scale, workspace,
                             stream=None, window: int = 0):
    """paged_kv_write followed by ragged_paged_attention, in one call (decode-class CTAs write their own
    rows; a batch of decodes is one launch).  Write errors go to the workspace's error word."""
    L = load()
    n, hq, d = q.shape
    nbt, bs, hkv, d2 = k_cache.shape
    if out.shape != q.shape or d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if k.shape != (n, hkv, d) or v.shape != k.shape or slot_mapping.numel() != n:
        raise ValueError("k, v must be [num_tokens, num_kv_heads, head_dim] with one slot per token")
    qsl_h = _host_i32(query_start_loc_host, "query_start_loc_host")
    sl_h = _host_i32(seq_lens_host, "seq_lens_host")
    if qsl_h.numel() != sl_h.numel() + 1:
        raise ValueError("query_start_loc needs num_reqs + 1 entries")
    _check_meta(query_start_loc, seq_lens, block_table, sl_h.numel())
    st = L.pkv_paged_kv_write_attention_ex(
        _dev(k, "k", torch.bfloat16), _dev(v, "v", torch.bfloat16),
        _dev(k_cache, "k_cache", torch.bfloat16), _dev(v_cache, "v_cache", torch.bfloat16),
        _dev(slot_mapping, "slot_mapping", torch.int64),
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16),
        _dev(query_start_loc, "query_start_loc", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        _dev(block_table, "block_table", torch.int32), block_table.shape[1],
        _c_p(qsl_h.data_ptr()), _c_p(sl_h.data_ptr()), sl_h.numel(), n, int(max_query_len), int(max_seq_len),
        hq, hkv, d, bs, nbt, float(scale), int(window), _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _opts(), _stream(stream))
    _check(st, "paged_kv_write_attention")


def clear_device_error(word: torch.Tensor, stream=None):
    """Zero a device error word (a CUDA int32 tensor, or the attention workspace)."""
    _check(load().pkv_clear_device_error(_c_p(word.data_ptr()), _stream(stream)), "clear_device_error")


def read_device_error(word: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the device error bits (0 when clean)."""
    flags = ctypes.c_uint32(0)
    st = load().pkv_read_device_error(_c_p(word.data_ptr()), ctypes.byref(flags), _stream(stream))
    if st not in (0, 5):
        _check(st, "read_device_error")
    return int(flags.value)


MAX_POOLS = 256


def _pool_array(pools):
    """Host array of the pools' device pointers; all pools share their block count and block bytes."""
    pools = list(pools)
    if not pools:
        raise ValueError("no pools")
    nbt = pools[0].shape[0]
    block_bytes = pools[0][0].numel() * pools[0].element_size()
    for i, t in enumerate(pools):
        _dev(t, f"pools[{i}]")
        if t.shape[0] != nbt or t[0].numel() * t.element_size() != block_bytes:
            raise ValueError("pools must share the number of blocks and the bytes per block")
    arr = (ctypes.c_void_p * len(pools))(*[t.data_ptr() for t in pools])
    return arr, len(pools), nbt, block_bytes


def _err(device_error):
    return _dev(device_error, "device_error", torch.int32) if device_error is not None else None


def _buf(t: torch.Tensor, name: str):
    """A device tensor, or pinned host memory the device can address."""
    if not isinstance(t, torch.Tensor) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor")
    if not t.is_cuda and not t.is_pinned():
        raise TypeError(f"{name} must be a CUDA tensor or pinned host memory")
    return _c_p(t.data_ptr())


def copy_blocks(pools, src_blocks, dst_blocks, device_error=None, stream=None):
    """Copy-on-write: block dst[i] := block src[i] in every pool ([nbt, ...] tensors)."""
    arr, n_pools, nbt, bb = _pool_array(pools)
    n = src_blocks.numel()
    if dst_blocks.numel() != n:
        raise ValueError("src_blocks and dst_blocks differ in length")
    _check(load().pkv_copy_blocks(arr, n_pools, _dev(src_blocks, "src_blocks", torch.int32),
                                  _dev(dst_blocks, "dst_blocks", torch.int32), n, nbt, bb, _err(device_error),
                                  _stream(stream)), "copy_blocks")


def gather_blocks(pools, blocks, out, device_error=None, stream=None):
    """Swap-out: out[q][i] = block blocks[i] of pool q; out holds len(pools) * len(blocks) blocks."""
    arr, n_pools, nbt, bb = _pool_array(pools)
    n = blocks.numel()
    if out.numel() * out.element_size() != n_pools * n * bb:
        raise ValueError("out must hold num_pools * num_blocks blocks")
    _check(load().pkv_gather_blocks(arr, n_pools, _dev(blocks, "blocks", torch.int32), n, nbt, bb,
                                    _buf(out, "out"), _err(device_error), _stream(stream)), "gather_blocks")


def scatter_blocks(pools, blocks, inp, device_error=None, stream=None):
    """Swap-in: block blocks[i] of pool q = inp[q][i] (the layout gather_blocks writes)."""
    arr, n_pools, nbt, bb = _pool_array(pools)
    n = blocks.numel()
    if inp.numel() * inp.element_size() != n_pools * n * bb:
        raise ValueError("inp must hold num_pools * num_blocks blocks")
    _check(load().pkv_scatter_blocks(arr, n_pools, _dev(blocks, "blocks", torch.int32), n, nbt, bb,
                                     _buf(inp, "inp"), _err(device_error), _stream(stream)), "scatter_blocks")



def paged_kv_write_attention_fp8(k, v, k_codes, v_codes, k_scale, v_scale, slot_mapping, out, q, query_start_loc,
                                 seq_lens, block_table, query_start_loc_host, seq_lens_host, max_query_len,
                                 max_seq_len, scale, workspace, stream=None, window: int = 0):
    """paged_kv_write_fp8 followed by ragged_paged_attention_fp8 in one call (decode CTAs quantize and
    write their own rows).  Write errors go to the workspace's error word."""
    L = load()
    n, hq, d = q.shape
    nbt, bs, hkv, d2 = k_codes.shape
    if out.shape != q.shape or d2 != d or v_codes.shape != k_codes.shape:
        raise ValueError("shape mismatch")
    if k.shape != (n, hkv, d) or v.shape != k.shape or slot_mapping.numel() != n:
        raise ValueError("k, v must be [num_tokens, num_kv_heads, head_dim] with one slot per token")
    if k_scale.shape != (nbt, bs, hkv) or v_scale.shape != k_scale.shape:
        raise ValueError("scales must be [num_blocks_total, block_size, num_kv_heads]")
    qsl_h = _host_i32(query_start_loc_host, "query_start_loc_host")
    sl_h = _host_i32(seq_lens_host, "seq_lens_host")
    if qsl_h.numel() != sl_h.numel() + 1:
        raise ValueError("query_start_loc needs num_reqs + 1 entries")
    _check_meta(query_start_loc, seq_lens, block_table, sl_h.numel())
    st = L.pkv_paged_kv_write_attention_fp8_ex(
        _dev(k, "k", torch.bfloat16), _dev(v, "v", torch.bfloat16),
        _dev(k_codes, "k_codes", torch.uint8), _dev(v_codes, "v_codes", torch.uint8),
        _dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32),
        _dev(slot_mapping, "slot_mapping", torch.int64),
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16),
        _dev(query_start_loc, "query_start_loc", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        _dev(block_table, "block_table", torch.int32), block_table.shape[1],
        _c_p(qsl_h.data_ptr()), _c_p(sl_h.data_ptr()), sl_h.numel(), n, int(max_query_len), int(max_seq_len),
        hq, hkv, d, bs, nbt, float(scale), int(window), _dev(workspace, "workspace", torch.uint8), workspace.numel(),
        _opts(), _stream(stream))
    _check(st, "paged_kv_write_attention_fp8")


def fp8_prefill_scratch_bytes(query_start_loc_host, seq_lens_host, num_q_heads, num_kv_heads, head_dim) -> int:
    """Extra workspace bytes that put this batch's quantized-pool prefill on the tcgen05 kernel."""
    qsl = _host_i32(query_start_loc_host, "query_start_loc_host")
    sl = _host_i32(seq_lens_host, "seq_lens_host")
    return int(load().pkv_fp8_prefill_scratch_bytes(_c_p(qsl.data_ptr()), _c_p(sl.data_ptr()), sl.numel(),
                                                    num_q_heads, num_kv_heads, head_dim))


def copy_async(dst, src, stream=None):
    """dst := src (same byte size) with a copy kernel; either may be a CUDA
    tensor or pinned host memory the device can address."""
    n = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != n:
        raise ValueError("dst and src differ in byte size")
    _check(load().pkv_copy_async(_buf(dst, "dst"), _buf(src, "src"), n, _stream(stream)), "copy_async")


def paged_kv_write_fp8(k, v, k_codes, v_codes, k_scale, v_scale, slot_mapping, device_error=None, stream=None):
    """Quantizing write: k, v bf16 [N, Hkv, d] -> E4M3 codes uint8 [nbt, bs, Hkv, d] and fp32 scales
    [nbt, bs, Hkv] at ``slot_mapping``."""
    L = load()
    n, hkv, d = k.shape
    nbt, bs, hkv2, d2 = k_codes.shape
    if (hkv2, d2) != (hkv, d) or v.shape != k.shape or v_codes.shape != k_codes.shape:
        raise ValueError("shape mismatch between k/v and the pools")
    if k_scale.shape != (nbt, bs, hkv) or v_scale.shape != (nbt, bs, hkv):
        raise ValueError("scale pools must be [num_blocks, block_size, num_kv_heads]")
    st = L.pkv_paged_kv_write_fp8(_dev(k, "k", torch.bfloat16), _dev(v, "v", torch.bfloat16),
                                  _dev(k_codes, "k_codes", torch.uint8), _dev(v_codes, "v_codes", torch.uint8),
                                  _dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32),
                                  _dev(slot_mapping, "slot_mapping", torch.int64), n, hkv, d, bs, nbt,
                                  _err(device_error), _stream(stream))
    _check(st, "paged_kv_write_fp8")


def ragged_paged_attention_fp8(out, q, k_codes, v_codes, k_scale, v_scale, query_start_loc, seq_lens,
                               block_table, query_start_loc_host, seq_lens_host, max_query_len, max_seq_len,
                               scale, workspace, stream=None, window: int = 0):
    """ragged_paged_attention over a quantized pool (E4M3 codes times per (slot, head) scales)."""
    L = load()
    n, hq, d = q.shape
    nbt, bs, hkv, d2 = k_codes.shape
    if out.shape != q.shape or d2 != d or v_codes.shape != k_codes.shape:
        raise ValueError("shape mismatch")
    qsl_h = _host_i32(query_start_loc_host, "query_start_loc_host")
    sl_h = _host_i32(seq_lens_host, "seq_lens_host")
    if qsl_h.numel() != sl_h.numel() + 1:
        raise ValueError("query_start_loc needs num_reqs + 1 entries")
    _check_meta(query_start_loc, seq_lens, block_table, sl_h.numel())
    st = L.pkv_ragged_paged_attention_fp8_ex(
        _dev(out, "out", torch.bfloat16), _dev(q, "q", torch.bfloat16),
        _dev(k_codes, "k_codes", torch.uint8), _dev(v_codes, "v_codes", torch.uint8),
        _dev(k_scale, "k_scale", torch.float32), _dev(v_scale, "v_scale", torch.float32),
        _dev(query_start_loc, "query_start_loc", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
        _dev(block_table, "block_table", torch.int32), block_table.shape[1],
        _c_p(qsl_h.data_ptr()), _c_p(sl_h.data_ptr()), sl_h.numel(), n, int(max_query_len), int(max_seq_len),
        hq, hkv, d, bs, nbt, float(scale), int(window), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), _opts(), _stream(stream))
    _check(st, "ragged_paged_attention_fp8")
