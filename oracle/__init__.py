"""Python handle on the CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use it; the library path never does.  It
shares no code with the CUDA library.  Arguments are CPU torch tensors
(bf16 values are passed as their raw 16-bit patterns).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
# A prebuilt oracle library to load instead (the mutation test points this
# at deliberately broken copies to show that the pins catch them).
_OVERRIDE = os.environ.get("PKV_ORACLE_LIB")
_lib = None

c_i32, c_i64, c_dbl, c_p = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc (plain -O2, OpenMP, no fast-math)."""
    if _OVERRIDE:
        return _OVERRIDE
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.oracle_slot.restype = c_i64
        L.oracle_slot.argtypes = [c_p, c_i64, c_i32]
        L.oracle_paged_kv_write.restype = ctypes.c_int
        L.oracle_paged_kv_write.argtypes = [c_p, c_p, c_p, c_p, c_p, c_i32, c_i32, c_i32, c_i32, c_i32]
        L.oracle_ragged_paged_attention.restype = ctypes.c_int
        L.oracle_ragged_paged_attention.argtypes = [c_p] + [c_p] * 3 + [c_p, c_p, c_p, c_i32] + \
            [c_i32] * 7 + [c_dbl, c_i32, c_i32]
        L.oracle_attention_rows.restype = ctypes.c_int
        L.oracle_attention_rows.argtypes = [c_p, c_p, c_p, c_i32] + [c_p] * 3 + [c_p, c_p, c_p, c_i32] + \
            [c_i32] * 7 + [c_dbl, c_i32, c_i32]
        L.oracle_max_threads.restype = ctypes.c_int
        L.oracle_max_threads.argtypes = []
        L.oracle_e4m3_decode.restype = c_dbl
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_paged_kv_write_fp8.restype = ctypes.c_int
        L.oracle_paged_kv_write_fp8.argtypes = [c_p] * 7 + [c_i32] * 5
        L.oracle_ragged_paged_attention_fp8.restype = ctypes.c_int
        L.oracle_ragged_paged_attention_fp8.argtypes = [c_p] * 6 + [c_p, c_p, c_p, c_i32] + [c_i32] * 7 + \
            [c_dbl, c_i32, c_i32]
        L.oracle_attention_rows_fp8.restype = ctypes.c_int
        L.oracle_attention_rows_fp8.argtypes = [c_p, c_p, c_p, c_i32] + [c_p] * 5 + [c_p, c_p, c_p, c_i32] + \
            [c_i32] * 7 + [c_dbl, c_i32, c_i32]
        for name in ("oracle_copy_blocks", "oracle_gather_blocks", "oracle_scatter_blocks"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [c_p, c_p, c_p, c_i32, c_i32, c_i64]
        _lib = L
    return _lib


def _ptr(t: torch.Tensor):
    assert t.device.type == "cpu" and t.is_contiguous()
    return ctypes.c_void_p(t.data_ptr())


def _bits(t: torch.Tensor) -> torch.Tensor:
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16)


def max_threads() -> int:
    return lib().oracle_max_threads()


def slot(table_row, p: int, block_size: int) -> int:
    t = torch.as_tensor(table_row, dtype=torch.int32).contiguous()
    return int(lib().oracle_slot(_ptr(t), p, block_size))


def paged_kv_write(k_cache, v_cache, k, v, slot_mapping, block_size=None):
    """In place on the CPU bf16 pools ``k_cache``/``v_cache`` [nbt, bs, Hkv, d]."""
    nbt, bs, hkv, d = k_cache.shape
    kb, vb = _bits(k), _bits(v)
    sm = slot_mapping.to(torch.int64).contiguous()
    rc = lib().oracle_paged_kv_write(_ptr(k_cache.view(torch.int16)), _ptr(v_cache.view(torch.int16)),
                                     _ptr(kb), _ptr(vb), _ptr(sm), sm.numel(), hkv, d, bs, nbt)
    if rc:
        raise ValueError(f"oracle_paged_kv_write: {rc}")


def _meta_tensors(query_start_loc, seq_lens, block_table):
    qsl = torch.as_tensor(query_start_loc, dtype=torch.int32).contiguous()
    sl = torch.as_tensor(seq_lens, dtype=torch.int32).contiguous()
    bt = block_table.to(torch.int32).contiguous()
    return qsl, sl, bt


def ragged_paged_attention(q, k_cache, v_cache, query_start_loc, seq_lens, block_table, scale,
                           threads: int = 1, window: int = 0) -> torch.Tensor:
    """Returns float64 [N, Hq, d]; ``window`` > 0 keeps only keys above position - window."""
    n, hq, d = q.shape
    nbt, bs, hkv, _ = k_cache.shape
    qsl, sl, bt = _meta_tensors(query_start_loc, seq_lens, block_table)
    out = torch.empty((n, hq, d), dtype=torch.float64)
    rc = lib().oracle_ragged_paged_attention(
        _ptr(out), _ptr(_bits(q)), _ptr(_bits(k_cache)), _ptr(_bits(v_cache)),
        _ptr(qsl), _ptr(sl), _ptr(bt), bt.shape[1], sl.numel(), n, hq, hkv, d, bs, nbt,
        float(scale), int(window), threads)
    if rc:
        raise ValueError(f"oracle_ragged_paged_attention: {rc}")
    return out


def attention_rows(tokens, heads, q, k_cache, v_cache, query_start_loc, seq_lens, block_table, scale,
                   threads: int = 1, window: int = 0) -> torch.Tensor:
    """Outputs of the listed (token, head) pairs only: float64 [len(tokens), d]."""
    n, hq, d = q.shape
    nbt, bs, hkv, _ = k_cache.shape
    qsl, sl, bt = _meta_tensors(query_start_loc, seq_lens, block_table)
    tk = torch.as_tensor(tokens, dtype=torch.int32).contiguous()
    hd = torch.as_tensor(heads, dtype=torch.int32).contiguous()
    out = torch.empty((tk.numel(), d), dtype=torch.float64)
    rc = lib().oracle_attention_rows(
        _ptr(out), _ptr(tk), _ptr(hd), tk.numel(), _ptr(_bits(q)), _ptr(_bits(k_cache)),
        _ptr(_bits(v_cache)), _ptr(qsl), _ptr(sl), _ptr(bt), bt.shape[1], sl.numel(), n, hq, hkv,
        d, bs, nbt, float(scale), int(window), threads)
    if rc:
        raise ValueError(f"oracle_attention_rows: {rc}")
    return out


def _pool_bytes(pool: torch.Tensor):
    """A CPU pool [nbt, ...] as raw bytes, with its block count and bytes per block."""
    assert pool.device.type == "cpu" and pool.is_contiguous()
    nbt = pool.shape[0]
    return pool.view(torch.uint8).view(nbt, -1), nbt, pool[0].numel() * pool.element_size()


def copy_blocks(pools, src_blocks, dst_blocks):
    """In every CPU pool, in list order: block dst[i] := block src[i]."""
    src = torch.as_tensor(src_blocks, dtype=torch.int32).contiguous()
    dst = torch.as_tensor(dst_blocks, dtype=torch.int32).contiguous()
    for pool in pools:
        raw, nbt, bb = _pool_bytes(pool)
        rc = lib().oracle_copy_blocks(_ptr(raw), _ptr(src), _ptr(dst), src.numel(), nbt, bb)
        if rc:
            raise ValueError(f"oracle_copy_blocks: {rc}")


def gather_blocks(pools, blocks) -> torch.Tensor:
    """uint8 [len(pools), len(blocks), bytes per block]: block blocks[i] of pool q."""
    ids = torch.as_tensor(blocks, dtype=torch.int32).contiguous()
    outs = []
    for pool in pools:
        raw, nbt, bb = _pool_bytes(pool)
        out = torch.empty((ids.numel(), bb), dtype=torch.uint8)
        rc = lib().oracle_gather_blocks(_ptr(out), _ptr(raw), _ptr(ids), ids.numel(), nbt, bb)
        if rc:
            raise ValueError(f"oracle_gather_blocks: {rc}")
        outs.append(out)
    return torch.stack(outs)


def scatter_blocks(pools, blocks, inp: torch.Tensor):
    """Block blocks[i] of pool q := inp[q][i] (uint8 [len(pools), len(blocks), bytes per block])."""
    ids = torch.as_tensor(blocks, dtype=torch.int32).contiguous()
    for q, pool in enumerate(pools):
        raw, nbt, bb = _pool_bytes(pool)
        src = inp[q].contiguous()
        rc = lib().oracle_scatter_blocks(_ptr(raw), _ptr(src), _ptr(ids), ids.numel(), nbt, bb)
        if rc:
            raise ValueError(f"oracle_scatter_blocks: {rc}")


# ---------------------------------------------------------------- quantized pools

def e4m3_encode(x: float) -> int:
    """fp32 value -> E4M3 code (round to nearest even, saturating at +-448)."""
    return int(lib().oracle_e4m3_encode(float(x)))


def e4m3_decode(code: int) -> float:
    return float(lib().oracle_e4m3_decode(int(code) & 0xFF))


def paged_kv_write_fp8(k_codes, v_codes, k_scale, v_scale, k, v, slot_mapping):
    """Quantizing write on CPU pools: codes uint8 [nbt, bs, Hkv, d], scales float32 [nbt, bs, Hkv]."""
    nbt, bs, hkv, d = k_codes.shape
    for t in (k_codes, v_codes, k_scale, v_scale):
        assert t.is_contiguous() and t.device.type == "cpu"
    sm = slot_mapping.to(torch.int64).contiguous()
    rc = lib().oracle_paged_kv_write_fp8(_ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
                                         _ptr(_bits(k)), _ptr(_bits(v)), _ptr(sm), sm.numel(), hkv, d, bs, nbt)
    if rc:
        raise ValueError(f"oracle_paged_kv_write_fp8: {rc}")


def ragged_paged_attention_fp8(q, k_codes, v_codes, k_scale, v_scale, query_start_loc, seq_lens, block_table,
                               scale, threads: int = 1, window: int = 0) -> torch.Tensor:
    """Attention over a quantized pool; returns float64 [N, Hq, d]."""
    n, hq, d = q.shape
    nbt, bs, hkv, _ = k_codes.shape
    qsl, sl, bt = _meta_tensors(query_start_loc, seq_lens, block_table)
    out = torch.empty((n, hq, d), dtype=torch.float64)
    rc = lib().oracle_ragged_paged_attention_fp8(
        _ptr(out), _ptr(_bits(q)), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
        _ptr(qsl), _ptr(sl), _ptr(bt), bt.shape[1], sl.numel(), n, hq, hkv, d, bs, nbt,
        float(scale), int(window), threads)
    if rc:
        raise ValueError(f"oracle_ragged_paged_attention_fp8: {rc}")
    return out


def attention_rows_fp8(tokens, heads, q, k_codes, v_codes, k_scale, v_scale, query_start_loc, seq_lens,
                       block_table, scale, threads: int = 1, window: int = 0) -> torch.Tensor:
    n, hq, d = q.shape
    nbt, bs, hkv, _ = k_codes.shape
    qsl, sl, bt = _meta_tensors(query_start_loc, seq_lens, block_table)
    tk = torch.as_tensor(tokens, dtype=torch.int32).contiguous()
    hd = torch.as_tensor(heads, dtype=torch.int32).contiguous()
    out = torch.empty((tk.numel(), d), dtype=torch.float64)
    rc = lib().oracle_attention_rows_fp8(
        _ptr(out), _ptr(tk), _ptr(hd), tk.numel(), _ptr(_bits(q)), _ptr(k_codes), _ptr(v_codes),
        _ptr(k_scale), _ptr(v_scale), _ptr(qsl), _ptr(sl), _ptr(bt), bt.shape[1], sl.numel(), n, hq, hkv,
        d, bs, nbt, float(scale), int(window), threads)
    if rc:
        raise ValueError(f"oracle_attention_rows_fp8: {rc}")
    return out
