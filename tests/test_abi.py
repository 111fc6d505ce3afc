"""The C ABI on a host without a GPU: the library loads, exports every
function include/pkv.h declares, and its host-only logic (status strings,
workspace sizing, request classification, argument validation) answers
without touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_84_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_two_calls():
    names = declared()
    assert "pkv_paged_kv_write" in names and "pkv_ragged_paged_attention" in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pkv_\w+)", out))
    assert set(declared()) <= exported


def test_header_compiles_as_c():
    src = '#include "pkv.h"\nint main(void){return (int)PKV_OK;}\n'
    r = subprocess.run(["gcc", "-x", "c", "-std=c99", "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
                        "-I", "/usr/local/cuda/include", "-"], input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_host_only_functions(lib):
    import paged_kv_cache_84_gb300 as pkv
    lib.pkv_status_string.restype = ctypes.c_char_p
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(3).startswith(b"workspace")
    assert pkv.attention_workspace_bytes(0, 0, 8, 64, 0) == pkv.WORKSPACE_MIN_BYTES
    small = pkv.attention_workspace_bytes(4, 9, 8, 48, 42)
    big = pkv.attention_workspace_bytes(32, 32, 64, 128, 32768)
    assert pkv.WORKSPACE_MIN_BYTES < small < big
    # layout example: every request is decode-class (t * g <= 16)
    assert pkv.plan_request_kernels([0, 3, 4, 5, 9], [9, 42, 10, 4], 8, 4, 48) == ["decode"] * 4
    # a 64-token chunk with g = 2 is a tensor-core tile job; seq_len 0 is padding; t = 0 is nothing
    assert pkv.plan_request_kernels([0, 64, 65, 65], [300, 0, 7], 8, 4, 48) == \
        ["prefill_tensor", "padding", "none"]
    # 18 rows (t = 6, g = 3) exceed a decode tile; g = 3 does not divide the
    # 128-row tensor-core tile, so the chunk runs on the warp-level MMA kernel
    assert pkv.plan_request_kernels([0, 6], [40], 9, 3, 64) == ["prefill_mma"]


def _attn_args(qsl, sl, R, N, maxq, maxl, hq=8, hkv=4, d=64, bs=16, stride=4, ws=1 << 20, window=0):
    fake = ctypes.c_void_p(1 << 20)                 # never dereferenced: validation fails first
    qsl_h = (ctypes.c_int32 * len(qsl))(*qsl)
    sl_h = (ctypes.c_int32 * max(1, len(sl)))(*sl)
    return [fake] * 7 + [stride, qsl_h, sl_h, R, N, maxq, maxl, hq, hkv, d, bs, 100, ctypes.c_float(0.1),
                         ctypes.c_int32(window), fake, ctypes.c_size_t(ws), None]


@pytest.mark.parametrize("qsl,sl,maxq,maxl,kw", [
    ([0, 3, 2, 5], [9, 9, 9], 3, 9, {}),             # not non-decreasing
    ([0, 3, 4, 6], [9, 9, 9], 3, 9, {}),             # does not end at N
    ([0, 3, 4, 5], [2, 9, 9], 3, 9, {}),             # t > L
    ([0, 3, 4, 5], [9, 99, 9], 3, 99, {}),           # table narrower than ceil(L / 16)
    ([0, 3, 4, 5], [9, 9, 9], 2, 9, {}),             # max_query_len below the data
    ([0, 3, 4, 5], [9, 9, 9], 3, 8, {}),             # max_seq_len below the data
    ([0, 3, 4, 5], [9, 9, 9], 3, 9, {"hkv": 3}),     # hq % hkv != 0
    ([0, 3, 4, 5], [9, 9, 9], 3, 9, {"window": -1}), # negative window
])
def test_attention_host_validation(lib, qsl, sl, maxq, maxl, kw):
    lib.pkv_ragged_paged_attention.restype = ctypes.c_int
    args = _attn_args(qsl, sl, len(sl), 5, maxq, maxl, **kw)
    assert lib.pkv_ragged_paged_attention(*args) == 1


def test_attention_unsupported_and_workspace(lib):
    lib.pkv_ragged_paged_attention.restype = ctypes.c_int
    assert lib.pkv_ragged_paged_attention(*_attn_args([0, 1], [5], 1, 1, 1, 5, d=96)) == 2
    assert lib.pkv_ragged_paged_attention(*_attn_args([0, 1], [5], 1, 1, 1, 5, bs=48)) == 2   # not 16 << k
    assert lib.pkv_ragged_paged_attention(*_attn_args([0, 1], [5], 1, 1, 1, 5, ws=64)) == 3


def test_write_host_validation(lib):
    lib.pkv_paged_kv_write.restype = ctypes.c_int
    fake = ctypes.c_void_p(1 << 20)
    assert lib.pkv_paged_kv_write(fake, fake, fake, fake, fake, -1, 4, 64, 16, 10, None, None) == 1
    assert lib.pkv_paged_kv_write(fake, fake, fake, fake, fake, 0, 4, 64, 16, 10, None, None) == 0
    assert lib.pkv_paged_kv_write(fake, fake, fake, fake, fake, 3, 4, 60, 16, 10, None, None) == 2
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert lib.pkv_paged_kv_write(odd, fake, fake, fake, fake, 3, 4, 64, 16, 10, None, None) == 2


def test_block_copy_validation_on_host(lib):
    """Block-copy calls reject bad arguments before touching the device."""
    P = ctypes.c_void_p
    fake = (P * 2)(1 << 20, 1 << 21)                 # never dereferenced: validation fails first
    ids = P(1 << 22)
    for fn in (lib.pkv_copy_blocks, lib.pkv_gather_blocks, lib.pkv_scatter_blocks):
        fn.restype = ctypes.c_int
    # zero pools, too many pools, zero block bytes: invalid
    assert lib.pkv_copy_blocks(fake, 0, ids, ids, 4, 10, ctypes.c_size_t(512), None, None) == 1
    assert lib.pkv_copy_blocks(fake, 257, ids, ids, 4, 10, ctypes.c_size_t(512), None, None) == 1
    assert lib.pkv_copy_blocks(fake, 2, ids, ids, 4, 10, ctypes.c_size_t(0), None, None) == 1
    # zero pairs: a no-op
    assert lib.pkv_copy_blocks(fake, 2, ids, ids, 0, 10, ctypes.c_size_t(512), None, None) == 0
    # missing destination list / buffer: invalid
    assert lib.pkv_copy_blocks(fake, 2, ids, None, 4, 10, ctypes.c_size_t(512), None, None) == 1
    assert lib.pkv_gather_blocks(fake, 2, ids, 4, 10, ctypes.c_size_t(512), None, None, None) == 1
    # block bytes not a multiple of 16, or a misaligned buffer: unsupported
    assert lib.pkv_copy_blocks(fake, 2, ids, ids, 4, 10, ctypes.c_size_t(520), None, None) == 2
    assert lib.pkv_scatter_blocks(fake, 2, ids, 4, 10, ctypes.c_size_t(512), P((1 << 22) + 8), None, None) == 2
    odd = (P * 2)(1 << 20, (1 << 21) + 4)
    assert lib.pkv_copy_blocks(odd, 2, ids, ids, 4, 10, ctypes.c_size_t(512), None, None) == 2


def test_copy_async_validation_on_host(lib):
    """pkv_copy_async rejects what it cannot copy before touching the device."""
    lib.pkv_copy_async.restype = ctypes.c_int
    lib.pkv_copy_async.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    a, b = 1 << 20, 1 << 24                                 # never dereferenced: validation fails first
    assert lib.pkv_copy_async(a, b, 0, None) == 0          # zero bytes: no-op
    assert lib.pkv_copy_async(None, b, 64, None) == 1
    assert lib.pkv_copy_async(a, None, 64, None) == 1
    assert lib.pkv_copy_async(a, a + 32, 64, None) == 1     # overlapping ranges
    assert lib.pkv_copy_async(a, b, 24, None) == 2          # not a multiple of 16 bytes
    assert lib.pkv_copy_async(a + 8, b, 64, None) == 2      # unaligned
    assert lib.pkv_copy_async(a, b + 8, 64, None) == 2



def test_fp8_prefill_scratch_bytes_on_host(lib):
    """The extra workspace for quantized prefill on tcgen05: bf16 K and V
    copies of the qualifying chunks' blocks plus a block table, 256-byte
    aligned parts; nothing for decodes, short chunks or head dims other
    than 128."""
    fn = lib.pkv_fp8_prefill_scratch_bytes
    fn.restype = ctypes.c_size_t
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]

    def call(qsl, sl, hq, hkv, d):
        q = (ctypes.c_int32 * len(qsl))(*qsl)
        s = (ctypes.c_int32 * len(sl))(*sl)
        return fn(q, s, len(sl), hq, hkv, d)

    # a 40-token chunk at 1000 keys (g = 4: 160 rows), a decode, a 3-token chunk (12 rows: decode class)
    qsl, sl = [0, 40, 41, 44], [1040, 77, 500]
    blocks, width = 65, 65                                 # ceil(1040 / 16)
    kv = blocks * 16 * 8 * 128 * 2
    want = 256 + 2 * ((kv + 255) // 256 * 256) + (3 * width * 4 + 255) // 256 * 256
    assert call(qsl, sl, 32, 8, 128) == want
    assert call([0, 1, 2], [77, 500], 32, 8, 128) == 0      # decodes only
    assert call(qsl, sl, 32, 8, 48) == 0                    # head dim 48: no tcgen05 path for codes
    assert call(qsl, sl, 24, 8, 128) == 0                   # g = 3 does not divide 128


def test_noalloc_scratch_fits_every_workload_plan(lib):
    """The no-allocation call's static scratch: its size as the header states
    it, and the planner's split plan for each of the five workloads fits it
    (the planner lengthens splits where the natural plan would not), so the
    call refuses none of them.  Host only."""
    fn = lib.pkv_noalloc_scratch_bytes
    fn.restype = ctypes.c_size_t
    fn.argtypes = []
    scratch = int(fn())
    assert scratch == 8 << 20
    assert re.search(r"#define PKV_NOALLOC_SCRATCH_BYTES \(8u << 20\)", open(HEADER).read())
    import paged_kv_cache_84_gb300 as pkv
    from workloads import build_meta, config_spec
    for cfg in range(1, 6):
        s = config_spec(cfg)
        m = build_meta(s)
        plan = pkv.plan_attention(m.query_start_loc, m.seq_lens, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                  workspace_bytes=scratch, num_sms=152)
        front = 256 + (65536 if plan["split_counters"] else 0)
        assert plan["partial_bytes"] + front <= scratch, cfg


def _c_layout(struct, fields, tmp_path):
    """sizeof and every field's offsetof of `struct` as the C compiler lays it
    out from include/pkv.h."""
    lines = [f'printf("%zu\\n", sizeof({struct}));']
    lines += [f'printf("%zu\\n", offsetof({struct}, {f}));' for f in fields]
    src = ('#include <stddef.h>\n#include <stdio.h>\n#include "pkv.h"\nint main(void){\n' + "\n".join(lines) +
           '\nreturn 0;}\n')
    exe = str(tmp_path / "layout")
    r = subprocess.run(["gcc", "-x", "c", "-std=c99", "-I", os.path.join(ROOT, "include"), "-I",
                        "/usr/local/cuda/include", "-o", exe, "-"], input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    vals = [int(v) for v in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    return vals[0], dict(zip(fields, vals[1:]))


@pytest.mark.parametrize("struct, name", [("pkv_attention_plan", "_Plan"),
                                          ("pkv_attention_options", "AttentionOptions")])
def test_binding_structs_match_the_header(struct, name, tmp_path):
    """The ctypes mirrors of the header's structs have the C layout: the same
    fields in the same order at the same offsets, and the same size."""
    import paged_kv_cache_84_gb300 as pkv
    cls = getattr(pkv, name)
    fields = [f for f, _ in cls._fields_]
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct %s \{(.*?)\}" % struct, text, flags=re.S).group(1)
    assert re.findall(r"\b(\w+);", body) == fields
    size, offsets = _c_layout(struct, fields, tmp_path)
    assert ctypes.sizeof(cls) == size
    assert {f: getattr(cls, f).offset for f in fields} == offsets
