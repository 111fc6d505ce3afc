"""The five synthetic workloads have the shapes they are built to have: the
pages' layout example, the 48-request engine step with a physically shared
256-token system prompt, the 256-request decode batch, the mixed chunked
prefill step and the 32-request long decode (head counts, head dim, block
size, context ranges, token budgets, pool sizes, block tables inside the
pool and private except for the shared prefix)."""
import math

import pytest

from workloads import build_meta, config_spec


def _tables_ok(spec, shared=0):
    seen = set()
    for r in spec.reqs:
        assert len(r.table) >= -(-r.seq_len // spec.block_size)
        assert all(0 <= b < spec.num_blocks for b in r.table)
        private = r.table[shared:]
        assert len(set(private)) == len(private) and not seen & set(private)
        seen.update(private)
    if shared:
        first = spec.reqs[0].table[:shared]
        assert all(r.table[:shared] == first for r in spec.reqs) and not seen & set(first)


def _common(spec, hq, hkv, d):
    assert (spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.block_size) == (hq, hkv, d, 16)
    assert spec.scale == pytest.approx(1.0 / math.sqrt(d))


def test_layout_example():
    spec = config_spec(1)
    _common(spec, 8, 4, 48)
    m = build_meta(spec)
    assert m.query_start_loc == [0, 3, 4, 5, 9] and m.seq_lens == [9, 42, 10, 4]
    assert spec.num_blocks == 64
    _tables_ok(spec)


def test_engine_step_with_shared_prefix():
    spec = config_spec(2)
    _common(spec, 8, 4, 48)
    chunks = [r for r in spec.reqs if r.new > 1]
    decodes = [r for r in spec.reqs if r.new == 1]
    assert len(spec.reqs) == 48 and len(chunks) == 16 and len(decodes) == 32
    assert all(r.new <= 64 and r.computed >= 256 and (r.computed - 256) % 64 == 0 for r in chunks)
    assert all(256 + 17 + 20 <= r.seq_len <= 256 + 251 + 192 for r in decodes)
    assert sum(r.new for r in spec.reqs) <= 2048
    _tables_ok(spec, shared=16)


def test_decode_batch():
    spec = config_spec(3)
    _common(spec, 32, 8, 128)
    assert len(spec.reqs) == 256 and all(r.new == 1 for r in spec.reqs)
    assert all(512 <= r.seq_len <= 8192 for r in spec.reqs)
    used = sum(-(-r.seq_len // 16) for r in spec.reqs)
    assert spec.num_blocks == math.ceil(1.1 * used)
    _tables_ok(spec)


def test_mixed_chunked_prefill_step():
    spec = config_spec(4)
    _common(spec, 32, 8, 128)
    chunk = [r for r in spec.reqs if r.new == 2048]
    fresh = [r for r in spec.reqs if r.new == 1024]
    decodes = [r for r in spec.reqs if r.new == 1]
    assert len(chunk) == 1 and chunk[0].computed == 16384 and chunk[0].seq_len == 18432
    assert len(fresh) == 2 and all(r.computed == 0 for r in fresh)
    assert len(decodes) == 64 and all(1024 <= r.seq_len <= 4096 for r in decodes)
    assert sum(r.new for r in spec.reqs) == 4160 <= 8192
    _tables_ok(spec)


def test_long_decode():
    spec = config_spec(5)
    _common(spec, 64, 8, 128)
    assert len(spec.reqs) == 32 and all(r.new == 1 and r.seq_len == 32768 for r in spec.reqs)
    assert all(len(r.table) == 2048 for r in spec.reqs) and spec.num_blocks == 70000
    _tables_ok(spec)
