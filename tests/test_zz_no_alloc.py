"""pkv_ragged_paged_attention_noalloc, called through the C ABI.

This entry point is for callers that cannot allocate device memory: plain C
hosts without a device allocator, and serving loops that must not call
cudaMalloc because it can synchronise the device or because their memory
budget is fixed at start-up.  It keeps its split-KV partials, split
counters and error word in a static array inside the library.  Its output
is checked against the oracle within the parity tolerance, and against the
workspace entry point, on calls made back to back that reuse the array.
This file is collected last, so that a run stopping at its first failure
has run every other test before it.
"""
import ctypes

import pytest
import torch

import oracle
import paged_kv_cache_84_gb300 as pkv
from workloads import config_spec, make_batch, random_spec
from _helpers import (DeviceStep, MAX_ERR, MEAN_ERR, assert_close, cpu_copy, oracle_full, oracle_write,
                      threads)

pytestmark = pytest.mark.gpu

_p, _i32 = ctypes.c_void_p, ctypes.c_int32


def _fn():
    fn = pkv.load().pkv_ragged_paged_attention_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [_p] * 7 + [_i32, _p, _p] + [_i32] * 9 + [ctypes.c_float, _i32, _p, _p]
    return fn


def _scratch_bytes():
    fn = pkv.load().pkv_noalloc_scratch_bytes
    fn.restype = ctypes.c_size_t
    fn.argtypes = []
    return int(fn())


def _call(dev: DeviceStep, bt=None, device_error=None):
    m, s = dev.batch.meta, dev.batch.spec
    bt = dev.bt if bt is None else bt
    qsl_h = torch.tensor(m.query_start_loc, dtype=torch.int32)
    sl_h = torch.tensor(m.seq_lens, dtype=torch.int32)
    out = torch.full_like(dev.q, float("nan"))
    st = _fn()(out.data_ptr(), dev.q.data_ptr(), dev.k_cache.data_ptr(), dev.v_cache.data_ptr(),
               dev.qsl.data_ptr(), dev.sl.data_ptr(), bt.data_ptr(), bt.shape[1], qsl_h.data_ptr(),
               sl_h.data_ptr(), m.num_reqs, m.num_tokens, m.max_query_len, m.max_seq_len, s.num_q_heads,
               s.num_kv_heads, s.head_dim, s.block_size, s.num_blocks_total, s.scale, 0,
               None if device_error is None else device_error.data_ptr(),
               torch.cuda.current_stream().cuda_stream)
    return st, out


def _close(a, b):
    d = (a.double() - b.double()).abs()
    return torch.isfinite(a.float()).all().item() and d.max().item() <= MAX_ERR and d.mean().item() <= MEAN_ERR


def _split_batch():
    # eight decodes over ~3000 keys: the planner splits each over many CTAs
    # (256-key splits merged by split counters), so the partials and the
    # counters really pass through the static array
    return random_spec(81, 8, 3200, 1, 32, 8, 128, decode_frac=1.0)


def test_noalloc_matches_oracle_on_two_calls_in_a_row():
    steps, refs = [], []
    for spec in (config_spec(2), _split_batch()):
        b = make_batch(spec, device="cpu")
        ref = cpu_copy(b)
        oracle_write(ref)
        dev = DeviceStep(b)
        dev.write()
        dev.attend()                                   # the workspace entry point, for comparison
        steps.append(dev)
        refs.append(oracle_full(ref))
    torch.cuda.synchronize()
    plan = pkv.plan_attention(steps[1].batch.meta.query_start_loc, steps[1].batch.meta.seq_lens, 32, 8, 128,
                              workspace_bytes=_scratch_bytes())
    assert plan["max_decode_splits"] > 1
    for order in (range(2), reversed(range(2))):      # twice, the second time after the other batch
        outs = {}
        pkv.profile_start(64)
        for i in order:
            st, out = _call(steps[i])
            assert st == 0
            outs[i] = out
        kernels = [name for name, _ in pkv.profile_stop()]
        assert "attn_mma_decode" in kernels
        for i, out in outs.items():
            assert_close(out, refs[i], f"no-allocation call, batch {i}")
            assert _close(out, steps[i].out)


@pytest.mark.parametrize("cfg", [3, 5], ids=["decode-256req", "long-decode-32req"])
def test_noalloc_full_size_decode_batches(cfg):
    """The two large decode batches need more than the array for their
    natural split plan; the planner splits them less and the results stay
    within the tolerance of the oracle (sampled rows) and of the workspace
    entry point."""
    spec = config_spec(cfg)
    b = make_batch(spec, device="cuda")
    ref = cpu_copy(b)
    oracle_write(ref)
    m = b.meta
    scratch = _scratch_bytes()
    assert pkv.attention_workspace_bytes(m.num_reqs, m.num_tokens, spec.num_q_heads, spec.head_dim,
                                         m.max_seq_len) > scratch
    plan = pkv.plan_attention(m.query_start_loc, m.seq_lens, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                              workspace_bytes=scratch)
    assert plan["partial_bytes"] <= scratch and plan["max_decode_splits"] > 1
    dev = DeviceStep(b)
    dev.write()
    dev.attend()
    err = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    for _ in range(2):
        st, out = _call(dev, device_error=err)
        assert st == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert _close(out, dev.out)
    gen = torch.Generator().manual_seed(300 + cfg)
    toks = list(range(m.num_tokens))
    heads = torch.randint(0, spec.num_q_heads, (len(toks),), generator=gen).tolist()
    want = oracle.attention_rows(toks, heads, ref.q, ref.k_cache, ref.v_cache, m.query_start_loc, m.seq_lens,
                                 m.block_table, spec.scale, threads())
    assert_close(out[torch.tensor(toks), torch.tensor(heads)], want, f"no-allocation call, {spec.name}")


def test_noalloc_reports_bounds_flags_per_call():
    b = make_batch(random_spec(82, 5, 400, 3, 8, 4, 64), device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    dev = DeviceStep(b)
    dev.write()
    err = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    bad = dev.bt.clone()
    bad[0, 0] = dev.batch.spec.num_blocks_total + 3
    st, _ = _call(dev, bt=bad, device_error=err)
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEVERR_BLOCK
    st, out = _call(dev, device_error=err)             # the word was cleared at the start of this call
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(out, oracle_full(ref), "no-allocation call after a flagged call")


def test_noalloc_blocks_of_64_slots():
    """Blocks of 64 slots: the array also holds the block table in 16-slot
    entries, and the results match the oracle and the workspace entry point."""
    b = make_batch(random_spec(83, 12, 3000, 1, 32, 8, 128, block_size=64, decode_frac=1.0, pad_rows=1),
                   device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    dev = DeviceStep(b)
    dev.write()
    dev.attend()
    for _ in range(2):
        st, out = _call(dev)
        assert st == 0
        torch.cuda.synchronize()
        assert_close(out, oracle_full(ref), "no-allocation call, blocks of 64 slots")
        assert _close(out, dev.out)
