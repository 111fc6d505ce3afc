"""pkv_ragged_paged_attention_noalloc, called through the C ABI.

This entry point is for callers that cannot allocate device memory (code
under a stream capture that forbids allocation, C hosts without a device
allocator, serving loops that must not call cudaMalloc because it can
synchronise the device).  It keeps its split-KV partials and error word in a
static array inside the library.  Its output must match the workspace entry
point's within the parity tolerance, on calls made back to back that reuse
the array.
"""
import ctypes

import pytest
import torch

import paged_kv_cache_84_gb300 as pkv
from workloads import config_spec, make_batch, random_spec
from _helpers import DeviceStep, MAX_ERR, MEAN_ERR

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20          # PKV_NOALLOC_SCRATCH_BYTES in include/pkv.h
_p, _i32 = ctypes.c_void_p, ctypes.c_int32


def _fn():
    fn = pkv.load().pkv_ragged_paged_attention_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [_p] * 7 + [_i32, _p, _p] + [_i32] * 9 + [ctypes.c_float, _i32, _p, _p]
    return fn


def _call(dev: DeviceStep, bt=None, device_error=None, max_seq_len=None):
    m, s = dev.batch.meta, dev.batch.spec
    bt = dev.bt if bt is None else bt
    qsl_h = torch.tensor(m.query_start_loc, dtype=torch.int32)
    sl_h = torch.tensor(m.seq_lens, dtype=torch.int32)
    out = torch.full_like(dev.q, float("nan"))
    st = _fn()(out.data_ptr(), dev.q.data_ptr(), dev.k_cache.data_ptr(), dev.v_cache.data_ptr(),
               dev.qsl.data_ptr(), dev.sl.data_ptr(), bt.data_ptr(), bt.shape[1], qsl_h.data_ptr(),
               sl_h.data_ptr(), m.num_reqs, m.num_tokens, m.max_query_len,
               m.max_seq_len if max_seq_len is None else max_seq_len, s.num_q_heads, s.num_kv_heads,
               s.head_dim, s.block_size, s.num_blocks_total, s.scale, 0,
               None if device_error is None else device_error.data_ptr(),
               torch.cuda.current_stream().cuda_stream)
    return st, out


def _close(a, b):
    d = (a.double() - b.double()).abs()
    return torch.isfinite(a.float()).all().item() and d.max().item() <= MAX_ERR and d.mean().item() <= MEAN_ERR


def _split_batch():
    # eight decodes over ~3000 keys: the planner splits each over many CTAs,
    # so the partials really pass through the static array
    return random_spec(81, 8, 3200, 1, 32, 8, 128, decode_frac=1.0)


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(monkeypatch):
    # keys split every 256 tokens: the second batch's decodes (~3000 keys)
    # run as many splits, combined in the kernel through the static array
    monkeypatch.setenv("PKV_SPLIT_TOKENS", "256")
    steps = []
    for spec in (config_spec(2), _split_batch()):
        dev = DeviceStep(make_batch(spec, device="cpu"))
        dev.write()
        dev.attend()
        steps.append(dev)
    torch.cuda.synchronize()
    outs = []
    pkv.profile_start(64)
    for dev in steps:                                  # two calls back to back on the same array
        st, out = _call(dev)
        assert st == 0
        outs.append(out)
    kernels = [name for name, _ in pkv.profile_stop()]
    assert "attn_mma_decode" in kernels
    for dev, out in zip(steps, outs):
        assert _close(out, dev.out)
    # and once more in reverse order, after the array holds the other batch's partials
    for dev in reversed(steps):
        st, out = _call(dev)
        assert st == 0 and _close(out, dev.out)


def test_noalloc_rejects_batches_beyond_the_scratch():
    dev = DeviceStep(make_batch(_split_batch(), device="cpu"))
    big_len = 1 << 20                                  # would need far more than the array holds
    m, s = dev.batch.meta, dev.batch.spec
    assert pkv.attention_workspace_bytes(m.num_reqs, m.num_tokens, s.num_q_heads, s.head_dim,
                                         big_len) > SCRATCH_BYTES
    before = pkv.launch_count()
    st, _ = _call(dev, max_seq_len=big_len)
    assert st == 3                                     # PKV_ERR_WORKSPACE, nothing enqueued
    assert pkv.launch_count() == before


def test_noalloc_reports_bounds_flags_per_call():
    dev = DeviceStep(make_batch(random_spec(82, 5, 400, 3, 8, 4, 64), device="cpu"))
    dev.write()
    err = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    bad = dev.bt.clone()
    bad[0, 0] = dev.batch.spec.num_blocks_total + 3
    st, _ = _call(dev, bt=bad, device_error=err)
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEVERR_BLOCK
    st, out = _call(dev, device_error=err)             # the word was reset after the first call
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    dev.attend()
    assert _close(out, dev.out)
