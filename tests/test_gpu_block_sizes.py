"""Block sizes other than 16 on the GPU, against the oracle.

"31. Engine v2", "Attention over the pool" and "Flattened ragged batches":
key j of a request lives in slot table[j // block_size] * block_size +
j % block_size; the vllm-lite README's test list checks results across block
sizes.  The kernels walk a block as sub-blocks of 16 slots (one TMA box
each), so every block size that is 16 times a power of two runs on every
path: the write (bit for bit) and attention on the decode kernels (slot ring
and streaming splits), the tcgen05 prefill (alone, with key pieces, and in
the one-launch mixed batch), the combined call, quantized pools, windows and
the replayed padded decode step.
"""
import math

import pytest
import torch

import oracle
import paged_kv_cache_84_gb300 as pkv
from workloads import Batch, Req, Spec, make_batch, random_spec
from _helpers import DeviceStep, assert_close, cpu_copy, oracle_full, oracle_write, threads

pytestmark = pytest.mark.gpu

COUNTERS = slice(256, 256 + 65536)


def _pool_bits(t):
    nbt, bs, hkv, d = t.shape
    return t.contiguous().view(torch.int16).view(nbt * bs, hkv * d)


def _check_pools(dev, ref):
    for got, want in ((dev.k_cache, ref.k_cache), (dev.v_cache, ref.v_cache)):
        assert torch.equal(_pool_bits(got.cpu())[:-1], _pool_bits(want)[:-1])


@pytest.mark.parametrize("combined", [False, True], ids=["two-calls", "combined"])
@pytest.mark.parametrize("bs", [32, 64, 128, 256])
@pytest.mark.parametrize("heads", [(32, 8, 128), (16, 4, 64), (8, 4, 48)], ids=["d128g4", "d64g4", "d48g2"])
def test_random_mix(heads, bs, combined):
    hq, hkv, d = heads
    spec = random_spec(700 + bs + d, 9, 2600, 300, hq, hkv, d, block_size=bs, pad_rows=1)
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    want = oracle_full(ref)
    dev = DeviceStep(b)
    dev.combined() if combined else dev.step()
    torch.cuda.synchronize()
    _check_pools(dev, ref)
    assert_close(dev.out, want, f"block size {bs}")
    assert pkv.read_device_error(dev.ws) == 0


@pytest.mark.parametrize("path", ["split256", "split1024", "mixed", "pieces", "window", "mma-prefill"])
@pytest.mark.parametrize("bs", [32, 64])
def test_kernel_paths(bs, path, attn_options):
    """Each arrangement the planner can choose, forced, at block sizes 32 and 64."""
    window = 0
    if path == "split256":
        attn_options(split_tokens=256)
    elif path == "split1024":
        attn_options(split_tokens=1024)
    elif path == "mixed":
        attn_options(mixed_launch=1)
    elif path == "pieces":
        attn_options(tc_key_pieces=3, mixed_launch=-1)
    elif path == "window":
        window = 450
    else:
        attn_options(disable_tcgen05=1)
    hq, hkv, d = 32, 8, 128
    reqs = [Req(1500, 260, list(range(0, 28))), Req(3000, 1, list(range(28, 76))), Req(40, 1, list(range(76, 77))),
            Req(0, 1, [], pad=True), Req(2000, 2, list(range(77, 109))), Req(700, 90, list(range(109, 122)))]
    scale = 1 / math.sqrt(d)
    # tables above are in blocks of 64 slots; for 32 slots give each request twice the blocks
    if bs == 32:
        reqs = [Req(r.computed, r.new, [2 * x for x in r.table] + [2 * x + 1 for x in r.table], r.pad) for r in reqs]
    spec = Spec(f"paths-bs{bs}", reqs, hq, hkv, d, bs, 250 * (64 // bs), scale, 40 + bs)
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    want = oracle_full(ref, window=window)
    dev = DeviceStep(b, window=window)
    dev.combined()
    torch.cuda.synchronize()
    _check_pools(dev, ref)
    assert_close(dev.out, want, f"block size {bs}, {path}")
    assert pkv.read_device_error(dev.ws) == 0
    assert int(dev.ws[COUNTERS].count_nonzero()) == 0


@pytest.mark.parametrize("bs", [32, 64])
def test_quantized_pool(bs):
    """E4M3 codes and scales in blocks of 32 or 64 slots: the quantizing
    write bit for bit, attention over codes x scales (decode kernels and
    the tcgen05 prefill over bf16 copies of the blocks)."""
    hq, hkv, d = 32, 8, 128
    spec = random_spec(800 + bs, 8, 2200, 200, hq, hkv, d, block_size=bs, pad_rows=1)
    b = make_batch(spec, device="cpu")
    m = b.meta
    nbt = spec.num_blocks_total
    pools = [torch.zeros((nbt, bs, hkv, d), dtype=torch.uint8) for _ in range(2)] + \
        [torch.zeros((nbt, bs, hkv), dtype=torch.float32) for _ in range(2)]
    every = torch.arange(nbt * bs, dtype=torch.int64)
    oracle.paged_kv_write_fp8(*pools, b.k_cache.view(-1, hkv, d), b.v_cache.view(-1, hkv, d), every)
    ref = [t.clone() for t in pools]
    oracle.paged_kv_write_fp8(*ref, b.k, b.v, m.slot_mapping)
    want = oracle.ragged_paged_attention_fp8(b.q, *ref, m.query_start_loc, m.seq_lens, m.block_table, spec.scale,
                                             threads())
    kc, vc, ks, vs = [t.cuda() for t in pools]
    q, k, v = b.q.cuda(), b.k.cuda(), b.v.cuda()
    out = torch.full_like(q, float("nan"))
    ws = pkv.make_workspace(pkv.attention_workspace_bytes(m.num_reqs, m.num_tokens, hq, d, m.max_seq_len) +
                            pkv.fp8_prefill_scratch_bytes(m.query_start_loc, m.seq_lens, hq, hkv, d), "cuda")
    pkv.paged_kv_write_attention_fp8(k, v, kc, vc, ks, vs, m.slot_mapping.cuda(), out, q,
                                     torch.tensor(m.query_start_loc, dtype=torch.int32, device="cuda"),
                                     torch.tensor(m.seq_lens, dtype=torch.int32, device="cuda"),
                                     m.block_table.cuda(), m.query_start_loc, m.seq_lens, m.max_query_len,
                                     m.max_seq_len, spec.scale, ws)
    torch.cuda.synchronize()
    for dv, r in zip((kc, vc, ks, vs), ref):
        n = dv.shape[0]
        assert torch.equal(dv.cpu().view(n, -1)[:-1].view(torch.uint8), r.view(n, -1)[:-1].view(torch.uint8))
    assert_close(out, want, f"quantized pool, block size {bs}")
    assert pkv.read_device_error(ws) == 0


def test_out_of_pool_block_id_is_flagged_at_block_size_64():
    """An id past the pool (in blocks of 64 slots) is reported, not read."""
    hq, hkv, d, bs = 16, 4, 64, 64
    spec = random_spec(901, 4, 900, 1, hq, hkv, d, block_size=bs, decode_frac=1.0)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.write()
    dev.bt[0, 0] = spec.num_blocks_total + 2
    dev.attend()
    torch.cuda.synchronize()
    assert pkv.read_device_error(dev.ws) & pkv.DEVERR_BLOCK
