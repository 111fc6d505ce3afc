"""One captured decode step replayed for other batches of its shape.

"31. Engine v2", "Flattened ragged batches": the batch builder pads a decode
batch to a fixed size (pad_to: padding rows with slot -1 and seq_len 0), so
that one captured step serves every batch of that size.  With the
device_lengths option the attention kernels read each request's context
length from the device seq_lens when they run; the host copies give the
capacity the launch is planned for.  These tests plan and capture the
combined write + attention call once, at capacity, then rewrite q, k, v,
seq_lens, block_table and slot_mapping in place for several batches (other
lengths, other block tables, padding rows that become requests and back) and
replay the graph: the pools bit for bit and the attention within the
tolerance of the oracle every time, the error word clear and the split
counters back at zero.
"""
import math
import random

import pytest
import torch

import oracle
import paged_kv_cache_84_gb300 as pkv
from workloads import Batch, Req, Spec, make_batch
from _helpers import assert_close, oracle_full, oracle_write, threads

pytestmark = pytest.mark.gpu

COUNTERS = slice(256, 256 + 65536)
BS = 16


def _batch_spec(seed, nreq, cap, hq, hkv, d, nblocks, pad_frac=0.15, bs=BS):
    """nreq decode requests of 1 new token each, context 1 .. cap (some
    padding rows), each on its own random blocks; tables cap/bs wide."""
    rnd = random.Random(seed)
    perm = list(range(nblocks))
    rnd.shuffle(perm)
    reqs, cur = [], 0
    for _ in range(nreq):
        if rnd.random() < pad_frac:
            reqs.append(Req(0, 1, [], pad=True))
            continue
        L = rnd.choice([1, 15, 16, 17, cap, rnd.randint(1, cap), rnd.randint(1, cap)])
        nb = -(-L // bs)
        reqs.append(Req(L - 1, 1, perm[cur:cur + nb]))
        cur += nb
    return Spec("graph-replay", reqs, hq, hkv, d, bs, nblocks, 1 / math.sqrt(d), seed, table_width=-(-cap // bs))


class Captured:
    """Device buffers of a padded decode step and the combined call captured
    over them once, planned at capacity `cap` for every row."""

    def __init__(self, nreq, cap, hq, hkv, d, pools, window=0, fp8=None, bs=BS):
        self.nreq, self.cap, self.window, self.fp8 = nreq, cap, window, fp8
        dev = torch.device("cuda")
        self.k_cache, self.v_cache = pools[0], pools[1]
        self.q = torch.zeros((nreq, hq, d), dtype=torch.bfloat16, device=dev)
        self.k = torch.zeros((nreq, hkv, d), dtype=torch.bfloat16, device=dev)
        self.v = torch.zeros_like(self.k)
        self.qsl = torch.arange(nreq + 1, dtype=torch.int32, device=dev)
        self.sl = torch.zeros(nreq, dtype=torch.int32, device=dev)
        self.bt = torch.zeros((nreq, -(-cap // bs)), dtype=torch.int32, device=dev)
        self.slots = torch.full((nreq,), -1, dtype=torch.int64, device=dev)
        self.out = torch.zeros_like(self.q)
        self.qsl_h = list(range(nreq + 1))
        self.sl_h = [cap] * nreq
        self.scale = 1 / math.sqrt(d)
        self.ws = pkv.make_workspace(pkv.attention_workspace_bytes(nreq, nreq, hq, d, cap), dev)
        self.graph = None

    def call(self):
        if self.fp8 is None:
            pkv.paged_kv_write_attention(self.k, self.v, self.k_cache, self.v_cache, self.slots, self.out, self.q,
                                         self.qsl, self.sl, self.bt, self.qsl_h, self.sl_h, 1, self.cap, self.scale,
                                         self.ws, window=self.window)
        else:
            ks, vs = self.fp8
            pkv.paged_kv_write_attention_fp8(self.k, self.v, self.k_cache, self.v_cache, ks, vs, self.slots, self.out,
                                             self.q, self.qsl, self.sl, self.bt, self.qsl_h, self.sl_h, 1, self.cap,
                                             self.scale, self.ws, window=self.window)

    def capture(self):
        self.call()                                       # first call outside the capture
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=side):
            self.call()
        torch.cuda.synchronize()

    def load(self, b: Batch):
        """Rewrite the step's inputs and metadata in place for batch b."""
        m = b.meta
        assert m.num_reqs == self.nreq and m.query_start_loc == self.qsl_h
        self.q.copy_(b.q)
        self.k.copy_(b.k)
        self.v.copy_(b.v)
        self.sl.copy_(torch.tensor(m.seq_lens, dtype=torch.int32))
        self.bt.copy_(m.block_table)
        self.slots.copy_(m.slot_mapping)
        self.out.fill_(float("nan"))
        torch.cuda.synchronize()


def _pool_bits(t):
    return t.contiguous().view(torch.int16).view(t.shape[0], -1)


@pytest.mark.parametrize("split", [0, 256, 1024], ids=["planner", "split256", "split1024"])
@pytest.mark.parametrize("heads", [(32, 8, 128), (16, 4, 64), (8, 4, 48), (64, 8, 128)],
                         ids=["d128g4", "d64g4", "d48g2", "d128g8"])
def test_padded_decode_step_replayed_for_other_batches(heads, split, attn_options):
    attn_options(device_lengths=1)
    if split:
        attn_options(split_tokens=split)
    hq, hkv, d = heads
    nreq, cap = 40, 2000
    nblocks = nreq * -(-cap // BS)
    first = make_batch(_batch_spec(500 + hq + d, nreq, cap, hq, hkv, d, nblocks), device="cpu")
    ref_k, ref_v = first.k_cache.clone(), first.v_cache.clone()
    cs = Captured(nreq, cap, hq, hkv, d, (first.k_cache.cuda(), first.v_cache.cuda()))
    plan = pkv.plan_attention(cs.qsl_h, cs.sl_h, hq, hkv, d, combined=True, workspace_bytes=cs.ws.numel())
    assert plan["decode_cluster"] == 0 and plan["split_counters"] == 1
    cs.load(first)
    cs.capture()
    for i in range(4):
        b = first if i == 0 else make_batch(_batch_spec(600 + 7 * i + hq, nreq, cap, hq, hkv, d, nblocks),
                                            device="cpu")
        cs.load(b)
        cs.graph.replay()
        torch.cuda.synchronize()
        ref = Batch(b.spec, b.meta, b.q, b.k, b.v, ref_k, ref_v)
        oracle_write(ref)                                 # the step's rows go into the running pools
        want = oracle_full(ref)
        assert_close(cs.out, want, f"replay {i} ({sum(r.pad for r in b.spec.reqs)} padding rows)")
        for got, w in ((cs.k_cache, ref_k), (cs.v_cache, ref_v)):
            assert torch.equal(_pool_bits(got.cpu())[:-1], _pool_bits(w)[:-1]), f"pool after replay {i}"
        assert pkv.read_device_error(cs.ws) == 0
        assert int(cs.ws[COUNTERS].count_nonzero()) == 0


def test_replay_with_a_window_and_eager_calls(attn_options):
    """A sliding window (the key range starts from each run's own length)
    and the same mode called eagerly, without a graph."""
    attn_options(device_lengths=1)
    hq, hkv, d, nreq, cap, window = 32, 8, 128, 24, 3000, 700
    nblocks = nreq * -(-cap // BS)
    first = make_batch(_batch_spec(71, nreq, cap, hq, hkv, d, nblocks), device="cpu")
    ref_k, ref_v = first.k_cache.clone(), first.v_cache.clone()
    cs = Captured(nreq, cap, hq, hkv, d, (first.k_cache.cuda(), first.v_cache.cuda()), window=window)
    cs.load(first)
    cs.capture()
    for i in range(3):
        b = first if i == 0 else make_batch(_batch_spec(80 + i, nreq, cap, hq, hkv, d, nblocks), device="cpu")
        cs.load(b)
        if i == 1:
            cs.call()                                     # eagerly
        else:
            cs.graph.replay()
        torch.cuda.synchronize()
        ref = Batch(b.spec, b.meta, b.q, b.k, b.v, ref_k, ref_v)
        oracle_write(ref)
        assert_close(cs.out, oracle_full(ref, window=window), f"window {window}, call {i}")
        assert pkv.read_device_error(cs.ws) == 0
        assert int(cs.ws[COUNTERS].count_nonzero()) == 0


def test_replay_on_a_quantized_pool(attn_options):
    """The quantized pool: the decode CTAs quantize and write their own rows
    (codes and scales bit for bit) and attend over codes x scales."""
    attn_options(device_lengths=1)
    hq, hkv, d, nreq, cap = 32, 8, 128, 32, 2500
    nblocks = nreq * -(-cap // BS)
    first = make_batch(_batch_spec(90, nreq, cap, hq, hkv, d, nblocks), device="cpu")
    # every slot of the pool quantized from the bf16 pool by the oracle's
    # write, so that whatever history a later batch's tables point at holds
    # values of the same scale as the new rows (junk codes with arbitrary
    # scales would make the attention ill-conditioned)
    nbt = first.spec.num_blocks_total
    pools = [torch.zeros((nbt, BS, hkv, d), dtype=torch.uint8) for _ in range(2)] + \
        [torch.zeros((nbt, BS, hkv), dtype=torch.float32) for _ in range(2)]
    every = torch.arange(nbt * BS, dtype=torch.int64)
    oracle.paged_kv_write_fp8(*pools, first.k_cache.view(-1, hkv, d), first.v_cache.view(-1, hkv, d), every)
    ref = [t.clone() for t in pools]
    kc, vc, ks, vs = [t.cuda() for t in pools]
    cs = Captured(nreq, cap, hq, hkv, d, (kc, vc), fp8=(ks, vs))
    cs.load(first)
    cs.capture()
    for i in range(3):
        b = first if i == 0 else make_batch(_batch_spec(95 + i, nreq, cap, hq, hkv, d, nblocks), device="cpu")
        cs.load(b)
        cs.graph.replay()
        torch.cuda.synchronize()
        m = b.meta
        oracle.paged_kv_write_fp8(ref[0], ref[1], ref[2], ref[3], b.k, b.v, m.slot_mapping)
        want = oracle.ragged_paged_attention_fp8(b.q, ref[0], ref[1], ref[2], ref[3], m.query_start_loc, m.seq_lens,
                                                 m.block_table, b.spec.scale, threads())
        assert_close(cs.out, want, f"quantized replay {i}")
        for dv, r in zip((kc, vc, ks, vs), ref):
            nbt = dv.shape[0]                             # the pools' last block is the scratch block
            assert torch.equal(dv.cpu().view(nbt, -1)[:-1].view(torch.uint8), r.view(nbt, -1)[:-1].view(torch.uint8))
        assert pkv.read_device_error(cs.ws) == 0


def test_longer_device_length_is_clamped_and_reported(attn_options):
    """A device length above the planned capacity is run at the capacity and
    flagged (PKV_DEVERR_META); the other rows are unaffected."""
    attn_options(device_lengths=1)
    hq, hkv, d, nreq, cap = 16, 4, 64, 8, 600
    nblocks = nreq * -(-cap // BS)
    b = make_batch(_batch_spec(33, nreq, cap, hq, hkv, d, nblocks, pad_frac=0.0), device="cpu")
    cs = Captured(nreq, cap, hq, hkv, d, (b.k_cache.cuda(), b.v_cache.cuda()))
    cs.load(b)
    cs.sl[0] = cap + 50
    cs.call()
    torch.cuda.synchronize()
    assert pkv.read_device_error(cs.ws) & pkv.DEVERR_META
    assert torch.isfinite(cs.out.float()).all()


@pytest.mark.parametrize("bs", [32, 64])
def test_replay_at_other_block_sizes(bs, attn_options):
    """The replayed padded step with blocks of 32 and 64 slots."""
    attn_options(device_lengths=1)
    hq, hkv, d, nreq, cap = 32, 8, 128, 24, 2100
    nblocks = nreq * -(-cap // bs)
    first = make_batch(_batch_spec(120 + bs, nreq, cap, hq, hkv, d, nblocks, bs=bs), device="cpu")
    ref_k, ref_v = first.k_cache.clone(), first.v_cache.clone()
    cs = Captured(nreq, cap, hq, hkv, d, (first.k_cache.cuda(), first.v_cache.cuda()), bs=bs)
    cs.load(first)
    cs.capture()
    for i in range(3):
        b = first if i == 0 else make_batch(_batch_spec(130 + bs + i, nreq, cap, hq, hkv, d, nblocks, bs=bs),
                                            device="cpu")
        cs.load(b)
        cs.graph.replay()
        torch.cuda.synchronize()
        ref = Batch(b.spec, b.meta, b.q, b.k, b.v, ref_k, ref_v)
        oracle_write(ref)
        assert_close(cs.out, oracle_full(ref), f"block size {bs}, replay {i}")
        assert pkv.read_device_error(cs.ws) == 0
        assert int(cs.ws[COUNTERS].count_nonzero()) == 0
