"""pkv_paged_kv_write_attention: the step's write and attention in one call.

The pools must come out bit-exact (whole pool except the scratch slot) and
the attention within the parity tolerance of the oracle, on every
arrangement the call makes: decode-class CTAs writing their own rows
(slot ring with split counters or clusters, streaming kernel, padding
requests, sliding window), the ranged scatter of prefill-class rows ahead of
the tcgen05 and warp-MMA prefill kernels, on one stream or two, eager and
from a CUDA graph.
"""
import math

import pytest
import torch

import paged_kv_cache_84_gb300 as pkv
from workloads import Req, Spec, config_spec, make_batch, random_spec
from _helpers import DeviceStep, assert_close, cpu_copy, oracle_full, oracle_write

pytestmark = pytest.mark.gpu


def _pool_bits(t):
    nbt, bs, hkv, d = t.shape
    return t.contiguous().view(torch.int16).view(nbt * bs, hkv * d)


def _check(dev, ref, window=0, what=""):
    for got, want in ((dev.k_cache, ref.k_cache), (dev.v_cache, ref.v_cache)):
        assert torch.equal(_pool_bits(got.cpu())[:-1], _pool_bits(want)[:-1]), f"pool {what}"
    assert_close(dev.out, oracle_full(ref, window=window), what)
    assert pkv.read_device_error(dev.ws) == 0


def _run(spec, window=0, what=""):
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    dev = DeviceStep(b, window=window)
    dev.combined()
    _check(dev, ref, window, what)
    return b, ref


@pytest.mark.parametrize("cfg", [1, 2])
def test_small_configs(cfg):
    _run(config_spec(cfg), what=f"config {cfg}")


def test_layout_example_is_one_launch():
    """The pages' layout example ("Flattened ragged batches": a 3-token chunk,
    two decodes and a 4-token prompt, g = 2) as one combined call is one
    library launch: its chunks are short enough for the decode kernel (at
    most 16/g tokens), whose CTAs write their own rows.  A second call writes
    the same rows again, so pools and output are checked after it."""
    b = make_batch(config_spec(1), device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    dev = DeviceStep(b)
    dev.combined()                       # the first call also sets kernel attributes
    torch.cuda.synchronize()
    before = pkv.launch_count()
    dev.combined()
    torch.cuda.synchronize()
    assert pkv.launch_count() - before == 1
    _check(dev, ref, 0, "layout example, one launch")


def test_engine_step_chunks_write_their_own_rows():
    """The 48-request engine step: every prefill chunk (at most 64 tokens,
    g = 2: one pair of 128-row tiles per KV head) is one tcgen05 CTA per KV
    head, which writes the chunk's new rows itself, so the call is two
    launches (the tcgen05 prefill and the decode kernel), no scatter."""
    b = make_batch(config_spec(2), device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    dev = DeviceStep(b)
    dev.combined()
    torch.cuda.synchronize()
    before = pkv.launch_count()
    dev.combined()
    torch.cuda.synchronize()
    assert pkv.launch_count() - before == 2
    _check(dev, ref, 0, "engine step, chunks writing their own rows")


@pytest.mark.parametrize("t", [1, 40, 64, 65, 130])
def test_chunk_rows_written_by_its_own_cta_or_the_scatter(t):
    """Chunks of t tokens (g = 4: 32 tokens per tile, 64 per pair) beside a
    decode: up to 64 tokens one tcgen05 CTA per KV head writes the chunk's
    rows (its first new key tile after older ones, or the first tile), above
    it the scatter does; pools bit-exact, attention within tolerance."""
    hq, hkv, d = 32, 8, 128
    reqs = [Req(300, t, list(range(0, 30))), Req(900, 1, list(range(30, 88))), Req(0, t, list(range(88, 98)))]
    spec = Spec(f"self-write-{t}", reqs, hq, hkv, d, 16, 120, 1 / math.sqrt(d), 61 + t)
    _run(spec, what=f"chunks of {t}")


@pytest.mark.parametrize("env", ["default", "no-overlap", "decode-side", "no-cluster", "separate", "no-tcgen05"])
def test_engine_step_arrangements(env, attn_options):
    """The 48-request engine step under every stream and kernel arrangement."""
    if env == "no-overlap":
        attn_options(no_overlap=1)
    elif env == "decode-side":
        attn_options(decode_main=-1)
    elif env == "no-cluster":
        attn_options(cluster=-1)
    elif env == "separate":
        attn_options(separate_write=1)
    elif env == "no-tcgen05":
        attn_options(disable_tcgen05=1)
    _run(config_spec(2), what=f"engine step {env}")


RANDOM = [
    # seed, reqs, max_ctx, max_new, hq, hkv, d, pad rows, decode fraction
    (0, 12, 700, 40, 16, 4, 64, 2, 0.5),
    (1, 20, 3000, 3, 32, 8, 128, 1, 0.9),
    (2, 8, 1500, 130, 8, 2, 48, 0, 0.5),
    (3, 30, 400, 8, 8, 8, 128, 3, 1.0),        # decodes and short chunks only: one launch
    (4, 6, 900, 300, 16, 2, 64, 0, 0.0),       # prefill chunks only: ranged scatter
    (5, 10, 2000, 60, 32, 8, 128, 1, 0.3),     # chunks of up to 64 tokens (g = 4) on tcgen05
]


@pytest.mark.parametrize("case", RANDOM, ids=[f"seed{c[0]}" for c in RANDOM])
@pytest.mark.parametrize("window", [0, 300])
def test_random_mixes(case, window):
    seed, reqs, max_ctx, max_new, hq, hkv, d, pad, frac = case
    spec = random_spec(300 + seed, reqs, max_ctx, max_new, hq, hkv, d, pad_rows=pad, decode_frac=frac)
    _run(spec, window, f"random {seed} window {window}")


@pytest.mark.parametrize("split", ["128", "1024"], ids=["slot-ring", "streaming"])
def test_split_decodes_write_their_rows(split, attn_options):
    """Splits whose ranges cut through a request's new rows (t up to 8) each
    write the rows in their own range."""
    attn_options(split_tokens=int(split))
    reqs, blk = [], 0
    for L, t in ((1030, 8), (2049, 3), (511, 5), (4000, 1), (129, 8), (0, 0)):
        if t == 0:
            reqs.append(Req(0, 1, [], pad=True))
            continue
        nb = (L + 15) // 16
        reqs.append(Req(L - t, t, list(range(blk, blk + nb))))
        blk += nb
    spec = Spec("split-writes", reqs, 16, 8, 128, 16, blk + 3, 1 / math.sqrt(128), 87)
    _run(spec, what=f"split {split}")


def test_graph_replays_and_repeated_calls():
    b = make_batch(config_spec(2), device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    dev = DeviceStep(b)
    for i in range(2):
        dev.out.fill_(float("nan"))
        dev.combined()
        _check(dev, ref, what=f"eager {i}")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dev.combined()
    torch.cuda.synchronize()
    for i in range(2):
        dev.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        _check(dev, ref, what=f"replay {i}")


def test_slot_mapping_that_disagrees_with_the_table_is_flagged():
    """A decode row whose slot differs from the block table's is written to
    its slot and reported (PKV_DEVERR_META); nothing faults."""
    spec = random_spec(310, 6, 500, 1, 8, 4, 64, decode_frac=1.0)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.slots[0] = (dev.slots[0] + 1) % (spec.num_blocks_total * spec.block_size - 1)
    dev.combined()
    assert pkv.read_device_error(dev.ws) & pkv.DEVERR_META


def test_out_of_pool_slot_is_skipped_and_flagged():
    spec = random_spec(311, 6, 500, 20, 8, 4, 64, decode_frac=0.5)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.slots[-1] = spec.num_blocks_total * spec.block_size + 5
    dev.combined()
    assert pkv.read_device_error(dev.ws) & pkv.DEVERR_SLOT
    torch.cuda.synchronize()


def test_more_requests_than_one_launch_lists():
    """600 decodes and 300 prefill chunks in one combined call: the decode
    class and the ranged scatter each run several launches of at most 256
    listed requests (or token ranges)."""
    gen = torch.Generator().manual_seed(88)
    reqs, blk = [], 0
    for i in range(900):
        if i % 3 == 2:
            t = int(torch.randint(9, 41, (1,), generator=gen))   # t * g > 16: prefill class
            c = int(torch.randint(0, 600, (1,), generator=gen))
        else:
            t, c = 1, int(torch.randint(0, 1500, (1,), generator=gen))
        nb = (c + t + 15) // 16
        reqs.append(Req(c, t, list(range(blk, blk + nb))))
        blk += nb
    spec = Spec("many", reqs, 8, 2, 64, 16, blk + 4, 0.125, 89)
    from workloads import build_meta
    m = build_meta(spec)
    classes = pkv.plan_request_kernels(m.query_start_loc, m.seq_lens, 8, 2, 64)
    assert sum(c != "decode" for c in classes) > 256
    _run(spec, what="900 requests, combined call")
