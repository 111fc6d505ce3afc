"""tcgen05 prefill pairs cut into key pieces, against the oracle.

A pair of 128-row query tiles may run as several CTAs over consecutive
ranges of its key tiles; each writes fp32 partials (unscaled O, running max,
weight sum) and the CTA that counts last on the pair's counter merges them
("FlashAttention is not PagedAttention": exact tiled attention, the split
form of the same identity).  The planner cuts heavy pairs that would start
in a later wave; the tc_key_pieces option forces k pieces on every pair so
that small batches reach the path: whole pairs and single-tile pairs,
head dims 48/64/128, group sizes 2/4/8, windows, the diagonal in the last
piece, repeated calls and graph replays (the counters return to zero).
"""
import math

import pytest
import torch

import oracle
import paged_kv_cache_84_gb300 as pkv
from workloads import Req, Spec, build_meta, config_spec, make_batch, subset_spec
from _helpers import DeviceStep, assert_close, cpu_copy, oracle_full, oracle_write, threads

pytestmark = pytest.mark.gpu

COUNTERS = slice(256, 256 + 65536)          # the split-counter region after the error word


def _spec(hq, hkv, d, seed):
    reqs = [Req(1000, 300, list(range(0, 82))), Req(0, 257, list(range(82, 99))),
            Req(5000, 64, list(range(99, 416))), Req(77, 1, list(range(416, 421))),
            Req(2000, 130, list(range(421, 555))), Req(900, 2, list(range(555, 612)))]
    return Spec("pieces", reqs, hq, hkv, d, 16, 620, 1 / math.sqrt(d), seed)


@pytest.mark.parametrize("window", [0, 300])
@pytest.mark.parametrize("pieces", [2, 3, 5])
@pytest.mark.parametrize("heads", [(32, 8, 128), (16, 4, 64), (8, 4, 48), (16, 2, 48)],
                         ids=["d128g4", "d64g4", "d48g2", "d48g8"])
def test_forced_key_pieces(heads, pieces, window, attn_options):
    attn_options(tc_key_pieces=pieces)
    hq, hkv, d = heads
    spec = _spec(hq, hkv, d, 90 + pieces)
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    want = oracle_full(ref, window=window)
    m = b.meta
    plan = pkv.plan_attention(m.query_start_loc, m.seq_lens, hq, hkv, d, window=window)
    assert plan["prefill_tensor_pieces"] > 0
    dev = DeviceStep(b, window=window)
    dev.write()
    for call in range(2):                                   # the second call reuses the reset counters
        dev.out.fill_(float("nan"))
        pkv.profile_start(32)
        dev.attend()
        names = {n for n, _ in pkv.profile_stop()}
        assert names & {"attn_tc_prefill", "attn_tc_mixed"}
        assert_close(dev.out, want, f"pieces {pieces} d{d} window {window} call {call}")
        assert pkv.read_device_error(dev.ws) == 0
        assert int(dev.ws[COUNTERS].count_nonzero()) == 0


def test_forced_key_pieces_combined_call_and_graph_replays(attn_options):
    attn_options(tc_key_pieces=4)
    spec = _spec(32, 8, 128, 97)
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    want = oracle_full(ref)
    dev = DeviceStep(b)
    dev.combined()
    assert_close(dev.out, want, "combined call with key pieces")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        dev.combined()
    for i in range(3):
        dev.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_close(dev.out, want, f"graph replay {i}")
    assert pkv.read_device_error(dev.ws) == 0
    assert int(dev.ws[COUNTERS].count_nonzero()) == 0


def _plan(spec, **kw):
    m = build_meta(spec)
    ws = pkv.attention_workspace_bytes(m.num_reqs, m.num_tokens, spec.num_q_heads, spec.head_dim, m.max_seq_len)
    return pkv.plan_attention(m.query_start_loc, m.seq_lens, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                              combined=True, workspace_bytes=ws, **kw)


def test_planner_cuts_heavy_pairs_only_without_decodes_beside():
    """The planner's own choice: the 2048-token chunk at 16384 alone (256
    heavy CTAs on 152 SMs) has its second-wave pairs cut; with the mixed
    step's 64 decodes (on the decode CTAs that open its launch) and in the
    engine step's short chunks nothing is cut."""
    assert _plan(subset_spec(config_spec(4), 1))["prefill_tensor_pieces"] > 0
    assert _plan(config_spec(4))["prefill_tensor_pieces"] == 0
    assert _plan(config_spec(2))["prefill_tensor_pieces"] == 0


def test_planner_pieces_on_the_long_chunk_full_size():
    """The 2048-token chunk at position 16384 alone, full size, with the
    planner's pieces (uneven two-piece cuts of the second-wave pairs):
    sampled rows of every pair against the oracle."""
    spec = subset_spec(config_spec(4), 1)
    b = make_batch(spec, device="cuda")
    ref = cpu_copy(b)
    oracle_write(ref)
    assert _plan(spec)["prefill_tensor_pieces"] > 0
    dev = DeviceStep(b)
    dev.combined()
    torch.cuda.synchronize()
    assert pkv.read_device_error(dev.ws) == 0
    assert int(dev.ws[COUNTERS].count_nonzero()) == 0
    gen = torch.Generator().manual_seed(5)
    toks = list(range(0, 2048, 13)) + [63, 64, 2047]
    heads = torch.randint(0, spec.num_q_heads, (len(toks),), generator=gen).tolist()
    m = ref.meta
    want = oracle.attention_rows(toks, heads, ref.q, ref.k_cache, ref.v_cache, m.query_start_loc, m.seq_lens,
                                 m.block_table, spec.scale, threads())
    assert_close(dev.out[torch.tensor(toks), torch.tensor(heads)], want, "long chunk with planner pieces")


def test_no_key_pieces_option(attn_options):
    attn_options(tc_key_pieces=-1)
    assert _plan(subset_spec(config_spec(4), 1))["prefill_tensor_pieces"] == 0
