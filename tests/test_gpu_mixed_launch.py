"""One launch for a mixed batch: the decode class inside the tcgen05 launch.

For a flattened batch of prefill chunks and decodes ("31. Engine v2",
"Flattened ragged batches"), the first CTAs of the tcgen05 launch are
decode CTAs: each of their warps runs decode items (request, KV head, key
split) over its own ring of KV stages, while the CTAs after them run the
prefill tiles.  The mixed_launch option forces the arrangement where it
applies; results must match the oracle like every other arrangement:
decodes of one and several splits (merged by the warp that counts last),
padding requests, windows, head dims 48/64/128, groups 2/4/8, the plain and
the combined call (decode items writing their own new rows), quantized
pools (decode items over E4M3 codes, the prefill over bf16 copies), graph
replays, and the counters back at zero after each call.
"""
import math

import pytest
import torch

import oracle
import paged_kv_cache_84_gb300 as pkv
from workloads import Req, Spec, build_meta, config_spec, make_batch
from _helpers import DeviceStep, assert_close, cpu_copy, oracle_full, oracle_write, quantized_pools, threads

pytestmark = pytest.mark.gpu

COUNTERS = slice(256, 256 + 65536)


def _pool_bits(t):
    nbt, bs, hkv, d = t.shape
    return t.contiguous().view(torch.int16).view(nbt * bs, hkv * d)


def _spec(hq, hkv, d, seed, pad=True):
    g = hq // hkv
    reqs = [Req(1000, 300, list(range(0, 82))), Req(0, 257, list(range(82, 99))),
            Req(3000, 1, list(range(99, 287))), Req(77, 1, list(range(287, 292))),
            Req(2600, 8 // g if g <= 8 else 1, list(range(292, 455))), Req(900, 1, list(range(455, 512)))]
    if pad:
        reqs.append(Req(0, 1, [], pad=True))
    return Spec("mixed-launch", reqs, hq, hkv, d, 16, 520, 1 / math.sqrt(d), seed)


@pytest.mark.parametrize("combined", [False, True], ids=["attention", "combined"])
@pytest.mark.parametrize("window", [0, 500])
@pytest.mark.parametrize("split", [0, 256])
@pytest.mark.parametrize("heads", [(32, 8, 128), (16, 4, 64), (8, 4, 48), (64, 8, 128)],
                         ids=["d128g4", "d64g4", "d48g2", "d128g8"])
def test_forced_mixed_launch(heads, split, window, combined, attn_options):
    attn_options(mixed_launch=1)
    if split:
        attn_options(split_tokens=split)
    hq, hkv, d = heads
    spec = _spec(hq, hkv, d, 60 + hq + d)
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    want = oracle_full(ref, window=window)
    m = b.meta
    plan = pkv.plan_attention(m.query_start_loc, m.seq_lens, hq, hkv, d, window=window, combined=combined)
    assert plan["mixed_launch"] == 1 and plan["mixed_decode_items"] > 0
    dev = DeviceStep(b, window=window)
    if not combined:
        dev.write()
    for call in range(2):
        dev.out.fill_(float("nan"))
        pkv.profile_start(32)
        dev.combined() if combined else dev.attend()
        names = [n for n, _ in pkv.profile_stop()]
        assert "attn_tc_mixed" in names and "attn_mma_decode" not in names, names
        assert_close(dev.out, want, f"mixed launch d{d} split {split} window {window} call {call}")
        assert pkv.read_device_error(dev.ws) == 0
        assert int(dev.ws[COUNTERS].count_nonzero()) == 0
    if combined:
        for got, w in ((dev.k_cache, ref.k_cache), (dev.v_cache, ref.v_cache)):
            assert torch.equal(_pool_bits(got.cpu())[:-1], _pool_bits(w)[:-1])


def test_mixed_launch_graph_replays_with_pieces(attn_options):
    """The mixed launch with the tcgen05 pairs cut into key pieces as well,
    captured once and replayed."""
    attn_options(mixed_launch=1, tc_key_pieces=3, split_tokens=512)
    spec = _spec(32, 8, 128, 77)
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    want = oracle_full(ref)
    dev = DeviceStep(b)
    dev.combined()
    assert_close(dev.out, want, "eager")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        dev.combined()
    for i in range(3):
        dev.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_close(dev.out, want, f"replay {i}")
    assert pkv.read_device_error(dev.ws) == 0
    assert int(dev.ws[COUNTERS].count_nonzero()) == 0


def test_mixed_launch_not_taken_where_it_does_not_apply(attn_options):
    """Decodes of more than 8 rows per KV head, or no tcgen05 prefill: the
    two-launch arrangement stays (the option cannot force it)."""
    attn_options(mixed_launch=1)
    p = pkv.plan_attention([0, 300, 302], [1300, 900], 64, 4, 128)   # t * g = 32 rows for the second
    assert p["mixed_launch"] == 0
    p = pkv.plan_attention([0, 1, 2], [1300, 900], 32, 8, 128)       # decodes only
    assert p["mixed_launch"] == 0


def test_mixed_step_full_size(attn_options):
    """The mixed 2048-token-chunk step in one launch (the 64 decodes on the
    launch's decode CTAs): pools bit-exact, sampled rows of every request
    and every head of the last decode against the oracle."""
    attn_options(mixed_launch=1)
    spec = config_spec(4)
    b = make_batch(spec, device="cuda")
    ref = cpu_copy(b)
    dev = DeviceStep(b)
    m = b.meta
    plan = pkv.plan_attention(m.query_start_loc, m.seq_lens, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                              combined=True, workspace_bytes=dev.ws.numel())
    assert plan["mixed_launch"] == 1
    dev.combined()
    torch.cuda.synchronize()
    oracle_write(ref)
    for got, w in ((dev.k_cache, ref.k_cache), (dev.v_cache, ref.v_cache)):
        assert torch.equal(_pool_bits(got.cpu())[:-1], _pool_bits(w)[:-1])
    assert pkv.read_device_error(dev.ws) == 0
    assert int(dev.ws[COUNTERS].count_nonzero()) == 0
    gen = torch.Generator().manual_seed(44)
    toks, heads = [], []
    for r in range(m.num_reqs):
        b0, t = m.query_start_loc[r], m.query_start_loc[r + 1] - m.query_start_loc[r]
        for i in sorted({0, t - 1, t // 2}):
            toks.append(b0 + i)
            heads.append(int(torch.randint(0, spec.num_q_heads, (1,), generator=gen)))
    last_dec = 2048 + 63
    toks += [last_dec] * spec.num_q_heads
    heads += list(range(spec.num_q_heads))
    want = oracle.attention_rows(toks, heads, ref.q, ref.k_cache, ref.v_cache, m.query_start_loc, m.seq_lens,
                                 m.block_table, spec.scale, threads())
    assert_close(dev.out[torch.tensor(toks), torch.tensor(heads)], want, "mixed step in one launch")


def _fp8_call(b, pools, combined, window, ws_bytes):
    spec, m = b.spec, b.meta
    kc, vc, ks, vs = [t.cuda() for t in pools]
    k, v, q = b.k.cuda(), b.v.cuda(), b.q.cuda()
    slots = m.slot_mapping.cuda()
    qsl = torch.tensor(m.query_start_loc, dtype=torch.int32, device="cuda")
    sl = torch.tensor(m.seq_lens, dtype=torch.int32, device="cuda")
    bt = m.block_table.cuda()
    ws = pkv.make_workspace(ws_bytes, "cuda")
    out = torch.full_like(q, float("nan"))
    if not combined:
        pkv.paged_kv_write_fp8(k, v, kc, vc, ks, vs, slots)
    pkv.profile_start(32)
    if combined:
        pkv.paged_kv_write_attention_fp8(k, v, kc, vc, ks, vs, slots, out, q, qsl, sl, bt, m.query_start_loc,
                                         m.seq_lens, m.max_query_len, m.max_seq_len, spec.scale, ws, window=window)
    else:
        pkv.ragged_paged_attention_fp8(out, q, kc, vc, ks, vs, qsl, sl, bt, m.query_start_loc, m.seq_lens,
                                       m.max_query_len, m.max_seq_len, spec.scale, ws, window=window)
    names = [n for n, _ in pkv.profile_stop()]
    torch.cuda.synchronize()
    return out, (kc, vc, ks, vs), ws, names


@pytest.mark.parametrize("combined", [False, True], ids=["attention", "combined"])
@pytest.mark.parametrize("window", [0, 500])
@pytest.mark.parametrize("split", [0, 256])
@pytest.mark.parametrize("heads", [(32, 8, 128), (64, 8, 128), (16, 8, 128)], ids=["g4", "g8", "g2"])
def test_forced_mixed_launch_quantized(heads, split, window, combined, attn_options):
    """Quantized pools: the decode CTAs read E4M3 codes and their scales,
    the prefill CTAs the bf16 copies of their blocks written by the
    dequantizing pass; codes and scales bit-exact, attention within the
    tolerance of the oracle's code * scale attention."""
    attn_options(mixed_launch=1)
    if split:
        attn_options(split_tokens=split)
    hq, hkv, d = heads
    spec = _spec(hq, hkv, d, 90 + hq)
    b = make_batch(spec, device="cpu")
    m = b.meta
    pools = quantized_pools(b, 91 + hq)
    ws_bytes = pkv.attention_workspace_bytes(m.num_reqs, m.num_tokens, hq, d, m.max_seq_len) + \
        pkv.fp8_prefill_scratch_bytes(m.query_start_loc, m.seq_lens, hq, hkv, d)
    plan = pkv.plan_attention(m.query_start_loc, m.seq_lens, hq, hkv, d, window=window, quantized=True,
                              combined=combined, workspace_bytes=ws_bytes)
    assert plan["mixed_launch"] == 1 and plan["mixed_decode_items"] > 0
    kc, vc, ks, vs = [t.clone() for t in pools]
    oracle.paged_kv_write_fp8(kc, vc, ks, vs, b.k, b.v, m.slot_mapping)
    want = oracle.ragged_paged_attention_fp8(b.q, kc, vc, ks, vs, m.query_start_loc, m.seq_lens, m.block_table,
                                             spec.scale, threads(), window=window)
    for call in range(2):
        got, dev_pools, ws, names = _fp8_call(b, pools, combined, window, ws_bytes)
        assert "attn_tc_mixed" in names and "attn_mma_decode" not in names, names
        assert_close(got, want, f"quantized mixed launch hq {hq} split {split} window {window} call {call}")
        assert pkv.read_device_error(ws) == 0
        assert int(ws[COUNTERS].count_nonzero()) == 0
        nbt = spec.num_blocks_total + 1
        for dv, r in zip(dev_pools, (kc, vc, ks, vs)):
            assert torch.equal(dv.cpu().view(nbt, -1)[:-1].view(torch.uint8), r.view(nbt, -1)[:-1].view(torch.uint8))


def test_quantized_mixed_step_full_size(attn_options):
    """The mixed 2048-token-chunk step on a quantized pool in one tcgen05
    launch after the dequantizing pass: sampled rows of every request and
    every head of the last decode against the oracle."""
    attn_options(mixed_launch=1)
    spec = config_spec(4)
    b = make_batch(spec, device="cpu")
    m = b.meta
    pools = quantized_pools(b, 93)
    ws_bytes = pkv.attention_workspace_bytes(m.num_reqs, m.num_tokens, spec.num_q_heads, spec.head_dim,
                                             m.max_seq_len) + \
        pkv.fp8_prefill_scratch_bytes(m.query_start_loc, m.seq_lens, spec.num_q_heads, spec.num_kv_heads, 128)
    got, dev_pools, ws, names = _fp8_call(b, pools, True, 0, ws_bytes)
    assert "attn_tc_mixed" in names, names
    assert pkv.read_device_error(ws) == 0
    assert int(ws[COUNTERS].count_nonzero()) == 0
    kc, vc, ks, vs = [t.clone() for t in pools]
    oracle.paged_kv_write_fp8(kc, vc, ks, vs, b.k, b.v, m.slot_mapping)
    nbt = spec.num_blocks_total + 1
    for dv, r in zip(dev_pools, (kc, vc, ks, vs)):
        assert torch.equal(dv.cpu().view(nbt, -1)[:-1].view(torch.uint8), r.view(nbt, -1)[:-1].view(torch.uint8))
    gen = torch.Generator().manual_seed(45)
    toks, heads = [], []
    for r in range(m.num_reqs):
        b0, t = m.query_start_loc[r], m.query_start_loc[r + 1] - m.query_start_loc[r]
        for i in sorted({0, t - 1, t // 2}):
            toks.append(b0 + i)
            heads.append(int(torch.randint(0, spec.num_q_heads, (1,), generator=gen)))
    last_dec = 2048 + 63
    toks += [last_dec] * spec.num_q_heads
    heads += list(range(spec.num_q_heads))
    want = oracle.attention_rows_fp8(toks, heads, b.q, kc, vc, ks, vs, m.query_start_loc, m.seq_lens,
                                     m.block_table, spec.scale, threads())
    assert_close(got[torch.tensor(toks), torch.tensor(heads)], want, "quantized mixed step in one launch")
