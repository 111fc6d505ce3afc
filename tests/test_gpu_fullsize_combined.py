"""The call the benchmark times, at full size, against the oracle.

``bench.py`` times one ``pkv_paged_kv_write_attention`` call per step (and
``pkv_paged_kv_write_attention_fp8`` on quantized pools), replayed from a
CUDA graph, with the workspace ``pkv_attention_workspace_bytes`` gives for
the batch.  These tests run that same call, captured and replayed the same
way, on the three large workloads at their full sizes:

- the pools after the step are compared bit for bit with the oracle's write
  (the whole pool except the scratch slot: "31. Engine v2", "Attention over
  the pool", ``write_kv``);
- sampled output rows are compared with the oracle's attention over the
  pool ("Attention over the pool", the reference backend's ``forward``):
  every request, the tile edges of the long chunk, every head of some rows.
  Only rows are sampled because the oracle's full step over these batches
  takes minutes; every row the oracle computes is compared.

In these batches the combined call splits the work in ways the small tests
do not reach: ten streaming splits of 3456 keys per 32768-key decode, merged
by the CTA that finishes last; 64 decodes that write their own rows, as
1024-key items on the decode CTAs that open the one launch of the mixed step,
ahead of the 2048-token chunk's tcgen05 pairs whose rows a ranged scatter
writes.
"""
import concurrent.futures as cf

import pytest
import torch

import oracle
import paged_kv_cache_84_gb300 as pkv
from workloads import config_spec, make_batch
from _helpers import DeviceStep, assert_close, cpu_copy, oracle_write, threads

pytestmark = pytest.mark.gpu


def _pool_bits(t):
    nbt, bs, hkv, d = t.shape
    return t.contiguous().view(torch.int16).view(nbt * bs, hkv * d)


def _rows_to_check(spec, meta, seed, per_req_heads):
    """Every request's first, middle and last new token (and the token at the
    128-row tile edge), with per_req_heads random heads each; for the mixed
    workload also the long chunk's tile edges and every head of the last row
    of the second fresh prompt."""
    gen = torch.Generator().manual_seed(seed)
    toks, heads = [], []
    for r, req in enumerate(spec.reqs):
        b, t = meta.query_start_loc[r], req.new
        for i in sorted({0, t - 1, t // 2, min(t - 1, 127), min(t - 1, 128)}):
            for h in torch.randint(0, spec.num_q_heads, (per_req_heads,), generator=gen).tolist():
                toks.append(b + i)
                heads.append(h)
    return toks, heads


def _mixed_extra_rows(spec, meta):
    """The 2048-token chunk's tile edges (32 tokens x 4 heads per tile, pairs of
    64 tokens per CTA) in several heads, and every head of the last row."""
    toks, heads = [], []
    for i in (31, 32, 63, 64, 65, 1000, 1023, 1024, 2047):
        for h in range(0, spec.num_q_heads, 7):
            toks.append(i)
            heads.append(h)
    last = meta.num_tokens - 1
    for h in range(spec.num_q_heads):
        toks.append(last)
        heads.append(h)
    return toks, heads


def _replay_in_graph(fn):
    """Run fn once captured in a CUDA graph and replayed, as the benchmark does."""
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fn()
    g.replay()
    torch.cuda.synchronize()
    del g


@pytest.mark.parametrize("cfg", [3, 4, 5], ids=["decode-256req", "mixed-chunk2048", "long-decode-32req"])
def test_combined_call_full_size(cfg):
    spec = config_spec(cfg)
    b = make_batch(spec, device="cuda")                 # values drawn on the device
    ref = cpu_copy(b)                                   # inputs, copied before any library kernel runs
    dev = DeviceStep(b)                                 # the benchmark's workspace size
    plan = pkv.plan_attention(b.meta.query_start_loc, b.meta.seq_lens, spec.num_q_heads, spec.num_kv_heads,
                              spec.head_dim, combined=True, workspace_bytes=dev.ws.numel())
    if cfg == 5:
        assert plan["max_decode_splits"] >= 8 and plan["decode_streaming"]
    if cfg == 4:                                        # one launch: decode CTAs ahead of the tcgen05 pairs
        assert plan["mixed_launch"] and plan["mixed_decode_ctas"] > 0 and plan["prefill_tensor_requests"] == 3
    _replay_in_graph(dev.combined)
    assert torch.isfinite(dev.out.float()).all()
    oracle_write(ref)
    for got, want in ((dev.k_cache, ref.k_cache), (dev.v_cache, ref.v_cache)):
        assert torch.equal(_pool_bits(got.cpu())[:-1], _pool_bits(want)[:-1])
    assert pkv.read_device_error(dev.ws) == 0
    toks, heads = _rows_to_check(spec, b.meta, cfg, per_req_heads=1 if cfg == 3 else 2)
    if cfg == 4:
        t2, h2 = _mixed_extra_rows(spec, b.meta)
        toks, heads = toks + t2, heads + h2
    want = oracle.attention_rows(toks, heads, ref.q, ref.k_cache, ref.v_cache, ref.meta.query_start_loc,
                                 ref.meta.seq_lens, ref.meta.block_table, spec.scale, threads())
    got = dev.out[torch.tensor(toks), torch.tensor(heads)]
    assert_close(got, want, f"combined call, {spec.name}, {len(toks)} sampled rows")


def _oracle_quantized_pool(k_pool, v_pool):
    """Codes and scales of a whole bf16 pool, written by the oracle's
    quantizing write slot by slot (disjoint slot ranges on several threads)."""
    nbt, bs, hkv, d = k_pool.shape
    kc = torch.empty((nbt, bs, hkv, d), dtype=torch.uint8)
    vc = torch.empty_like(kc)
    ks = torch.empty((nbt, bs, hkv), dtype=torch.float32)
    vs = torch.empty_like(ks)
    n = nbt * bs
    kf, vf = k_pool.view(n, hkv, d), v_pool.view(n, hkv, d)
    step = (n + 63) // 64

    def part(s0):
        s1 = min(n, s0 + step)
        oracle.paged_kv_write_fp8(kc, vc, ks, vs, kf[s0:s1], vf[s0:s1], torch.arange(s0, s1, dtype=torch.int64))

    with cf.ThreadPoolExecutor(threads()) as ex:
        list(ex.map(part, range(0, n, step)))
    return kc, vc, ks, vs


@pytest.mark.parametrize("cfg", [3, 5], ids=["decode-256req", "long-decode-32req"])
def test_combined_call_quantized_pool_full_size(cfg):
    """The same on a quantized (E4M3) pool: every slot holds the oracle's codes
    of N(0,1) values; the call quantizes and writes the step's rows and
    attends over codes times scales."""
    spec = config_spec(cfg)
    b = make_batch(spec, device="cuda")
    m = b.meta
    k_host, v_host = b.k_cache.cpu(), b.v_cache.cpu()
    del b.k_cache, b.v_cache
    torch.cuda.empty_cache()
    pools = _oracle_quantized_pool(k_host, v_host)
    del k_host, v_host
    kc, vc, ks, vs = [t.cuda() for t in pools]
    q, k, v = b.q, b.k, b.v
    slots = m.slot_mapping.cuda()
    qsl = torch.tensor(m.query_start_loc, dtype=torch.int32, device="cuda")
    sln = torch.tensor(m.seq_lens, dtype=torch.int32, device="cuda")
    bt = m.block_table.cuda()
    out = torch.full_like(q, float("nan"))
    extra = pkv.fp8_prefill_scratch_bytes(m.query_start_loc, m.seq_lens, spec.num_q_heads, spec.num_kv_heads, 128)
    ws = pkv.make_workspace(pkv.attention_workspace_bytes(m.num_reqs, m.num_tokens, spec.num_q_heads, 128,
                                                          m.max_seq_len) + extra, "cuda")

    def step():
        pkv.paged_kv_write_attention_fp8(k, v, kc, vc, ks, vs, slots, out, q, qsl, sln, bt, m.query_start_loc,
                                         m.seq_lens, m.max_query_len, m.max_seq_len, spec.scale, ws)

    _replay_in_graph(step)
    assert pkv.read_device_error(ws) == 0
    rk, rv, rks, rvs = pools
    oracle.paged_kv_write_fp8(rk, rv, rks, rvs, k.cpu(), v.cpu(), m.slot_mapping)
    nbt = spec.num_blocks_total
    for got, want in zip((kc, vc, ks, vs), (rk, rv, rks, rvs)):
        g = got.cpu().view(nbt, -1)[:-1].contiguous().view(torch.uint8)
        w = want.view(nbt, -1)[:-1].contiguous().view(torch.uint8)
        assert torch.equal(g, w)
    toks, heads = _rows_to_check(spec, m, 100 + cfg, per_req_heads=1 if cfg == 3 else 2)
    want = oracle.attention_rows_fp8(toks, heads, q.cpu(), rk, rv, rks, rvs, m.query_start_loc, m.seq_lens,
                                     m.block_table, spec.scale, threads())
    got = out[torch.tensor(toks), torch.tensor(heads)]
    assert_close(got, want, f"quantized combined call, {spec.name}, {len(toks)} sampled rows")
