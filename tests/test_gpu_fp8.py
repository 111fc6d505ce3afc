"""Quantized (FP8 E4M3) pools on the GPU against the oracle: the quantizing
write bit for bit, attention within the usual tolerance ("31. Engine v2",
"Attention over the pool": per (slot, head) scales beside K and V)."""
import math

import pytest
import torch

import oracle
import paged_kv_cache_84_gb300 as pkv
from workloads import Req, Spec, build_meta, config_spec, make_batch, random_spec, subset_spec
from _helpers import MAX_ERR, MEAN_ERR, assert_close, quantized_pools as _quantized_pools, threads

pytestmark = pytest.mark.gpu


def _run(batch, pools, window=0, workspace_bytes=None):
    spec, m = batch.spec, batch.meta
    kc, vc, ks, vs = [t.cuda() for t in pools]
    k, v, q = batch.k.cuda(), batch.v.cuda(), batch.q.cuda()
    slots = m.slot_mapping.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_write_fp8(k, v, kc, vc, ks, vs, slots, err)
    out = torch.full_like(q, float("nan"))
    ws = pkv.make_workspace(workspace_bytes or pkv.attention_workspace_bytes(
        max(1, m.num_reqs), max(1, m.num_tokens), spec.num_q_heads, spec.head_dim, max(1, m.max_seq_len)), "cuda")
    pkv.ragged_paged_attention_fp8(out, q, kc, vc, ks, vs, torch.tensor(m.query_start_loc, dtype=torch.int32,
                                   device="cuda"), torch.tensor(m.seq_lens, dtype=torch.int32, device="cuda"),
                                   m.block_table.cuda(), m.query_start_loc, m.seq_lens, m.max_query_len,
                                   m.max_seq_len, spec.scale, ws, window=window)
    torch.cuda.synchronize()
    return out, (kc, vc, ks, vs), err, ws


def _oracle(batch, pools, window=0):
    spec, m = batch.spec, batch.meta
    kc, vc, ks, vs = [t.clone() for t in pools]
    oracle.paged_kv_write_fp8(kc, vc, ks, vs, batch.k, batch.v, m.slot_mapping)
    out = oracle.ragged_paged_attention_fp8(batch.q, kc, vc, ks, vs, m.query_start_loc, m.seq_lens, m.block_table,
                                            spec.scale, threads(), window=window)
    return out, (kc, vc, ks, vs)


FP8_CASES = [
    # seed, reqs, max_ctx, max_new, hq, hkv, pad rows
    (0, 8, 700, 40, 32, 8, 1),
    (1, 6, 3000, 3, 16, 4, 0),
    (2, 5, 1500, 130, 8, 8, 0),
    (3, 12, 400, 20, 64, 8, 2),
    (4, 4, 5000, 1, 32, 4, 0),
    (5, 4, 900, 2, 32, 16, 0),
    (6, 3, 2600, 1, 64, 32, 1),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=[f"seed{c[0]}" for c in FP8_CASES])
def test_fp8_write_bit_exact_and_attention_parity(case):
    seed, reqs, max_ctx, max_new, hq, hkv, pad = case
    spec = random_spec(200 + seed, reqs, max_ctx, max_new, hq, hkv, 128, pad_rows=pad)
    b = make_batch(spec, device="cpu")
    pools = _quantized_pools(b, seed)
    got, dev_pools, err, ws = _run(b, pools)
    want, ref_pools = _oracle(b, pools)
    nbt = spec.num_blocks_total + 1
    for d, r in zip(dev_pools, ref_pools):
        d = d.cpu()
        # the whole pool except the scratch block is bit-exact
        assert torch.equal(d.view(nbt, -1)[:-1].view(torch.uint8), r.view(nbt, -1)[:-1].view(torch.uint8))
    assert pkv.read_device_error(err) == 0
    assert_close(got, want, f"fp8 seed {seed}")
    assert pkv.read_device_error(ws) == 0


@pytest.mark.parametrize("row_tiles", ["0", "1"], ids=["key-major", "row-tiles"])
@pytest.mark.parametrize("split", ["128", "1024", "cluster"])
@pytest.mark.parametrize("window", [0, 300])
def test_fp8_split_paths_and_window(split, window, row_tiles, attn_options):
    """Decode splits on the slot-ring (128, split counters; "cluster": four
    splits per request combined in a thread-block cluster) and the streaming
    kernel (1024), in key-major and in 16-row tiles, with and without a
    sliding window."""
    if split == "cluster":
        attn_options(cluster=4)
        split = "256"
    attn_options(split_tokens=int(split))
    attn_options(decode_row_tiles=int(row_tiles))
    reqs = [Req(3000, 1, list(range(0, 188))), Req(700, 40, list(range(188, 235))),
            Req(2500, 2, list(range(235, 392))), Req(5000, 1, list(range(392, 705)))]
    spec = Spec("fp8-paths", reqs, 32, 8, 128, 16, 710, 1 / math.sqrt(128), 71)
    b = make_batch(spec, device="cpu")
    pools = _quantized_pools(b, 72)
    got, _, _, _ = _run(b, pools, window=window)
    want, _ = _oracle(b, pools, window=window)
    assert_close(got, want, f"fp8 split {split} window {window}")


HEAD_PAIR_CASES = [
    # hq, hkv, (computed, new) per request: every request has t * g <= 8 rows
    # per KV head, so the streaming kernel runs key-major tiles two KV heads
    # per CTA; ragged tails, a padding request, t > 1 rows per head
    (8, 8, [(2500, 8), (1033, 3), (4000, 1), (0, 0)]),
    (32, 16, [(3001, 4), (1700, 1), (2222, 2)]),
    (16, 4, [(2900, 2), (1111, 1), (0, 0), (3500, 2)]),
    (64, 8, [(5000, 1), (1800, 1)]),
]


@pytest.mark.parametrize("window", [0, 700])
@pytest.mark.parametrize("case", HEAD_PAIR_CASES, ids=[f"hq{c[0]}-hkv{c[1]}" for c in HEAD_PAIR_CASES])
def test_fp8_streaming_head_pairs(case, window, attn_options):
    """Quantized pools on the streaming kernel (splits of 1024 keys): key-major
    tiles with two KV heads per CTA, every group size the kernel stages."""
    attn_options(split_tokens=1024)
    hq, hkv, plan = case
    reqs, nxt = [], 0
    for computed, new in plan:
        if new == 0:
            reqs.append(Req(0, 1, [], pad=True))
            continue
        nb = (computed + new + 15) // 16
        reqs.append(Req(computed, new, list(range(nxt, nxt + nb))))
        nxt += nb
    spec = Spec("fp8-head-pairs", reqs, hq, hkv, 128, 16, nxt + 5, 1 / math.sqrt(128), 80 + hq)
    b = make_batch(spec, device="cpu")
    pools = _quantized_pools(b, 81)
    got, _, err, ws = _run(b, pools, window=window)
    want, _ = _oracle(b, pools, window=window)
    assert pkv.read_device_error(err) == 0
    assert pkv.read_device_error(ws) == 0
    assert_close(got, want, f"fp8 head pairs hq {hq} hkv {hkv} window {window}")


def test_fp8_long_decodes_sampled():
    """The 32 x 32768 decode shape (4 requests), the streaming kernel."""
    spec = subset_spec(config_spec(5), 4)
    b = make_batch(spec, device="cpu")
    pools = _quantized_pools(b, 73)
    got, _, _, _ = _run(b, pools)
    m = b.meta
    kc, vc, ks, vs = [t.clone() for t in pools]
    oracle.paged_kv_write_fp8(kc, vc, ks, vs, b.k, b.v, m.slot_mapping)
    toks = [0, 1, 2, 3, 0, 3]
    heads = [0, 17, 40, 63, 63, 5]
    want = oracle.attention_rows_fp8(toks, heads, b.q, kc, vc, ks, vs, m.query_start_loc, m.seq_lens,
                                     m.block_table, spec.scale, threads())
    assert_close(got[torch.tensor(toks), torch.tensor(heads)], want, "fp8 long decodes")


def test_fp8_unsupported_shapes_are_rejected():
    spec = random_spec(230, 3, 100, 1, 8, 2, 128)          # 2 KV heads: not a multiple of 4
    b = make_batch(spec, device="cpu")
    pools = _quantized_pools(b, 74)
    with pytest.raises(pkv.PkvError) as e:
        _run(b, pools)
    assert e.value.status == 2


@pytest.mark.parametrize("window", [0, 300])
@pytest.mark.parametrize("case", [FP8_CASES[0], FP8_CASES[2], FP8_CASES[3]], ids=["seed0", "seed2", "seed3"])
def test_fp8_prefill_on_tensor_cores(case, window):
    """With the extra workspace, quantized-pool prefill chunks attend over bf16
    copies of their blocks on the tcgen05 kernel: parity with the oracle's
    code * scale attention, and the same pools as with the plain workspace."""
    seed, reqs, max_ctx, max_new, hq, hkv, pad = case
    spec = random_spec(200 + seed, reqs, max_ctx, max_new, hq, hkv, 128, pad_rows=pad)
    b = make_batch(spec, device="cpu")
    m = b.meta
    extra = pkv.fp8_prefill_scratch_bytes(m.query_start_loc, m.seq_lens, hq, hkv, 128)
    assert extra > 0
    base = pkv.attention_workspace_bytes(max(1, m.num_reqs), max(1, m.num_tokens), hq, 128, max(1, m.max_seq_len))
    pools = _quantized_pools(b, seed)
    got, _, err, ws = _run(b, pools, window=window, workspace_bytes=base + extra)
    want, _ = _oracle(b, pools, window=window)
    assert pkv.read_device_error(err) == 0
    assert pkv.read_device_error(ws) == 0
    assert_close(got, want, f"fp8 tcgen05 prefill seed {seed} window {window}")


def test_fp8_mixed_chunk_step_sampled_on_tensor_cores():
    """The mixed 2048-token-chunk step (a subset: the chunk at 16384 and 10
    decodes) on a quantized pool with the tcgen05 scratch: sampled rows of
    the chunk and of the decodes."""
    spec = subset_spec(config_spec(4), 11)
    b = make_batch(spec, device="cpu")
    m = b.meta
    extra = pkv.fp8_prefill_scratch_bytes(m.query_start_loc, m.seq_lens, spec.num_q_heads, spec.num_kv_heads, 128)
    base = pkv.attention_workspace_bytes(m.num_reqs, m.num_tokens, spec.num_q_heads, 128, m.max_seq_len)
    pools = _quantized_pools(b, 74)
    got, _, _, ws = _run(b, pools, workspace_bytes=base + extra)
    assert pkv.read_device_error(ws) == 0
    kc, vc, ks, vs = [t.clone() for t in pools]
    oracle.paged_kv_write_fp8(kc, vc, ks, vs, b.k, b.v, m.slot_mapping)
    n = m.num_tokens
    toks = [0, 1, 777, 1500, 2047, 2048, 2052, n - 3, n - 2, n - 1]
    heads = [0, 31, 5, 17, 3, 30, 12, 7, 22, 1]
    want = oracle.attention_rows_fp8(toks, heads, b.q, kc, vc, ks, vs, m.query_start_loc, m.seq_lens,
                                     m.block_table, spec.scale, threads())
    assert_close(got[torch.tensor(toks), torch.tensor(heads)], want, "fp8 mixed step on tcgen05")



def _run_combined(batch, pools, window=0, workspace_bytes=None):
    spec, m = batch.spec, batch.meta
    kc, vc, ks, vs = [t.cuda() for t in pools]
    k, v, q = batch.k.cuda(), batch.v.cuda(), batch.q.cuda()
    slots = m.slot_mapping.cuda()
    out = torch.full_like(q, float("nan"))
    ws = pkv.make_workspace(workspace_bytes or pkv.attention_workspace_bytes(
        max(1, m.num_reqs), max(1, m.num_tokens), spec.num_q_heads, spec.head_dim, max(1, m.max_seq_len)), "cuda")
    pkv.paged_kv_write_attention_fp8(k, v, kc, vc, ks, vs, slots, out, q,
                                     torch.tensor(m.query_start_loc, dtype=torch.int32, device="cuda"),
                                     torch.tensor(m.seq_lens, dtype=torch.int32, device="cuda"),
                                     m.block_table.cuda(), m.query_start_loc, m.seq_lens, m.max_query_len,
                                     m.max_seq_len, spec.scale, ws, window=window)
    torch.cuda.synchronize()
    return out, (kc, vc, ks, vs), ws


@pytest.mark.parametrize("mode", ["combined", "tcgen05-scratch", "separate"])
@pytest.mark.parametrize("case", FP8_CASES[:4], ids=[f"seed{c[0]}" for c in FP8_CASES[:4]])
def test_fp8_combined_write_and_attention(case, mode, attn_options):
    """pkv_paged_kv_write_attention_fp8: decode CTAs quantize and write their
    own rows, the prefill rows go through the ranged quantizing scatter; codes
    and scales bit-exact (whole pool except the scratch block), attention
    within the tolerance; with the tcgen05 prefill scratch; and as the full
    scatter followed by the attention (the separate_write option)."""
    if mode == "separate":
        attn_options(separate_write=1)
    seed, reqs, max_ctx, max_new, hq, hkv, pad = case
    spec = random_spec(200 + seed, reqs, max_ctx, max_new, hq, hkv, 128, pad_rows=pad)
    b = make_batch(spec, device="cpu")
    m = b.meta
    wsb = None
    if mode == "tcgen05-scratch":
        wsb = pkv.attention_workspace_bytes(max(1, m.num_reqs), max(1, m.num_tokens), hq, 128,
                                            max(1, m.max_seq_len)) + \
            pkv.fp8_prefill_scratch_bytes(m.query_start_loc, m.seq_lens, hq, hkv, 128)
    pools = _quantized_pools(b, seed)
    for window in (0, 300):
        got, dev_pools, ws = _run_combined(b, pools, window=window, workspace_bytes=wsb)
        want, ref_pools = _oracle(b, pools, window=window)
        nbt = spec.num_blocks_total + 1
        for d, r in zip(dev_pools, ref_pools):
            assert torch.equal(d.cpu().view(nbt, -1)[:-1].view(torch.uint8), r.view(nbt, -1)[:-1].view(torch.uint8))
        assert pkv.read_device_error(ws) == 0
        assert_close(got, want, f"fp8 combined {mode} seed {seed} window {window}")


def test_fp8_combined_long_decodes_one_launch():
    """Decode-only batch on the streaming kernel (two KV heads per CTA): one
    launch writes and attends."""
    spec = subset_spec(config_spec(5), 4)
    b = make_batch(spec, device="cpu")
    pools = _quantized_pools(b, 75)
    before = pkv.launch_count()
    got, dev_pools, ws = _run_combined(b, pools)
    assert pkv.launch_count() - before == 1
    m = b.meta
    kc, vc, ks, vs = [t.clone() for t in pools]
    oracle.paged_kv_write_fp8(kc, vc, ks, vs, b.k, b.v, m.slot_mapping)
    for d, r in zip(dev_pools, (kc, vc, ks, vs)):
        nbt = spec.num_blocks_total + 1
        assert torch.equal(d.cpu().view(nbt, -1)[:-1].view(torch.uint8), r.view(nbt, -1)[:-1].view(torch.uint8))
    toks, heads = [0, 1, 2, 3], [0, 21, 42, 63]
    want = oracle.attention_rows_fp8(toks, heads, b.q, kc, vc, ks, vs, m.query_start_loc, m.seq_lens,
                                     m.block_table, spec.scale, threads())
    assert_close(got[torch.tensor(toks), torch.tensor(heads)], want, "fp8 combined long decodes")
    assert pkv.read_device_error(ws) == 0


def _midpoint_rows(shape, seed):
    """bf16 rows [N, Hkv, 128] whose quotients by their scale are exactly E4M3
    rounding midpoints, where the code is decided by the tie rule alone.  A
    row's largest magnitude is 7 * o * 2^(a+6), in [0.5, 2) (the size of the
    other tests' values, so that the attention check's absolute tolerance
    means the same), so its scale max/448 = o * 2^a is exact (o = 3, 5 or 7);
    every other value is +-o * m * 2^p with m odd in 17..31, whose quotient
    m * 2^(p-a) lies halfway between two neighbouring E4M3 values."""
    import numpy as np
    rng = np.random.default_rng(seed)
    n, hkv, d = shape
    rows = np.empty((n * hkv, d), dtype=np.float32)
    for i in range(n * hkv):
        o = int(rng.choice([3, 5, 7]))
        a = int(rng.integers(0, 2)) - math.ceil(math.log2(7 * o)) - 6     # max in [0.5, 2)
        ms = np.array([m for m in range(17, 32, 2) if o * m <= 255])
        x = o * rng.choice(ms, d) * np.exp2(rng.integers(a - 4, a + 4, d))
        x[rng.integers(0, d)] = 7 * o * 2.0 ** (a + 6)
        rows[i] = x * np.where(rng.random(d) < 0.5, -1.0, 1.0)
    return torch.from_numpy(rows).to(torch.bfloat16).view(n, hkv, d)


def _share_on_midpoints(x):
    """Share of the values of bf16 rows x [R, 128] whose quotient by the row's
    scale (fp32, as the write computes it) is an E4M3 rounding midpoint: a
    5-bit significand ending in a one, in E4M3's normal range."""
    import numpy as np
    f = x.to(torch.float32).numpy()
    s = np.abs(f).max(axis=1, keepdims=True) / np.float32(448.0)
    q = np.abs(f / s).astype(np.float32)
    man, ex = np.frexp(q.astype(np.float64))                 # q = man * 2^ex, man in [0.5, 1)
    sig = man * 32.0                                         # 5 significant bits
    return float(np.mean((sig == np.round(sig)) & (np.round(sig) % 2 == 1) & (q >= 2.0 ** -6)))


@pytest.mark.parametrize("mode", ["write", "combined"])
def test_fp8_write_ties_on_rounding_midpoints(mode):
    """Values whose quotient by the scale sits exactly halfway between two
    E4M3 values: the quantizing write (and the combined call: decode CTAs and
    the ranged scatter) takes the even code, bit for bit as the oracle."""
    spec = random_spec(410, 6, 1500, 90, 32, 8, 128, pad_rows=1)
    b = make_batch(spec, device="cpu")
    b.k = _midpoint_rows(tuple(b.k.shape), 411)
    b.v = _midpoint_rows(tuple(b.v.shape), 412)
    assert _share_on_midpoints(b.k.view(-1, 128)) > 0.9
    pools = _quantized_pools(b, 413)
    if mode == "write":
        got, dev_pools, err, ws = _run(b, pools)
        assert pkv.read_device_error(err) == 0
    else:
        got, dev_pools, ws = _run_combined(b, pools)
    want, ref_pools = _oracle(b, pools)
    nbt = spec.num_blocks_total + 1
    for d, r in zip(dev_pools, ref_pools):
        assert torch.equal(d.cpu().view(nbt, -1)[:-1].view(torch.uint8), r.view(nbt, -1)[:-1].view(torch.uint8))
    assert pkv.read_device_error(ws) == 0
    assert_close(got, want, f"fp8 midpoint rows, {mode}")
