"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: the checks are the pages'
printed worked examples (tests/golden/), brute-force dense attention through
torch's scaled_dot_product_attention (a library routine) on contiguous
per-request K/V, closed forms, and invariances that the pages state for the
engine (block sizes 1/4/16/64, chunk budgets 8/33/64/4096, prefix sharing,
batch composition; vllm-lite README, test list) and for the block table
(physical permutation of blocks; "vLLM: LLM Inference as a memory and
scheduling problem", "PagedAttention: virtual memory, but for tokens").
"""
import math
import os

import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import Req, Spec, build_meta, config_spec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        rows.setdefault(key, []).append([int(v) for v in vals])
    return rows


def _bf16(shape, gen):
    return torch.randn(shape, generator=gen).to(torch.bfloat16)


# ---------------------------------------------------------------- slot formula

def test_slot_formula_block_table_example():
    g = _golden("block_table_example.txt")
    bs = g["block_size"][0][0]
    table = g["table"][0]
    for p, want in g["slot"]:
        assert oracle.slot(table, p, bs) == want


def test_layout_example_metadata():
    g = _golden("layout_example.txt")
    meta = build_meta(config_spec(1))
    assert meta.query_start_loc == g["query_start_loc"][0]
    assert meta.seq_lens == g["seq_lens"][0]
    assert meta.positions == g["positions"][0]


@pytest.mark.parametrize("cfg", [1, 2])
def test_generator_slots_follow_oracle_slot(cfg):
    spec = config_spec(cfg)
    meta = build_meta(spec)
    for r, req in enumerate(spec.reqs):
        b = meta.query_start_loc[r]
        for i in range(req.new):
            p = req.computed + i
            assert int(meta.slot_mapping[b + i]) == oracle.slot(req.table, p, spec.block_size)


# ---------------------------------------------------------------- write

def test_write_small_worked_case():
    # pool of 4 blocks x 2 slots, 1 KV head, d 2 -> flat slots 0..7, scratch = 7
    kc = torch.zeros((4, 2, 1, 2), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    k = torch.tensor([[[1.0, 2.0]], [[3.0, 4.0]], [[5.0, 6.0]]], dtype=torch.bfloat16)
    v = -k
    oracle.paged_kv_write(kc, vc, k, v, torch.tensor([5, -1, 0]))
    flat_k = kc.view(8, 2).float()
    assert flat_k[5].tolist() == [1.0, 2.0]
    assert flat_k[7].tolist() == [3.0, 4.0]          # padding row -> last slot
    assert flat_k[0].tolist() == [5.0, 6.0]
    assert flat_k[[1, 2, 3, 4, 6]].abs().sum().item() == 0.0
    assert vc.view(8, 2).float()[5].tolist() == [-1.0, -2.0]


@pytest.mark.parametrize("seed", range(3))
def test_write_matches_index_copy_on_sentinel_pool(seed):
    gen = torch.Generator().manual_seed(seed)
    nbt, bs, hkv, d = 37, 16, 4, 48
    n = 100
    slots = torch.randperm(nbt * bs - 1, generator=gen)[:n]          # distinct real slots
    slots[::17] = -1                                                   # some padding rows
    k, v = _bf16((n, hkv, d), gen), _bf16((n, hkv, d), gen)
    kc = torch.empty((nbt, bs, hkv, d), dtype=torch.bfloat16)
    kc.view(torch.int16).fill_(0x7F7F)
    vc = kc.clone()
    exp_k, exp_v = kc.clone(), vc.clone()
    real = slots >= 0
    exp_k.view(-1, hkv, d).view(torch.int16)[slots[real]] = k.view(torch.int16)[real]
    exp_v.view(-1, hkv, d).view(torch.int16)[slots[real]] = v.view(torch.int16)[real]
    oracle.paged_kv_write(kc, vc, k, v, slots)
    # every slot but the scratch one is bit-exact; scratch holds one of the padding rows
    assert torch.equal(kc.view(torch.int16).view(-1, hkv * d)[:-1], exp_k.view(torch.int16).view(-1, hkv * d)[:-1])
    assert torch.equal(vc.view(torch.int16).view(-1, hkv * d)[:-1], exp_v.view(torch.int16).view(-1, hkv * d)[:-1])
    pad_rows = k.view(torch.int16)[~real].view(-1, hkv * d)
    scratch = kc.view(torch.int16).view(-1, hkv * d)[-1]
    assert any(torch.equal(scratch, r) for r in pad_rows)


def test_write_rejects_slot_outside_pool():
    kc = torch.zeros((2, 4, 1, 8), dtype=torch.bfloat16)
    k = torch.zeros((1, 1, 8), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle.paged_kv_write(kc, kc.clone(), k, k, torch.tensor([8]))


# ---------------------------------------------------------------- dense brute force

class Problem:
    """Requests with dense per-request K/V, stored in a permuted paged pool by
    two oracle writes (history, then this step's rows)."""

    def __init__(self, plan, hq, hkv, d, bs, seed, spare=3, shared_prefix_blocks=0, junk=True,
                 kv=None, q=None):
        gen = torch.Generator().manual_seed(seed)
        self.plan, self.hq, self.hkv, self.d, self.bs = plan, hq, hkv, d, bs
        nblk = [-(-(c + t) // bs) for c, t in plan]
        shared = shared_prefix_blocks
        used = shared + sum(n - shared for n in nblk)
        nb = used + spare
        perm = torch.randperm(nb, generator=gen).tolist()
        pre, cur = perm[:shared], shared
        tables = []
        for n in nblk:
            tables.append(pre + perm[cur:cur + n - shared])
            cur += n - shared
        self.tables = tables
        # dense logical K/V per request; requests sharing prefix blocks share those rows
        if kv is None:
            prefix_k = _bf16((shared * bs, hkv, d), gen)
            prefix_v = _bf16((shared * bs, hkv, d), gen)
            self.K, self.V = [], []
            for c, t in plan:
                L = c + t
                k = _bf16((L, hkv, d), gen)
                v = _bf16((L, hkv, d), gen)
                k[:min(L, shared * bs)] = prefix_k[:min(L, shared * bs)]
                v[:min(L, shared * bs)] = prefix_v[:min(L, shared * bs)]
                self.K.append(k)
                self.V.append(v)
        else:
            self.K, self.V = kv
        reqs = [Req(c, t, tab) for (c, t), tab in zip(plan, tables)]
        self.spec = Spec("pin", reqs, hq, hkv, d, bs, nb, 1.0 / math.sqrt(d), seed)
        self.meta = build_meta(self.spec)
        n = self.meta.num_tokens
        self.Q = q if q is not None else _bf16((n, hq, d), gen)
        shape = (nb + 1, bs, hkv, d)
        self.kc = _bf16(shape, gen) if junk else torch.zeros(shape, dtype=torch.bfloat16)
        self.vc = _bf16(shape, gen) if junk else torch.zeros(shape, dtype=torch.bfloat16)
        # history: positions 0..c-1 of every request
        hist = build_meta(Spec("hist", [Req(0, c, tab) for (c, t), tab in zip(plan, tables)],
                               hq, hkv, d, bs, nb, 1.0, seed))
        hk = torch.cat([k[:c] for k, (c, t) in zip(self.K, plan)]) if hist.num_tokens else None
        hv = torch.cat([v[:c] for v, (c, t) in zip(self.V, plan)]) if hist.num_tokens else None
        if hist.num_tokens:
            oracle.paged_kv_write(self.kc, self.vc, hk, hv, hist.slot_mapping)
        # this step's rows
        self.k_new = torch.cat([k[c:] for k, (c, t) in zip(self.K, plan)])
        self.v_new = torch.cat([v[c:] for v, (c, t) in zip(self.V, plan)])
        oracle.paged_kv_write(self.kc, self.vc, self.k_new, self.v_new, self.meta.slot_mapping)

    def oracle_out(self, threads=1, window=0):
        return oracle.ragged_paged_attention(self.Q, self.kc, self.vc, self.meta.query_start_loc,
                                             self.meta.seq_lens, self.meta.block_table,
                                             self.spec.scale, threads, window=window)

    def brute_force(self, window=0):
        """torch SDPA in float64 on contiguous K/V, explicit offset-causal mask
        (restricted to keys above position - window when window > 0), GQA by
        repeating each KV head over its contiguous group of query heads."""
        g = self.hq // self.hkv
        out = torch.zeros((self.meta.num_tokens, self.hq, self.d), dtype=torch.float64)
        for r, (c, t) in enumerate(self.plan):
            b = self.meta.query_start_loc[r]
            L = c + t
            if t == 0 or L == 0:
                continue
            q = self.Q[b:b + t].double().transpose(0, 1)                       # [hq, t, d]
            k = self.K[r].double().repeat_interleave(g, dim=1).transpose(0, 1)  # [hq, L, d]
            v = self.V[r].double().repeat_interleave(g, dim=1).transpose(0, 1)
            qpos = torch.arange(L - t, L)[:, None]
            kpos = torch.arange(L)[None, :]
            allowed = kpos <= qpos
            if window > 0:
                allowed = allowed & (kpos > qpos - window)
            y = F.scaled_dot_product_attention(q[None], k[None], v[None], attn_mask=allowed,
                                               scale=self.spec.scale)
            out[b:b + t] = y[0].transpose(0, 1)
        return out


GQA = [(8, 8), (8, 4), (8, 2), (8, 1)]          # g = 1, 2, 4, 8


@pytest.mark.parametrize("hq,hkv", GQA)
@pytest.mark.parametrize("bs", [1, 4, 16])
def test_oracle_matches_dense_brute_force(hq, hkv, bs):
    plan = [(6, 3), (41, 1), (9, 1), (0, 4), (0, 1), (17, 15), (31, 2)]
    P = Problem(plan, hq, hkv, 48, bs, seed=hq * 10 + hkv + bs)
    got = P.oracle_out()
    want = P.brute_force()
    assert (got - want).abs().max().item() < 1e-10


def test_fresh_prompt_is_standard_causal_attention():
    """t == L: textbook causal attention (SDPA with is_causal, no explicit mask)."""
    L, hq, hkv, d = 37, 4, 2, 64
    P = Problem([(0, L)], hq, hkv, d, 16, seed=5)
    got = P.oracle_out()
    q = P.Q.double().transpose(0, 1)[None]
    k = P.K[0].double().repeat_interleave(2, dim=1).transpose(0, 1)[None]
    v = P.V[0].double().repeat_interleave(2, dim=1).transpose(0, 1)[None]
    want = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=1 / math.sqrt(d))[0].transpose(0, 1)
    assert (got - want).abs().max().item() < 1e-10


def test_multithreaded_matches_single_thread():
    P = Problem([(100, 20), (7, 1), (0, 33)], 8, 2, 48, 16, seed=9)
    assert torch.equal(P.oracle_out(1), P.oracle_out(4))


# ---------------------------------------------------------------- closed forms

def test_single_key_returns_its_value():
    """L = 1: the only weight is 1, so the output is v0 exactly."""
    P = Problem([(0, 1)], 4, 2, 48, 16, seed=3)
    got = P.oracle_out()
    want = P.V[0][0].double().repeat_interleave(2, dim=0)
    assert torch.equal(got[0], want)


def test_equal_keys_give_mean_of_visible_values():
    plan = [(20, 5)]
    gen = torch.Generator().manual_seed(11)
    L, hkv, d = 25, 2, 48
    krow = _bf16((1, hkv, d), gen)
    K = krow.expand(L, hkv, d).clone()
    V = _bf16((L, hkv, d), gen)
    P = Problem(plan, 4, hkv, d, 16, seed=11, kv=([K], [V]))
    got = P.oracle_out()
    for i in range(5):
        p = 20 + i
        want = V[:p + 1].double().mean(0).repeat_interleave(2, dim=0)
        assert (got[i] - want).abs().max().item() < 1e-12


def test_one_dominant_key_selects_its_value():
    gen = torch.Generator().manual_seed(12)
    L, hkv, d = 40, 1, 16
    K = torch.zeros((L, hkv, d), dtype=torch.bfloat16)
    K[13, 0, 0] = 64.0
    V = _bf16((L, hkv, d), gen)
    q = torch.zeros((1, 1, d), dtype=torch.bfloat16)
    q[0, 0, 0] = 64.0
    P = Problem([(L - 1, 1)], 1, hkv, d, 16, seed=12, kv=([K], [V]), q=q)
    got = P.oracle_out()
    # score gap 64*64/4 = 1024 against every other key: weights e^-1024 ~ 0
    assert (got[0, 0] - V[13, 0].double()).abs().max().item() < 1e-300 + 1e-12


def test_padding_request_gives_zero_rows():
    P = Problem([(5, 2)], 4, 2, 48, 16, seed=2)
    qsl = P.meta.query_start_loc + [P.meta.query_start_loc[-1] + 1]
    sl = P.meta.seq_lens + [0]
    bt = torch.cat([P.meta.block_table, torch.zeros((1, P.meta.block_table.shape[1]), dtype=torch.int32)])
    q = torch.cat([P.Q, _bf16((1, 4, 48), torch.Generator().manual_seed(0))])
    out = oracle.ragged_paged_attention(q, P.kc, P.vc, qsl, sl, bt, P.spec.scale)
    assert out[-1].abs().sum().item() == 0.0
    assert torch.equal(out[:-1], P.oracle_out())


# ---------------------------------------------------------------- invariances (bit-identical)

def test_physical_block_permutation_invariance():
    P = Problem([(50, 3), (17, 1), (0, 20)], 8, 4, 48, 16, seed=21)
    base = P.oracle_out()
    nbt = P.kc.shape[0]
    gen = torch.Generator().manual_seed(99)
    perm = torch.randperm(nbt - 1, generator=gen)       # physical block b moves to perm[b]
    kc2, vc2 = P.kc.clone(), P.vc.clone()
    kc2[perm] = P.kc[:nbt - 1]
    vc2[perm] = P.vc[:nbt - 1]
    bt2 = perm[P.meta.block_table.long()].to(torch.int32)
    out2 = oracle.ragged_paged_attention(P.Q, kc2, vc2, P.meta.query_start_loc, P.meta.seq_lens,
                                         bt2, P.spec.scale)
    assert torch.equal(base, out2)


def _chunked_run(prompt_len, chunk, K, V, Q, hq, hkv, d, bs):
    """Prefill one prompt in chunks over successive write+attend steps;
    returns the output of every position."""
    nb = -(-prompt_len // bs) + 2
    table = list(range(nb - 1, -1, -1))[: -(-prompt_len // bs)]        # reversed physical order
    kc = torch.zeros((nb + 1, bs, hkv, d), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    outs = []
    c = 0
    while c < prompt_len:
        t = min(chunk, prompt_len - c)
        spec = Spec("chunk", [Req(c, t, table)], hq, hkv, d, bs, nb, 1 / math.sqrt(d), 0)
        meta = build_meta(spec)
        oracle.paged_kv_write(kc, vc, K[c:c + t], V[c:c + t], meta.slot_mapping)
        outs.append(oracle.ragged_paged_attention(Q[c:c + t], kc, vc, meta.query_start_loc,
                                                  meta.seq_lens, meta.block_table, spec.scale))
        c += t
    return torch.cat(outs)


def test_chunked_prefill_budget_invariance():
    gen = torch.Generator().manual_seed(31)
    L, hq, hkv, d = 150, 8, 2, 48
    K, V, Q = _bf16((L, hkv, d), gen), _bf16((L, hkv, d), gen), _bf16((L, hq, d), gen)
    runs = [_chunked_run(L, c, K, V, Q, hq, hkv, d, 16) for c in (8, 33, 64, 4096)]
    for r in runs[1:]:
        assert torch.equal(runs[0], r)


def test_block_size_invariance():
    gen = torch.Generator().manual_seed(32)
    L, hq, hkv, d = 130, 8, 4, 48
    K, V, Q = _bf16((L, hkv, d), gen), _bf16((L, hkv, d), gen), _bf16((L, hq, d), gen)
    runs = [_chunked_run(L, 40, K, V, Q, hq, hkv, d, bs) for bs in (1, 4, 16, 64)]
    for r in runs[1:]:
        assert torch.equal(runs[0], r)


def test_shared_prefix_blocks_match_private_copies():
    plan = [(70, 1), (40, 8), (33, 1), (64, 1)]
    shared = Problem(plan, 8, 4, 48, 16, seed=41, shared_prefix_blocks=2)
    private = Problem(plan, 8, 4, 48, 16, seed=41, shared_prefix_blocks=0,
                      kv=(shared.K, shared.V), q=shared.Q)
    # shared tables really do point at the same physical blocks
    assert all(t[:2] == shared.tables[0][:2] for t in shared.tables)
    assert len({tuple(t[:2]) for t in private.tables}) == len(plan)
    assert torch.equal(shared.oracle_out(), private.oracle_out())


def test_alone_vs_batched_with_seven_others():
    gen = torch.Generator().manual_seed(51)
    others = [(int(torch.randint(0, 90, (1,), generator=gen)), int(torch.randint(1, 12, (1,), generator=gen)))
              for _ in range(7)]
    plan = others[:3] + [(60, 6)] + others[3:]
    batched = Problem(plan, 8, 2, 48, 16, seed=52)
    b = batched.meta.query_start_loc[3]
    alone = Problem([(60, 6)], 8, 2, 48, 16, seed=53, kv=([batched.K[3]], [batched.V[3]]),
                    q=batched.Q[b:b + 6].clone())
    assert torch.equal(batched.oracle_out()[b:b + 6], alone.oracle_out())


# ---------------------------------------------------------------- sampled rows, errors

def test_rows_entry_matches_full_entry():
    P = Problem([(30, 4), (9, 1), (0, 12)], 8, 4, 48, 16, seed=61)
    full = P.oracle_out()
    toks = [0, 3, 4, 5, 16, 10]
    heads = [0, 7, 3, 5, 2, 6]
    rows = oracle.attention_rows(toks, heads, P.Q, P.kc, P.vc, P.meta.query_start_loc,
                                 P.meta.seq_lens, P.meta.block_table, P.spec.scale)
    for k, (n, h) in enumerate(zip(toks, heads)):
        assert torch.equal(rows[k], full[n, h])


def test_inconsistent_metadata_is_rejected():
    P = Problem([(5, 2)], 4, 2, 48, 16, seed=1)
    with pytest.raises(ValueError):                  # t > seq_len
        oracle.ragged_paged_attention(P.Q, P.kc, P.vc, [0, 2], [1], P.meta.block_table, 0.1)
    bad = P.meta.block_table.clone()
    bad[0, 0] = P.kc.shape[0]                        # block id outside the pool
    with pytest.raises(ValueError):
        oracle.ragged_paged_attention(P.Q, P.kc, P.vc, P.meta.query_start_loc, P.meta.seq_lens, bad, 0.1)


# ---------------------------------------------------------------- block copies
# Copy-on-write and swap-out / swap-in of whole blocks ("vllm-lite README";
# "31. Engine v2", "Preemption: recompute or swap").

def _example_pool(nb, bb):
    return torch.tensor([[10 * b + i for i in range(bb)] for b in range(nb)], dtype=torch.uint8)


def test_block_copies_match_the_worked_example():
    g = _golden("block_copy_example.txt")
    nb, bb = g["blocks"][0][0], g["bytes"][0][0]
    pool = _example_pool(nb, bb)
    pairs = g["pair"]
    oracle.copy_blocks([pool], [p[0] for p in pairs], [p[1] for p in pairs])
    for row in g["after"]:
        assert pool[row[0]].tolist() == row[1:]
    pool = _example_pool(nb, bb)
    out = oracle.gather_blocks([pool], g["gather"][0])
    assert out[0].tolist() == g["gathered"]
    pool = _example_pool(nb, bb)
    oracle.scatter_blocks([pool], g["scatter"][0], torch.tensor([g["saved"]], dtype=torch.uint8))
    for row in g["scattered"]:
        assert pool[row[0]].tolist() == row[1:]


def test_block_copies_against_torch_indexing_on_several_pools():
    gen = torch.Generator().manual_seed(7)
    # a layer's K and V pools (bf16, [nbt, bs, Hkv, d]); scale pools (fp32 [nbt, bs, Hkv])
    # have other block bytes and go through their own call
    groups = [[_bf16((12, 16, 2, 8), gen) for _ in range(2)],
              [torch.rand((12, 16, 2), generator=gen) for _ in range(2)]]
    for pools in groups:
        ref = [p.clone() for p in pools]
        src, dst = [3, 7, 11], [0, 5, 9]
        oracle.copy_blocks(pools, src, dst)
        for p, r in zip(pools, ref):
            r.index_copy_(0, torch.tensor(dst), r.index_select(0, torch.tensor(src)))
            assert torch.equal(p.view(torch.uint8), r.view(torch.uint8))
        ids = [8, 2, 2, 10]
        out = oracle.gather_blocks(pools, ids)
        for q, p in enumerate(pools):
            want = p.index_select(0, torch.tensor(ids)).contiguous().view(torch.uint8).view(len(ids), -1)
            assert torch.equal(out[q], want)
        # swap-out then swap-in into other blocks copies those blocks and nothing else
        fresh = [p.clone() for p in pools]
        oracle.scatter_blocks(fresh, [1, 4, 6, 0], out)
        for p, f in zip(pools, fresh):
            for a, b in zip(ids, [1, 4, 6, 0]):
                assert torch.equal(f[b].view(torch.uint8), p[a].view(torch.uint8))
            for b in set(range(12)) - {1, 4, 6, 0}:
                assert torch.equal(f[b].view(torch.uint8), p[b].view(torch.uint8))
    with pytest.raises(ValueError):
        oracle.copy_blocks(groups[0], [12], [0])
    with pytest.raises(ValueError):
        oracle.gather_blocks(groups[0], [-1])



# ---------------------------------------------------------------- sliding window
# "31. Engine v2", "Attention over the pool": with a sliding window w > 0 a
# query at position p sees only the keys above p - w (and, causally, up to p).

@pytest.mark.parametrize("window", [1, 3, 16, 40, 1000])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2)])
def test_sliding_window_matches_dense_brute_force(window, hq, hkv):
    plan = [(6, 3), (41, 1), (9, 1), (0, 4), (17, 15), (31, 2), (60, 20)]
    P = Problem(plan, hq, hkv, 48, 16, seed=window + hq + hkv)
    got = P.oracle_out(window=window)
    want = P.brute_force(window=window)
    assert (got - want).abs().max().item() < 1e-10


def test_window_one_returns_own_value_and_wide_window_is_no_window():
    P = Problem([(20, 5), (50, 1), (0, 9)], 4, 2, 64, 16, seed=44)
    got = P.oracle_out(window=1)
    g = 2
    for r, (c, t) in enumerate(P.plan):
        b = P.meta.query_start_loc[r]
        for i in range(t):
            for h in range(4):
                # the only visible key is the query's own position c + i
                assert torch.equal(got[b + i, h], P.V[r][c + i, h // g].double())
    assert torch.equal(P.oracle_out(window=10 ** 6), P.oracle_out())
    assert torch.equal(P.oracle_out(window=60), P.oracle_out())           # 60 > every position


def test_sliding_window_chunk_invariance():
    gen = torch.Generator().manual_seed(45)
    L, hq, hkv, d, w = 150, 8, 2, 48, 37
    K, V, Q = _bf16((L, hkv, d), gen), _bf16((L, hkv, d), gen), _bf16((L, hq, d), gen)
    runs = []
    for chunk in (8, 33, 4096):
        nb = -(-L // 16) + 2
        table = list(range(nb - 1, -1, -1))[: -(-L // 16)]
        kc = torch.zeros((nb + 1, 16, hkv, d), dtype=torch.bfloat16)
        vc = torch.zeros_like(kc)
        outs, c = [], 0
        while c < L:
            t = min(chunk, L - c)
            spec = Spec("chunk", [Req(c, t, table)], hq, hkv, d, 16, nb, 1 / math.sqrt(d), 0)
            meta = build_meta(spec)
            oracle.paged_kv_write(kc, vc, K[c:c + t], V[c:c + t], meta.slot_mapping)
            outs.append(oracle.ragged_paged_attention(Q[c:c + t], kc, vc, meta.query_start_loc, meta.seq_lens,
                                                      meta.block_table, spec.scale, window=w))
            c += t
        runs.append(torch.cat(outs))
    for r in runs[1:]:
        assert torch.equal(runs[0], r)


# ---------------------------------------------------------------- quantized pool
# "31. Engine v2", "Attention over the pool": quantized pools carry per
# (slot, head) scales beside K and V, dequantized as code * scale.  Codes are
# FP8 E4M3 (reading of the pages' open kv_cache_dtype); the write uses
# scale = max|x| / 448 and rounds x / scale to nearest even.

def test_e4m3_worked_examples():
    rows = []
    for line in open(os.path.join(GOLDEN, "e4m3_examples.txt")):
        if line.startswith("value"):
            _, v, c, d = line.split()
            rows.append((float(v), int(c, 16), float(d)))
    for v, c, d in rows:
        assert oracle.e4m3_encode(v) == c, v
        assert oracle.e4m3_decode(c) == d, c


def test_e4m3_decode_matches_torch_float8_on_every_finite_code():
    codes = torch.tensor([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64)
    got = torch.tensor([oracle.e4m3_decode(int(c)) for c in codes], dtype=torch.float64)
    assert torch.equal(got, want)


def test_e4m3_encode_matches_torch_float8_below_saturation():
    gen = torch.Generator().manual_seed(61)
    mags = torch.cat([torch.rand(3000, generator=gen) * 447.0,
                      torch.exp2(torch.rand(3000, generator=gen) * 18 - 12)])   # 2^-12 .. 2^6
    xs = mags * torch.where(torch.rand(6000, generator=gen) < 0.5, -1.0, 1.0)
    xs = xs.to(torch.float32)
    want = xs.to(torch.float8_e4m3fn).view(torch.uint8)
    got = torch.tensor([oracle.e4m3_encode(float(x)) for x in xs], dtype=torch.uint8)
    assert torch.equal(got, want)


def test_quantizing_write_against_torch():
    gen = torch.Generator().manual_seed(62)
    nbt, bs, hkv, d, n = 9, 16, 4, 64, 30
    k, v = _bf16((n, hkv, d), gen) * 3, _bf16((n, hkv, d), gen)
    k[3, 1] = 0                                               # an all-zero row: scale 0, codes 0
    slots = torch.randperm(nbt * bs - 1, generator=gen)[:n]
    pools = [torch.zeros((nbt, bs, hkv, d), dtype=torch.uint8) for _ in range(2)] + \
            [torch.zeros((nbt, bs, hkv), dtype=torch.float32) for _ in range(2)]
    oracle.paged_kv_write_fp8(pools[0], pools[1], pools[2], pools[3], k, v, slots)
    for x, codes, scales in ((k, pools[0], pools[2]), (v, pools[1], pools[3])):
        xf = x.float()
        amax = xf.abs().amax(dim=-1)
        sc = amax / 448.0                                      # fp32, as the pages' scales
        q = torch.where(sc[..., None] > 0, xf / torch.where(sc > 0, sc, 1.0)[..., None], 0.0)
        want = q.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        flat_c = codes.view(-1, hkv, d)[slots]
        flat_s = scales.view(-1, hkv)[slots]
        assert torch.equal(flat_c, want)
        assert torch.equal(flat_s, sc)
    # dequantized values are within half a code step of the inputs: 2^-4 of
    # the value for normal codes, half the smallest subnormal (2^-10) times
    # the scale below them
    sc = pools[2].view(-1, hkv)[slots][..., None].double()
    deq = pools[0].view(-1, hkv, d)[slots].view(torch.float8_e4m3fn).double() * sc
    assert ((deq - k.double()).abs() <= k.double().abs() / 16 + sc * 2.0 ** -10).all()


def _fp8_problem(plan, hq, hkv, d, seed):
    """A quantized pool written by the oracle's quantizing write from random
    bf16 K/V (history, then this step's rows); returns everything the
    attention needs and the dequantized dense K/V per request."""
    gen = torch.Generator().manual_seed(seed)
    bs = 16
    nblk = [-(-(c + t) // bs) for c, t in plan]
    nb = sum(nblk) + 2
    perm = torch.randperm(nb, generator=gen).tolist()
    tables, cur = [], 0
    for n in nblk:
        tables.append(perm[cur:cur + n])
        cur += n
    reqs = [Req(c, t, tab) for (c, t), tab in zip(plan, tables)]
    spec = Spec("fp8", reqs, hq, hkv, d, bs, nb, 1.0 / math.sqrt(d), seed)
    meta = build_meta(spec)
    kc = torch.randint(0, 255, (nb + 1, bs, hkv, d), generator=gen, dtype=torch.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0                               # junk codes, never NaN
    vc = torch.randint(0, 255, (nb + 1, bs, hkv, d), generator=gen, dtype=torch.uint8)
    vc[(vc & 0x7F) == 0x7F] = 0
    ks = torch.rand((nb + 1, bs, hkv), generator=gen)
    vs = torch.rand((nb + 1, bs, hkv), generator=gen)
    K = [_bf16((c + t, hkv, d), gen) for c, t in plan]
    V = [_bf16((c + t, hkv, d), gen) for c, t in plan]
    hist = build_meta(Spec("hist", [Req(0, c, tab) for (c, t), tab in zip(plan, tables)], hq, hkv, d, bs, nb, 1.0, 0))
    if hist.num_tokens:
        oracle.paged_kv_write_fp8(kc, vc, ks, vs, torch.cat([k[:c] for k, (c, t) in zip(K, plan)]),
                                  torch.cat([v[:c] for v, (c, t) in zip(V, plan)]), hist.slot_mapping)
    oracle.paged_kv_write_fp8(kc, vc, ks, vs, torch.cat([k[c:] for k, (c, t) in zip(K, plan)]),
                              torch.cat([v[c:] for v, (c, t) in zip(V, plan)]), meta.slot_mapping)
    q = _bf16((meta.num_tokens, hq, d), gen)
    return spec, meta, q, kc, vc, ks, vs


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 2)])
def test_fp8_attention_matches_dense_dequantized_brute_force(hq, hkv):
    plan = [(6, 3), (41, 1), (0, 4), (17, 15), (60, 1)]
    spec, meta, q, kc, vc, ks, vs = _fp8_problem(plan, hq, hkv, 64, 63 + hq + hkv)
    got = oracle.ragged_paged_attention_fp8(q, kc, vc, ks, vs, meta.query_start_loc, meta.seq_lens,
                                            meta.block_table, spec.scale)
    g = hq // hkv
    for r, (c, t) in enumerate(plan):
        L, b = c + t, meta.query_start_loc[r]
        slots = [meta.block_table[r, j // 16].item() * 16 + j % 16 for j in range(L)]
        # dequantize through torch's float8 type, independently of the oracle
        k = kc.view(-1, hkv, 64)[slots].view(torch.float8_e4m3fn).double() * ks.view(-1, hkv)[slots][..., None].double()
        v = vc.view(-1, hkv, 64)[slots].view(torch.float8_e4m3fn).double() * vs.view(-1, hkv)[slots][..., None].double()
        qq = q[b:b + t].double().transpose(0, 1)[None]
        kk = k.repeat_interleave(g, dim=1).transpose(0, 1)[None]
        vv = v.repeat_interleave(g, dim=1).transpose(0, 1)[None]
        mask = torch.arange(L)[None, :] <= torch.arange(L - t, L)[:, None]
        want = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=spec.scale)[0].transpose(0, 1)
        assert (got[b:b + t] - want).abs().max().item() < 1e-10
    # sampled rows equal the full computation
    rows = oracle.attention_rows_fp8([0, 5, 12], [1, 0, hq - 1], q, kc, vc, ks, vs, meta.query_start_loc,
                                     meta.seq_lens, meta.block_table, spec.scale)
    assert torch.equal(rows, torch.stack([got[0, 1], got[5, 0], got[12, hq - 1]]))
