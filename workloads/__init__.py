"""Seeded synthetic ragged batches for the paged KV write and ragged paged attention.

This module only builds inputs.  It draws request lengths, block tables and
N(0,1) bf16 values, and lays a step out as one flattened ragged batch the way
the engine's batch builder does ("31. Engine v2: one core for every request",
sections "Flattened ragged batches" and the ``build_batch`` listing): rows of
all scheduled tokens concatenated, ``query_start_loc``/``seq_lens`` per
request, a zero-padded int32 block table and an int64 slot per new token.
It holds none of the attention arithmetic and none of the pool write: the CPU
oracle and the CUDA library both consume what it produces, and neither is
imported here.

Workload shapes follow the pages' workloads (the layout example of "Flattened
ragged batches"; the 48-request lognormal benchmark with a shared 256-token
system prompt from the vllm-lite README; decode/prefill mixes from
"vLLM: LLM Inference as a memory and scheduling problem").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = [
    "Req", "Spec", "Meta", "Batch", "build_meta", "make_batch", "config_spec",
    "CONFIG_NAMES", "fill_normal_bf16", "subset_spec", "random_spec",
]


@dataclass
class Req:
    """One scheduled request: ``computed`` tokens already in the pool, ``new``
    tokens scheduled this step, ``table`` its physical blocks in logical order.
    A padding row (the batch builder's ``pad_to``) is ``Req(0, 1, [], pad=True)``.
    """
    computed: int
    new: int
    table: list
    pad: bool = False

    @property
    def seq_len(self) -> int:
        return 0 if self.pad else self.computed + self.new


@dataclass
class Spec:
    name: str
    reqs: list
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int          # blocks the allocator may hand out; the pool holds one more (scratch)
    scale: float
    seed: int
    table_width: int = 0     # 0: as wide as the longest table (at least 1)

    @property
    def num_blocks_total(self) -> int:
        return self.num_blocks + 1

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


@dataclass
class Meta:
    """Flat batch metadata, host side (torch CPU tensors and Python lists)."""
    query_start_loc: list
    seq_lens: list
    block_table: torch.Tensor      # int32 [R, W], zero padded
    slot_mapping: torch.Tensor     # int64 [N], -1 for padding rows
    positions: list                # position of every row (for reference and tests)
    max_query_len: int
    max_seq_len: int

    @property
    def num_reqs(self) -> int:
        return len(self.seq_lens)

    @property
    def num_tokens(self) -> int:
        return self.query_start_loc[-1]


def build_meta(spec: Spec) -> Meta:
    """Lay out the scheduled requests as one flattened batch.

    Request r's new tokens sit at positions c .. c+t-1 (c = tokens already
    computed) and position p goes to slot ``table[p // bs] * bs + p % bs``
    ("31. Engine v2", "Flattened ragged batches", the batch builder listing).
    Padding rows get slot -1 and length 0, as the builder's ``pad_to`` does.
    """
    bs = spec.block_size
    starts, lengths, slots, positions, tables = [0], [], [], [], []
    for r in spec.reqs:
        if r.pad:
            starts.append(starts[-1] + r.new)
            lengths.append(0)
            slots.extend([-1] * r.new)
            positions.extend([0] * r.new)
            tables.append([])
            continue
        c, t = r.computed, r.new
        need = -(-(c + t) // bs)
        if len(r.table) < need:
            raise ValueError(f"{spec.name}: table of {len(r.table)} blocks for {c + t} tokens")
        for p in range(c, c + t):
            slots.append(r.table[p // bs] * bs + p % bs)
            positions.append(p)
        starts.append(starts[-1] + t)
        lengths.append(c + t)
        tables.append(list(r.table))
    width = max(1, max((len(t) for t in tables), default=1), spec.table_width)
    bt = torch.zeros((len(tables), width), dtype=torch.int32)
    for i, t in enumerate(tables):
        if t:
            bt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
    qlens = [b - a for a, b in zip(starts, starts[1:])]
    return Meta(
        query_start_loc=starts, seq_lens=lengths, block_table=bt,
        slot_mapping=torch.tensor(slots, dtype=torch.int64),
        positions=positions,
        max_query_len=max(qlens) if qlens else 0,
        max_seq_len=max(lengths) if lengths else 0,
    )


def fill_normal_bf16(t: torch.Tensor, gen: torch.Generator, chunk: int = 1 << 26) -> torch.Tensor:
    """Fill a bf16 tensor with N(0,1) draws made in fp32 and rounded to bf16
    (round to nearest even), ``chunk`` elements at a time."""
    flat = t.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        flat[s:e] = torch.randn(e - s, generator=gen, device=t.device, dtype=torch.float32).to(torch.bfloat16)
    return t


@dataclass
class Batch:
    spec: Spec
    meta: Meta
    q: torch.Tensor          # bf16 [N, Hq, d]
    k: torch.Tensor          # bf16 [N, Hkv, d]   new keys of this step
    v: torch.Tensor          # bf16 [N, Hkv, d]
    k_cache: torch.Tensor    # bf16 [nb+1, bs, Hkv, d]
    v_cache: torch.Tensor
    extras: dict = field(default_factory=dict)


def make_batch(spec: Spec, device="cpu", pool_fill: str = "normal", value_seed: int | None = None) -> Batch:
    """Draw the values of one step on ``device``.

    The pool is filled with N(0,1) bf16 everywhere (``pool_fill="normal"``), so
    the tails of partial blocks and unused blocks hold junk that attention must
    never read; ``pool_fill="zeros"`` gives an all-zero pool and ``"sentinel"``
    a pool of one recognisable bit pattern (0x7F7F), for write tests.
    Q and the step's new K/V are N(0,1) bf16.
    """
    meta = build_meta(spec)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(spec.seed * 7919 + 17 if value_seed is None else value_seed)
    n = meta.num_tokens
    shape_pool = (spec.num_blocks_total, spec.block_size, spec.num_kv_heads, spec.head_dim)
    k_cache = torch.empty(shape_pool, dtype=torch.bfloat16, device=dev)
    v_cache = torch.empty(shape_pool, dtype=torch.bfloat16, device=dev)
    if pool_fill == "normal":
        fill_normal_bf16(k_cache, gen)
        fill_normal_bf16(v_cache, gen)
    elif pool_fill == "zeros":
        k_cache.zero_()
        v_cache.zero_()
    elif pool_fill == "sentinel":
        k_cache.view(torch.int16).fill_(0x7F7F)
        v_cache.view(torch.int16).fill_(0x7F7F)
    else:
        raise ValueError(pool_fill)
    q = fill_normal_bf16(torch.empty((n, spec.num_q_heads, spec.head_dim), dtype=torch.bfloat16, device=dev), gen)
    k = fill_normal_bf16(torch.empty((n, spec.num_kv_heads, spec.head_dim), dtype=torch.bfloat16, device=dev), gen)
    v = fill_normal_bf16(torch.empty((n, spec.num_kv_heads, spec.head_dim), dtype=torch.bfloat16, device=dev), gen)
    return Batch(spec, meta, q, k, v, k_cache, v_cache)


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

CONFIG_NAMES = {
    1: "layout-example-N9",
    2: "engine-step-48req-shared-prefix",
    3: "decode-256req-ctx512-8192",
    4: "mixed-chunk2048-at16384+2x1024+64dec",
    5: "long-decode-32req-ctx32768-g8",
}


def _randint(gen, lo, hi):
    """Uniform integer in [lo, hi] (both ends included)."""
    return int(torch.randint(lo, hi + 1, (1,), generator=gen).item())


def _blocks(n_tokens, bs):
    return -(-n_tokens // bs)


def _take(perm, cursor, n):
    return [int(x) for x in perm[cursor:cursor + n]], cursor + n


def config_spec(cfg: int, seed: int | None = None) -> Spec:
    """The metadata of workload ``cfg`` (1..5) for ``seed`` (default 1000+cfg)."""
    seed = 1000 + cfg if seed is None else seed
    gen = torch.Generator().manual_seed(seed)
    bs = 16
    if cfg == 1:
        # The layout example: a (chunk of 3 at 6..8), b (decode at 41),
        # c (decode at 9), d (new prompt of 4).
        nb = 64
        perm = torch.randperm(nb, generator=gen)
        cur = 0
        reqs = []
        for c, t in ((6, 3), (41, 1), (9, 1), (0, 4)):
            tab, cur = _take(perm, cur, _blocks(c + t, bs))
            reqs.append(Req(c, t, tab))
        return Spec(CONFIG_NAMES[1], reqs, 8, 4, 48, bs, nb, 1.0 / math.sqrt(48), seed)
    if cfg == 2:
        # 48 requests behind one 256-token system prompt (16 shared blocks).
        # Prompt tail lengths: lognormal with mu, sigma chosen so that the
        # 17..251 range spans about +-2 sigma; rounded and clipped.
        mu = 0.5 * (math.log(17) + math.log(251))
        sigma = math.log(251 / 17) / 4
        tails = torch.exp(torch.randn(48, generator=gen, dtype=torch.float64) * sigma + mu)
        tails = [min(251, max(17, int(round(float(x))))) for x in tails]
        plan = []
        for i, lq in enumerate(tails):
            prompt = 256 + lq
            if i < 16:
                kk = _randint(gen, 0, -(-lq // 64) - 1)
                c = 256 + 64 * kk
                t = min(64, prompt - c)
                plan.append((c, t))
            else:
                seq = prompt + _randint(gen, 20, 192)
                plan.append((seq - 1, 1))
        used = 16 + sum(_blocks(c + t, bs) - 16 for c, t in plan)
        nb = math.ceil(1.1 * used)
        perm = torch.randperm(nb, generator=gen)
        shared, cur = _take(perm, 0, 16)
        reqs = []
        for c, t in plan:
            priv, cur = _take(perm, cur, _blocks(c + t, bs) - 16)
            reqs.append(Req(c, t, shared + priv))
        order = torch.randperm(48, generator=gen).tolist()
        reqs = [reqs[i] for i in order]
        return Spec(CONFIG_NAMES[2], reqs, 8, 4, 48, bs, nb, 1.0 / math.sqrt(48), seed)
    if cfg == 3:
        lens = [_randint(gen, 512, 8192) for _ in range(256)]
        used = sum(_blocks(L, bs) for L in lens)
        nb = math.ceil(1.1 * used)
        perm = torch.randperm(nb, generator=gen)
        cur, reqs = 0, []
        for L in lens:
            tab, cur = _take(perm, cur, _blocks(L, bs))
            reqs.append(Req(L - 1, 1, tab))
        return Spec(CONFIG_NAMES[3], reqs, 32, 8, 128, bs, nb, 1.0 / math.sqrt(128), seed)
    if cfg == 4:
        plan = [(16384, 2048)]
        plan += [(L - 1, 1) for L in (_randint(gen, 1024, 4096) for _ in range(64))]
        plan += [(0, 1024), (0, 1024)]
        used = sum(_blocks(c + t, bs) for c, t in plan)
        nb = math.ceil(1.1 * used)
        perm = torch.randperm(nb, generator=gen)
        cur, reqs = 0, []
        for c, t in plan:
            tab, cur = _take(perm, cur, _blocks(c + t, bs))
            reqs.append(Req(c, t, tab))
        return Spec(CONFIG_NAMES[4], reqs, 32, 8, 128, bs, nb, 1.0 / math.sqrt(128), seed)
    if cfg == 5:
        nb = 70000
        perm = torch.randperm(nb, generator=gen)[:65536]
        cur, reqs = 0, []
        for _ in range(32):
            tab, cur = _take(perm, cur, 2048)
            reqs.append(Req(32767, 1, tab))
        return Spec(CONFIG_NAMES[5], reqs, 64, 8, 128, bs, nb, 1.0 / math.sqrt(128), seed)
    raise ValueError(f"unknown workload {cfg}")


def subset_spec(spec: Spec, n: int) -> Spec:
    """The first ``n`` requests of ``spec`` on a pool of their own: their blocks
    renumbered in order of first use, the pool sized to the blocks used plus
    10%.  A smaller instance of the same workload shape (for profiling)."""
    reqs = spec.reqs[:n]
    remap = {}
    for r in reqs:
        for blk in r.table:
            remap.setdefault(blk, len(remap))
    gen = torch.Generator().manual_seed(spec.seed)
    nb = math.ceil(1.1 * max(1, len(remap)))
    perm = torch.randperm(nb, generator=gen).tolist()
    new = [Req(r.computed, r.new, [perm[remap[b]] for b in r.table], r.pad) for r in reqs]
    return Spec(f"{spec.name}[:{n}]", new, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                spec.block_size, nb, spec.scale, spec.seed)


def random_spec(seed: int, num_reqs: int, max_ctx: int, max_new: int, num_q_heads: int,
                num_kv_heads: int, head_dim: int, block_size: int = 16, decode_frac: float = 0.5,
                spare_blocks: int = 3, pad_rows: int = 0, name: str = "random") -> Spec:
    """A small random mix of decodes and prefill chunks over a permuted pool
    (for parity tests)."""
    gen = torch.Generator().manual_seed(seed)
    plan = []
    for _ in range(num_reqs):
        if torch.rand(1, generator=gen).item() < decode_frac:
            L = _randint(gen, 1, max_ctx)
            plan.append((L - 1, 1))
        else:
            t = _randint(gen, 1, max_new)
            c = _randint(gen, 0, max(0, max_ctx - t))
            plan.append((c, t))
    used = sum(_blocks(c + t, block_size) for c, t in plan)
    nb = used + spare_blocks
    perm = torch.randperm(nb, generator=gen)
    cur, reqs = 0, []
    for c, t in plan:
        tab, cur = _take(perm, cur, _blocks(c + t, block_size))
        reqs.append(Req(c, t, tab))
    for _ in range(pad_rows):
        reqs.append(Req(0, 1, [], pad=True))
    return Spec(name, reqs, num_q_heads, num_kv_heads, head_dim, block_size, nb,
                1.0 / math.sqrt(head_dim), seed)
