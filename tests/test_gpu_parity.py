"""CUDA library vs the CPU oracle, element by element, on the same seeded inputs.

paged_kv_write and all indexing: bit-exact (whole pool except the scratch
slot).  Attention (bf16 in, fp32 accumulate) against the fp64 oracle:
max |err| <= 2e-2 and mean |err| <= 2e-3.
"""
import math

import pytest
import torch

import oracle
import paged_kv_cache_84_gb300 as pkv
from workloads import Batch, Req, Spec, build_meta, config_spec, make_batch, random_spec
from _helpers import (DeviceStep, assert_close, cpu_copy, device_batch, oracle_full, oracle_rows,
                      oracle_write)

pytestmark = pytest.mark.gpu

# the tcgen05 prefill kernel, alone or with a batch's decodes in its launch
TC_KERNELS = {"attn_tc_prefill", "attn_tc_mixed"}


def _pool_bits(t):
    nbt, bs, hkv, d = t.shape
    return t.contiguous().view(torch.int16).view(nbt * bs, hkv * d)


def _check_write(dev: DeviceStep, ref_cpu):
    """Whole pool except the scratch slot, bit for bit."""
    for got, want in ((dev.k_cache, ref_cpu.k_cache), (dev.v_cache, ref_cpu.v_cache)):
        g = _pool_bits(got.cpu())[:-1]
        w = _pool_bits(want)[:-1]
        assert torch.equal(g, w)
    assert pkv.read_device_error(dev.write_err) == 0


# ------------------------------------------------------------------ small configs: full compare

@pytest.mark.parametrize("cfg", [1, 2])
def test_config_full_parity(cfg):
    spec = config_spec(cfg)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.step()
    torch.cuda.synchronize()
    ref = cpu_copy(b)
    oracle_write(ref)
    _check_write(dev, ref)
    want = oracle_full(ref)
    assert_close(dev.out, want, f"config {cfg}")
    assert pkv.read_device_error(dev.ws) == 0


RANDOM_CASES = [
    # seed, reqs, max_ctx, max_new, hq, hkv, d, pad rows
    (0, 6, 300, 40, 8, 8, 48, 0),
    (1, 9, 700, 70, 8, 4, 64, 2),
    (2, 5, 1200, 130, 32, 8, 128, 1),
    (3, 12, 2500, 33, 16, 2, 128, 0),
    (4, 7, 90, 90, 8, 1, 64, 3),
    (5, 4, 4100, 300, 64, 8, 128, 0),
    (6, 16, 600, 1, 32, 8, 128, 0),
    (7, 3, 33, 33, 4, 4, 48, 1),
    (8, 4, 700, 260, 8, 8, 128, 0),       # g = 1 tensor-core tiles
    (9, 3, 500, 200, 16, 1, 128, 1),      # g = 16
    (10, 5, 900, 300, 16, 8, 128, 0),     # g = 2
]


@pytest.mark.parametrize("case", RANDOM_CASES, ids=[f"seed{c[0]}" for c in RANDOM_CASES])
def test_random_mixes_full_parity(case):
    seed, reqs, ctx, new, hq, hkv, d, pad = case
    spec = random_spec(seed, reqs, ctx, new, hq, hkv, d, pad_rows=pad)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.step()
    torch.cuda.synchronize()
    ref = cpu_copy(b)
    oracle_write(ref)
    _check_write(dev, ref)
    assert_close(dev.out, oracle_full(ref), f"random {seed}")


@pytest.mark.parametrize("disable_tc", [False, True])
@pytest.mark.parametrize("heads", [(32, 8, 128), (16, 4, 64), (8, 4, 48), (16, 2, 48)], ids=["d128g4", "d64g4", "d48g2", "d48g8"])
def test_long_chunks_tensor_core_path(disable_tc, heads, attn_options):
    """Prefill chunks of 128+ rows go to the tcgen05 kernel (head dims below 64
    padded to 64 columns); the same batch with it disabled runs on the
    warp-level MMA kernel.  Both match the oracle."""
    if disable_tc:
        attn_options(disable_tcgen05=1)
    hq, hkv, d = heads
    reqs = [Req(1000, 300, list(range(0, 82))), Req(0, 257, list(range(82, 99))), Req(77, 1, list(range(99, 104))),
            Req(5000, 64, list(range(104, 421)))]
    spec = Spec("chunks", reqs, hq, hkv, d, 16, 430, 1 / math.sqrt(d), 17)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    pkv.profile_start(16)
    dev.step()
    names = {n for n, _ in pkv.profile_stop()}
    assert bool(names & TC_KERNELS) != disable_tc
    ref = cpu_copy(b)
    oracle_write(ref)
    assert_close(dev.out, oracle_full(ref), "chunks")
    assert pkv.read_device_error(dev.ws) == 0


def _mixed_spec():
    reqs = [Req(3000, 512, list(range(0, 220))), Req(0, 300, list(range(220, 239)))]
    reqs += [Req(700 + 97 * i, 1, list(range(239 + 111 * i, 239 + 111 * (i + 1)))) for i in range(12)]
    return Spec("mixed", reqs, 32, 8, 128, 16, 1600, 1 / math.sqrt(128), 23)


@pytest.mark.parametrize("shape", ["long-chunks", "engine-step"])
@pytest.mark.parametrize("overlap", [True, False])
def test_mixed_step_side_stream_and_cuda_graph(overlap, shape, attn_options):
    """Decodes next to prefill chunks: the decode kernels run on a forked side
    stream (or, with the no_overlap option, on the caller's stream); in the small
    engine step the short prefill tiles are split over keys and all split
    partials are merged by one combine launch.  The step is also captured in
    a CUDA graph and replayed; every result matches the oracle."""
    if not overlap:
        attn_options(no_overlap=1)
    spec = _mixed_spec() if shape == "long-chunks" else config_spec(2)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.step()
    ref = cpu_copy(b)
    oracle_write(ref)
    want = oracle_full(ref)
    assert_close(dev.out, want, "eager")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        dev.step()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            dev.step()
    torch.cuda.synchronize()
    dev.out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert_close(dev.out, want, "graph replay")
    assert pkv.read_device_error(dev.ws) == 0


@pytest.mark.parametrize("pdl", [True, False])
def test_programmatic_launch_and_padding_only_decodes(pdl, attn_options):
    """Kernels launched with programmatic stream serialization wait in-kernel
    for the pool write.  A batch whose decode-class requests are all padding,
    next to a prefill chunk, must still see the step's K/V (the no_pdl option gives
    plain stream order)."""
    if not pdl:
        attn_options(no_pdl=1)
    reqs = [Req(0, 1, [], pad=True), Req(200, 90, list(range(0, 19))), Req(0, 1, [], pad=True)]
    spec = Spec("pad-mix", reqs, 8, 4, 64, 16, 24, 0.125, 31)
    b = make_batch(spec, device="cpu")
    for _ in range(3):
        dev = DeviceStep(b)
        dev.step()
        ref = cpu_copy(b)
        oracle_write(ref)
        assert_close(dev.out, oracle_full(ref), "padding-only decodes")
        assert dev.out[0].abs().sum().item() == 0 and dev.out[-1].abs().sum().item() == 0


@pytest.mark.parametrize("prefill_split", [False, True])
def test_engine_step_prefill_split_toggle(prefill_split, attn_options):
    """The small engine step on the warp-level MMA kernels only (tensor cores
    off), with and without key splits of its short prefill tiles
    (the prefill_key_splits option)."""
    attn_options(disable_tcgen05=1)
    if prefill_split:
        attn_options(prefill_key_splits=1)
    b = make_batch(config_spec(2), device="cpu")
    dev = DeviceStep(b)
    dev.step()
    ref = cpu_copy(b)
    oracle_write(ref)
    assert_close(dev.out, oracle_full(ref), "engine step")


@pytest.mark.parametrize("split", [256, 512, 4096])
def test_forced_split_sizes(split, attn_options):
    attn_options(split_tokens=split)
    spec = random_spec(11, 10, 3000, 3, 32, 8, 128, decode_frac=0.8)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.step()
    ref = cpu_copy(b)
    oracle_write(ref)
    assert_close(dev.out, oracle_full(ref), f"split {split}")


def test_minimum_workspace_disables_splitting():
    spec = random_spec(12, 6, 5000, 1, 64, 8, 128, decode_frac=1.0)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b, workspace_bytes=pkv.WORKSPACE_MIN_BYTES)
    dev.step()
    ref = cpu_copy(b)
    oracle_write(ref)
    assert_close(dev.out, oracle_full(ref), "min workspace")


# ------------------------------------------------------------------ full-size configs: sampled rows

def _sample_rows(spec, meta, gen, per_req_heads=1, extra=()):
    toks, heads = [], []
    for r, req in enumerate(spec.reqs):
        b = meta.query_start_loc[r]
        t = req.new
        picks = sorted({0, t - 1, t // 2, min(t - 1, 127), min(t - 1, 128)})
        for i in picks:
            for h in torch.randint(0, spec.num_q_heads, (per_req_heads,), generator=gen).tolist():
                toks.append(b + i)
                heads.append(h)
    for tok, h in extra:
        toks.append(tok)
        heads.append(h)
    return toks, heads


@pytest.mark.parametrize("cfg", [3, 4, 5])
def test_config_full_size_sampled_parity(cfg):
    spec = config_spec(cfg)
    b = device_batch(spec)
    ref = cpu_copy(b)                     # inputs, copied before any library kernel runs
    dev = DeviceStep(b)
    dev.step()
    torch.cuda.synchronize()
    assert torch.isfinite(dev.out.float()).all()
    oracle_write(ref)
    _check_write(dev, ref)
    gen = torch.Generator().manual_seed(cfg)
    extra = []
    if cfg == 4:                          # tile edges of the long chunk, every head of one row
        extra = [(i, h) for i in (31, 32, 63, 64, 1000, 2047) for h in range(0, 32, 7)]
        extra += [(2048 + 64 + 1023, h) for h in range(32)]
    toks, heads = _sample_rows(spec, b.meta, gen, per_req_heads=2 if cfg != 3 else 1, extra=extra)
    want = oracle_rows(ref, toks, heads)
    got = dev.out[torch.tensor(toks), torch.tensor(heads)]
    assert_close(got, want, f"config {cfg} sampled")
    assert pkv.read_device_error(dev.ws) == 0


# ------------------------------------------------------------------ invariances through the GPU path

def test_chunked_prefill_steps_match_oracle():
    """One prompt in chunks of 8/33/64/4096 over successive write+attend steps."""
    L, hq, hkv, d, bs = 300, 32, 8, 128, 16
    gen = torch.Generator().manual_seed(71)
    K = torch.randn((L, hkv, d), generator=gen).to(torch.bfloat16)
    V = torch.randn((L, hkv, d), generator=gen).to(torch.bfloat16)
    Q = torch.randn((L, hq, d), generator=gen).to(torch.bfloat16)
    nb = -(-L // bs) + 3
    table = torch.randperm(nb, generator=gen)[: -(-L // bs)].tolist()
    outs = {}
    for chunk in (8, 33, 64, 4096):
        kc = torch.zeros((nb + 1, bs, hkv, d), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        kc_ref = kc.cpu()
        vc_ref = vc.cpu()
        got = []
        c = 0
        while c < L:
            t = min(chunk, L - c)
            spec = Spec("chunk", [Req(c, t, table)], hq, hkv, d, bs, nb, 1 / math.sqrt(d), 0)
            meta = build_meta(spec)
            step = DeviceStep(Batch(spec, meta, Q[c:c + t], K[c:c + t], V[c:c + t], kc_ref, vc_ref),
                              pools=(kc, vc))
            step.step()
            oracle.paged_kv_write(kc_ref, vc_ref, K[c:c + t], V[c:c + t], meta.slot_mapping)
            want = oracle.ragged_paged_attention(Q[c:c + t], kc_ref, vc_ref, meta.query_start_loc,
                                                 meta.seq_lens, meta.block_table, spec.scale, 8)
            assert_close(step.out, want, f"chunk {chunk} at {c}")
            got.append(step.out.float().cpu())
            c += t
        outs[chunk] = torch.cat(got)
    base = outs[8]
    for chunk, o in outs.items():
        assert (o - base).abs().max().item() <= 2 * 2e-2


def test_block_permutation_and_shared_prefix():
    """Shared prefix blocks vs private copies, and a physical permutation of the pool."""
    spec = config_spec(2)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.step()
    base = dev.out.float().cpu()
    # permute physical blocks (scratch block stays last)
    nbt = b.k_cache.shape[0]
    perm = torch.randperm(nbt - 1, generator=torch.Generator().manual_seed(5))
    kc2, vc2 = b.k_cache.clone(), b.v_cache.clone()
    kc2[perm] = b.k_cache[:nbt - 1]
    vc2[perm] = b.v_cache[:nbt - 1]
    reqs2 = [Req(r.computed, r.new, [int(perm[x]) for x in r.table]) for r in spec.reqs]
    spec2 = Spec(spec.name, reqs2, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.block_size,
                 spec.num_blocks, spec.scale, spec.seed)
    b2 = Batch(spec2, build_meta(spec2), b.q, b.k, b.v, kc2, vc2)
    dev2 = DeviceStep(b2)
    dev2.step()
    ref2 = cpu_copy(b2)
    oracle_write(ref2)
    assert_close(dev2.out, oracle_full(ref2), "permuted")
    assert (dev2.out.float().cpu() - base).abs().max().item() <= 2 * 2e-2


# ------------------------------------------------------------------ edge cases

def test_empty_batch_is_a_noop():
    spec = Spec("empty", [], 8, 4, 64, 16, 4, 0.125, 0)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    before = pkv.launch_count()
    dev.step()
    torch.cuda.synchronize()
    assert pkv.launch_count() == before


def test_padding_requests_give_zero_rows():
    reqs = [Req(10, 2, [0]), Req(0, 1, [], pad=True), Req(20, 1, [1, 2]), Req(0, 1, [], pad=True)]
    spec = Spec("pad", reqs, 8, 2, 64, 16, 4, 0.125, 3)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.step()
    ref = cpu_copy(b)
    oracle_write(ref)
    want = oracle_full(ref)
    assert_close(dev.out, want, "padding")
    assert dev.out[2].abs().sum().item() == 0 and dev.out[4].abs().sum().item() == 0
    # padding rows wrote to the scratch slot only
    _check_write(dev, ref)


def test_invalid_metadata_is_rejected_on_host():
    spec = Spec("bad", [Req(5, 3, [0]), Req(20, 1, [1, 2]), Req(0, 4, [3])], 8, 4, 64, 16, 5, 0.125, 0)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    m = b.meta

    def call(qsl=m.query_start_loc, sl=m.seq_lens, bt=dev.bt, maxq=m.max_query_len, maxl=m.max_seq_len):
        pkv.ragged_paged_attention(dev.out, dev.q, dev.k_cache, dev.v_cache, dev.qsl, dev.sl, bt,
                                   qsl, sl, maxq, maxl, 0.1, dev.ws)

    before = pkv.launch_count()
    cases = [
        dict(sl=[2, 21, 4]),                                  # t = 3 > seq_len = 2
        dict(bt=dev.bt[:, :1].contiguous()),                  # table narrower than ceil(L / 16)
        dict(qsl=[0, 4, 3, 8]),                               # query_start_loc not non-decreasing
        dict(qsl=[0, 3, 4, 7]),                               # does not end at num_tokens
        dict(maxl=10),                                        # max_seq_len below the data
    ]
    for kw in cases:
        with pytest.raises(pkv.PkvError) as e:
            call(**kw)
        assert e.value.status == 1, kw
    assert pkv.launch_count() == before
    call()                                                    # the valid call still works
    assert pkv.launch_count() > before


def test_unsupported_head_dim():
    spec = Spec("d96", [Req(3, 1, [0])], 4, 2, 96, 16, 2, 0.1, 0)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    with pytest.raises(pkv.PkvError) as e:
        dev.attend()
    assert e.value.status == 2


def test_out_of_pool_block_id_sets_flag_without_fault():
    spec = random_spec(21, 4, 200, 4, 8, 4, 64)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.write()
    bt = dev.bt.clone()
    bt[0, 0] = spec.num_blocks_total + 5          # the device table points outside the pool
    dev.bt = bt
    pkv.clear_device_error(dev.ws)
    dev.attend()
    assert pkv.read_device_error(dev.ws) & pkv.DEVERR_BLOCK
    torch.cuda.synchronize()                      # the context is still usable
    dev.bt = b.meta.block_table.cuda()
    pkv.clear_device_error(dev.ws)
    dev.attend()
    assert pkv.read_device_error(dev.ws) == 0


def test_out_of_pool_slot_sets_flag_and_skips():
    spec = random_spec(22, 3, 100, 4, 8, 4, 64)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    before = dev.k_cache.clone()
    dev.slots = dev.slots.clone()
    dev.slots[0] = spec.num_blocks_total * spec.block_size + 3
    dev.write()
    assert pkv.read_device_error(dev.write_err) & pkv.DEVERR_SLOT
    ref = cpu_copy(b)
    sm = b.meta.slot_mapping.clone()
    keep = torch.ones(sm.numel(), dtype=torch.bool)
    keep[0] = False
    oracle.paged_kv_write(ref.k_cache, ref.v_cache, b.k[keep], b.v[keep], sm[keep])
    assert torch.equal(_pool_bits(dev.k_cache.cpu())[:-1], _pool_bits(ref.k_cache)[:-1])
    del before


@pytest.mark.parametrize("path", ["default", "no-tcgen05"])
def test_device_metadata_differing_from_host_copies_is_flagged(path, attn_options):
    """The kernels take each request's rows and context length from the host
    copies they were planned with; device arrays that disagree set
    DEVERR_META and change nothing else (prefill on tcgen05, and on the
    warp-MMA kernel)."""
    if path == "no-tcgen05":
        attn_options(disable_tcgen05=1)
    # decodes, short chunks and one tensor-core-sized chunk (t*g >= 128, d 128)
    reqs = [Req(300, 1, list(range(0, 19))), Req(40, 24, list(range(19, 23))),
            Req(100, 64, list(range(23, 34)))]
    spec = Spec("meta", reqs, 8, 2, 128, 16, 40, 1.0 / math.sqrt(128), 5)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.write()
    pkv.clear_device_error(dev.ws)
    dev.attend()
    assert pkv.read_device_error(dev.ws) == 0
    ref = cpu_copy(b)
    oracle_write(ref)
    want = oracle_full(ref)
    for r in range(len(reqs)):                    # each request is checked by the kernel serving it
        dev.sl = torch.tensor(b.meta.seq_lens, dtype=torch.int32, device="cuda")
        dev.sl[r] -= 1                            # the device copy disagrees with the host copy
        dev.out.fill_(float("nan"))
        pkv.clear_device_error(dev.ws)
        dev.attend()
        assert pkv.read_device_error(dev.ws) & pkv.DEVERR_META, f"request {r}"
        assert_close(dev.out.cpu(), want, f"planned metadata, request {r} altered")


COUNTER_BYTES = 65536          # split-counter region after the 256-byte error word


@pytest.mark.parametrize("split", [128, 1024])
@pytest.mark.parametrize("d", [48, 128])
def test_in_kernel_split_combine_repeats_and_leaves_counters_zero(split, d, attn_options):
    """Split decodes combine inside the kernel (the CTA finishing the last
    split of a request and KV head); repeated calls, eager and replayed from a
    CUDA graph, stay exact, and every call leaves the counters at zero."""
    attn_options(split_tokens=split)
    spec = random_spec(31, 12, 4000, 3, 16 if d == 128 else 8, 4 if d == 128 else 2, d, decode_frac=0.85)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.write()
    ref = cpu_copy(b)
    oracle_write(ref)
    want = oracle_full(ref)
    for i in range(3):
        dev.out.fill_(float("nan"))
        dev.attend()
        assert_close(dev.out, want, f"eager call {i}")
    assert int(dev.ws[256:256 + COUNTER_BYTES].count_nonzero()) == 0
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dev.attend()
    torch.cuda.synchronize()
    for i in range(3):
        dev.out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_close(dev.out, want, f"graph replay {i}")
    assert int(dev.ws[256:256 + COUNTER_BYTES].count_nonzero()) == 0
    assert pkv.read_device_error(dev.ws) == 0


def test_workspace_without_counter_room_uses_the_combine_kernel(attn_options):
    """A workspace too small for the counter region still splits (partials
    after the error word) and combines with the separate kernel (clusters
    off: they would combine without partials)."""
    attn_options(split_tokens=256)
    attn_options(cluster=-1)
    # one decode at L = 1500: 8 partial rows of 264 bytes per split, so the
    # 12 KiB workspace holds 5 splits (of 512 keys: 3 splits)
    spec = Spec("ws", [Req(1499, 1, list(range(94)))], 8, 2, 64, 16, 100, 0.125, 32)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b, workspace_bytes=12 * 1024)
    before = pkv.launch_count()
    dev.step()
    ref = cpu_copy(b)
    oracle_write(ref)
    assert_close(dev.out, oracle_full(ref), "small workspace")
    assert pkv.launch_count() - before >= 3              # write, attention, combine


def test_nonzero_split_counter_is_flagged(attn_options):
    """A workspace whose counter region was not zero-filled is reported
    (split counters: clusters off)."""
    attn_options(split_tokens=256)
    attn_options(cluster=-1)
    spec = random_spec(33, 4, 2000, 1, 8, 2, 64, decode_frac=1.0)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    dev.write()
    dev.ws[256:256 + COUNTER_BYTES] = 0x7f
    dev.attend()
    assert pkv.read_device_error(dev.ws) & pkv.DEVERR_COUNTER
    torch.cuda.synchronize()                              # no fault, the context is usable



@pytest.mark.parametrize("d", [48, 64, 128])
def test_short_chunks_on_tensor_cores(d, attn_options):
    """With the row threshold lowered, chunks that fill only part of a 128-row
    tile (ragged token counts, unaligned contexts) run on the tcgen05 kernel."""
    attn_options(tc_min_rows=16)
    reqs = [Req(256 + 64 * k, t, list(range(40 * k, 40 * k + 40))) for k, t in enumerate((64, 17, 33, 5, 1, 40))]
    reqs[4] = Req(300, 1, list(range(160, 200)))                  # a decode stays on the decode kernel
    spec = Spec("short", reqs, 8, 2 if d == 128 else 4, d, 16, 250, 1 / math.sqrt(d), 41)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b)
    pkv.profile_start(16)
    dev.step()
    names = {n for n, _ in pkv.profile_stop()}
    assert names & TC_KERNELS
    ref = cpu_copy(b)
    oracle_write(ref)
    assert_close(dev.out, oracle_full(ref), f"short chunks d{d}")
    assert pkv.read_device_error(dev.ws) == 0


# ------------------------------------------------------------------ sliding window

WINDOW_CASES = [
    # (random case index, window)
    (0, 1), (1, 7), (2, 64), (3, 300), (5, 1000), (6, 100), (8, 129), (9, 40), (10, 256),
]


@pytest.mark.parametrize("case,window", WINDOW_CASES, ids=[f"seed{RANDOM_CASES[c][0]}-w{w}" for c, w in WINDOW_CASES])
def test_sliding_window_random_mixes(case, window):
    """The reference backend's window: the query at position p sees keys above
    p - window.  Decodes (split and unsplit), warp-MMA and tcgen05 prefill."""
    seed, reqs, max_ctx, max_new, hq, hkv, d, pad = RANDOM_CASES[case]
    spec = random_spec(100 + seed, reqs, max_ctx, max_new, hq, hkv, d, pad_rows=pad)
    b = make_batch(spec, device="cpu")
    dev = DeviceStep(b, window=window)
    dev.step()
    ref = cpu_copy(b)
    oracle_write(ref)
    assert_close(dev.out, oracle_full(ref, window=window), f"window {window}")
    assert pkv.read_device_error(dev.ws) == 0


@pytest.mark.parametrize("path", ["split64", "split1024", "prefill-split", "no-tcgen05"])
def test_sliding_window_on_every_kernel_path(path, attn_options):
    if path == "split64":
        attn_options(split_tokens=64)          # many decode splits, in-kernel combine
    elif path == "split1024":
        attn_options(split_tokens=1024)        # streaming decode kernel
    elif path == "prefill-split":
        attn_options(disable_tcgen05=1)
        attn_options(prefill_key_splits=1)
        attn_options(split_tokens=128)
    else:
        attn_options(disable_tcgen05=1)
    reqs = [Req(3000, 1, list(range(0, 188))), Req(700, 40, list(range(188, 235))),
            Req(2500, 3, list(range(235, 392))), Req(0, 300, list(range(392, 411))),
            Req(5000, 1, list(range(411, 724)))]
    spec = Spec("window-paths", reqs, 16, 4, 128, 16, 730, 1 / math.sqrt(128), 51)
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    for window in (33, 500):
        dev = DeviceStep(b, window=window)
        dev.step()
        assert_close(dev.out, oracle_full(ref, window=window), f"{path} window {window}")


def test_negative_window_is_rejected():
    b = make_batch(config_spec(1), device="cpu")
    dev = DeviceStep(b, window=-1)
    with pytest.raises(pkv.PkvError) as e:
        dev.attend()
    assert e.value.status == 1


def test_long_decodes_with_window_sampled():
    """The 32 x 32768 decode shape (8 requests) with a 4096-key window: each
    decode reads only its last 4096 keys."""
    from workloads import subset_spec
    spec = subset_spec(config_spec(5), 8)
    b = device_batch(spec)
    ref = cpu_copy(b)
    dev = DeviceStep(b, window=4096)
    dev.step()
    oracle_write(ref)
    gen = torch.Generator().manual_seed(5)
    toks, heads = _sample_rows(spec, b.meta, gen, per_req_heads=3)
    want = oracle_rows(ref, toks, heads, window=4096)
    got = dev.out[torch.tensor(toks), torch.tensor(heads)]
    assert_close(got, want, "long decodes, window 4096")


@pytest.mark.parametrize("d,hq,hkv", [(64, 16, 4), (128, 32, 8)])
def test_short_decodes_head_dims_and_windows(d, hq, hkv):
    reqs = [Req(L - 1, 1, list(range(64 * i, 64 * i + 64))) for i, L in enumerate((17, 300, 1000, 1024, 640, 1))]
    spec = Spec("decodes", reqs, hq, hkv, d, 16, 64 * 6 + 2, 1 / math.sqrt(d), 81)
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    for window in (0, 100):
        dev = DeviceStep(b, window=window)
        dev.step()
        assert_close(dev.out, oracle_full(ref, window=window), f"decodes d{d} window {window}")


@pytest.mark.parametrize("row_tiles", [0, 1], ids=["key-major", "row-tiles"])
@pytest.mark.parametrize("split", [128, 1024], ids=["slot-ring", "streaming"])
@pytest.mark.parametrize("d,hq,hkv", [(48, 8, 4), (64, 16, 4), (128, 64, 8)])
def test_decode_tile_forms(d, hq, hkv, split, row_tiles, attn_options):
    """Decode CTAs of at most 8 rows per KV head run key-major tiles (keys in
    the MMA's M dimension); the decode_row_tiles option keeps the 16-row tiles.
    Both forms, both decode kernels, t = 1 and 2 where g allows, a window."""
    attn_options(split_tokens=split)
    attn_options(decode_row_tiles=row_tiles)
    g = hq // hkv
    lens = (17, 300, 1000, 2048, 2500, 1, 5000)
    reqs, blk = [], 0
    for i, L in enumerate(lens):
        t = 2 if (g * 2 <= 8 and i % 2 == 1 and L > 1) else 1
        nb = (L + 15) // 16
        reqs.append(Req(L - t, t, list(range(blk, blk + nb))))
        blk += nb
    spec = Spec("decode-tiles", reqs, hq, hkv, d, 16, blk + 2, 1 / math.sqrt(d), 83)
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    for window in (0, 700):
        dev = DeviceStep(b, window=window)
        dev.step()
        assert_close(dev.out, oracle_full(ref, window=window), f"decode tiles d{d} split {split} window {window}")
        assert pkv.read_device_error(dev.ws) == 0


CLUSTER_LENS = (17, 40, 300, 700, 1000, 1999, 33)


@pytest.mark.parametrize("window", [0, 500])
@pytest.mark.parametrize("cs", [2, 3, 8])
@pytest.mark.parametrize("d,hq,hkv,row_tiles", [(48, 8, 4, 0), (128, 32, 8, 0), (64, 16, 4, 1), (128, 64, 8, 1)],
                         ids=["d48g2", "d128g4", "d64g4-rows", "d128g8-rows"])
def test_cluster_split_combine(d, hq, hkv, row_tiles, cs, window, attn_options):
    """Short split decodes whose splits run as one thread-block cluster and
    combine through distributed shared memory: cs CTAs per request and KV
    head, keys divided evenly (short requests leave empty trailing splits),
    key-major and 16-row tiles, t = 1 and 2, a padding request; two eager calls
    and two CUDA-graph replays give the same result."""
    attn_options(split_tokens=256)
    attn_options(cluster=cs)
    attn_options(decode_row_tiles=row_tiles)
    g = hq // hkv
    reqs, blk = [], 0
    for i, L in enumerate(CLUSTER_LENS):
        t = 2 if (i % 2 == 1 and 2 * g <= 16) else 1
        nb = (L + 15) // 16
        reqs.append(Req(L - t, t, list(range(blk, blk + nb))))
        blk += nb
    reqs.insert(3, Req(0, 1, [], pad=True))
    spec = Spec("cluster", reqs, hq, hkv, d, 16, blk + 2, 1 / math.sqrt(d), 84)
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    want = oracle_full(ref, window=window)
    dev = DeviceStep(b, window=window)
    dev.write()
    for i in range(2):
        dev.out.fill_(float("nan"))
        dev.attend()
        assert_close(dev.out, want, f"cluster {cs} d{d} window {window} call {i}")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        dev.attend()
    torch.cuda.synchronize()
    for i in range(2):
        dev.out.fill_(float("nan"))
        gr.replay()
        torch.cuda.synchronize()
        assert_close(dev.out, want, f"cluster {cs} d{d} window {window} replay {i}")
    assert pkv.read_device_error(dev.ws) == 0


@pytest.mark.parametrize("cluster", [-1, 0], ids=["counters", "cluster"])
def test_engine_step_split_combine_both_ways(cluster, attn_options):
    """The 48-request engine step with its short decode splits combined by
    the split counters (cluster option -1) and by clusters (the default)."""
    attn_options(cluster=cluster)
    b = make_batch(config_spec(2), device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    dev = DeviceStep(b)
    dev.step()
    _check_write(dev, ref)
    assert_close(dev.out, oracle_full(ref), f"engine step cluster={cluster}")
    assert pkv.read_device_error(dev.ws) == 0


@pytest.mark.parametrize("cluster", [0, -1], ids=["clusters", "counters"])
def test_more_requests_than_one_launch_lists(cluster, attn_options):
    """600 decode requests and 300 prefill chunks: every kernel class runs
    several launches of at most 256 listed requests, each launch with its own
    plan (split counts, cluster size); short and long contexts mixed."""
    attn_options(cluster=cluster)
    gen = torch.Generator().manual_seed(85)
    reqs, blk = [], 0
    for i in range(900):
        if i % 3 == 2:                                   # prefill chunk of 2..40 tokens
            t = int(torch.randint(2, 41, (1,), generator=gen))
            c = int(torch.randint(0, 600, (1,), generator=gen))
        else:                                            # decode over 1..1500 keys
            t = 1
            c = int(torch.randint(0, 1500, (1,), generator=gen))
        nb = (c + t + 15) // 16
        reqs.append(Req(c, t, list(range(blk, blk + nb))))
        blk += nb
    spec = Spec("many", reqs, 8, 2, 64, 16, blk + 4, 0.125, 86)
    b = make_batch(spec, device="cpu")
    ref = cpu_copy(b)
    oracle_write(ref)
    dev = DeviceStep(b)
    dev.step()
    _check_write(dev, ref)
    assert_close(dev.out, oracle_full(ref), f"900 requests, cluster={cluster}")
    assert pkv.read_device_error(dev.ws) == 0
