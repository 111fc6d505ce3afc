"""The attention planner's decisions on a host without a GPU
(pkv_plan_attention, include/pkv.h), for the five workload shapes and the
rules the header states: request classes, one decode split length (about 16
CTAs per SM over the decode keys, 4 beside a longer prefill, at least 256
keys, a multiple of 128, at most 32 streaming splits per request, doubled
until the split partials fit the workspace), short splits merged in
thread-block clusters (at most two beside prefill work), long ones on the
streaming kernel, and the two-stream overlap of the decode and prefill
classes of one flattened ragged batch ("31. Engine v2", "Flattened ragged
batches").  The expected split lengths restate those rules here."""
import math

import pytest

import paged_kv_cache_84_gb300 as pkv
from workloads import config_spec

SMS = 152
BIG_WS = 1 << 30


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_84_gb300 import build
    build.build()
    pkv.load()


@pytest.fixture(autouse=True)
def _planner_choices():
    pkv.reset_options()
    yield
    pkv.reset_options()


def meta(cfg):
    spec = config_spec(cfg)
    qsl = [0]
    for r in spec.reqs:
        qsl.append(qsl[-1] + r.new)
    return spec, qsl, [r.seq_len for r in spec.reqs]


def plan(cfg, mixed=-1, **kw):
    """The plan for workload cfg; by default with the single mixed launch
    ruled out, so that the two-stream rules below are what is checked."""
    spec, qsl, sl = meta(cfg)
    kw.setdefault("num_sms", SMS)
    kw.setdefault("workspace_bytes", BIG_WS)
    with pkv.options(mixed_launch=mixed):
        return pkv.plan_attention(qsl, sl, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, **kw)


def rule_split(keys, head_ctas, ctas_per_sm, sms=SMS, max_keys=0):
    """The documented split rule, restated: keys x KV-head CTAs spread over
    ctas_per_sm CTAs per SM, at least 256, rounded up to 128; a streaming
    split (>= 512 keys) is long enough for at most 32 splits per request."""
    s = max(256, math.ceil(keys * head_ctas / (sms * ctas_per_sm)))
    s = -(-s // 128) * 128
    if s >= 512:
        s = max(s, -(-math.ceil(max_keys / 32) // 128) * 128)
    return s


def test_layout_example_is_all_decode():
    p = plan(1)
    assert (p["decode_requests"], p["prefill_tensor_requests"], p["prefill_mma_requests"]) == (4, 0, 0)
    assert p["decode_split_tokens"] == 256 and p["max_decode_splits"] == 1
    assert p["decode_cluster"] == 0 and not p["decode_streaming"] and not p["overlap"]
    assert p["partial_bytes"] == 0


def test_long_decode_streams_ten_splits_per_request():
    spec, qsl, sl = meta(5)
    p = plan(5)
    split = rule_split(sum(sl), spec.num_kv_heads, 16, max_keys=max(sl))
    assert p["decode_split_tokens"] == split == 3456
    assert p["max_decode_splits"] == math.ceil(32768 / split) == 10
    assert p["decode_streaming"] and p["decode_cluster"] == 0 and p["split_counters"]
    rows = 32 * 10 * spec.num_q_heads                 # S x t x hq partial rows per request
    assert p["partial_bytes"] == rows * spec.head_dim * 4 + rows * 8


def test_split_grows_until_the_partials_fit():
    spec, qsl, sl = meta(5)
    base = plan(5)["decode_split_tokens"]
    p = plan(5, workspace_bytes=4 << 20)
    assert p["partial_bytes"] <= 4 << 20
    assert p["decode_split_tokens"] in [base << k for k in range(1, 6)]
    assert p["max_decode_splits"] == math.ceil(32768 / p["decode_split_tokens"]) == 3
    # a workspace too small for any partial: nothing is split, no counters
    q = plan(5, workspace_bytes=pkv.WORKSPACE_MIN_BYTES)
    assert q["max_decode_splits"] == 1 and q["partial_bytes"] == 0 and not q["split_counters"]


def test_decode_batch_uses_sixteen_ctas_per_sm():
    spec, qsl, sl = meta(3)
    p = plan(3)
    split = rule_split(sum(sl), spec.num_kv_heads, 16, max_keys=max(sl))
    assert p["decode_split_tokens"] == split
    assert p["max_decode_splits"] == math.ceil(max(sl) / split)
    assert p["decode_requests"] == 256 and not p["overlap"]
    assert p["decode_streaming"] == (split >= 512)
    # half the SMs: about twice the keys per split
    h = plan(3, num_sms=SMS // 2)
    assert h["decode_split_tokens"] == rule_split(sum(sl), spec.num_kv_heads, 16, sms=SMS // 2, max_keys=max(sl))
    assert h["decode_split_tokens"] > split


def test_engine_step_overlaps_classes_with_clusters_of_two():
    spec, qsl, sl = meta(2)
    p = plan(2, combined=True)
    assert (p["decode_requests"], p["prefill_tensor_requests"], p["prefill_mma_requests"]) == (32, 16, 0)
    assert p["overlap"] and p["decode_on_caller_stream"]     # the decodes' K/V bytes outweigh the chunks
    assert p["decode_split_tokens"] == 256
    assert p["max_decode_splits"] >= 2 and p["decode_cluster"] == 2 and not p["decode_streaming"]
    assert p["partial_bytes"] > 0                               # reserved, although clusters merge on chip


def test_chunks_that_are_one_cta_per_kv_head_write_their_own_rows():
    """Combined call, bf16 pool: a tcgen05 request whose rows of each KV
    head fit one pair of 128-row tiles (t * g <= 256) and are not cut into
    key pieces is written by its own CTAs, not by the scatter; never on a
    quantized pool, in a mixed launch, or outside the combined call."""
    p = plan(2, combined=True)
    assert p["prefill_tensor_own_rows"] == p["prefill_tensor_requests"] == 16   # chunks of <= 64 tokens, g = 2
    assert plan(2, combined=False)["prefill_tensor_own_rows"] == 0
    assert plan(4, mixed=0, combined=True)["prefill_tensor_own_rows"] == 0       # one mixed launch
    assert plan(4, combined=True)["prefill_tensor_own_rows"] == 0                # 2048- and 1024-token chunks
    # g = 4: 64 tokens per pair; a 64-token and a 65-token chunk beside a decode
    for t, own in ((64, 1), (65, 0)):
        qsl, sl = [0, t, t + 1], [300 + t, 900]
        q = pkv.plan_attention(qsl, sl, 32, 8, 128, combined=True, num_sms=SMS, workspace_bytes=BIG_WS)
        assert (q["prefill_tensor_requests"], q["prefill_tensor_own_rows"]) == (1, own), t
        q = pkv.plan_attention(qsl, sl, 32, 8, 128, quantized=True, combined=True, num_sms=SMS,
                               workspace_bytes=BIG_WS)                     # quantized pool (head dim 128)
        assert (q["prefill_tensor_requests"], q["prefill_tensor_own_rows"]) == (1, 0), t
    with pkv.options(tc_key_pieces=2):                                         # a pair cut into pieces
        q = pkv.plan_attention([0, 64, 65], [8192, 900], 32, 8, 128, combined=True, num_sms=SMS,
                               workspace_bytes=BIG_WS)
        assert q["prefill_tensor_pieces"] > 0 and q["prefill_tensor_own_rows"] == 0


def test_decodes_beside_a_long_prefill_take_longer_splits():
    spec, qsl, sl = meta(4)
    p = plan(4, combined=True)
    assert (p["decode_requests"], p["prefill_tensor_requests"]) == (64, 3)
    assert p["overlap"] and not p["decode_on_caller_stream"]   # the 2048-token chunk at 16384 dominates
    dec = [L for L, a, b in zip(sl, qsl, qsl[1:]) if b - a == 1]
    assert p["decode_split_tokens"] == rule_split(sum(dec), spec.num_kv_heads, 4, max_keys=max(dec))
    # the same decodes alone spread over 16 CTAs per SM
    alone_qsl = list(range(len(dec) + 1))
    a = pkv.plan_attention(alone_qsl, dec, 32, 8, 128, workspace_bytes=BIG_WS, num_sms=SMS)
    assert a["decode_split_tokens"] == rule_split(sum(dec), 8, 16, max_keys=max(dec))
    assert p["decode_split_tokens"] >= 3 * a["decode_split_tokens"]


def test_options():
    """Each option overrides its planner choice (pkv_attention_options)."""
    with pkv.options(no_overlap=1):
        assert not plan(2)["overlap"]
    with pkv.options(decode_main=-1):
        p = plan(2)
        assert p["overlap"] and not p["decode_on_caller_stream"]
    with pkv.options(cluster=-1):
        assert plan(2)["decode_cluster"] == 0
    with pkv.options(cluster=4):
        assert plan(2)["decode_cluster"] == 4
    with pkv.options(split_tokens=512):
        p = plan(3)
        assert p["decode_split_tokens"] == 512 and p["decode_streaming"]
    with pkv.options(disable_tcgen05=1):
        p = plan(2)
        assert p["prefill_tensor_requests"] == 0 and p["prefill_mma_requests"] == 16
    with pkv.options(tc_min_rows=1000):
        p = plan(2)                                      # chunks of <= 64 tokens x g 2 stay below it
        assert p["prefill_tensor_requests"] == 0 and p["prefill_mma_requests"] == 16
    with pkv.options(prefill_key_splits=1, disable_tcgen05=1):
        assert plan(2)["prefill_key_splits"]
    spec, qsl, sl = meta(4)
    extra = pkv.fp8_prefill_scratch_bytes(qsl, sl, 32, 8, 128)
    with pkv.options(fp8_prefill_on_mma=1):
        p = plan(4, quantized=True, workspace_bytes=BIG_WS + extra)
        assert p["prefill_tensor_requests"] == 0 and p["quantized_prefill_scratch"] == 0
    assert pkv.current_options() == {}
    with pytest.raises(TypeError):
        pkv.set_options(no_such_option=1)


def test_library_reads_no_environment():
    """The library's planner does not change with environment variables."""
    import os
    import subprocess
    import sys
    code = ("import json, paged_kv_cache_84_gb300 as pkv; from workloads import config_spec; "
            "s = config_spec(2); q = [0]; [q.append(q[-1] + r.new) for r in s.reqs]; "
            "print(json.dumps(pkv.plan_attention(q, [r.seq_len for r in s.reqs], 8, 4, 48, "
            "workspace_bytes=1 << 30, num_sms=152)))")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    base = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True)
    env.update(PKV_NO_OVERLAP="1", PKV_CLUSTER="0", PKV_SPLIT_TOKENS="512", PKV_DISABLE_TCGEN05="1")
    other = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True)
    assert base.returncode == 0 and other.returncode == 0, base.stderr + other.stderr
    assert base.stdout == other.stdout
    csrc = os.path.join(root, "paged_kv_cache_84_gb300", "csrc")
    for name in os.listdir(csrc):
        assert "getenv" not in open(os.path.join(csrc, name)).read(), name


def test_quantized_prefill_on_tcgen05_needs_the_scratch():
    spec, qsl, sl = meta(4)
    ws = 8 << 20
    extra = pkv.fp8_prefill_scratch_bytes(qsl, sl, 32, 8, 128)
    assert extra > ws
    p = plan(4, quantized=True, workspace_bytes=ws)
    assert p["prefill_tensor_requests"] == 0 and p["prefill_mma_requests"] == 3
    assert p["quantized_prefill_scratch"] == 0
    q = plan(4, quantized=True, workspace_bytes=ws + extra)
    assert q["prefill_tensor_requests"] == 3 and q["prefill_mma_requests"] == 0
    assert q["quantized_prefill_scratch"] == extra
    # two KV heads per streaming CTA: half the CTAs per split than bf16
    dec = [L for L, a, b in zip(sl, qsl, qsl[1:]) if b - a == 1]
    assert q["decode_split_tokens"] == rule_split(sum(dec), 8 // 2, 4, max_keys=max(dec))


def test_sliding_window_limits_the_decode_keys():
    p = plan(5, window=4096)
    keys = 32 * 4096
    split = rule_split(keys, 8, 16, max_keys=4096)
    assert p["decode_split_tokens"] == split == 512
    assert p["max_decode_splits"] == 4096 // split


@pytest.mark.parametrize("args,status", [
    (dict(num_q_heads=8, num_kv_heads=3), 1),           # heads do not group
    (dict(seq_lens=[2]), 1),                            # t > seq_len
    (dict(window=-1), 1),
    (dict(block_size=48), 2),                           # not 16 times a power of two
    (dict(block_size=8), 2),
    (dict(block_size=512), 2),
    (dict(head_dim=96), 2),
    (dict(quantized=True), 2),                          # quantized pools need head_dim 128
])
def test_rejections(args, status):
    kw = dict(query_start_loc_host=[0, 3], seq_lens=[9], num_q_heads=8, num_kv_heads=4, head_dim=64)
    kw.update(args)
    qsl, sl = kw.pop("query_start_loc_host"), kw.pop("seq_lens")
    with pytest.raises(pkv.PkvError) as e:
        pkv.plan_attention(qsl, sl, kw.pop("num_q_heads"), kw.pop("num_kv_heads"), kw.pop("head_dim"),
                           num_sms=SMS, **kw)
    assert e.value.status == status


def test_mixed_launch_choice():
    """The planner's choice of one launch for both classes (decode CTAs ahead
    of the tcgen05 prefill CTAs): taken for the mixed 2048-token-chunk step,
    whose decodes are long (items of 1024 keys dealt to the decode CTAs'
    warps), not for the engine step's short decodes (one latency-bound item
    per warp would outlast the whole two-stream step) nor where there is no
    tcgen05 prefill."""
    p = plan(4, mixed=0, combined=True)
    spec, qsl, sl = meta(4)
    dec = [L for L, a, b in zip(sl, qsl, qsl[1:]) if b - a == 1]
    assert p["mixed_launch"] == 1 and not p["overlap"]
    assert p["decode_split_tokens"] == 1024
    assert p["mixed_decode_items"] == sum(-(-L // 1024) for L in dec) * spec.num_kv_heads
    assert 8 <= p["mixed_decode_ctas"] <= SMS // 2 and p["mixed_decode_ctas"] % spec.num_kv_heads == 0
    for cfg in (1, 2, 3, 5):
        assert plan(cfg, mixed=0, combined=True)["mixed_launch"] == 0, cfg
    with pkv.options(mixed_decode_ctas=40):
        q = plan(4, mixed=1, combined=True)
    assert q["mixed_launch"] == 1 and q["mixed_decode_ctas"] == 40
    assert q["mixed_predicted_us"] == 0 and p["mixed_predicted_us"] > 0
    # beside decode CTAs no pair is cut into key pieces unless asked
    assert p["prefill_tensor_pieces"] == 0
    with pkv.options(tc_key_pieces=3):
        assert plan(4, mixed=1, combined=True)["prefill_tensor_pieces"] > 0


def test_mixed_launch_choice_quantized():
    """Quantized pools: with room for the bf16 copies of the prefill blocks,
    the mixed step runs as one tcgen05 launch whose decode CTAs read the
    codes; without that room the prefill stays on the warp-MMA kernel and
    there is no mixed launch."""
    spec, qsl, sl = meta(4)
    extra = pkv.fp8_prefill_scratch_bytes(qsl, sl, spec.num_q_heads, spec.num_kv_heads, 128)
    p = plan(4, mixed=0, combined=True, quantized=True, workspace_bytes=BIG_WS + extra)
    assert p["mixed_launch"] == 1 and p["quantized_prefill_scratch"] == extra
    assert p["mixed_decode_ctas"] % spec.num_kv_heads == 0 and p["prefill_tensor_pieces"] == 0
    q = plan(4, mixed=0, combined=True, quantized=True, workspace_bytes=32 << 20)   # no room for the copies
    assert q["mixed_launch"] == 0 and q["quantized_prefill_scratch"] == 0 and q["prefill_mma_requests"] > 0


def test_device_lengths_plan_decode_batches_only():
    """With device lengths (a padded decode step planned at capacity) only
    decode-class batches are accepted: a prefill chunk, whose tiles are
    planned from its own length, is refused before anything is enqueued;
    split decodes merge through the counters, never clusters."""
    with pkv.options(device_lengths=1):
        with pytest.raises(pkv.PkvError):
            pkv.plan_attention([0, 1, 65], [500, 300], 32, 8, 128, num_sms=SMS)
        p = pkv.plan_attention(list(range(49)), [4096] * 48, 8, 4, 48, num_sms=SMS)
    assert p["decode_requests"] == 48 and p["decode_cluster"] == 0
    q = pkv.plan_attention(list(range(49)), [4096] * 48, 8, 4, 48, num_sms=SMS)
    assert q["decode_requests"] == 48


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
def test_block_sizes_the_kernels_walk(bs):
    """Blocks of 16 times a power of two slots (up to 256) are planned: the
    kernels walk a block as sub-blocks of 16 slots."""
    p = pkv.plan_attention([0, 1, 300], [100, 2000], 32, 8, 128, block_size=bs, num_sms=SMS)
    assert p["decode_requests"] == 1 and p["prefill_tensor_requests"] == 1
    assert p["decode_split_tokens"] % bs == 0
