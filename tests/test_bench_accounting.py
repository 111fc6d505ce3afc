"""bench.py's roofline arithmetic on CPU: the algorithmic bytes and FLOPs of
a step (every pool slot a request reads counted once, shared prefix blocks
once for the whole batch; 4 * d * Hq FLOPs per unmasked query-key pair),
their split between kernels, the achieved/peak fraction, and the rule that
stored ncu traffic is used only while the kernel's sources are unchanged.
The expected values are computed here from the workload metadata by other
routes: query positions for the causal pairs, block tables for the prefix
sharing."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import paged_kv_cache_84_gb300 as pkv  # noqa: E402
from workloads import build_meta, config_spec  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_84_gb300 import build
    build.build()
    pkv.load()


def step_accounting(cfg):
    spec = config_spec(cfg)
    meta = build_meta(spec)
    classes = pkv.plan_request_kernels(meta.query_start_loc, meta.seq_lens, spec.num_q_heads,
                                       spec.num_kv_heads, spec.head_dim)
    return spec, meta, classes, bench.accounting(spec, meta, classes)


def test_layout_example_by_hand():
    spec, meta, classes, acc = step_accounting(1)
    slot = 4 * 48 * 2 * 2                                # K and V of one slot: Hkv x d bf16, twice
    assert acc["unique_kv_bytes"] == (9 + 42 + 10 + 4) * slot
    assert acc["q_out_bytes"] == 2 * 9 * 8 * 48 * 2
    assert acc["write_bytes"] == 9 * slot * 2 + 9 * 8     # new rows read and written, int64 slots
    # causal pairs from the query positions: a query at position p sees p + 1 keys
    pairs = sum(p + 1 for p in meta.positions)
    assert pairs == 24 + 42 + 10 + 10
    assert acc["flops"] == pytest.approx(4 * 48 * 8 * pairs)


def test_causal_pairs_of_every_workload_shape():
    for cfg in (2, 3, 4):
        spec, meta, classes, acc = step_accounting(cfg)
        pairs = sum(p + 1 for p, s in zip(meta.positions, meta.slot_mapping.tolist()) if s >= 0)
        assert acc["flops"] == pytest.approx(4 * spec.head_dim * spec.num_q_heads * pairs, rel=1e-12)


def test_shared_prefix_blocks_count_once():
    spec, meta, classes, acc = step_accounting(2)
    slot = spec.num_kv_heads * spec.head_dim * 2 * 2
    # the 16 system-prompt blocks are the same physical blocks in all 48 tables
    first = [tuple(r.table[:16]) for r in spec.reqs]
    assert len(set(first)) == 1
    private = set()
    for r in spec.reqs:
        private.update(r.table[16:])
    assert not private & set(first[0])
    assert acc["logical_kv_bytes"] == sum(meta.seq_lens) * slot
    assert acc["unique_kv_bytes"] == acc["logical_kv_bytes"] - 47 * 256 * slot


def test_write_bytes_split_between_scatter_and_decode_kernels():
    spec, meta, classes, acc = step_accounting(2)
    scatter, _ = bench.kernel_work("paged_kv_write", acc, combined=True)
    dec_b, _ = bench.kernel_work("attn_mma_decode", acc, combined=True)
    dec_plain, _ = bench.kernel_work("attn_mma_decode", acc, combined=False)
    dec_writes = dec_b - dec_plain
    assert scatter + dec_writes == acc["write_bytes"]
    assert bench.kernel_work("paged_kv_write", acc, combined=False)[0] == acc["write_bytes"]
    t_dec = sum(b - a for (a, b), c in zip(zip(meta.query_start_loc, meta.query_start_loc[1:]), classes)
                if c in ("decode", "padding"))
    row = spec.num_kv_heads * spec.head_dim * 2 * 2
    assert dec_writes == t_dec * (row * 2 + 8)


def test_roofline_fraction_and_bound():
    acc = {"per_class": {"decode": {"kv_bytes": 6.0e9, "q_out_bytes": 0.0, "write_bytes": 0.0, "flops": 1.0e9}},
           "write_bytes": 0.0}
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "source": "measured", "sm_max_mhz": 2070.0}
    r = bench.roofline("attn_mma_decode", 1.25e-3, 1, acc, peaks, "cfgX")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(6.0e9 / 1.25e-3 / 1e9)          # 4800 GB/s
    assert r["frac"] == pytest.approx(0.8)
    assert r["traffic"] is None
    # a tensor-class kernel that is nearer its HBM roofline reports that one
    acc2 = {"per_class": {"prefill_tensor": {"kv_bytes": 6.0e9, "q_out_bytes": 0.0, "write_bytes": 0.0,
                                             "flops": 1.0e9}}, "write_bytes": 0.0}
    r2 = bench.roofline("attn_tc_prefill", 1.25e-3, 2, acc2, peaks, "cfgX")
    assert r2["bound"] == "hbm" and r2["frac"] == pytest.approx(0.4)          # two launches per step
    acc3 = {"per_class": {"prefill_tensor": {"kv_bytes": 1.0e6, "q_out_bytes": 0.0, "write_bytes": 0.0,
                                             "flops": 2.0e12}}, "write_bytes": 0.0}
    r3 = bench.roofline("attn_tc_prefill", 1.25e-3, 1, acc3, peaks, "cfgX")
    assert r3["bound"] == "tensor" and r3["achieved"] == pytest.approx(1600.0) and r3["frac"] == pytest.approx(0.8)


def test_stored_traffic_only_while_sources_unchanged(tmp_path, monkeypatch):
    csrc = tmp_path / "paged_kv_cache_84_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name, text in (("attn_tc.cu", "kernel v1\n"), ("common.cuh", "common\n"), ("sm100.cuh", "sm100\n")):
        (csrc / name).write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.source_hash("attn_tc_prefill")
    assert h is not None and len(h) == 12
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(
        "# kernel workload bytes hash\n"
        f"attn_tc_prefill cfg4 209576448 {h}\n"
        "attn_mma_decode cfg4 123 000000000000\n")
    assert bench.stored_traffic("attn_tc_prefill", "cfg4") == 209576448.0
    assert bench.stored_traffic("attn_tc_prefill", "cfg2") is None             # no line for it
    assert bench.stored_traffic("attn_mma_decode", "cfg4") is None             # its source file is absent
    (csrc / "common.cuh").write_text("common, edited\n")
    assert bench.stored_traffic("attn_tc_prefill", "cfg4") is None             # stale once a source changes


def test_clock_summary_of_the_timed_region():
    """The clocks line: median SM clock and the throttle reasons seen inside
    the timed region (samples just outside it are ignored)."""
    s = bench.ClockSampler(0)

    def row(sm, reason_hw="Not Active", power="150.5"):
        return ["0", str(sm), "2070", power, "0x0", reason_hw, "Not Active", "Not Active", "Not Active"]

    s.samples = [(9.0, row(1000, "Active")),                       # before the timed region
                 (10.0, row(2070)), (10.1, row(2055, power="300.0")), (10.2, row(2070)),
                 (12.0, row(900, "Active"))]                       # after it
    out = s.summary(10.0, 10.2)
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070 and out["samples"] == 3
    assert out["reasons"] == [] and out["power_w_max"] == 300.0 and out["window"] == "timed region"
    s.samples.append((10.15, row(1500, "Active")))
    assert s.summary(10.0, 10.2)["reasons"] == ["hw_slowdown"]
    # a timed region shorter than the sampling interval falls back to every sample
    assert s.summary(20.0, 20.01)["window"].startswith("whole GPU phase")
