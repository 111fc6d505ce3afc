"""Shared pieces of the GPU tests: run one step through the CUDA library and
the same step through the CPU oracle, on the same seeded inputs."""
from __future__ import annotations

import os

import torch

import oracle
import paged_kv_cache_84_gb300 as pkv
from workloads import Batch, Req, Spec, build_meta, make_batch

MAX_ERR = 2e-2       # max |float(out_bf16) - oracle|
MEAN_ERR = 2e-3      # mean |float(out_bf16) - oracle|


def threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


class DeviceStep:
    """One batch resident on the GPU: pools, new rows, metadata, output, workspace."""

    def __init__(self, batch: Batch, device="cuda", workspace_bytes=None, pools=None, window=0):
        self.batch = batch
        self.window = window
        spec, meta = batch.spec, batch.meta
        dev = torch.device(device)
        if pools is None:
            self.k_cache = batch.k_cache.to(dev).contiguous()
            self.v_cache = batch.v_cache.to(dev).contiguous()
        else:                                   # pools already on the device, shared across steps
            self.k_cache, self.v_cache = pools
        self.q = batch.q.to(dev).contiguous()
        self.k = batch.k.to(dev).contiguous()
        self.v = batch.v.to(dev).contiguous()
        self.qsl = torch.tensor(meta.query_start_loc, dtype=torch.int32, device=dev)
        self.sl = torch.tensor(meta.seq_lens, dtype=torch.int32, device=dev)
        self.bt = meta.block_table.to(dev).contiguous()
        self.slots = meta.slot_mapping.to(dev).contiguous()
        self.out = torch.full_like(self.q, float("nan"))
        if workspace_bytes is None:
            workspace_bytes = pkv.attention_workspace_bytes(
                max(1, meta.num_reqs), max(1, meta.num_tokens), spec.num_q_heads, spec.head_dim,
                max(1, meta.max_seq_len))
        self.ws = pkv.make_workspace(workspace_bytes, dev)
        self.write_err = torch.zeros(1, dtype=torch.int32, device=dev)

    def write(self):
        pkv.paged_kv_write(self.k, self.v, self.k_cache, self.v_cache, self.slots, self.write_err)

    def attend(self):
        b = self.batch
        pkv.ragged_paged_attention(self.out, self.q, self.k_cache, self.v_cache, self.qsl, self.sl, self.bt,
                                   b.meta.query_start_loc, b.meta.seq_lens, b.meta.max_query_len,
                                   b.meta.max_seq_len, b.spec.scale, self.ws, window=self.window)

    def step(self):
        self.write()
        self.attend()
        return self.out

    def combined(self):
        """The step as one pkv_paged_kv_write_attention call."""
        b = self.batch
        pkv.paged_kv_write_attention(self.k, self.v, self.k_cache, self.v_cache, self.slots, self.out, self.q,
                                     self.qsl, self.sl, self.bt, b.meta.query_start_loc, b.meta.seq_lens,
                                     b.meta.max_query_len, b.meta.max_seq_len, b.spec.scale, self.ws,
                                     window=self.window)
        return self.out


def device_batch(spec, device="cuda") -> Batch:
    """Values drawn on the device (fast for multi-GB pools)."""
    return make_batch(spec, device=device)


def cpu_copy(batch: Batch) -> Batch:
    return Batch(batch.spec, batch.meta, batch.q.cpu(), batch.k.cpu(), batch.v.cpu(),
                 batch.k_cache.cpu(), batch.v_cache.cpu())


def oracle_write(batch_cpu: Batch):
    """The step's write on the CPU pools (in place)."""
    oracle.paged_kv_write(batch_cpu.k_cache, batch_cpu.v_cache, batch_cpu.k, batch_cpu.v,
                          batch_cpu.meta.slot_mapping)


def oracle_full(batch_cpu: Batch, window: int = 0) -> torch.Tensor:
    m = batch_cpu.meta
    return oracle.ragged_paged_attention(batch_cpu.q, batch_cpu.k_cache, batch_cpu.v_cache, m.query_start_loc,
                                         m.seq_lens, m.block_table, batch_cpu.spec.scale, threads(), window=window)


def oracle_rows(batch_cpu: Batch, tokens, heads, window: int = 0) -> torch.Tensor:
    m = batch_cpu.meta
    return oracle.attention_rows(tokens, heads, batch_cpu.q, batch_cpu.k_cache, batch_cpu.v_cache,
                                 m.query_start_loc, m.seq_lens, m.block_table, batch_cpu.spec.scale, threads(),
                                 window=window)


def errors(got_bf16: torch.Tensor, want: torch.Tensor):
    diff = (got_bf16.double().cpu() - want).abs()
    return diff.max().item(), diff.mean().item()


def assert_close(got_bf16, want, what=""):
    got = got_bf16.double().cpu()
    assert torch.isfinite(got).all(), f"{what}: non-finite output"
    mx, mean = errors(got_bf16, want)
    assert mx <= MAX_ERR and mean <= MEAN_ERR, f"{what}: max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def quantized_pools(batch, seed):
    """Junk codes and scales everywhere (never NaN codes), then the history of
    every request written by the oracle's quantizing write from bf16 values."""
    spec, m = batch.spec, batch.meta
    nbt = spec.num_blocks_total + 1
    g = torch.Generator().manual_seed(seed)
    shape = (nbt, spec.block_size, spec.num_kv_heads, spec.head_dim)
    kc = torch.randint(0, 255, shape, generator=g, dtype=torch.uint8)
    vc = torch.randint(0, 255, shape, generator=g, dtype=torch.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0
    vc[(vc & 0x7F) == 0x7F] = 0
    ks = torch.rand(shape[:3], generator=g)
    vs = torch.rand(shape[:3], generator=g)
    # history rows (positions 0 .. c-1) from the batch's bf16 pools
    hist = build_meta(Spec("hist", [Req(0, r.computed, r.table) for r in spec.reqs if not r.pad],
                           spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.block_size,
                           spec.num_blocks_total, 1.0, 0))
    if hist.num_tokens:
        sm = hist.slot_mapping
        kh = batch.k_cache.view(-1, spec.num_kv_heads, spec.head_dim)[sm]
        vh = batch.v_cache.view(-1, spec.num_kv_heads, spec.head_dim)[sm]
        oracle.paged_kv_write_fp8(kc, vc, ks, vs, kh, vh, sm)
    return kc, vc, ks, vs
