"""Block copies on the GPU (copy-on-write, swap-out, swap-in) against the
oracle, bit for bit ("vllm-lite README": copy-on-write of a shared block;
"31. Engine v2", "Preemption: recompute or swap")."""
import pytest
import torch

import oracle
import paged_kv_cache_84_gb300 as pkv

pytestmark = pytest.mark.gpu


def _pools(n_layers, nbt, bs, hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((nbt, bs, hkv, d), generator=g).to(torch.bfloat16) for _ in range(2 * n_layers)]


def _bits(t):
    return t.contiguous().view(torch.uint8)


@pytest.mark.parametrize("shape", [(3, 64, 16, 4, 48), (2, 300, 16, 8, 128)])
def test_copy_on_write_matches_oracle(shape):
    n_layers, nbt, bs, hkv, d = shape
    host = _pools(n_layers, nbt, bs, hkv, d, 1)
    dev = [p.cuda() for p in host]
    g = torch.Generator().manual_seed(2)
    perm = torch.randperm(nbt, generator=g)
    src, dst = perm[:nbt // 3].to(torch.int32), perm[nbt // 3:2 * (nbt // 3)].to(torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(dev, src.cuda(), dst.cuda(), err)
    oracle.copy_blocks(host, src, dst)
    for h, dv in zip(host, dev):
        assert torch.equal(_bits(dv.cpu()), _bits(h))
    assert pkv.read_device_error(err) == 0


@pytest.mark.parametrize("where", ["device", "pinned-host"])
def test_swap_out_and_in_match_oracle(where):
    nbt, bs, hkv, d = 200, 16, 8, 128
    host = _pools(4, nbt, bs, hkv, d, 3)
    dev = [p.cuda() for p in host]
    g = torch.Generator().manual_seed(4)
    ids = torch.randperm(nbt, generator=g)[:37].to(torch.int32)
    bb = bs * hkv * d * 2
    buf = torch.empty((len(dev), ids.numel(), bb), dtype=torch.uint8,
                      device="cuda" if where == "device" else "cpu")
    if where != "device":
        buf = buf.pin_memory()
    pkv.gather_blocks(dev, ids.cuda(), buf)
    torch.cuda.synchronize()
    want = oracle.gather_blocks(host, ids)
    assert torch.equal(buf.cpu(), want)
    # swap back in to newly allocated blocks of fresh pools
    new_ids = torch.randperm(nbt, generator=g)[:37].to(torch.int32)
    fresh_host = _pools(4, nbt, bs, hkv, d, 5)
    fresh_dev = [p.cuda() for p in fresh_host]
    pkv.scatter_blocks(fresh_dev, new_ids.cuda(), buf)
    oracle.scatter_blocks(fresh_host, new_ids, want)
    for h, dv in zip(fresh_host, fresh_dev):
        assert torch.equal(_bits(dv.cpu()), _bits(h))


def test_out_of_pool_ids_are_skipped_and_flagged():
    host = _pools(1, 32, 16, 2, 64, 6)
    dev = [p.cuda() for p in host]
    src = torch.tensor([1, 40, 3], dtype=torch.int32)
    dst = torch.tensor([5, 6, -1], dtype=torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(dev, src.cuda(), dst.cuda(), err)
    assert pkv.read_device_error(err) & pkv.DEVERR_BLOCK
    oracle.copy_blocks(host, [1], [5])                 # only the valid pair lands
    for h, dv in zip(host, dev):
        assert torch.equal(_bits(dv.cpu()), _bits(h))
    torch.cuda.synchronize()


def test_block_copy_in_a_cuda_graph():
    host = _pools(2, 64, 16, 4, 64, 7)
    dev = [p.cuda() for p in host]
    src = torch.tensor([0, 1, 2, 3], dtype=torch.int32, device="cuda")
    dst = torch.tensor([10, 11, 12, 13], dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pkv.copy_blocks(dev, src, dst)
    graph.replay()
    torch.cuda.synchronize()
    oracle.copy_blocks(host, src.cpu(), dst.cpu())
    for h, dv in zip(host, dev):
        assert torch.equal(_bits(dv.cpu()), _bits(h))


@pytest.mark.parametrize("nbytes", [16, 4096, (1 << 20) + 48, 7 << 20, (8 << 20) + 48, 51 << 20])
def test_copy_async_host_device_round_trip(nbytes):
    """pkv_copy_async: pinned host -> device, device -> device, device ->
    pinned host, bit for bit, inside one stream and in a CUDA graph (copies
    across the link of 8 MiB or more go to the copy engine)."""
    g = torch.Generator().manual_seed(nbytes % 1000)
    src = torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8).pin_memory()
    d1 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d2 = torch.empty_like(d1)
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    pkv.copy_async(d1, src)
    pkv.copy_async(d2, d1)
    pkv.copy_async(back, d2)
    torch.cuda.synchronize()
    assert torch.equal(d1.cpu(), src) and torch.equal(back, src)
    back.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        pkv.copy_async(d2, src)
        pkv.copy_async(back, d2)
    gr.replay()
    torch.cuda.synchronize()
    assert torch.equal(back, src)


def test_copy_async_interior_of_pinned_buffers():
    """Copies between device memory and 16-byte-aligned interiors of larger
    pinned buffers (how a step's packed inputs are laid out), at a size that
    takes host-link copies through several grid-stride rounds and a ragged
    last round, leaving the bytes around the copied range untouched."""
    n = (12 * 2048 * 2 + 77) * 16
    g = torch.Generator().manual_seed(7)
    big = torch.randint(0, 256, (n + 4096,), generator=g, dtype=torch.uint8).pin_memory()
    d = torch.zeros(n + 512, dtype=torch.uint8, device="cuda")
    pkv.copy_async(d[256:256 + n], big[1024:1024 + n])
    torch.cuda.synchronize()
    got = d.cpu()
    assert torch.equal(got[256:256 + n], big[1024:1024 + n])
    assert not got[:256].any() and not got[256 + n:].any()
    back = torch.full((n + 4096,), 0xA5, dtype=torch.uint8).pin_memory()
    pkv.copy_async(back[2048:2048 + n], d[256:256 + n])
    torch.cuda.synchronize()
    assert torch.equal(back[2048:2048 + n], big[1024:1024 + n])
    assert bool((back[:2048] == 0xA5).all()) and bool((back[2048 + n:] == 0xA5).all())


def test_copy_async_rejects_unaligned_and_odd_sizes():
    d = torch.empty(4096, dtype=torch.uint8, device="cuda")
    h = torch.empty(4096, dtype=torch.uint8).pin_memory()
    with pytest.raises(pkv.PkvError):
        pkv.copy_async(d[8:8 + 64], h[:64])                  # unaligned device side
    with pytest.raises(pkv.PkvError):
        pkv.copy_async(d[:24], h[:24])                       # not a multiple of 16 bytes
    pkv.copy_async(d[:0], h[:0])                             # zero bytes: no-op
    torch.cuda.synchronize()

