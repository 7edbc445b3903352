"""One captured decode step per bucket replays correctly for every length.

The step is the SenseNova-style shape (32 q / 8 kv heads, head_dim 128,
bf16) over the growth schedule 512..8192.  For every seqused in a bucket the
replay must be bit-identical to the eager launches, and at a stride (plus the
bucket edges) it must match the fp64 oracle run on a host mirror of the cache
that the oracle's own append keeps up to date.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

HQ, HKV, D = 32, 8, 128


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_13_gb300 as m
    return m


class Mirror:
    """Host copy of the cache inputs, advanced only by the oracle's append."""

    def __init__(self, k_host, v_host, bt_host):
        self.k = [t.view(torch.int16).numpy().copy() for t in k_host]
        self.v = [t.view(torch.int16).numpy().copy() for t in v_host]
        self.bt = bt_host.numpy()

    def append(self, layer, si, kn, vn):
        err = O.append(self.k[layer], self.v[layer], self.bt, si, kn.view(torch.int16).numpy(),
                       vn.view(torch.int16).numpy())
        assert err == 0

    def attend(self, layer, q, si, scale):
        kp = torch.from_numpy(self.k[layer]).view(torch.bfloat16).double().numpy()
        vp = torch.from_numpy(self.v[layer]).view(torch.bfloat16).double().numpy()
        out, lse, err = O.attend(q.double().numpy(), kp, vp, self.bt, si, scale)
        assert err == 0
        return out, lse


def sweep_bucket(pkv, runner, mirror, lengths, sample, gen, layers):
    st = runner.step_bufs
    for L in lengths:
        si = np.array([[0, 1, 0, L]], np.int32)
        qs = [torch.randn(1, HQ, D, generator=gen).to(torch.bfloat16) for _ in range(layers)]
        ks = [(torch.randn(1, HKV, D, generator=gen) / math.sqrt(D)).to(torch.bfloat16) for _ in range(layers)]
        vs = [(torch.randn(1, HKV, D, generator=gen) / math.sqrt(D)).to(torch.bfloat16) for _ in range(layers)]
        st.seq_info.copy_(torch.from_numpy(si))
        for layer in range(layers):
            st.q[layer].copy_(qs[layer])
            st.k_new[layer].copy_(ks[layer])
            st.v_new[layer].copy_(vs[layer])
        runner.step()
        replay = [o.clone() for o in st.out]
        st.run()                                   # eager: same launches, same inputs
        for layer in range(layers):
            assert torch.equal(replay[layer], st.out[layer]), f"replay != eager at length {L}"
            mirror.append(layer, si, ks[layer], vs[layer])
        if L in sample:
            torch.cuda.synchronize()
            for layer in range(layers):
                ref, _ = mirror.attend(layer, qs[layer], si, st.scale)
                diff = float(np.abs(U.f64(replay[layer]) - ref).max())
                assert diff <= 2e-3, f"length {L} layer {layer}: {diff}"
    assert int(st.err.item()) == 0


def test_one_capture_per_bucket_serves_every_length(pkv):
    from paged_kv_decode_13_gb300.graph import DecodeGraphRunner, DecodeStep
    layers = 2
    gen = torch.Generator().manual_seed(0)
    cache = pkv.PagedKVCache.allocate(layers, HKV, D, 512)
    host = [(torch.randn(t.shape, generator=gen) / math.sqrt(D)).to(torch.bfloat16) for t in cache.k + cache.v]
    for t, h in zip(cache.k + cache.v, host):
        t.copy_(h)
    runner = DecodeGraphRunner(DecodeStep(cache, HQ))
    mirror = Mirror(host[:layers], host[layers:], torch.arange(512 // 16, dtype=torch.int32)[None])
    prev = 0
    length = 0
    for bucket in (512, 1024, 2048, 4096, 8192):
        if bucket != cache.bucket:
            new = pkv.PagedKVCache.allocate(layers, HKV, D, pkv.bucket_for(length + 1),
                                            generation=cache.generation)
            assert new.bucket == bucket
            assert pkv.resize_bucket(cache, new, length) == 0
            assert new.generation == cache.generation + 1
            cache = new
            runner.rebind(cache)
            # the mirror grows with the new buffers (tail stays zero, as in the new allocation)
            for layer in range(layers):
                for arr_name in ("k", "v"):
                    old = getattr(mirror, arr_name)[layer]
                    grown = np.zeros((bucket // 16,) + old.shape[1:], old.dtype)
                    grown.reshape(-1, HKV, D)[:length] = old.reshape(-1, HKV, D)[:length]
                    getattr(mirror, arr_name)[layer] = grown
            mirror.bt = torch.arange(bucket // 16, dtype=torch.int32)[None].numpy()
        lengths = list(range(prev + 1, bucket + 1))
        sample = set(lengths[::61]) | {prev + 1, prev + 2, bucket - 1, bucket}
        sweep_bucket(pkv, runner, mirror, lengths, sample, gen, layers)
        length = bucket
        prev = bucket
    assert runner.captures == 5


def test_full_step_42_layers_bucket_8192(pkv):
    """The benchmark's launch configuration: 42 fused launches with PDL, one graph."""
    from paged_kv_decode_13_gb300.graph import DecodeGraphRunner, DecodeStep
    import workloads
    layers, bucket = 42, 8192
    w = workloads.sensenova(bucket, bucket, num_layers=layers, seed=1, device="cuda")
    sampled = (0, 21, 41)
    bt_host = torch.arange(bucket // 16, dtype=torch.int32)[None]
    mirror = Mirror([w.k[i].cpu() for i in sampled], [w.v[i].cpu() for i in sampled], bt_host)
    cache = pkv.PagedKVCache(w.k, w.v, w.block_table, bucket=bucket)
    step = DecodeStep(cache, HQ)
    runner = DecodeGraphRunner(step)
    for layer in range(layers):
        step.q[layer].copy_(w.q[layer])
        step.k_new[layer].copy_(w.k_new[layer])
        step.v_new[layer].copy_(w.v_new[layer])
    for L in (4096, 8192, 1, 777):
        si = np.array([[0, 1, 0, L]], np.int32)
        step.seq_info.copy_(torch.from_numpy(si))
        runner.step()
        torch.cuda.synchronize()
        assert int(step.err.item()) == 0
        for m, layer in enumerate(sampled):
            mirror.append(m, si, w.k_new[layer].cpu(), w.v_new[layer].cpu())
            ref, _ = mirror.attend(m, w.q[layer].cpu(), si, 1 / math.sqrt(D))
            diff = float(np.abs(U.f64(step.out[layer]) - ref).max())
            assert diff <= 2e-3, (L, layer, diff)
            flat_k = cache.k[layer].view(-1, HKV, D)
            assert torch.equal(flat_k[L - 1].cpu(), w.k_new[layer][0].cpu())
    assert runner.captures == 1


def test_graph_pool_does_not_grow_across_requests(pkv):
    from paged_kv_decode_13_gb300.graph import DecodeGraphRunner, DecodeStep
    reserved = []
    for it in range(8):
        cache = pkv.PagedKVCache.allocate(4, HKV, D, 1024)
        runner = DecodeGraphRunner(DecodeStep(cache, HQ))
        runner.step_bufs.seq_info.copy_(torch.tensor([[0, 1, 0, 100 + it]], dtype=torch.int32))
        runner.step()
        torch.cuda.synchronize()
        del runner, cache
        torch.cuda.synchronize()
        reserved.append(torch.cuda.memory_reserved())
    # After the first requests have warmed the allocator, memory stays level.
    assert reserved[-1] <= reserved[2], reserved


def test_batched_left_padding_one_capture(pkv):
    """A batched step over a left-padded batch: one capture, replayed while the
    lengths grow and each sequence's first valid position changes (the graph
    holds the descriptor's pointer, the values are read at run time)."""
    from paged_kv_decode_13_gb300.graph import DecodeGraphRunner, DecodeStep
    import workloads
    S = 4
    base = np.array([1500, 300, 1900, 40])
    w = workloads.batched(S=S, max_len=2048, seed=5, lengths=base.tolist())
    dev = torch.device("cuda")
    fv = torch.zeros(S, dtype=torch.int32, device=dev)
    cache = pkv.PagedKVCache([t.to(dev) for t in w.k], [t.to(dev) for t in w.v], w.block_table.to(dev),
                             bucket=w.bucket, first_valid=fv)
    step = DecodeStep(cache, w.q_heads, rows=S, num_segments=S, max_kv=w.bucket)
    runner = DecodeGraphRunner(step)
    kp = w.k[0].view(torch.int16).numpy().copy()
    vp = w.v[0].view(torch.int16).numpy().copy()
    bt = w.block_table.numpy()
    gen = torch.Generator().manual_seed(3)
    firsts = ([0, 0, 0, 0], [700, 299, 1950, 10], [1501, 0, 100, 41], [3, 150, 1901, 0])
    for it, first in enumerate(firsts):
        si = np.array([[s, 1, s, base[s] + it] for s in range(S)], np.int32)
        q = torch.randn(S, w.q_heads, D, generator=gen).to(torch.bfloat16)
        kn = (torch.randn(S, w.kv_heads, D, generator=gen) / math.sqrt(D)).to(torch.bfloat16)
        vn = (torch.randn(S, w.kv_heads, D, generator=gen) / math.sqrt(D)).to(torch.bfloat16)
        step.seq_info.copy_(torch.from_numpy(si))
        step.q[0].copy_(q)
        step.k_new[0].copy_(kn)
        step.v_new[0].copy_(vn)
        fv.copy_(torch.tensor(first, dtype=torch.int32))
        runner.step()
        torch.cuda.synchronize()
        assert int(step.err.item()) == 0
        assert O.append(kp, vp, bt, si, kn.view(torch.int16).numpy(), vn.view(torch.int16).numpy()) == 0
        kpf = torch.from_numpy(kp).view(torch.bfloat16).double().numpy()
        vpf = torch.from_numpy(vp).view(torch.bfloat16).double().numpy()
        ref, _, e = O.attend(q.double().numpy(), kpf, vpf, bt, si, step.scale,
                             first_valid=np.array(first, np.int32))
        assert e == 0
        diff = float(np.abs(U.f64(step.out[0]) - ref).max())
        assert diff <= 2e-3, (it, diff)
    assert runner.captures == 1


def test_replays_advance_lengths_on_the_device(pkv):
    """DecodeStep(advance=True): the segment table is written once by the host;
    each replay appends and attends at the current length and then moves
    kv_end on by q_len on the device (tiny-llm kv_cache.py, SlotKVCache.end_step).
    N replays with only q / k_new / v_new copied in match N oracle steps on a
    host mirror whose lengths the test advances itself, and the table reads
    back kv_end + N."""
    from paged_kv_decode_13_gb300.graph import DecodeGraphRunner, DecodeStep
    layers, bucket, L0, N = 2, 1024, 990, 34    # crosses two page boundaries, ends at the bucket edge
    gen = torch.Generator().manual_seed(11)
    cache = pkv.PagedKVCache.allocate(layers, HKV, D, bucket)
    host = [(torch.randn(t.shape, generator=gen) / math.sqrt(D)).to(torch.bfloat16) for t in cache.k + cache.v]
    for t, h in zip(cache.k + cache.v, host):
        t.copy_(h)
    mirror = Mirror(host[:layers], host[layers:], torch.arange(bucket // 16, dtype=torch.int32)[None])
    step = DecodeStep(cache, HQ, advance=True)
    runner = DecodeGraphRunner(step)
    assert step.launch_count() == layers + 1
    step.seq_info.copy_(torch.tensor([[0, 1, 0, L0]], dtype=torch.int32))
    for n in range(N):
        qs = [torch.randn(1, HQ, D, generator=gen).to(torch.bfloat16) for _ in range(layers)]
        ks = [(torch.randn(1, HKV, D, generator=gen) / math.sqrt(D)).to(torch.bfloat16) for _ in range(layers)]
        vs = [(torch.randn(1, HKV, D, generator=gen) / math.sqrt(D)).to(torch.bfloat16) for _ in range(layers)]
        # one host -> device copy of the step's rows; the segment table is not written
        host_in = torch.cat([t.view(torch.uint8).reshape(-1) for t in qs + ks + vs])
        assert host_in.numel() == step.step_inputs.numel()
        step.step_inputs.copy_(host_in)
        runner.step()
        torch.cuda.synchronize()
        si = np.array([[0, 1, 0, L0 + n]], np.int32)   # the host's own copy of the lengths
        for layer in range(layers):
            mirror.append(layer, si, ks[layer], vs[layer])
            ref, _ = mirror.attend(layer, qs[layer], si, step.scale)
            diff = float(np.abs(U.f64(step.out[layer]) - ref).max())
            assert diff <= 2e-3, (n, layer, diff)
    assert int(step.err.item()) == 0
    assert step.seq_info.cpu().tolist() == [[0, 1, 0, L0 + N]]
    assert runner.captures == 1
    # the pools hold exactly the mirror's appended rows
    for layer in range(layers):
        assert U.pool_bytes(cache.k[layer]) == mirror.k[layer].tobytes()
        assert U.pool_bytes(cache.v[layer]) == mirror.v[layer].tobytes()
