"""DecodeStep's static buffers, checked on the CPU: the per-layer inputs and
outputs are 16-byte aligned, non-overlapping views of one input and one
output buffer, in the documented order."""
import pytest
import torch


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_13_gb300 as m
    return m


@pytest.mark.parametrize("rows,segs,with_lse", [(1, 1, False), (5, 3, True)])
def test_step_buffers_are_views_of_one_buffer(pkv, rows, segs, with_lse):
    from paged_kv_decode_13_gb300.graph import DecodeStep
    L, Hkv, D, Hq = 3, 2, 72, 8
    k = [torch.zeros(4, 16, Hkv, D, dtype=torch.bfloat16) for _ in range(L)]
    v = [torch.zeros(4, 16, Hkv, D, dtype=torch.bfloat16) for _ in range(L)]
    cache = pkv.PagedKVCache(k, v, torch.zeros(2, 4, dtype=torch.int32))
    st = DecodeStep(cache, Hq, rows=rows, num_segments=segs, with_lse=with_lse)
    ins = st.q + st.k_new + st.v_new + [st.seq_info]
    outs = st.out + (st.lse if with_lse else [])
    for buf, views in ((st.inputs, ins), (st.outputs, outs)):
        base, end = buf.data_ptr(), buf.data_ptr() + buf.numel()
        spans = []
        for t in views:
            a = t.data_ptr()
            assert a % 16 == 0 and base <= a and a + t.numel() * t.element_size() <= end
            assert t.is_contiguous()
            spans.append((a, a + t.numel() * t.element_size()))
        assert spans == sorted(spans)                       # layer order, q then k_new then v_new then table
        assert all(e <= s for (_, e), (s, _) in zip(spans, spans[1:]))  # no overlap
    assert st.q[0].shape == (rows, Hq, D) and st.k_new[0].shape == (rows, Hkv, D)
    assert st.seq_info.shape == (segs, 4) and st.seq_info.dtype == torch.int32
    assert st.out[0].dtype == torch.float32 and (not with_lse or st.lse[0].shape == (rows, Hq))
    # writing through a view lands in the shared buffer
    st.k_new[1].fill_(1.0)
    # (bf16 1.0 is 0x3f80: both bytes nonzero)
    assert int(st.inputs.count_nonzero()) == rows * Hkv * D * 2
