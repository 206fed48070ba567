"""The seeded input generator shared by the oracle and the CUDA path: draws are
reproducible, chunking never changes an input (the draw order depends only on
the prompt length), and the named workloads have the shapes of their
definitions (prefix pooled rows = offset / ratio, the 127 raw window rows)."""
import torch

from deepseek_v4_sparse_ratio_gb300 import inputs


def test_draws_are_reproducible():
    a = inputs.draw(inputs.small(5, [37, 11], index_topk=8))
    b = inputs.draw(inputs.small(5, [37, 11], index_topk=8))
    for key in a.t:
        assert torch.equal(a.t[key], b.t[key]), key


def test_chunking_never_changes_an_input():
    whole = inputs.draw(inputs.small(9, [48], index_topk=8))
    for chunks in ([10, 6, 32], [1] * 48, [47, 1]):
        cut = inputs.draw(inputs.small(9, chunks, index_topk=8))
        for key in ("raw_ik", "raw_kv", "q_idx", "w", "q"):
            assert torch.equal(whole.t[key], cut.t[key]), (chunks, key)


def test_named_workload_shapes():
    for name in inputs.WORKLOADS + inputs.COMPRESSED_WORKLOADS + inputs.SHORT_WORKLOADS:
        wl = inputs.workload(name)
        assert wl.off0 % wl.ratio == 0 or wl.off0 == 0, name
        assert wl.prefix_pooled == wl.off0 // wl.ratio, name
        assert wl.index_topk > 0 and wl.window == 128, name
    wl = inputs.draw(inputs.workload("band_128k"))
    L, P = wl.total, wl.prefix_pooled
    assert wl.t["q_idx"].shape == (L, 64, 128) and wl.t["q"].shape == (L, 64, 512)
    assert wl.t["raw_kv"].shape == (L, 512) and wl.t["raw_ik"].shape == (L, 128)
    assert wl.t["w"].dtype == torch.float32 and wl.t["q"].dtype == torch.bfloat16
    assert wl.t["prefix_kv"].shape == (P, 512) and wl.t["prefix_ik"].shape == (P, 128)
    assert wl.t["prefix_win"].shape == (127, 512)
