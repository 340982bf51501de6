"""The paged-pool builder used by the tests and the bench: every key and
value lands in the page and slot the page table names, and no page is used
twice. Host only."""
import torch

from gqa_attention_softmax_gb300 import workloads


def test_to_paged_places_every_key_where_the_page_table_says():
    Hkv, P = 2, 16
    inp = workloads.explicit_inputs([5, 0, 40, 1], [70, 0, 40, 33], 8, Hkv, 64, seed=1)
    pg = workloads.to_paged(inp, Hkv, P, seed=3, spare_pages=2)
    ind = pg["page_indptr"].tolist()
    idx = pg["page_indices"].tolist()
    cu = inp["cu_k"].tolist()
    assert ind == [0, 5, 5, 8, 11]
    assert len(set(idx)) == len(idx) and all(0 <= i < pg["k_pages"].shape[0] for i in idx)
    assert pg["k_pages"].shape == (13, Hkv, P, 64)
    for b, L in enumerate(inp["kv_lens"]):
        blk_k = inp["k"][Hkv * cu[b]:Hkv * cu[b + 1]].view(Hkv, L, 64)
        blk_v = inp["v"][Hkv * cu[b]:Hkv * cu[b + 1]].view(Hkv, L, 64)
        for t in range(L):
            page = idx[ind[b] + t // P]
            assert torch.equal(pg["k_pages"][page, :, t % P], blk_k[:, t])
            assert torch.equal(pg["v_pages"][page, :, t % P], blk_v[:, t])


def test_to_paged_fills_unused_slots_with_large_finite_values():
    inp = workloads.explicit_inputs([3], [3], 4, 1, 64, seed=2)
    pg = workloads.to_paged(inp, 1, 16, seed=0, spare_pages=1)
    page = pg["page_indices"][0].item()
    tail = pg["k_pages"][page, 0, 3:].float()
    assert torch.isfinite(tail).all() and tail.abs().max() > 50
