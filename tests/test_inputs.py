"""The seeded input builders (CPU): what the parity tests and the bench rely on about their
shapes, index structure and poisoning."""
import numpy as np
import pytest
import torch

import mla_inputs


def _pages_of(case, b):
    s, e = int(case.kv_indptr[b]), int(case.kv_indptr[b + 1])
    return case.kv_indices[s:e].tolist()


@pytest.mark.parametrize("page_size", [2, 16, 128])
def test_paged_lengths_and_last_pages(page_size):
    lens = [1, page_size, page_size + 1, 5 * page_size - 3, 0, 1000]
    case = mla_inputs.make_paged(lens, H=12, page_size=page_size, seed=3)
    assert case.kv.shape[1:] == (page_size, 1, 576) and case.kv.dtype == torch.uint8
    for b, L in enumerate(lens):
        n = int(case.kv_indptr[b + 1] - case.kv_indptr[b])
        last = int(case.kv_last_page_lens[b])
        assert n == (L + page_size - 1) // page_size
        if n:
            assert 1 <= last <= page_size and (n - 1) * page_size + last == L
    assert case.meta["page_size"] == page_size
    assert int(case.kv_indptr[-1]) <= case.kv_indices.numel()


def test_paged_pages_are_distinct_except_the_shared_prefix():
    ps, P = 64, 2048
    lens = [P + 100 * i + 7 for i in range(6)]
    case = mla_inputs.make_paged(lens, H=12, page_size=ps, seed=4, shared_prefix=P)
    lead = _pages_of(case, 0)[:P // ps]
    seen = set(lead)
    for b in range(len(lens)):
        pages = _pages_of(case, b)
        assert pages[:P // ps] == lead                     # the prefix's whole pages shared
        own = pages[P // ps:]
        assert not (set(own) & seen)                       # every other page its own
        seen |= set(own)
        assert all(0 <= p < case.kv.shape[0] for p in pages)
    with pytest.raises(ValueError):
        mla_inputs.make_paged(lens, page_size=ps, shared_prefix=P + 1)


def test_paged_poison_marks_exactly_the_unattended_slots():
    ps = 16
    lens = [37, 16, 5]
    case = mla_inputs.make_paged(lens, H=12, page_size=ps, seed=5, poison=True, index_buffer=40)
    kv = case.kv.reshape(case.kv.shape[0], ps, 576)
    used = np.zeros((case.kv.shape[0], ps), dtype=bool)
    for b, L in enumerate(lens):
        for j in range(L):
            used[_pages_of(case, b)[j // ps], j % ps] = True
    nan_rows = (kv == mla_inputs.POISON_FP8).all(dim=2).numpy()
    assert not nan_rows[used].any()
    assert nan_rows[~used].all()
    tail = case.kv_indices[int(case.kv_indptr[-1]):]
    assert tail.numel() == 40 - int(case.kv_indptr[-1]) and (tail >= case.kv.shape[0]).all()


def test_paged_workloads_follow_the_token_workloads():
    # c16p128 takes c16's lengths (the same length draw) and its pool in 128-token pages;
    # the full builds hold 3 GB each, so the check reads the recipe's parts
    lens = mla_inputs._shared_prefix_lens(16, 0)
    assert len(lens) == 16 and all(63_911 + 4_089 <= L < 63_911 + 4_089 + 350 for L in lens)
    assert 41_280 * 128 == 5_283_840 and 63_872 == 499 * 128 <= 63_911
    lp = mla_inputs.make_case("longp128")
    assert lp.kv_lens == [142000] and int(lp.kv_indptr[-1]) == 1110
    assert int(lp.kv_last_page_lens[0]) == 48


def test_vproj_inputs():
    o, w = mla_inputs.make_vproj(16, 12, seed=1)
    assert o.shape == (16, 12, 512) and w.shape == (12, 512, 128)
    assert o.dtype == w.dtype == torch.bfloat16
    assert 0.9 < float(o.float().std()) < 1.1
    assert abs(float(w.float().std()) * 512 ** 0.5 - 1.0) < 0.05
    o2, w2 = mla_inputs.make_vproj(16, 12, seed=1)
    assert torch.equal(o, o2) and torch.equal(w, w2)
