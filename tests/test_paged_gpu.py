"""Parity of the CUDA decode path with the FP64 oracle on caches of several tokens a page.

kv is (n_pages, page_size, 1, 576); kv_indptr counts pages and kv_last_page_lens gives the
fill of each request's last page ("Scaling Kimi K3 on AMD Instinct MI355X", §4.1 argument
list; the page axis is the one the paged-attention reading of the cache gives).  Cases span
several tiles, ragged last pages, poisoned unattended slots, causal drafts, split policies
and the shared-prefix entry point, which runs its plain path on such caches.
"""
import numpy as np
import pytest
import torch

import mla_inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

LENS = [1000, 2500, 130, 1, 257, 64, 65, 1024, 3001]


@pytest.fixture(scope="module")
def pm():
    import paged_mla_latent_gb300 as m
    return m


def _check(case, **kw):
    case = gu.to_device(case)
    o, lse, status = gu.run_gpu(case, **kw)
    assert status == 0, f"device error {status}"
    o_ref, lse_ref = gu.run_oracle(case)
    return gu.compare(o, lse, o_ref, lse_ref, what=case.name)


@pytest.mark.parametrize("page_size", [2, 16, 64, 128, 1024])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_page_sizes_ragged_last_pages(pm, page_size, splits):
    case = mla_inputs.make_paged(LENS, H=12, page_size=page_size, seed=page_size + splits,
                                 q_scale=1.0, kv_scale=1.0, poison=True,
                                 name=f"ps{page_size}")
    _check(case, num_kv_splits=splits)


@pytest.mark.parametrize("page_size", [16, 64])
@pytest.mark.parametrize("scales", [(0.05, 0.1), (1.0, 1.0)])
def test_paged_causal_drafts(pm, page_size, scales):
    case = mla_inputs.make_paged([700, 1300, 5, 64, 129], q_lens=[2, 4, 1, 3, 4], H=12,
                                 page_size=page_size, seed=21, q_scale=scales[0],
                                 kv_scale=scales[1], poison=True, name="paged-drafts")
    _check(case)


@pytest.mark.parametrize("H", [16, 96])
def test_paged_head_counts(pm, H):
    case = mla_inputs.make_paged([900, 33, 2048], H=H, page_size=32, seed=H, q_scale=1.0,
                                 kv_scale=1.0, poison=True, name=f"paged-h{H}")
    _check(case)


def test_paged_fp32_output(pm):
    case = mla_inputs.make_paged([640, 17], H=12, page_size=16, seed=5, q_scale=1.0,
                                 kv_scale=1.0, name="paged-fp32")
    _check(case, o_dtype=torch.float32)


def test_paged_index_buffer_tail(pm):
    """kv_indices longer than kv_indptr[B], its tail pointing past the pool: never read."""
    case = mla_inputs.make_paged([300, 1200], H=12, page_size=64, seed=8, poison=True,
                                 index_buffer=200, name="paged-tail")
    _check(case)


@pytest.mark.parametrize("page_size,call_prefix", [(64, 2048), (64, 2000), (128, 2048),
                                                   (16, 1030), (1024, 2048)])
@pytest.mark.parametrize("scales", [(0.05, 0.1), (1.0, 1.0)])
def test_shared_prefix_cascade_on_pages(pm, page_size, call_prefix, scales):
    """The cascade over whole shared pages: the prefix units take the largest whole number
    of pages within the declared prefix (2000 -> 31 pages of 64; 1030 -> 64 pages of 16)
    and each request's own units the rest, last page ragged; results as the oracle."""
    case = mla_inputs.make_paged([2048 + 100 * i + 7 for i in range(16)], H=12,
                                 page_size=page_size, seed=11 + page_size,
                                 q_scale=scales[0], kv_scale=scales[1], poison=True,
                                 shared_prefix=2048, name=f"paged-shared{page_size}")
    _check(case, shared_prefix=call_prefix)


@pytest.mark.parametrize("q_len", [1, 2, 4])
def test_shared_prefix_cascade_on_pages_with_drafts(pm, q_len):
    lens = [4096 + 61 * i + q_len for i in range(9)]
    case = mla_inputs.make_paged(lens, q_lens=[q_len] * 9, H=12, page_size=128, seed=40 + q_len,
                                 q_scale=1.0, kv_scale=1.0, poison=True, shared_prefix=4096,
                                 name=f"paged-shared-drafts{q_len}")
    _check(case, shared_prefix=4096)


def test_shared_prefix_below_a_page_runs_plain(pm):
    """A declared prefix of less than one whole page (1000 positions of 1024-token pages)
    leaves the cascade nothing to share: the plain decode runs, same results."""
    case = mla_inputs.make_paged([3000 + 9 * i for i in range(8)], H=12, page_size=1024,
                                 seed=12, q_scale=1.0, kv_scale=1.0, poison=True,
                                 shared_prefix=2048, name="paged-shared-small")
    _check(case, shared_prefix=1000)


def test_padded_page_and_slot_pitch(pm):
    """kv as a view of a wider buffer: slots 640 bytes apart and one spare slot a page."""
    case = gu.to_device(mla_inputs.make_paged([900, 130, 1], H=12, page_size=16, seed=13,
                                              q_scale=1.0, kv_scale=1.0, name="paged-pitch"))
    n_pages = case.kv.shape[0]
    wide = torch.zeros((n_pages, 17, 1, 640), dtype=torch.uint8, device="cuda")
    wide[:, :16, :, :576] = case.kv
    view = wide[:, :16, :, :576]
    o, lse, status = gu.run_gpu(case, kv_view=view)
    assert status == 0
    o_ref, lse_ref = gu.run_oracle(case)
    gu.compare(o, lse, o_ref, lse_ref, what=case.name)


@pytest.mark.parametrize("page_size", [16, 128])
def test_paged_equals_token_view_bitwise(pm, page_size):
    """With one piece per (request, row group) the paged call and a one-token-a-page call
    over the same rows run the same tiles: outputs agree bit for bit."""
    case = gu.to_device(mla_inputs.make_paged([1500, 77, 2049], q_lens=[1, 3, 2], H=12,
                                              page_size=page_size, seed=17, q_scale=1.0,
                                              kv_scale=1.0, name="paged-vs-token"))
    o_p, lse_p, st = gu.run_gpu(case, num_kv_splits=1)
    assert st == 0
    kvp = case.kv_indptr.cpu().numpy()
    last = case.kv_last_page_lens.cpu().numpy()
    pages = case.kv_indices.cpu().numpy()
    tok_ids, tok_ptr = [], [0]
    for b in range(case.B):
        pg = pages[kvp[b]:kvp[b + 1]].astype(np.int64)
        L = (len(pg) - 1) * page_size + int(last[b]) if len(pg) else 0
        ids = (pg[:, None] * page_size + np.arange(page_size)[None, :]).reshape(-1)[:L]
        tok_ids.append(ids)
        tok_ptr.append(tok_ptr[-1] + L)
    flat = case.kv.reshape(-1, 1, 1, 576)
    tok = mla_inputs.Case(**{**case.__dict__})
    tok.kv = flat
    tok.kv_indices = torch.tensor(np.concatenate(tok_ids).astype(np.int32), device="cuda")
    tok.kv_indptr = torch.tensor(np.array(tok_ptr, dtype=np.int32), device="cuda")
    tok.kv_last_page_lens = torch.ones(case.B, dtype=torch.int32, device="cuda")
    tok.meta = {**case.meta, "page_size": 1}
    o_t, lse_t, st = gu.run_gpu(tok, num_kv_splits=1)
    assert st == 0
    assert torch.equal(o_p.view(torch.int16), o_t.view(torch.int16))
    assert torch.equal(lse_p, lse_t)


def test_paged_empty_request(pm):
    """A request with no pages: zero output and lse -inf; its neighbours as the oracle."""
    case = gu.to_device(mla_inputs.make_paged([0, 400, 0], H=12, page_size=64, seed=14,
                                              poison=True))
    for splits in (0, 1, 4):
        o, lse, st = gu.run_gpu(case, num_kv_splits=splits, o_dtype=torch.float32)
        assert st == 0
        assert torch.equal(o[0], torch.zeros_like(o[0])) and torch.equal(o[2], torch.zeros_like(o[2]))
        assert torch.isneginf(lse[0]).all() and torch.isneginf(lse[2]).all()
        one = mla_inputs.Case(**{**case.__dict__})
        one.q, one.kv_lens, one.q_lens = case.q[1:2], [400], [1]
        one.qo_indptr = torch.tensor([0, 1], dtype=torch.int32)
        base = int(case.kv_indptr[1])
        one.kv_indptr = case.kv_indptr[1:3].cpu() - base
        one.kv_indices = case.kv_indices[base:].cpu()
        one.kv_last_page_lens = case.kv_last_page_lens[1:2].cpu()
        o_ref, lse_ref = gu.run_oracle(one)
        gu.compare(o[1:2], lse[1:2], o_ref, lse_ref, what="paged-empty")


def test_paged_validate(pm):
    case = gu.to_device(mla_inputs.make_paged([500, 300], q_lens=[1, 2], H=12, page_size=64,
                                              seed=16))
    ws = pm.make_workspace(case.B, 12, 2, 0, "cuda")
    args = (case.q, case.kv, case.qo_indptr, case.kv_indptr, case.kv_indices)
    assert pm.mla_validate(*args, case.kv_last_page_lens, ws) == 0
    for v in (0, 65, -3):
        bad = case.kv_last_page_lens.clone()
        bad[1] = v
        assert pm.mla_validate(*args, bad, ws) == 7, v
    # one page holding one token against a two-token query
    short_ptr = torch.tensor([0, 8, 9], dtype=torch.int32, device="cuda")
    one = torch.tensor([52, 1], dtype=torch.int32, device="cuda")
    assert pm.mla_validate(case.q, case.kv, case.qo_indptr, short_ptr, case.kv_indices,
                           one, ws) == 7
