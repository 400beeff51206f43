"""Full-size workloads, in the launch configuration bench.py times (automatic split-KV,
bf16 o, fp32 lse, CUDA stream of the caller), checked against the oracle on every query
token and head of every request the test names: every request of the concurrency-16/24
batches (so every slot of every shared-prefix group: 96 rows, 8 requests x 12 heads), all
12 heads of the 142K-position request unsplit and split, all drafts and heads of the shortest, the longest and
four more multi-token requests, and all 96 heads of the 8-shard merge.
"""
import functools

import numpy as np
import pytest
import torch

import mla_inputs
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def pm():
    import paged_mla_latent_gb300 as m
    return m


def _run(pm, case, shared_prefix=None, num_kv_splits=0):
    n_tok, H = case.q.shape[0], case.q.shape[1]
    o = torch.full((n_tok, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((n_tok, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = pm.make_workspace(case.B, H, case.max_seqlen_q, num_kv_splits, "cuda",
                           shared_prefix=shared_prefix is not None)
    if shared_prefix is None:
        pm.mla_decode(case.q, case.kv, o, case.qo_indptr, case.kv_indptr, case.kv_indices,
                      case.kv_last_page_lens, case.max_seqlen_q, case.sm_scale, case.q_scale,
                      case.kv_scale, num_kv_splits=num_kv_splits, lse_out=lse, workspace=ws)
    else:
        pm.mla_decode_shared_prefix(case.q, case.kv, o, case.qo_indptr, case.kv_indptr,
                                    case.kv_indices, case.kv_last_page_lens, case.max_seqlen_q,
                                    case.sm_scale, case.q_scale, case.kv_scale, shared_prefix,
                                    lse_out=lse, workspace=ws)
    torch.cuda.synchronize()
    assert pm.mla_check_error(ws) == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    return o, lse


@functools.lru_cache(maxsize=2)
def _case_and_refs(name, scales, reqs=None):
    """A full-size workload on the device and the oracle of the named requests (all of
    them when reqs is None); cached so that both entry points check against one oracle."""
    case = mla_inputs.make_case(name, seed=0, device="cuda", q_scale=scales[0], kv_scale=scales[1])
    reqs = range(case.B) if reqs is None else reqs
    return case, gu.oracle_requests(case, reqs)


@pytest.mark.parametrize("name", ["c16", "c24"])
@pytest.mark.parametrize("scales", [(0.05, 0.1), (1.0, 1.0)])
@pytest.mark.parametrize("entry", ["plain", "shared_prefix"])
def test_shared_prefix_workloads_every_request(pm, name, scales, entry):
    case, refs = _case_and_refs(name, scales)
    assert len(refs) == case.B
    o, lse = _run(pm, case, case.meta["shared_prefix"] if entry == "shared_prefix" else None)
    gu.compare_requests(case, o, lse, refs, what=f"{name} {entry} {scales}")


@pytest.mark.parametrize("scales", [(0.05, 0.1), (1.0, 1.0)])
@pytest.mark.parametrize("splits", [0, 1])
def test_long_context_all_heads(pm, scales, splits):
    """The 142K-position request decoded split (automatic) and unsplit, all 12 heads."""
    case, refs = _case_and_refs("long", scales)
    o, lse = _run(pm, case, num_kv_splits=splits)
    gu.compare_requests(case, o, lse, refs, what=f"long splits={splits} {scales}")


def test_mtp_causal_requests(pm):
    """All 4 drafts x 12 heads of the shortest, the longest and four other requests."""
    case = mla_inputs.make_case("mtp", seed=0, device="cuda", q_scale=1.0, kv_scale=1.0)
    lens = np.asarray(case.kv_lens)
    reqs = sorted({int(lens.argmin()), int(lens.argmax()), 0, 17, 40, case.B - 1})
    refs = gu.oracle_requests(case, reqs)
    o, lse = _run(pm, case)
    gu.compare_requests(case, o, lse, refs, what="mtp")


def test_context_shard_merge_full_size(pm):
    """8 context shards of 17,750 positions, 96 heads per shard call, merged by
    mla_merge_partials, equals the unsplit 96-head call and the oracle on all 96 heads."""
    case = mla_inputs.make_case("long96", seed=0, device="cuda", q_scale=1.0, kv_scale=1.0)
    refs = gu.oracle_requests(case, [0])
    o_full, lse_full = _run(pm, case)
    gu.compare_requests(case, o_full, lse_full, refs, what="long96 unsplit call")
    shards = mla_inputs.shard_views(case, 8)
    assert all(lens == [17750] for _, _, lens in shards)
    o_parts = torch.empty((8, 96, 512), dtype=torch.float32, device="cuda")
    lse_parts = torch.empty((8, 96), dtype=torch.float32, device="cuda")
    ws = pm.make_workspace(1, 96, 1, 0, "cuda")
    for s, (ip, idx, _) in enumerate(shards):
        pm.mla_decode(case.q, case.kv, o_parts[s:s + 1], case.qo_indptr, ip, idx,
                      case.kv_last_page_lens, 1, case.sm_scale, case.q_scale, case.kv_scale,
                      lse_out=lse_parts[s:s + 1], workspace=ws)
    o = torch.empty((1, 96, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 96), dtype=torch.float32, device="cuda")
    pm.mla_merge_partials(o_parts, lse_parts, torch.tensor([0, 8], dtype=torch.int32, device="cuda"),
                          torch.arange(8, dtype=torch.int32, device="cuda"), o, lse)
    torch.cuda.synchronize()
    assert pm.mla_check_error(ws) == 0
    assert torch.allclose(o.float(), o_full.float(), atol=1e-2, rtol=1e-2)
    assert torch.allclose(lse, lse_full, atol=1e-3)
    gu.compare_requests(case, o, lse, refs, what="long96 8-shard merge")
