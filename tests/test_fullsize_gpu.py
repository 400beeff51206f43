"""Full-size workloads, in the launch configuration bench.py times (automatic split-KV,
bf16 o, fp32 lse, CUDA stream of the caller), checked on sampled outputs the oracle
computes one by one, and on properties that hold at any size.
"""
import numpy as np
import pytest
import torch

import mla_inputs
import oracle
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def pm():
    import paged_mla_latent_gb300 as m
    return m


def _run(pm, case, shared_prefix=None):
    n_tok, H = case.q.shape[0], case.q.shape[1]
    o = torch.full((n_tok, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((n_tok, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = pm.make_workspace(case.B, H, case.max_seqlen_q, 0, "cuda",
                           shared_prefix=shared_prefix is not None)
    if shared_prefix is None:
        pm.mla_decode(case.q, case.kv, o, case.qo_indptr, case.kv_indptr, case.kv_indices,
                      case.kv_last_page_lens, case.max_seqlen_q, case.sm_scale, case.q_scale,
                      case.kv_scale, lse_out=lse, workspace=ws)
    else:
        pm.mla_decode_shared_prefix(case.q, case.kv, o, case.qo_indptr, case.kv_indptr,
                                    case.kv_indices, case.kv_last_page_lens, case.max_seqlen_q,
                                    case.sm_scale, case.q_scale, case.kv_scale, shared_prefix,
                                    lse_out=lse, workspace=ws)
    torch.cuda.synchronize()
    assert pm.mla_check_error(ws) == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    return o, lse


def _check_samples(case, o, lse, samples):
    ref = gu.oracle_sampled(case, samples)
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    for r, h, o_ref, lse_ref in ref:
        d = np.abs(og[r, h] - o_ref)
        assert (d <= gu.O_ATOL + gu.O_RTOL * np.abs(o_ref)).all(), (r, h, float(d.max()))
        assert abs(lg[r, h] - lse_ref) <= gu.LSE_ATOL, (r, h, lg[r, h], lse_ref)


@pytest.mark.parametrize("name", ["c16", "c24"])
@pytest.mark.parametrize("scales", [(0.05, 0.1), (1.0, 1.0)])
@pytest.mark.parametrize("entry", ["plain", "shared_prefix"])
def test_shared_prefix_workloads_sampled(pm, name, scales, entry):
    case = mla_inputs.make_case(name, seed=0, device="cuda", q_scale=scales[0], kv_scale=scales[1])
    o, lse = _run(pm, case, case.meta["shared_prefix"] if entry == "shared_prefix" else None)
    B = case.B
    _check_samples(case, o, lse, [(0, 0, 0), (0, 0, 11), (B // 2, 0, 5), (B - 1, 0, 7)])


@pytest.mark.parametrize("scales", [(0.05, 0.1), (1.0, 1.0)])
def test_long_context_sampled(pm, scales):
    case = mla_inputs.make_case("long", seed=0, device="cuda", q_scale=scales[0], kv_scale=scales[1])
    o, lse = _run(pm, case)
    _check_samples(case, o, lse, [(0, 0, h) for h in (0, 3, 6, 11)])


def test_mtp_causal_sampled(pm):
    case = mla_inputs.make_case("mtp", seed=0, device="cuda", q_scale=1.0, kv_scale=1.0)
    o, lse = _run(pm, case)
    _check_samples(case, o, lse, [(0, 0, 0), (0, 3, 0), (17, 1, 4), (63, 3, 11), (63, 0, 2)])


def test_context_shard_merge_full_size(pm):
    """8 context shards of 17,750 positions, 96 heads per shard call, merged by
    mla_merge_partials, equals the unsplit 96-head call and the oracle."""
    case = mla_inputs.make_case("long96", seed=0, device="cuda", q_scale=1.0, kv_scale=1.0)
    o_full, lse_full = _run(pm, case)
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
    _check_samples(case, o, lse, [(0, 0, h) for h in (0, 47, 48, 95)])
