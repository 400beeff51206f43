"""mla_decode_noalloc (the entry point for callers that cannot allocate device memory)
against mla_decode (the entry point with a caller-provided workspace).

Such callers, e.g. code inside a framework that owns all device memory through its own
allocator, get their scratch from the library's fixed device array instead of a
workspace.  Both entry points must give the same answer; the array keeps the previous
call's contents, so every case is run twice in a row.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import mla_inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pm():
    import paged_mla_latent_gb300 as m
    return m


def _both(pm, case, splits):
    n_tok, H = case.q.shape[0], case.q.shape[1]
    args = (case.q, case.kv)
    tail = (case.qo_indptr, case.kv_indptr, case.kv_indices, case.kv_last_page_lens,
            case.max_seqlen_q, case.sm_scale, case.q_scale, case.kv_scale)
    o_ref = torch.empty((n_tok, H, 512), dtype=torch.bfloat16, device="cuda")
    l_ref = torch.empty((n_tok, H), dtype=torch.float32, device="cuda")
    ws = pm.make_workspace(case.B, H, case.max_seqlen_q, splits, "cuda")
    pm.mla_decode(*args, o_ref, *tail, num_kv_splits=splits, lse_out=l_ref, workspace=ws)
    outs = []
    for _ in range(2):   # two calls in a row on the shared scratch array
        o = torch.full((n_tok, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((n_tok, H), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        pm.mla_decode_noalloc(*args, o, *tail, num_kv_splits=splits, lse_out=lse, error_out=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append((o, lse))
    assert pm.mla_check_error(ws) == 0
    return (o_ref, l_ref), outs


@pytest.mark.parametrize("splits", [0, 1, 3])
def test_noalloc_matches_workspace_entry_point(pm, splits):
    case = gu.to_device(mla_inputs.make_custom([1500, 333, 2049, 1], q_lens=[1, 1, 4, 1], H=12,
                                               seed=21, q_scale=1.0, kv_scale=1.0))
    (o_ref, l_ref), outs = _both(pm, case, splits)
    ref = o_ref.float().cpu().numpy().astype(np.float64)
    for o, lse in outs:
        got = o.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert (np.abs(got - ref) <= gu.O_ATOL + gu.O_RTOL * np.abs(ref)).all()
        assert (np.abs(lse.cpu().numpy() - l_ref.cpu().numpy()) <= gu.LSE_ATOL).all()


def test_noalloc_tiny_workload(pm):
    case = gu.to_device(mla_inputs.make_case("tiny", seed=2))
    (o_ref, l_ref), outs = _both(pm, case, 0)
    for o, lse in outs:
        assert torch.allclose(o.float(), o_ref.float(), atol=gu.O_ATOL, rtol=gu.O_RTOL)
        assert torch.allclose(lse, l_ref, atol=gu.LSE_ATOL)


def test_noalloc_rejects_calls_larger_than_its_array(pm):
    # 96 heads x 64 requests with automatic splitting needs far more than the fixed array
    case = gu.to_device(mla_inputs.make_custom([200] * 64, H=96, seed=22))
    need = pm.mla_get_workspace_size(case.B, 96, 1, 0)
    assert need > (16 << 20)
    o = torch.empty((64, 96, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pm.MlaError) as e:
        pm.mla_decode_noalloc(case.q, case.kv, o, case.qo_indptr, case.kv_indptr,
                              case.kv_indices, case.kv_last_page_lens, 1, case.sm_scale,
                              case.q_scale, case.kv_scale)
    assert e.value.status == 3   # MLA_ERR_WORKSPACE_TOO_SMALL
