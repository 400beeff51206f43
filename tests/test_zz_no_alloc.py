"""mla_decode_noalloc, the decode entry point for callers that cannot allocate device
memory, against the oracle and against mla_decode (the entry point with a caller-provided
workspace).

Such callers (code inside a framework that owns all device memory through its own
allocator, or a hook handed only its input and output tensors) get their scratch from the
library's fixed device array instead of a workspace.  The array keeps the previous call's
contents, so the cases below alternate between two different batches (other lengths,
seeds and split policies) on the same array, and every result is checked against the
oracle and against the workspace entry point.  This file is collected last.
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


def _tail(case):
    return (case.qo_indptr, case.kv_indptr, case.kv_indices, case.kv_last_page_lens,
            case.max_seqlen_q, case.sm_scale, case.q_scale, case.kv_scale)


def _workspace_call(pm, case, splits):
    n_tok, H = case.q.shape[0], case.q.shape[1]
    o = torch.empty((n_tok, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((n_tok, H), dtype=torch.float32, device="cuda")
    ws = pm.make_workspace(case.B, H, case.max_seqlen_q, splits, "cuda")
    pm.mla_decode(case.q, case.kv, o, *_tail(case), num_kv_splits=splits, lse_out=lse,
                  workspace=ws)
    torch.cuda.synchronize()
    assert pm.mla_check_error(ws) == 0
    return o, lse


def _noalloc_call(pm, case, splits):
    n_tok, H = case.q.shape[0], case.q.shape[1]
    o = torch.full((n_tok, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((n_tok, H), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    pm.mla_decode_noalloc(case.q, case.kv, o, *_tail(case), num_kv_splits=splits, lse_out=lse,
                          error_out=err)
    torch.cuda.synchronize()
    return o, lse, int(err.item())


def _case_a():
    return mla_inputs.make_custom([1500, 333, 2049, 1], q_lens=[1, 1, 4, 1], H=12, seed=21,
                                  q_scale=1.0, kv_scale=1.0)


def _case_b():
    # other lengths, another seed, 16 heads and a request of 7,000 positions (many pieces)
    return mla_inputs.make_custom([7000, 129, 4096], q_lens=[2, 1, 1], H=16, seed=23,
                                  q_scale=1.0, kv_scale=1.0)


@pytest.fixture(scope="module")
def cases():
    out = []
    for make in (_case_a, _case_b):
        host = make()
        o_ref, lse_ref = gu.run_oracle(host)
        out.append((gu.to_device(host), o_ref, lse_ref))
    return out


@pytest.mark.parametrize("splits_a,splits_b", [(0, 3), (3, 0), (1, 0)])
def test_noalloc_alternating_cases_match_oracle_and_workspace_entry(pm, cases, splits_a, splits_b):
    """a, b, a, b on the shared array: each call equals the oracle and the workspace call."""
    plan = [(0, splits_a), (1, splits_b), (0, splits_a), (1, splits_b)]
    for which, splits in plan:
        case, o_ref, lse_ref = cases[which]
        o_ws, lse_ws = _workspace_call(pm, case, splits)
        o, lse, err = _noalloc_call(pm, case, splits)
        assert err == 0
        gu.compare(o, lse, o_ref, lse_ref, what=f"noalloc case {which} splits {splits}")
        got = o.float().cpu().numpy().astype(np.float64)
        ref = o_ws.float().cpu().numpy().astype(np.float64)
        assert (np.abs(got - ref) <= gu.O_ATOL + gu.O_RTOL * np.abs(ref)).all()
        assert (np.abs(lse.cpu().numpy() - lse_ws.cpu().numpy()) <= gu.LSE_ATOL).all()


def test_noalloc_tiny_workload(pm):
    host = mla_inputs.make_case("tiny", seed=2)
    o_ref, lse_ref = gu.run_oracle(host)
    case = gu.to_device(host)
    o_ws, lse_ws = _workspace_call(pm, case, 0)
    for _ in range(2):
        o, lse, err = _noalloc_call(pm, case, 0)
        assert err == 0
        gu.compare(o, lse, o_ref, lse_ref, what="noalloc tiny")
        assert torch.allclose(o.float(), o_ws.float(), atol=gu.O_ATOL, rtol=gu.O_RTOL)
        assert torch.allclose(lse, lse_ws, atol=gu.LSE_ATOL)


def test_noalloc_reports_a_bad_index_then_a_clean_call(pm, cases):
    """A row id outside the cache is skipped and flagged (no fault) in that call's
    error_out; the next clean call reports 0 (every call clears the array's error words)."""
    host = mla_inputs.make_custom([500, 300], H=12, seed=15)
    host.kv_indices[10] = host.kv.shape[0] + 123
    bad = gu.to_device(host)
    _, _, err = _noalloc_call(pm, bad, 0)
    assert err != 0
    case, o_ref, lse_ref = cases[0]
    o, lse, err = _noalloc_call(pm, case, 0)
    assert err == 0
    gu.compare(o, lse, o_ref, lse_ref, what="noalloc after a flagged call")


def test_noalloc_rejects_calls_larger_than_its_array(pm):
    # 96 heads x 64 requests with automatic splitting needs far more than the fixed array
    case = gu.to_device(mla_inputs.make_custom([200] * 64, H=96, seed=22))
    need = pm.mla_get_workspace_size(case.B, 96, 1, 0)
    assert need > (16 << 20)
    o = torch.empty((64, 96, 512), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pm.MlaError) as e:
        pm.mla_decode_noalloc(case.q, case.kv, o, *_tail(case)[:4], 1, case.sm_scale,
                              case.q_scale, case.kv_scale)
    assert e.value.status == 3   # MLA_ERR_WORKSPACE_TOO_SMALL


def test_noalloc_rejects_bad_arguments_before_enqueuing(pm, cases):
    case, _, _ = cases[0]
    n_tok, H = case.q.shape[0], case.q.shape[1]
    o_bad = torch.empty((n_tok, H, 256), dtype=torch.bfloat16, device="cuda")
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(pm.MlaError) as e:
        pm.mla_decode_noalloc(case.q, case.kv, o_bad, *_tail(case), error_out=err)
    assert e.value.status == 1   # MLA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(err.item()) == -1   # nothing was enqueued, error_out untouched
    o = torch.empty((n_tok, H, 512), dtype=torch.bfloat16, device="cuda")
    for bad_err in (torch.zeros(1, dtype=torch.int64, device="cuda"),
                    torch.zeros(1, dtype=torch.int32),
                    torch.zeros(0, dtype=torch.int32, device="cuda")):
        with pytest.raises(ValueError):
            pm.mla_decode_noalloc(case.q, case.kv, o, *_tail(case), error_out=bad_err)
