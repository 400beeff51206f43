"""mla_expand_shared_prefix_indices: the full page table of a shared-prefix batch built on
the device from the shared pages (once) and each request's own pages.  Index work, so the
result must be bit-exact: checked against the table written out in numpy, with an offset
own_indptr, empty own lists, no shared pages, a table too small for the result (entries
past its end untouched, flagged) and a decreasing own_indptr (flagged); and the decode on
an expanded table against the oracle."""
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


def _reference(shared, own_ptr, own):
    B = len(own_ptr) - 1
    S = len(shared)
    kvp = [b * S + (own_ptr[b] - own_ptr[0]) for b in range(B + 1)]
    idx = []
    for b in range(B):
        idx.extend(shared)
        idx.extend(own[own_ptr[b]:own_ptr[b + 1]])
    return np.array(kvp, dtype=np.int32), np.array(idx, dtype=np.int32)


@pytest.mark.parametrize("B,S,base", [(1, 0, 0), (1, 7, 0), (5, 1000, 3), (16, 63911, 0),
                                      (33, 129, 11), (3, 0, 5)])
def test_matches_the_table_written_out(pm, B, S, base):
    rng = np.random.default_rng(B * 100 + S)
    lens = [int(x) for x in rng.integers(0, 300, size=B)]
    if B > 1:
        lens[1] = 0                                     # a request with no own pages
    own_ptr = [base]
    for L in lens:
        own_ptr.append(own_ptr[-1] + L)
    own = rng.integers(0, 1 << 30, size=own_ptr[-1] + 4, dtype=np.int64).astype(np.int32)
    shared = rng.integers(0, 1 << 30, size=S, dtype=np.int64).astype(np.int32)
    kvp_ref, idx_ref = _reference(shared, own_ptr, own)
    dev = "cuda"
    d_sh = torch.from_numpy(shared).to(dev)
    d_ptr = torch.tensor(own_ptr, dtype=torch.int32, device=dev)
    d_own = torch.from_numpy(own).to(dev)
    d_kvp = torch.full((B + 1,), -7, dtype=torch.int32, device=dev)
    d_idx = torch.full((len(idx_ref) + 5,), -7, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pm.mla_expand_shared_prefix_indices(d_sh, d_ptr, d_own, d_kvp, d_idx, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(d_kvp.cpu().numpy(), kvp_ref)
    got = d_idx.cpu().numpy()
    assert np.array_equal(got[:len(idx_ref)], idx_ref)
    assert (got[len(idx_ref):] == -7).all()


def test_a_table_too_small_is_flagged_and_not_overrun(pm):
    dev = "cuda"
    shared = torch.arange(100, dtype=torch.int32, device=dev)
    own_ptr = torch.tensor([0, 50, 120], dtype=torch.int32, device=dev)
    own = torch.arange(1000, 1120, dtype=torch.int32, device=dev)
    need = 2 * 100 + 120
    buf = torch.full((need,), -7, dtype=torch.int32, device=dev)
    view = buf[:need - 30]                              # 30 entries short
    kvp = torch.zeros(3, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pm.mla_expand_shared_prefix_indices(shared, own_ptr, own, kvp, view, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 8
    _, idx_ref = _reference(shared.cpu().numpy(), [0, 50, 120], own.cpu().numpy())
    got = buf.cpu().numpy()
    assert np.array_equal(got[:need - 30], idx_ref[:need - 30])
    assert (got[need - 30:] == -7).all()


def test_a_decreasing_own_indptr_is_flagged(pm):
    dev = "cuda"
    shared = torch.arange(10, dtype=torch.int32, device=dev)
    own_ptr = torch.tensor([0, 40, 20], dtype=torch.int32, device=dev)
    own = torch.arange(40, dtype=torch.int32, device=dev)
    kvp = torch.zeros(3, dtype=torch.int32, device=dev)
    idx = torch.zeros(100, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pm.mla_expand_shared_prefix_indices(shared, own_ptr, own, kvp, idx, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 2


@pytest.mark.parametrize("page_size", [1, 16])
def test_decode_on_the_expanded_table(pm, page_size):
    """A shared-prefix batch: its page table in compact form, expanded on the device, then
    mla_decode_shared_prefix on the result against the oracle on the original table."""
    lens = [2048 + 37 * i + 5 for i in range(9)]
    P = 2048
    if page_size == 1:
        case = mla_inputs.make_custom(lens, H=12, seed=61, shared_prefix=P, q_scale=1.0,
                                      kv_scale=1.0, name="expand")
    else:
        case = mla_inputs.make_paged(lens, H=12, page_size=page_size, seed=62, shared_prefix=P,
                                     q_scale=1.0, kv_scale=1.0, name="expand-paged")
    case = gu.to_device(case)
    S = P // page_size
    kvp = [int(x) for x in case.kv_indptr.cpu()]
    idx = case.kv_indices.cpu()
    shared = idx[kvp[0]:kvp[0] + S]
    owns = [idx[kvp[b] + S:kvp[b + 1]] for b in range(case.B)]
    own_ptr = [0]
    for x in owns:
        own_ptr.append(own_ptr[-1] + x.numel())
    d_kvp = torch.empty(case.B + 1, dtype=torch.int32, device="cuda")
    d_idx = torch.empty(case.B * S + own_ptr[-1], dtype=torch.int32, device="cuda")
    pm.mla_expand_shared_prefix_indices(shared.cuda(), torch.tensor(own_ptr, dtype=torch.int32,
                                                                    device="cuda"),
                                        torch.cat(owns).cuda(), d_kvp, d_idx)
    torch.cuda.synchronize()
    assert torch.equal(d_kvp.cpu(), case.kv_indptr.cpu() - kvp[0])
    assert torch.equal(d_idx.cpu(), idx[kvp[0]:kvp[-1]])
    o_ref, lse_ref = gu.run_oracle(case)
    case.kv_indptr, case.kv_indices = d_kvp, d_idx
    o, lse, status = gu.run_gpu(case, shared_prefix=P)
    assert status == 0
    gu.compare(o, lse, o_ref, lse_ref, what=case.name)


def test_prepared_decode_with_the_compact_table(pm):
    """PreparedDecode given the compact page table rebuilds the full one in run() before
    the shared-prefix decode; fresh compact data in the same tensors is picked up."""
    lens = [1500 + 53 * i for i in range(8)]
    P = 1200
    case = gu.to_device(mla_inputs.make_custom(lens, H=12, seed=71, shared_prefix=P, q_scale=1.0,
                                               kv_scale=1.0, name="prep-compact"))
    kvp = [int(x) for x in case.kv_indptr.cpu()]
    idx = case.kv_indices.cpu()
    shared = idx[:P].cuda()
    owns = [idx[kvp[b] + P:kvp[b + 1]] for b in range(case.B)]
    own_ptr = [0]
    for x in owns:
        own_ptr.append(own_ptr[-1] + x.numel())
    optr = torch.tensor(own_ptr, dtype=torch.int32, device="cuda")
    own = torch.cat(owns).cuda()
    d_kvp = torch.full((case.B + 1,), -1, dtype=torch.int32, device="cuda")
    d_idx = torch.full((case.B * P + own_ptr[-1],), -1, dtype=torch.int32, device="cuda")
    o = torch.empty((case.q.shape[0], 12, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((case.q.shape[0], 12), dtype=torch.float32, device="cuda")
    prep = pm.PreparedDecode(case.q, case.kv, o, case.qo_indptr, d_kvp, d_idx,
                             case.kv_last_page_lens, case.max_seqlen_q, case.sm_scale,
                             case.q_scale, case.kv_scale, lse_out=lse, shared_prefix_len=P,
                             compact_page_table=(shared, optr, own))
    o_ref, lse_ref = gu.run_oracle(case)
    for step in range(2):
        ws = prep.run()
        torch.cuda.synchronize()
        assert pm.mla_check_error(ws) == 0
        gu.compare(o, lse, o_ref, lse_ref, what=f"prepared compact step {step}")
    # new own ids in place (request 3 attends another request's rows): picked up by run()
    own2 = own.clone()
    s3, e3 = own_ptr[3], own_ptr[4]
    own2[s3:e3] = own[own_ptr[0]:own_ptr[0] + (e3 - s3)]
    own.copy_(own2)
    case2 = case
    idx2 = idx.clone()
    idx2[kvp[3] + P:kvp[4]] = own2[s3:e3].cpu()
    case2.kv_indices = idx2.cuda()
    o_ref2, lse_ref2 = gu.run_oracle(case2)
    ws = prep.run()
    torch.cuda.synchronize()
    assert pm.mla_check_error(ws) == 0
    gu.compare(o, lse, o_ref2, lse_ref2, what="prepared compact, new ids")
