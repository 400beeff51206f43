"""Parity of the 96-row decode kernel (query rows on the tensor-memory lanes, the hi and lo
planes of P in one accumulator through block-scaled FP8 MMAs) with the FP64 oracle: every
group depth from 49 to 96 rows and two-group calls, causal drafts whose limits differ row by
row, split policies, the lazy reference max moved on every tile, the precision envelope of
P (a sink far above a uniform bulk, a logit jump inside the headroom), strided and fp32
outputs, the shared-prefix cascade in 96-row groups of 2, 4 and 8 requests (and the 48-row
cascade kept for 4..7 small requests), pages of several tokens, empty requests and a bad
index.  Tolerances are the suite's (tests/gpu_util.py)."""
import numpy as np
import pytest
import torch

import mla_inputs
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pm():
    import paged_mla_latent_gb300 as m
    return m


def _f8(x):
    return torch.tensor([x]).to(torch.float8_e4m3fn).view(torch.uint8).item()


def _check(case, **kw):
    case = gu.to_device(case)
    o, lse, status = gu.run_gpu(case, **kw)
    assert status == 0, f"device error {status}"
    o_ref, lse_ref = gu.run_oracle(case)
    return gu.compare(o, lse, o_ref, lse_ref, what=case.name)


@pytest.mark.parametrize("H,T", [(49, 1), (52, 1), (64, 1), (80, 1), (96, 1), (16, 4), (24, 3),
                                 (12, 8), (32, 3), (128, 1), (40, 3), (200, 1)])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_group_depths(pm, H, T, splits):
    """One 96-row group 49..96 rows deep, or two groups (128 = 96 + 32, 120 = 96 + 24,
    200 = 96 + 96 + 8); draft boundaries fall inside the group wherever H does not divide 96."""
    case = mla_inputs.make_custom([T, 70, 700, 1500], q_lens=[T] * 4, H=H, seed=H * 7 + T,
                                  q_scale=1.0, kv_scale=1.0, name=f"rows96 H{H} T{T}")
    _check(case, num_kv_splits=splits)


@pytest.mark.parametrize("scales", [(0.05, 0.1), (1.0, 1.0)])
def test_causal_drafts_long(pm, scales):
    """Eight drafts of 12 heads (96 rows, each draft's limit one position further) over
    histories of many 64-position tiles, with the drafts' last positions at every offset."""
    case = mla_inputs.make_custom([8, 9, 63, 64, 65, 1000, 2047], q_lens=[8] * 7, H=12, seed=31,
                                  q_scale=scales[0], kv_scale=scales[1], name="drafts96")
    for splits in (0, 2):
        _check(case, num_kv_splits=splits)


@pytest.mark.parametrize("splits", [0, 1, 3])
def test_running_max_rescale_every_tile(pm, splits):
    """96 heads; cache rows rise every 64 positions so that for heads 0-47 each tile's logits
    exceed the previous tile's by more than the reference headroom (the kernel moves the
    reference and rescales those rows' accumulated output on every tile), while heads 48-95
    see a slow rise.  The value columns stay random."""
    L = 24 * 64 + 19
    case = mla_inputs.make_custom([L, 200], H=96, seed=37, q_scale=1.0, kv_scale=1.0,
                                  name="rescale96")
    idx = case.kv_indices[:L].long()
    rise = torch.tensor([_f8(0.25 * min(j // 64, 15)) for j in range(L)], dtype=torch.uint8)
    keys = case.kv.clone()
    keys[idx, :] = rise[:, None].expand(L, 576)
    keys[idx, 300:512] = case.kv[idx, 300:512]
    q = case.q.clone()
    q[0, :48, :] = _f8(1.0)
    q[0, 48:, :] = _f8(0.125)
    q[0, :, 300:512] = 0
    case.kv = keys
    case.q = q
    _check(case, num_kv_splits=splits)


@pytest.mark.parametrize("splits", [0, 1])
def test_sink_over_uniform_bulk(pm, splits):
    """The sink of the 16/32/48-row suite at 96 heads: a sink ~11 log2 units above 2,000
    identical rows.  The lo plane reaches the accumulator at 2^-4 through its block scale
    factor; a wrong factor misweights the bulk by far more than the tolerance."""
    L = 2001
    case = mla_inputs.make_custom([L], H=96, seed=41, q_scale=1.0, kv_scale=1.0, name="sink96")
    idx = case.kv_indices[:L].long()
    keys = case.kv.clone()
    keys[idx, :] = _f8(2.0)
    keys[idx, 512:] = 0
    keys[idx[0], :512] = 0
    keys[idx[0], 512:] = _f8(1.75)
    q = case.q.clone()
    q[0, :, :512] = 0
    for h in range(96):
        q[0, h, 512:] = _f8([0.9375, 0.875, 1.0, 0.8125][h % 4])
    case.kv = keys
    case.q = q
    _check(case, num_kv_splits=splits)


@pytest.mark.parametrize("splits", [0, 1])
def test_logit_jump_within_reference_headroom(pm, splits):
    """A position 5-7.5 log2 units above every earlier logit, with large values: its weight
    must reach the tensor core with the hi/lo precision."""
    L = 12 * 64 + 11
    spike = 700
    case = mla_inputs.make_custom([L], H=96, seed=43, q_scale=1.0, kv_scale=1.0, name="jump96")
    idx = case.kv_indices[:L].long()
    keys = case.kv.clone()
    keys[idx, 512:] = 0
    keys[idx[spike], 512:] = _f8(1.0)
    keys[idx[spike], :512] = _f8(320.0)
    q = case.q.clone()
    q[0, :, :512] = 0
    qvs = [0.75, 0.8125, 0.875, 0.9375, 1.0, 1.125]
    for h in range(96):
        q[0, h, 512:] = _f8(qvs[h % 6])
    case.kv = keys
    case.q = q
    _check(case, num_kv_splits=splits)


@pytest.mark.parametrize("dtype,width", [(torch.bfloat16, 512), (torch.bfloat16, 516),
                                          (torch.bfloat16, 520), (torch.float32, 514),
                                          (torch.float32, 516)])
def test_output_row_strides(pm, dtype, width):
    """o as a view of a wider buffer, written directly by the 96-row kernel (one split) and
    through the merge (automatic split): 16-byte and scalar store paths write exactly o's
    columns."""
    case = gu.to_device(mla_inputs.make_custom([700, 300, 2], q_lens=[1, 2, 1], H=96, seed=47,
                                               q_scale=1.0, kv_scale=1.0, name="strided96"))
    n_tok = case.q.shape[0]
    base = torch.full((n_tok, 96, width), 7.0, dtype=dtype, device="cuda")
    o = base[:, :, :512]
    lse = torch.empty((n_tok, 96), dtype=torch.float32, device="cuda")
    o_ref, lse_ref = gu.run_oracle(case)
    for splits in (0, 1):
        ws = pm.make_workspace(case.B, 96, case.max_seqlen_q, splits, "cuda")
        pm.mla_decode(case.q, case.kv, o, case.qo_indptr, case.kv_indptr, case.kv_indices,
                      case.kv_last_page_lens, case.max_seqlen_q, case.sm_scale, case.q_scale,
                      case.kv_scale, num_kv_splits=splits, lse_out=lse, workspace=ws)
        torch.cuda.synchronize()
        assert pm.mla_check_error(ws) == 0
        gu.compare(o, lse, o_ref, lse_ref, what=f"strided96 {width} splits {splits}")
        assert bool((base[:, :, 512:] == 7.0).all()), "write past the row's 512 columns"


@pytest.mark.parametrize("H,T,B,prefix", [(12, 1, 8, 1024), (12, 1, 11, 2500), (12, 1, 17, 1100),
                                          (12, 2, 4, 2048), (12, 2, 7, 1024), (12, 4, 2, 1500),
                                          (12, 4, 5, 2048), (8, 1, 12, 1024), (24, 1, 4, 3000),
                                          (48, 1, 3, 1024), (12, 1, 5, 2048), (16, 1, 3, 1024)])
@pytest.mark.parametrize("scales", [(0.05, 0.1), (1.0, 1.0)])
def test_shared_prefix_cascade(pm, H, T, B, prefix, scales):
    """Prefix units of 96 rows: 8 requests of 12 heads (with a partial last group), groups of
    4 (24 rows) and 2 (48 rows, mtp-like drafts), 12 requests of 8 heads, 48 heads in pairs;
    and the 48-row cascade for 4..7 requests of 12 heads (12 x 5) or 3 of 16."""
    rng = np.random.default_rng(H * 1000 + B)
    lens = [prefix + T + int(x) for x in rng.integers(0, 700, size=B)]
    case = mla_inputs.make_custom(lens, q_lens=[T] * B, H=H, seed=B + T, shared_prefix=prefix,
                                  q_scale=scales[0], kv_scale=scales[1], poison=True,
                                  index_buffer=sum(lens) + 32, name=f"casc96 H{H} T{T} B{B}")
    _check(case, shared_prefix=prefix)


@pytest.mark.parametrize("page_size", [2, 16, 128])
def test_shared_prefix_cascade_on_pages(pm, page_size):
    """The paged cascade in 96-row groups: 9 requests of 12 heads on pages of several
    tokens, the prefix a whole number of pages, ragged last pages."""
    lens = [2048 + 100 * i + 7 for i in range(9)]
    case = mla_inputs.make_paged(lens, H=12, page_size=page_size, seed=page_size + 5,
                                 q_scale=1.0, kv_scale=1.0, shared_prefix=2048,
                                 name=f"paged-casc96-{page_size}")
    _check(case, shared_prefix=2048)


@pytest.mark.parametrize("page_size", [16, 64])
def test_paged_96_heads(pm, page_size):
    case = mla_inputs.make_paged([900, 33, 2048, 5], H=96, page_size=page_size, seed=page_size,
                                 q_scale=1.0, kv_scale=1.0, poison=True, name=f"paged96-{page_size}")
    for splits in (0, 1, 2):
        _check(case, num_kv_splits=splits)


def test_empty_request_gives_zero_and_neg_inf(pm):
    case = gu.to_device(mla_inputs.make_custom([0, 400, 0], q_lens=[1, 1, 1], H=96, seed=53))
    for splits in (0, 1, 4):
        o, lse, st = gu.run_gpu(case, num_kv_splits=splits, o_dtype=torch.float32)
        assert st == 0
        assert torch.equal(o[0], torch.zeros_like(o[0])) and torch.equal(o[2], torch.zeros_like(o[2]))
        assert torch.isneginf(lse[0]).all() and torch.isneginf(lse[2]).all()
        # (the oracle's batch entry rejects kv_len < q_len: the live request head by head)
        rows = gu.gather_rows(case, 1)
        for h in (0, 37, 95):
            o_ref, lse_ref = oracle.attend_one(case.q[1, h].cpu().numpy(), rows,
                                               np.arange(400, dtype=np.int32), *case.scales())
            assert np.allclose(o[1, h].cpu().numpy(), o_ref, atol=1e-2, rtol=1e-2)
            assert abs(float(lse[1, h]) - lse_ref) <= 1e-3


def test_bad_index_is_flagged_without_fault(pm):
    case = mla_inputs.make_custom([500, 300], H=96, seed=59)
    case.kv_indices[10] = case.kv.shape[0] + 123
    case = gu.to_device(case)
    o, lse, st = gu.run_gpu(case)
    assert st == 5   # MLA_ERR_BAD_INDEX
    torch.cuda.synchronize()   # the context is still usable
    _check(mla_inputs.make_custom([500, 300], H=96, seed=60, name="after-bad-index"))
