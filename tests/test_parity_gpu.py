"""Parity of the CUDA decode path (through the C ABI) with the FP64 oracle.

Small cases are compared element by element; they span several 128-position tiles, a
ragged tail, every row-group size (16 / 32 / 48 / 96 rows), causal drafts, split policies and
poisoned memory.  Full-size workloads are checked on sampled outputs and invariants.
"""
import math

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


def _check(case, **kw):
    case = gu.to_device(case)
    o, lse, status = gu.run_gpu(case, **kw)
    assert status == 0, f"device error {status}"
    o_ref, lse_ref = gu.run_oracle(case)
    return gu.compare(o, lse, o_ref, lse_ref, what=case.name)


def test_tiny_workload(pm):
    _check(mla_inputs.make_case("tiny", seed=0))


@pytest.mark.parametrize("stress", [False, True])
def test_tiny_workload_stress_scales(pm, stress):
    s = 1.0 if stress else 0.05
    _check(mla_inputs.make_case("tiny", seed=1, q_scale=s, kv_scale=1.0 if stress else 0.1))


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("scales", [(0.05, 0.1), (1.0, 1.0)])
def test_multi_tile_ragged(pm, seed, scales):
    case = mla_inputs.make_custom([1000, 2500, 130, 1, 257], H=12, seed=seed,
                                  q_scale=scales[0], kv_scale=scales[1], name="ragged")
    _check(case)


@pytest.mark.parametrize("splits", [0, 1, 2, 7])
def test_split_policies_agree_with_oracle(pm, splits):
    case = mla_inputs.make_custom([3000, 700, 129], H=12, seed=3, q_scale=1.0, kv_scale=1.0,
                                  name=f"splits{splits}")
    _check(case, num_kv_splits=splits)


def test_fp32_output(pm):
    case = mla_inputs.make_custom([900, 40], H=12, seed=4, q_scale=1.0, kv_scale=1.0, name="fp32o")
    _check(case, o_dtype=torch.float32)


@pytest.mark.parametrize("dtype,width", [(torch.bfloat16, 516), (torch.bfloat16, 520),
                                          (torch.float32, 514), (torch.float32, 516)])
def test_output_row_strides(pm, dtype, width):
    """o as a view of a wider buffer: head strides that do (520, 516 fp32) and do not (516
    bf16, 514 fp32) allow 16-byte stores; both store paths must write exactly o's columns."""
    case = gu.to_device(mla_inputs.make_custom([700, 300, 1], q_lens=[1, 2, 1], H=12, seed=9,
                                               q_scale=1.0, kv_scale=1.0, name="strided"))
    n_tok = case.q.shape[0]
    base = torch.full((n_tok, 12, width), 7.0, dtype=dtype, device="cuda")
    o = base[:, :, :512]
    lse = torch.empty((n_tok, 12), dtype=torch.float32, device="cuda")
    for splits in (0, 1):
        ws = pm.make_workspace(case.B, 12, case.max_seqlen_q, splits, "cuda")
        pm.mla_decode(case.q, case.kv, o, case.qo_indptr, case.kv_indptr, case.kv_indices,
                      case.kv_last_page_lens, case.max_seqlen_q, case.sm_scale, case.q_scale,
                      case.kv_scale, num_kv_splits=splits, lse_out=lse, workspace=ws)
        torch.cuda.synchronize()
        assert pm.mla_check_error(ws) == 0
        o_ref, lse_ref = gu.run_oracle(case)
        gu.compare(o, lse, o_ref, lse_ref, what=f"strided {width} splits {splits}")
        assert bool((base[:, :, 512:] == 7.0).all()), "write past the row's 512 columns"


def _many_rows_case():
    # 64 requests x 4 drafts x 12 heads = 3,072 merged rows; ~10 tiles each over 152 CTAs
    # gives each row ~3 partials, so the merge runs one warp per row
    rng = np.random.default_rng(41)
    kv_lens = [int(x) for x in rng.integers(900, 1600, size=64)]
    return gu.to_device(mla_inputs.make_custom(kv_lens, q_lens=[4] * 64, H=12, seed=41,
                                               q_scale=1.0, kv_scale=1.0, name="rows"))


@pytest.mark.parametrize("dtype,width,with_lse", [(torch.bfloat16, 512, True),
                                                   (torch.bfloat16, 516, False),
                                                   (torch.float32, 512, True),
                                                   (torch.float32, 514, True)])
def test_many_rows_few_partials(pm, dtype, width, with_lse):
    """Thousands of merged rows with a few partials each (the warp-per-row merge): aligned
    and unaligned o rows, bf16 and fp32, with and without lse."""
    case = _many_rows_case()
    n_tok = case.q.shape[0]
    base = torch.full((n_tok, 12, width), 7.0, dtype=dtype, device="cuda")
    o = base[:, :, :512]
    lse = torch.empty((n_tok, 12), dtype=torch.float32, device="cuda") if with_lse else None
    ws = pm.make_workspace(case.B, 12, case.max_seqlen_q, 0, "cuda")
    pm.mla_decode(case.q, case.kv, o, case.qo_indptr, case.kv_indptr, case.kv_indices,
                  case.kv_last_page_lens, case.max_seqlen_q, case.sm_scale, case.q_scale,
                  case.kv_scale, lse_out=lse, workspace=ws)
    torch.cuda.synchronize()
    assert pm.mla_check_error(ws) == 0
    o_ref, lse_ref = gu.run_oracle(case)
    gu.compare(o, lse, o_ref, lse_ref if with_lse else None, what=f"rows {dtype} {width}")
    assert bool((base[:, :, 512:] == 7.0).all()), "write past the row's 512 columns"


def test_shared_prefix_cascade_many_requests(pm):
    """64 requests of one shared prefix: 768 merged rows with ~15 partials each, merged one
    warp per row."""
    rng = np.random.default_rng(42)
    lens = [1100 + int(x) for x in rng.integers(0, 300, size=64)]
    case = gu.to_device(mla_inputs.make_custom(lens, H=12, seed=42, shared_prefix=1024,
                                               q_scale=1.0, kv_scale=1.0, poison=True,
                                               index_buffer=sum(lens) + 64, name="c64"))
    o, lse, status = gu.run_gpu(case, shared_prefix=1024)
    assert status == 0, f"device error {status}"
    o_ref, lse_ref = gu.run_oracle(case)
    gu.compare(o, lse, o_ref, lse_ref, what="cascade, 64 requests")


@pytest.mark.parametrize("H", [16, 24, 40, 96])
def test_head_counts(pm, H):
    """16 -> one 16-row group, 24 -> 32-row group, 40 -> 48-row group, 96 -> one 96-row group
    (the kernel with the query rows on the tensor-memory lanes)."""
    case = mla_inputs.make_custom([1500, 333], H=H, seed=5, q_scale=1.0, kv_scale=1.0, name=f"H{H}")
    _check(case)


@pytest.mark.parametrize("scales", [(0.05, 0.1), (1.0, 1.0)])
def test_causal_drafts(pm, scales):
    """q_len 4 (MTP): draft t attends positions 0 .. L-4+t; includes L == T and ragged tails."""
    case = mla_inputs.make_custom([4, 130, 1000, 2049], q_lens=[4, 4, 4, 4], H=12, seed=6,
                                  q_scale=scales[0], kv_scale=scales[1], name="mtp-small")
    _check(case)


@pytest.mark.parametrize("H,T", [(24, 2), (16, 3), (8, 4), (20, 2), (40, 3)])
def test_causal_drafts_other_head_counts(pm, H, T):
    """Draft boundaries that fall inside a 16-row softmax chunk at other alignments than
    12 heads give (rows t * H of a group), short last chunks, and groups of 32 and 48
    rows; a request shorter than its drafts' window (L == T) included."""
    case = mla_inputs.make_custom([T, 97, 700], q_lens=[T] * 3, H=H, seed=17 + H + T,
                                  q_scale=1.0, kv_scale=1.0, name=f"mtp-H{H}-T{T}")
    _check(case)


def test_mixed_query_lengths(pm):
    case = mla_inputs.make_custom([300, 800, 50, 1200], q_lens=[1, 3, 2, 4], H=12, seed=7,
                                  q_scale=1.0, kv_scale=1.0, name="mixed-q")
    _check(case)


def test_shared_prefix(pm):
    case = mla_inputs.make_custom([2000, 2100, 2222, 1900], H=12, seed=8, shared_prefix=1700,
                                  index_buffer=10000, name="prefix")
    _check(case)


@pytest.mark.parametrize("kv_lens,q_lens,prefix", [
    ([3000, 3100, 2900, 3050, 3200], [1] * 5, 2048),         # 2 groups (4 + 1)
    ([2500] * 9, [1] * 9, 2500),                             # whole requests shared
    ([2600, 2100, 3300, 2100, 2800, 2200], [1] * 6, 2100),   # some suffixes empty
    ([4000, 4500, 3900, 4100], [2] * 4, 3000),               # 2 queries each, causal tail
    ([3000, 3000, 3000, 3000], [1, 2, 1, 1], 2999),          # prefix up to the causal cap
    ([1500, 1700, 1600, 1800], [1] * 4, 900),                # too short: plain decode
    ([2000, 2100, 2200], [1] * 3, 1500),                     # under one group: plain decode
])
@pytest.mark.parametrize("scales", [(0.05, 0.1), (1.0, 1.0)])
def test_shared_prefix_cascade(pm, kv_lens, q_lens, prefix, scales):
    """mla_decode_shared_prefix: the shared rows are attended in groups of requests (prefix
    units), each request's own rows separately (own units, same launch), and the two
    merged; the result must equal the oracle.  Unattended rows are poisoned."""
    case = gu.to_device(mla_inputs.make_custom(kv_lens, q_lens=q_lens, H=12, seed=31,
                                               shared_prefix=prefix, q_scale=scales[0],
                                               kv_scale=scales[1], poison=True,
                                               index_buffer=sum(kv_lens) + 64, name="cascade"))
    o, lse, status = gu.run_gpu(case, shared_prefix=prefix)
    assert status == 0, f"device error {status}"
    o_ref, lse_ref = gu.run_oracle(case)
    gu.compare(o, lse, o_ref, lse_ref, what="cascade")


@pytest.mark.parametrize("shared", [None, 2048])
def test_prepared_call(pm, shared):
    """PreparedDecode: descriptors built once, run() twice; the second run after new q
    data written in place gives that data's answer, equal to the one-shot call's."""
    case = gu.to_device(mla_inputs.make_custom([3000, 3100, 2900, 3050, 3200], H=12, seed=34,
                                               shared_prefix=2048 if shared else 0,
                                               q_scale=1.0, kv_scale=1.0, name="prepared"))
    n_tok = case.q.shape[0]
    q = case.q.clone()
    o = torch.empty((n_tok, 12, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((n_tok, 12), dtype=torch.float32, device="cuda")
    prep = pm.PreparedDecode(q, case.kv, o, case.qo_indptr, case.kv_indptr, case.kv_indices,
                             case.kv_last_page_lens, case.max_seqlen_q, case.sm_scale,
                             case.q_scale, case.kv_scale, lse_out=lse, shared_prefix_len=shared)
    prep.run()
    torch.cuda.synchronize()
    o_one, lse_one, st = gu.run_gpu(case, shared_prefix=shared)
    assert st == 0 and pm.mla_check_error(prep.workspace) == 0
    assert torch.equal(o, o_one) and torch.equal(lse, lse_one)
    q2 = torch.flip(case.q, dims=[1]).contiguous()
    q.copy_(q2)
    prep.run()
    torch.cuda.synchronize()
    o2, lse2, st2 = gu.run_gpu(case, shared_prefix=shared, q_override=q2)
    assert st2 == 0 and torch.equal(o, o2) and torch.equal(lse, lse2)
    assert not torch.equal(o2, o_one)


def test_shared_prefix_with_the_plain_workspace(pm):
    """With only the plain decode's workspace the call runs the plain decode: same answer."""
    case = gu.to_device(mla_inputs.make_custom([3000] * 5, H=12, seed=32, shared_prefix=2500,
                                               q_scale=1.0, kv_scale=1.0))
    plain = pm.mla_get_workspace_size(case.B, 12, 1, 0)
    assert plain < pm.mla_get_shared_prefix_workspace_size(case.B, 12, 1)
    ws = torch.zeros(plain, dtype=torch.uint8, device="cuda")
    o, lse, status = gu.run_gpu(case, workspace=ws, shared_prefix=2500)
    assert status == 0
    o_ref, lse_ref = gu.run_oracle(case)
    gu.compare(o, lse, o_ref, lse_ref, what="plain path")


def test_shared_prefix_beyond_a_query_is_flagged(pm):
    """A claimed prefix that the second draft of a request could not see in full (P > kv_len
    - q_len + 1) is reported as bad input; the kernels finish normally."""
    case = gu.to_device(mla_inputs.make_custom([3000, 3000, 3000, 3000], q_lens=[1, 2, 1, 1],
                                               H=12, seed=33, shared_prefix=3000))
    o, lse, status = gu.run_gpu(case, shared_prefix=3000)
    assert status == 7   # MLA_ERR_BAD_INPUT


def test_poisoned_rows_and_index_tail(pm):
    """Unattended rows hold fp8 NaN and the index buffer tail points outside the pool:
    any stray read would surface as NaN or a device error."""
    case = mla_inputs.make_custom([700, 129, 1], q_lens=[1, 4, 1], H=12, seed=9, poison=True,
                                  index_buffer=5000, q_scale=1.0, kv_scale=1.0, name="poison")
    _check(case)
    for splits in (1, 3):
        _check(case, num_kv_splits=splits)


def test_zero_padded_heads_are_bit_identical(pm):
    """P6: 12 heads vs the same 12 heads + 4 zero heads; real heads' o and lse identical."""
    case = gu.to_device(mla_inputs.make_custom([1000, 300], H=12, seed=10, q_scale=1.0,
                                               kv_scale=1.0))
    o12, lse12, st = gu.run_gpu(case)
    assert st == 0
    q16 = torch.zeros((case.q.shape[0], 16, 576), dtype=torch.uint8, device="cuda")
    q16[:, :12] = case.q
    o16, lse16, st = gu.run_gpu(case, q_override=q16)
    assert st == 0
    assert torch.equal(o16[:, :12], o12)
    assert torch.equal(lse16[:, :12], lse12)


def test_identical_rows_mean_and_exact_counts(pm):
    """P2: all attended rows equal -> o = kv_scale * v and exp(lse - s) = attended count,
    which pins the attended set of every (request, draft) bit-exactly."""
    lens, qlens = [1000, 37, 300], [1, 4, 2]
    case = mla_inputs.make_custom(lens, q_lens=qlens, H=12, seed=11, q_scale=0.5, kv_scale=0.25)
    row = case.kv[0].clone()
    case.kv[:] = row
    case = gu.to_device(case)
    o, lse, st = gu.run_gpu(case, o_dtype=torch.float32)
    assert st == 0
    from tests import brute
    v = brute.fp8_decode(row.numpy())
    sm, qs, ks = case.scales()
    o = o.cpu().numpy()
    lse = lse.cpu().numpy()
    qh = case.q.cpu().numpy()
    for b, (L, T) in enumerate(zip(lens, qlens)):
        for t in range(T):
            r = int(case.qo_indptr[b]) + t
            for h in range(12):
                assert np.allclose(o[r, h], ks * v[:512], rtol=1e-2, atol=1e-4)
                s = sm * qs * ks * float(brute.fp8_decode(qh[r, h]) @ v)
                count = math.exp(lse[r, h] - s)
                assert round(count) == L - T + t + 1, (b, t, h, count)


def test_constant_logit_shift(pm):
    """P3: every row shares its rope block; changing q's rope block shifts all logits of a
    head by the same delta: o unchanged, lse moves by delta."""
    case = mla_inputs.make_custom([900, 200], H=12, seed=12, q_scale=1.0, kv_scale=1.0)
    case.kv[:, 512:] = case.kv[0, 512:]
    q2 = case.q.clone()
    q2[:, :, 512:] = torch.flip(case.q[:, :, 512:], dims=[1])
    case = gu.to_device(case)
    o1, l1, _ = gu.run_gpu(case, o_dtype=torch.float32)
    o2, l2, _ = gu.run_gpu(case, o_dtype=torch.float32, q_override=q2.cuda())
    from tests import brute
    sm, qs, ks = case.scales()
    kr = brute.fp8_decode(case.kv[0, 512:].cpu().numpy())
    q1h, q2h = case.q.cpu().numpy(), q2.numpy()
    for r in range(2):
        for h in range(12):
            delta = sm * qs * ks * (float(brute.fp8_decode(q2h[r, h, 512:]) @ kr) -
                                    float(brute.fp8_decode(q1h[r, h, 512:]) @ kr))
            assert abs((l2[r, h] - l1[r, h]).item() - delta) < 2e-3
    assert torch.allclose(o1, o2, atol=2e-3, rtol=1e-2)


def test_needle_position_and_causal_limit(pm):
    """One row with a dominant logit and a one-hot value reveals which positions each
    draft attends."""
    L, T = 300, 4
    case = mla_inputs.make_custom([L], q_lens=[T], H=12, seed=13, q_scale=1.0, kv_scale=1.0)
    case.kv.zero_()
    case.q.zero_()
    big = torch.tensor([16.0]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    one = torch.tensor([1.0]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    case.q[:, :, 0] = big
    needle_pos = L - 2
    row = int(case.kv_indices[needle_pos])
    case.kv[row, 0] = big
    case.kv[row, 100] = one
    case = gu.to_device(case)
    o, lse, st = gu.run_gpu(case, o_dtype=torch.float32)
    assert st == 0
    for t in range(T):
        sees = needle_pos <= L - T + t
        for h in range(12):
            val = o[t, h, 100].item()
            assert (val > 0.99) == sees, (t, h, val)


def test_empty_request_gives_zero_and_neg_inf(pm):
    case = mla_inputs.make_custom([0, 400, 0], q_lens=[1, 1, 1], H=12, seed=14)
    case = gu.to_device(case)
    for splits in (0, 1, 4):
        o, lse, st = gu.run_gpu(case, num_kv_splits=splits, o_dtype=torch.float32)
        assert st == 0
        assert torch.equal(o[0], torch.zeros_like(o[0])) and torch.equal(o[2], torch.zeros_like(o[2]))
        assert torch.isneginf(lse[0]).all() and torch.isneginf(lse[2]).all()
        o_ref, lse_ref = oracle.attend_one(case.q[1, 3].cpu().numpy(),
                                           gu.gather_rows(case, 1), np.arange(400, dtype=np.int32),
                                           *case.scales())
        assert np.allclose(o[1, 3].cpu().numpy(), o_ref, atol=1e-2, rtol=1e-2)


def test_bad_index_is_flagged_without_fault(pm):
    case = mla_inputs.make_custom([500, 300], H=12, seed=15)
    case.kv_indices[10] = case.kv.shape[0] + 123
    case = gu.to_device(case)
    o, lse, st = gu.run_gpu(case)
    assert st == 5   # MLA_ERR_BAD_INDEX
    torch.cuda.synchronize()   # the context is still usable
    ws = pm.make_workspace(case.B, 12, 1, 0, "cuda")
    assert pm.mla_validate(case.q, case.kv, case.qo_indptr, case.kv_indptr, case.kv_indices,
                           case.kv_last_page_lens, ws) == 5


def test_validate(pm):
    case = gu.to_device(mla_inputs.make_custom([500, 300], q_lens=[1, 2], H=12, seed=16))
    ws = pm.make_workspace(case.B, 12, 2, 0, "cuda")
    assert pm.mla_validate(case.q, case.kv, case.qo_indptr, case.kv_indptr, case.kv_indices,
                           case.kv_last_page_lens, ws) == 0
    bad = case.kv_last_page_lens.clone()
    bad[1] = 128
    assert pm.mla_validate(case.q, case.kv, case.qo_indptr, case.kv_indptr, case.kv_indices,
                           bad, ws) == 7
    short = torch.tensor([0, 500, 501], dtype=torch.int32, device="cuda")   # kv_len 1 < q_len 2
    assert pm.mla_validate(case.q, case.kv, case.qo_indptr, short, case.kv_indices,
                           case.kv_last_page_lens, ws) == 7


def test_merge_partials_csr(pm):
    """mla_merge_partials == oracle merge on random partials, including -inf ones and an
    output row with no partials at all."""
    rng = np.random.default_rng(17)
    P, H = 9, 12
    o_parts = rng.standard_normal((P, H, 512)).astype(np.float32)
    lse_parts = (rng.standard_normal((P, H)) * 3).astype(np.float32)
    lse_parts[2, :] = -np.inf
    indptr = np.array([0, 3, 3, 9], dtype=np.int32)
    idx = np.array([4, 2, 0, 1, 3, 5, 6, 7, 8], dtype=np.int32)
    dev = lambda a: torch.from_numpy(a).cuda()
    o = torch.empty((3, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((3, H), dtype=torch.float32, device="cuda")
    pm.mla_merge_partials(dev(o_parts), dev(lse_parts), dev(indptr), dev(idx), o, lse)
    torch.cuda.synchronize()
    for r in range(3):
        sel = idx[indptr[r]:indptr[r + 1]]
        for h in range(H):
            if sel.size == 0:
                assert torch.equal(o[r, h].cpu(), torch.zeros(512))
                assert math.isinf(lse[r, h].item()) and lse[r, h].item() < 0
                continue
            ro, rl = oracle.merge(o_parts[sel, h].astype(np.float64), lse_parts[sel, h].astype(np.float64))
            assert np.allclose(o[r, h].cpu().numpy(), ro, rtol=1e-5, atol=1e-5)
            assert abs(lse[r, h].item() - rl) < 1e-4


def test_context_shard_merge_small(pm):
    """8 context shards x 96 heads, each shard's partial (fp32 o, lse) merged by
    mla_merge_partials, equals the unsplit 96-head call and the oracle."""
    case = gu.to_device(mla_inputs.make_custom([4000], H=96, seed=18, q_scale=1.0, kv_scale=1.0))
    o_ref, lse_ref = gu.run_oracle(case)
    o_full, lse_full, st = gu.run_gpu(case, o_dtype=torch.float32)
    assert st == 0
    shards = mla_inputs.shard_views(case, 8)
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
    gu.compare(o, lse, o_ref, lse_ref, what="shard-merge")
    assert torch.allclose(o.float(), o_full, atol=1e-2, rtol=1e-2)
    assert torch.allclose(lse, lse_full, atol=1e-3)


@pytest.mark.parametrize("splits", [0, 1, 3])
def test_running_max_rescale_every_tile(pm, splits):
    """Cache rows rise tile by tile so that, for heads 0-5, every 128-position tile's logits
    exceed the previous tile's by ~10 nats (more than the headroom of the reference
    max): the kernel must move its reference and rescale the accumulated output on every
    tile.  Heads 6-11 see a slow rise (no rescale).  Values carry random latent parts."""
    L = 15 * 128 + 37
    case = mla_inputs.make_custom([L, 300], H=12, seed=19, q_scale=1.0, kv_scale=1.0)
    f8 = lambda x: torch.tensor([x]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    idx = case.kv_indices[:L].long()
    rise = torch.tensor([f8(0.25 * min(j // 128, 15)) for j in range(L)], dtype=torch.uint8)
    keys = case.kv.clone()
    keys[idx, :] = rise[:, None].expand(L, 576)          # constant rows rising per tile
    keys[idx, 300:512] = case.kv[idx, 300:512]           # random value columns (not in logits)
    q = case.q.clone()
    q[0, :6, :] = f8(1.0)
    q[0, 6:, :] = f8(0.125)
    q[0, :, 300:512] = 0                                  # those columns do not enter the logits
    case.kv = keys
    case.q = q
    _check(case, num_kv_splits=splits)


@pytest.mark.parametrize("splits", [0, 1])
def test_logit_jump_within_reference_headroom(pm, splits):
    """A position in a later tile whose logit is 5-7.5 log2 units above every earlier one
    and whose values are large.  However the kernel treats the jump (moving its reference
    max, or keeping it and giving the position a weight p = 2^5..2^7.5), the weight must
    reach the tensor core with the hi/lo precision: a lo plane 256 (p - hi) that saturates
    at the e4m3 maximum misweights such a position by a few percent.  No head's jump is
    large enough to force a move on its own (a move for one head moves its whole
    16-column chunk)."""
    L = 6 * 128 + 11
    spike = 700
    case = mla_inputs.make_custom([L], H=12, seed=23, q_scale=1.0, kv_scale=1.0)
    f8 = lambda x: torch.tensor([x]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    idx = case.kv_indices[:L].long()
    keys = case.kv.clone()
    keys[idx, 512:] = 0                                   # rope columns: logits 0 ...
    keys[idx[spike], 512:] = f8(1.0)                      # ... except at the jump
    keys[idx[spike], :512] = f8(320.0)                    # large values at the jump
    q = case.q.clone()
    q[0, :, :512] = 0                                     # logits from the rope part only
    qvs = [0.75, 0.8125, 0.875, 0.9375, 1.0, 1.125, 1.125, 1.0, 0.9375, 0.875, 0.8125, 0.75]
    for h, qv in enumerate(qvs):
        q[0, h, 512:] = f8(qv)                            # jump = 6.66 * qv log2 units
    case.kv = keys
    case.q = q
    _check(case, num_kv_splits=splits)


@pytest.mark.parametrize("splits", [0, 1])
def test_sink_over_uniform_bulk(pm, splits):
    """An attention sink at position 0 whose logit is ~11 log2 units above 2,000 identical
    bulk positions: each bulk weight is ~2^-11 of the sink's, but together they carry about
    half of the mass, and identical rows make any rounding of their weights systematic.  The
    weights must keep the hi/lo precision even that far below the reference max."""
    L = 2001
    case = mla_inputs.make_custom([L], H=12, seed=29, q_scale=1.0, kv_scale=1.0)
    f8 = lambda x: torch.tensor([x]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    idx = case.kv_indices[:L].long()
    keys = case.kv.clone()
    keys[idx, :] = f8(2.0)                                # bulk: identical rows, values 2
    keys[idx, 512:] = 0                                   # bulk rope 0
    keys[idx[0], :512] = 0                                # sink: values 0 ...
    keys[idx[0], 512:] = f8(1.75)                         # ... rope 1.75
    q = case.q.clone()
    q[0, :, :512] = 0
    qvs = [0.9375, 0.875, 1.0, 0.8125, 0.9375, 0.875, 1.0, 0.8125, 0.9375, 0.875, 1.0, 0.8125]
    for h, qv in enumerate(qvs):
        q[0, h, 512:] = f8(qv)                            # sink - bulk = 11.66 * qv log2 units
    case.kv = keys
    case.q = q
    _check(case, num_kv_splits=splits)
