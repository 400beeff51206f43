"""Pins of the FP64 oracle against things other than itself (CPU only).

Each test fixes a part of the oracle with brute force, a closed form, an invariant or a
figure printed on the pages, chosen so that a dropped term, a wrong sign or index, or a
transposed operand fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import mla_inputs
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")


def _np(case):
    return dict(q=case.q.numpy(), kv=case.kv.numpy(), qo=case.qo_indptr.numpy(),
                kvp=case.kv_indptr.numpy(), idx=case.kv_indices.numpy())


def _oracle(case):
    a = _np(case)
    sm, qs, ks = case.scales()
    return oracle.decode(a["q"], a["kv"], a["qo"], a["kvp"], a["idx"], sm, qs, ks)


# ---------------------------------------------------------------- P7: FP8 decode table

def test_fp8_table_matches_torch_cast():
    """All 256 codes agree with torch's independent e4m3fn -> float64 cast (NaNs at the same codes)."""
    ours = oracle.fp8_e4m3fn_table()
    ref = brute.fp8_decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_fp8_table_format_anchors():
    """Anchors of the e4m3fn format (OCP 8-bit floating point): bias 7, no infinities."""
    t = oracle.fp8_e4m3fn_table()
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0          # largest finite
    assert t[0x38] == 1.0 and t[0xB8] == -1.0              # exponent field 7 = 2^0
    assert t[0x08] == 2.0 ** -6                            # smallest normal
    assert t[0x01] == 2.0 ** -9                            # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9                        # largest subnormal
    assert t[0x00] == 0.0 and math.copysign(1.0, t[0x80]) == -1.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isnan(t).sum() == 2                          # only S.1111.111 is NaN
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)                        # codes 0..126 strictly increase
    assert np.array_equal(t[0x80:0xFF], -t[:0x7F])         # sign-magnitude


def test_fp8_roundtrip_through_torch_encoder():
    t = oracle.fp8_e4m3fn_table()
    codes = np.array([c for c in range(256) if not np.isnan(t[c])], dtype=np.uint8)
    enc = torch.from_numpy(t[codes]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # -0.0 and +0.0 both encode faithfully
    assert np.array_equal(enc, codes)


# ---------------------------------------------------------------- P1: brute force

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_oracle_matches_brute_force_tiny(seed):
    case = mla_inputs.make_custom([5, 17, 1, 40], q_lens=[1, 3, 1, 2], H=3, seed=seed,
                                  q_scale=0.7, kv_scale=0.9)
    o, lse = _oracle(case)
    a = _np(case)
    sm, qs, ks = case.scales()
    bo, blse = brute.decode(a["q"], a["kv"], a["qo"], a["kvp"], a["idx"], sm, qs, ks)
    assert np.allclose(o, bo, rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, blse, rtol=1e-12, atol=1e-12)


def test_oracle_matches_brute_force_on_tiny_workload():
    case = mla_inputs.make_case("tiny", seed=3)
    o, lse = _oracle(case)
    a = _np(case)
    sm, qs, ks = case.scales()
    bo, blse = brute.decode(a["q"], a["kv"], a["qo"], a["kvp"], a["idx"], sm, qs, ks)
    assert np.allclose(o, bo, rtol=1e-12, atol=1e-15)
    assert np.allclose(lse, blse, rtol=1e-12, atol=1e-12)


def _rows(rng, n):
    x = rng.standard_normal((n, 576)).clip(-448, 448)
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_closed_form_single_position():
    """L = 1: o = kv_scale * v exactly and lse = s_0."""
    rng = np.random.default_rng(7)
    kv = _rows(rng, 4)
    q = _rows(rng, 1)[0]
    sm, qs, ks = 0.0721, 0.5, 0.25
    o, lse = oracle.attend_one(q, kv, [2], sm, qs, ks)
    v = brute.fp8_decode(kv[2])
    assert np.array_equal(o, ks * v[:512])
    s0 = sm * qs * ks * float(brute.fp8_decode(q) @ v)
    assert lse == pytest.approx(s0, rel=1e-13, abs=1e-13)


def test_closed_form_two_positions():
    """L = 2: o = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1, lse = logaddexp(s0, s1)."""
    rng = np.random.default_rng(8)
    kv = _rows(rng, 3)
    q = _rows(rng, 1)[0]
    sm, qs, ks = 0.0721, 1.0, 1.0
    o, lse = oracle.attend_one(q, kv, [0, 2], sm, qs, ks)
    qf = brute.fp8_decode(q)
    v0, v2 = brute.fp8_decode(kv[0]), brute.fp8_decode(kv[2])
    s0, s1 = sm * float(qf @ v0), sm * float(qf @ v2)
    sig = 1.0 / (1.0 + math.exp(-(s0 - s1)))
    assert np.allclose(o, sig * v0[:512] + (1 - sig) * v2[:512], rtol=1e-12, atol=1e-13)
    assert lse == pytest.approx(np.logaddexp(s0, s1), rel=1e-13)


# ---------------------------------------------------------------- P2: identical rows

@pytest.mark.parametrize("T", [1, 4])
def test_identical_rows_give_mean_and_exact_count(T):
    """Every attended row identical: o = kv_scale * v, and exp(lse - s) = number attended."""
    rng = np.random.default_rng(11)
    row = _rows(rng, 1)[0]
    L = 37
    kv = np.tile(row, (L + 5, 1))
    q = _rows(rng, T * 2).reshape(T, 2, 576)
    sm, qs, ks = 0.0722, 0.3, 0.6
    o, lse = oracle.decode(q, kv, [0, T], [0, L], np.arange(L, dtype=np.int32), sm, qs, ks)
    v = brute.fp8_decode(row)
    for t in range(T):
        for h in range(2):
            assert np.allclose(o[t, h], ks * v[:512], rtol=1e-13, atol=1e-15)
            s = sm * qs * ks * float(brute.fp8_decode(q[t, h]) @ v)
            count = math.exp(lse[t, h] - s)
            assert round(count) == L - T + t + 1
            assert abs(count - round(count)) < 1e-9


# ---------------------------------------------------------------- P3: constant logit shift

def test_constant_logit_shift_leaves_o_unchanged():
    """All rows share one rope block; changing q's rope block shifts every logit by the
    same delta = c * q_rope . k_rope, so o is unchanged and lse moves by exactly delta."""
    rng = np.random.default_rng(12)
    L = 50
    kv = _rows(rng, L)
    kv[:, 512:] = kv[0, 512:]
    q1 = _rows(rng, 1)[0]
    q2 = q1.copy()
    q2[512:] = _rows(rng, 1)[0][512:]
    sm, qs, ks = 0.0722, 1.0, 1.0
    rows = np.arange(L, dtype=np.int32)
    o1, lse1 = oracle.attend_one(q1, kv, rows, sm, qs, ks)
    o2, lse2 = oracle.attend_one(q2, kv, rows, sm, qs, ks)
    kr = brute.fp8_decode(kv[0, 512:])
    delta = sm * (float(brute.fp8_decode(q2[512:]) @ kr) - float(brute.fp8_decode(q1[512:]) @ kr))
    assert abs(delta) > 1e-3
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-14)
    assert lse2 - lse1 == pytest.approx(delta, rel=1e-10, abs=1e-12)


# ---------------------------------------------------------------- P4: split + merge

@pytest.mark.parametrize("seed", [0, 1])
def test_any_split_merged_equals_unsplit(seed):
    rng = np.random.default_rng(100 + seed)
    L = 300
    kv = _rows(rng, L + 10)
    q = _rows(rng, 1)[0]
    rows = rng.permutation(L + 10)[:L].astype(np.int32)
    sm, qs, ks = 0.0722, 1.0, 1.0
    o_ref, lse_ref = oracle.attend_one(q, kv, rows, sm, qs, ks)
    for n_parts in (1, 2, 7, 33):
        cuts = np.sort(rng.integers(0, L + 1, size=n_parts - 1))
        bounds = np.concatenate([[0], cuts, [L]])
        parts = [oracle.attend_one(q, kv, rows[a:b], sm, qs, ks) for a, b in zip(bounds[:-1], bounds[1:])]
        o, lse = oracle.merge(np.stack([p[0] for p in parts]), np.array([p[1] for p in parts]))
        assert np.allclose(o, o_ref, rtol=1e-11, atol=1e-14)
        assert lse == pytest.approx(lse_ref, rel=1e-12, abs=1e-12)


def test_merge_special_cases():
    a = np.arange(6.0).reshape(1, 6)
    o, lse = oracle.merge(a, [1.5])
    assert np.array_equal(o, a[0]) and lse == 1.5
    o, lse = oracle.merge(np.stack([a[0], 100 + a[0]]), [-np.inf, 0.25])
    assert np.array_equal(o, 100 + a[0]) and lse == 0.25
    o, lse = oracle.merge(np.stack([a[0], 2 * a[0]]), [0.5, 0.5])      # equal weights: mean
    assert np.allclose(o, 1.5 * a[0]) and lse == pytest.approx(0.5 + math.log(2))
    o, lse = oracle.merge(np.stack([a[0], a[0]]), [-np.inf, -np.inf])   # nothing attended
    assert np.array_equal(o, np.zeros(6)) and lse == -np.inf
    # weights e^lse: lse = (0, ln 3) -> weights 1:3
    o, lse = oracle.merge(np.stack([np.zeros(6), 4 * np.ones(6)]), [0.0, math.log(3.0)])
    assert np.allclose(o, 3.0) and lse == pytest.approx(math.log(4.0))


# ---------------------------------------------------------------- P5: index handling

def test_poisoned_rows_and_tail_are_never_read():
    case = mla_inputs.make_custom([33, 64, 5], q_lens=[1, 4, 2], H=2, seed=5, poison=True,
                                  index_buffer=200)
    kv = case.kv.numpy()
    assert (kv == mla_inputs.POISON_FP8).all(axis=1).sum() > 0
    o, lse = _oracle(case)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


def test_out_of_range_index_is_an_error():
    rng = np.random.default_rng(1)
    kv = _rows(rng, 8)
    q = _rows(rng, 1)[0]
    with pytest.raises(ValueError):
        oracle.attend_one(q, kv, [0, 8], 0.07, 1.0, 1.0)


def test_needle_identifies_attended_position_and_causal_limit():
    """One row with a dominant logit and a one-hot value: o points at that row only when
    the row's position is inside the query's attended set."""
    L, T = 20, 4
    kv = np.zeros((L, 576), dtype=np.uint8)          # fp8 zero rows: logit 0, value 0
    q = np.zeros((T, 1, 576), dtype=np.uint8)
    one = torch.tensor([1.0]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    big = torch.tensor([16.0]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    q[:, 0, 0] = big
    needle_pos = L - 2                               # seen by drafts t >= T - 2
    perm = np.random.default_rng(3).permutation(L).astype(np.int32)
    needle_row = perm[needle_pos]
    kv[needle_row, 0] = big                          # logit = c * 256
    kv[needle_row, 100] = one                        # one-hot value at column 100
    o, lse = oracle.decode(q, kv, [0, T], [0, L], perm, 1.0, 1.0, 1.0)
    for t in range(T):
        sees = needle_pos <= L - T + t
        assert (o[t, 0, 100] > 0.999) == sees
        if not sees:
            assert np.array_equal(o[t, 0], np.zeros(512))
            assert lse[t, 0] == pytest.approx(math.log(L - T + t + 1))


# ---------------------------------------------------------------- P6: head independence

def test_zero_padded_heads_leave_real_heads_bit_identical():
    case = mla_inputs.make_custom([70, 9], H=12, seed=9)
    a = _np(case)
    sm, qs, ks = case.scales()
    o12, lse12 = oracle.decode(a["q"], a["kv"], a["qo"], a["kvp"], a["idx"], sm, qs, ks)
    q16 = np.zeros((a["q"].shape[0], 16, 576), dtype=np.uint8)
    q16[:, :12] = a["q"]
    o16, lse16 = oracle.decode(q16, a["kv"], a["qo"], a["kvp"], a["idx"], sm, qs, ks)
    assert np.array_equal(o16[:, :12], o12) and np.array_equal(lse16[:, :12], lse12)


# ---------------------------------------------------------------- edge cases

def test_empty_and_short_requests():
    case = mla_inputs.make_custom([0, 3], q_lens=[0, 3], H=2, seed=4)
    o, lse = _oracle(case)
    assert o.shape == (3, 2, 512)
    # T = L = 3: draft 0 attends exactly one position
    a = _np(case)
    sm, qs, ks = case.scales()
    r0 = int(a["idx"][0])
    v = brute.fp8_decode(a["kv"][r0])
    assert np.allclose(o[0, 0], ks * v[:512], rtol=1e-13)
    with pytest.raises(ValueError):   # kv_len < q_len is rejected
        oracle.decode(a["q"], a["kv"], [0, 3], [0, 2], a["idx"], sm, qs, ks)


# ---------------------------------------------------------------- figures on the pages

def test_page_constants_and_accounting():
    g = json.load(open(GOLDEN))
    assert mla_inputs.SM_SCALE == g["sm_scale"]["value"]
    assert mla_inputs.SM_SCALE == pytest.approx(1.0 / math.sqrt(g["sm_scale"]["qk_head_dim"]), rel=1e-15)
    assert np.float32(mla_inputs.SM_SCALE) == np.float32(1.0 / math.sqrt(192.0))
    geo = g["geometry"]
    assert mla_inputs.D == geo["kv_entry_width"] == geo["kv_lora_rank"] + geo["qk_rope_head_dim"]
    assert mla_inputs.DV == geo["kv_lora_rank"]
    for key in ("c16_late_step", "c24_late_step"):
        f = g[key]
        n = f["kv_len_sum"]
        assert mla_inputs.gathered_kv_bytes([n]) / 2**20 == pytest.approx(f["kv_bytes_mib"], abs=0.5)
        assert 4 * n / 2**20 == pytest.approx(f["index_bytes_mib"], abs=0.05)
        assert mla_inputs.useful_flops([n], [1], 16) / 1e9 == pytest.approx(f["gflop_padded_16_heads"], abs=0.05)
        assert mla_inputs.useful_flops([n], [1], 12) / 1e9 == pytest.approx(f["gflop_useful_12_heads"], abs=0.05)
    kb = g["kv_buffer"]
    assert kb["rows"] * 576 / 1e9 == pytest.approx(kb["bytes_gb"], abs=0.005)
    lc = g["long_context"]
    assert lc["layers"] * lc["positions"] * 576 / 1e9 == pytest.approx(lc["payload_gb"], abs=0.005)


def test_workload_shapes():
    t = mla_inputs.make_case("tiny")
    assert t.q.shape == (2, 12, 576) and t.kv.shape == (1024, 576)
    assert t.kv_indptr.tolist() == [0, 256, 556] and t.kv_indices.numel() == 1024
    assert sorted(t.kv_indices.tolist()) == list(range(1024))
    lens = mla_inputs._shared_prefix_lens(16, 0)
    assert all(68000 <= L < 68350 for L in lens)
    m = mla_inputs._mtp_lens(64, 0)
    assert all(2048 <= L <= 65536 for L in m)


# ---------------------------------------------------------------- paged caches (page_size > 1)

def test_expand_pages_hand_example():
    """Pages [3, 0] with 2 slots used in the last, then page [5] full, at 4 slots a page."""
    ptr, rows = oracle.expand_pages([0, 2, 3], [3, 0, 5], [2, 4], 4)
    assert ptr.tolist() == [0, 6, 10]
    assert rows.tolist() == [12, 13, 14, 15, 0, 1, 20, 21, 22, 23]
    with pytest.raises(ValueError):
        oracle.expand_pages([0, 1], [0], [5], 4)      # more slots than a page holds
    with pytest.raises(ValueError):
        oracle.expand_pages([0, 1], [0], [0], 4)      # an empty last page


def _paged_case(seed, page_size, lens, q_lens, H=3, n_pages=40):
    rng = np.random.default_rng(seed)
    kv = _rows(rng, n_pages * page_size).reshape(n_pages, page_size, 576)
    perm = rng.permutation(n_pages)
    counts = [(L + page_size - 1) // page_size for L in lens]
    kvp = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    idx = perm[:kvp[-1]].astype(np.int32)
    last = np.array([L - (c - 1) * page_size for L, c in zip(lens, counts)], dtype=np.int32)
    qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = _rows(rng, int(qo[-1]) * H).reshape(int(qo[-1]), H, 576)
    return q, kv, qo, kvp, idx, last


@pytest.mark.parametrize("page_size", [4, 16])
def test_paged_decode_matches_brute_force(page_size):
    """Brute force gathers each request's rows by the page axis of the cache
    (kv[pages].reshape(-1, 576)[:L]), not by row arithmetic."""
    lens, q_lens = [37, 5, 64, 17], [1, 3, 2, 1]
    q, kv, qo, kvp, idx, last = _paged_case(11 + page_size, page_size, lens, q_lens)
    sm, qs, ks = 0.11, 0.8, 0.9
    o, lse = oracle.decode_paged(q, kv, qo, kvp, idx, last, page_size, sm, qs, ks)
    for b, (L, T) in enumerate(zip(lens, q_lens)):
        rows_b = kv[idx[kvp[b]:kvp[b + 1]]].reshape(-1, 576)[:L]
        for t in range(T):
            r = qo[b] + t
            for h in range(q.shape[1]):
                bo, blse = brute.attend(q[r, h], rows_b[:L - T + t + 1], sm * qs * ks, ks)
                assert np.allclose(o[r, h], bo, rtol=1e-12, atol=1e-14)
                assert abs(lse[r, h] - blse) < 1e-12


def test_paged_page_size_one_is_the_token_decode():
    q, kv, qo, kvp, idx, last = _paged_case(5, 1, [9, 30, 2], [1, 2, 1], n_pages=64)
    a = oracle.decode_paged(q, kv, qo, kvp, idx, last, 1, 0.2, 1.0, 1.0)
    b = oracle.decode(q, kv.reshape(-1, 576), qo, kvp, idx, 0.2, 1.0, 1.0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_paged_unused_slots_are_never_attended():
    """Filling the unused slots of every last page with the largest finite e4m3 value
    (logits far above the rest) leaves the result unchanged."""
    page_size, lens = 8, [13, 3, 24]
    q, kv, qo, kvp, idx, last = _paged_case(7, page_size, lens, [1, 1, 2])
    base = oracle.decode_paged(q, kv, qo, kvp, idx, last, page_size, 0.3, 1.0, 1.0)
    kv2 = kv.copy()
    for b in range(len(lens)):
        pg = idx[kvp[b + 1] - 1]
        kv2[pg, last[b]:, :] = 0x7E   # 448
    poisoned = oracle.decode_paged(q, kv2, qo, kvp, idx, last, page_size, 0.3, 1.0, 1.0)
    assert np.array_equal(base[0], poisoned[0]) and np.array_equal(base[1], poisoned[1])


# ---------------------------------------------------------------- latent o -> v_head_dim

def test_bf16_decode_exact_values():
    """bf16 words of known values: 1, -2, 0.5, the smallest normal, the largest finite,
    +inf and a value with every mantissa bit set."""
    words = np.array([0x3F80, 0xC000, 0x3F00, 0x0080, 0x7F7F, 0x7F80, 0x3FFF], dtype=np.uint16)
    got = oracle.bf16_to_f64(words)
    want = [1.0, -2.0, 0.5, 2.0 ** -126, (2 - 2 ** -7) * 2.0 ** 127, np.inf, 1 + (2 ** 7 - 1) / 2 ** 7]
    assert list(got) == want
    # agrees with torch's own bf16 -> float conversion on random words
    rng = np.random.default_rng(3)
    w = rng.integers(0, 1 << 16, size=4096, dtype=np.uint32).astype(np.uint16)
    w = w[(w & 0x7F80) != 0x7F80]            # finite values only
    ref = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.bf16_to_f64(w), ref)


def test_latent_to_v_brute_force():
    """Triple loop over (t, h, n) with a running sum over k, on small random sizes."""
    rng = np.random.default_rng(21)
    T, H, K, N = 3, 4, 7, 5
    o = rng.standard_normal((T, H, K))
    w = rng.standard_normal((H, K, N))
    got = oracle.latent_to_v(o, w)
    for t in range(T):
        for h in range(H):
            for n in range(N):
                acc = 0.0
                for k in range(K):
                    acc += o[t, h, k] * w[h, k, n]
                assert abs(got[t, h, n] - acc) <= 1e-12 * (1 + abs(acc))


def test_latent_to_v_closed_forms():
    rng = np.random.default_rng(22)
    T, H, K, N = 2, 3, 512, 128
    w = rng.standard_normal((H, K, N))
    # a one-hot latent row picks row k0 of its own head's matrix
    o = np.zeros((T, H, K))
    o[1, 2, 300] = 1.0
    v = oracle.latent_to_v(o, w)
    assert np.array_equal(v[1, 2], w[2, 300]) and not v[0].any() and not v[1, :2].any()
    # identity matrices (w[h, k, n] = [k == n]) return the first N latent columns
    eye = np.zeros((H, K, N))
    eye[:, np.arange(N), np.arange(N)] = 1.0
    o = rng.standard_normal((T, H, K))
    assert np.array_equal(oracle.latent_to_v(o, eye), o[:, :, :N])
    # heads are independent: permuting the matrices permutes the outputs head by head
    perm = np.array([2, 0, 1])
    o_same = np.repeat(o[:, :1, :], H, axis=1)   # every head sees the same latent row
    v1 = oracle.latent_to_v(o_same, w)
    v2 = oracle.latent_to_v(o_same, w[perm])
    assert np.allclose(v2, v1[:, perm], rtol=0, atol=1e-12)
    # linear in o
    o2 = rng.standard_normal((T, H, K))
    assert np.allclose(oracle.latent_to_v(2 * o - o2, w),
                       2 * oracle.latent_to_v(o, w) - oracle.latent_to_v(o2, w), atol=1e-9)
