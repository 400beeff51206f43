"""Pins of the oracle of the fused step before the decode (q rope + concat + fp8 cache
write, "[Kimi-K3 MLA TP8] MLA performance" §3 "Entry point", §2 geometry 512 + 64): each
check ties oracle.rope_concat_cache or oracle.e4m3_encode to something other than itself --
torch's own e4m3fn cast, exact complex multiplication, closed forms of special tables, a
permutation identity between the two pair conventions, and the cache's page axis."""
import numpy as np
import pytest
import torch

import oracle

D = 576


def torch_e4m3(x):
    """torch's independent e4m3fn encoder (round to nearest even) on float32 values."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def bf16_bits(x):
    """bf16 bit patterns (uint16) of float values, rounded by torch."""
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def bf16_vals(bits):
    return oracle.bf16_to_f64(bits).astype(np.float32)


def test_encoder_matches_torch_on_random_values():
    rng = np.random.default_rng(0)
    mags = np.exp2(rng.uniform(-12, np.log2(460.0), 4000))
    x = (mags * rng.choice([-1.0, 1.0], mags.size)).astype(np.float32)
    ours = np.array([oracle.e4m3_encode(float(v)) for v in x], dtype=np.uint8)
    assert (ours == torch_e4m3(x)).all()


def test_encoder_ties_go_to_the_even_code_and_saturates():
    table = oracle.fp8_e4m3fn_table()
    for c in range(0, 0x7E):
        mid = (table[c] + table[c + 1]) / 2.0          # exact in fp32 (few bits)
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even
        assert oracle.e4m3_encode(-mid) == 0x80 | even
        assert torch_e4m3([mid])[0] == even
    for big in (448.0, 449.0, 464.0, 500.0, 1e6, float("inf")):
        assert oracle.e4m3_encode(big) == 0x7E
        assert oracle.e4m3_encode(-big) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    assert oracle.e4m3_encode(-0.0) == 0x80 and oracle.e4m3_encode(-1e-12) == 0x80


def test_encoder_round_trips_every_finite_code():
    table = oracle.fp8_e4m3fn_table()
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(table[c]) == c


def _inputs(T, H, seed, lo=None, hi=None, max_pos=64):
    rng = np.random.default_rng(seed)

    def vals(*shape):
        v = rng.standard_normal(shape).astype(np.float32)
        if lo is not None:   # magnitudes in [lo, hi): few exponents, for exact products
            v = np.sign(v + 1e-9) * rng.uniform(lo, hi, shape).astype(np.float32)
        return bf16_bits(v)

    return dict(q_nope=vals(T, H, 512), q_pe=vals(T, H, 64), kv_c=vals(T, 512), k_pe=vals(T, 64),
                positions=rng.integers(0, max_pos, T).astype(np.int32))


def _run(inp, cos_sin, neox, slots, q_scale, kv_scale, cache):
    return oracle.rope_concat_cache(inp["q_nope"], inp["q_pe"], inp["kv_c"], inp["k_pe"],
                                    inp["positions"], cos_sin, neox, slots, q_scale, kv_scale,
                                    cache)


def _table(cos, sin, max_pos=64):
    t = np.zeros((max_pos, 64), np.float32)
    t[:, :32] = cos
    t[:, 32:] = sin
    return t


def _pairs(neox):
    i = np.arange(32)
    return (i, i + 32) if neox else (2 * i, 2 * i + 1)


@pytest.mark.parametrize("neox", [0, 1])
def test_identity_table_is_plain_concat_and_quantise(neox):
    T, H, qs, ks = 5, 3, np.float32(0.05), np.float32(0.1)
    inp = _inputs(T, H, 1)
    cache = np.full((16, D), 0x7F, np.uint8)
    slots = np.array([3, -1, 0, 15, 7], np.int32)
    q_out, new_cache, err = _run(inp, _table(1.0, 0.0), neox, slots, qs, ks, cache)
    assert err == 0
    want_q = np.concatenate([torch_e4m3(bf16_vals(inp["q_nope"]) / qs),
                             torch_e4m3(bf16_vals(inp["q_pe"]) / qs)], axis=2)
    assert (q_out == want_q).all()
    want_rows = np.concatenate([torch_e4m3(bf16_vals(inp["kv_c"]) / ks),
                                torch_e4m3(bf16_vals(inp["k_pe"]) / ks)], axis=1)
    for t, s in enumerate(slots):
        if s >= 0:
            assert (new_cache[s] == want_rows[t]).all()
    untouched = np.setdiff1d(np.arange(16), slots[slots >= 0])
    assert (new_cache[untouched] == 0x7F).all()


@pytest.mark.parametrize("neox", [0, 1])
def test_quarter_turn_swaps_each_pair_with_a_sign(neox):
    """cos 0, sin 1: (x, y) -> (-y, x) for every pair of the convention."""
    T, H, qs, ks = 3, 2, np.float32(0.5), np.float32(0.25)
    inp = _inputs(T, H, 2)
    q_out, cache, err = _run(inp, _table(0.0, 1.0), neox, np.arange(T, dtype=np.int32), qs, ks,
                             np.zeros((T, D), np.uint8))
    assert err == 0
    a, b = _pairs(neox)
    x = bf16_vals(inp["q_pe"])
    assert (q_out[..., 512 + a] == torch_e4m3(-x[..., b] / qs)).all()
    assert (q_out[..., 512 + b] == torch_e4m3(x[..., a] / qs)).all()
    k = bf16_vals(inp["k_pe"])
    assert (cache[:, 512 + a] == torch_e4m3(-k[:, b] / ks)).all()
    assert (cache[:, 512 + b] == torch_e4m3(k[:, a] / ks)).all()


@pytest.mark.parametrize("neox", [0, 1])
def test_rotation_equals_exact_complex_product(neox):
    """With dyadic cos/sin of few bits, inputs of a few binades and power-of-two scales,
    every fp32 operation is exact, so the codes must equal the e4m3 of the exact complex
    product (x + iy)(cos + i sin) / scale."""
    T, H, max_pos = 6, 4, 8
    qs, ks = np.float32(0.5), np.float32(0.125)
    rng = np.random.default_rng(3)
    choices = np.array([0.5, 0.625, 0.75, 0.875, 1.0, -0.5, -0.75, -1.0], np.float32)
    cs = np.zeros((max_pos, 64), np.float32)
    cs[:, :32] = rng.choice(choices, (max_pos, 32))
    cs[:, 32:] = rng.choice(choices, (max_pos, 32))
    inp = _inputs(T, H, 4, lo=0.25, hi=4.0, max_pos=max_pos)
    q_out, cache, err = _run(inp, cs, neox, np.arange(T, dtype=np.int32), qs, ks,
                             np.zeros((T, D), np.uint8))
    assert err == 0
    a, b = _pairs(neox)
    for src, scale, got in ((bf16_vals(inp["q_pe"]), qs, q_out[..., 512:]),
                            (bf16_vals(inp["k_pe"])[:, None, :], ks, cache[:, None, 512:])):
        z = src[..., a].astype(np.float64) + 1j * src[..., b].astype(np.float64)
        rot = cs[inp["positions"]].astype(np.float64)
        w = rot[:, None, :32] + 1j * rot[:, None, 32:]
        r = z * w / float(scale)
        want = np.empty(got.shape, np.uint8)
        want[..., a] = torch_e4m3(r.real.astype(np.float32))
        want[..., b] = torch_e4m3(r.imag.astype(np.float32))
        assert (got == want).all()


@pytest.mark.parametrize("neox", [0, 1])
def test_rotation_near_exact_on_random_tables(neox):
    """Random angles: the codes equal the e4m3 of the fp64 complex product except where
    that value lies within fp32 rounding (2^-20 relative) of a rounding boundary."""
    T, H, max_pos = 8, 4, 32
    qs, ks = np.float32(0.05), np.float32(0.1)
    rng = np.random.default_rng(5)
    th = rng.uniform(-np.pi, np.pi, (max_pos, 32))
    cs = _table(0, 0, max_pos)
    cs[:, :32], cs[:, 32:] = np.cos(th), np.sin(th)
    inp = _inputs(T, H, 6, max_pos=max_pos)
    q_out, _, err = _run(inp, cs, neox, np.full(T, -1, np.int32), qs, ks,
                         np.zeros((1, D), np.uint8))
    assert err == 0
    a, b = _pairs(neox)
    x = bf16_vals(inp["q_pe"]).astype(np.float64)
    rot = cs[inp["positions"]].astype(np.float64)
    c, s = rot[:, None, :32], rot[:, None, 32:]
    ra = (x[..., a] * c - x[..., b] * s) / float(qs)
    rb = (x[..., b] * c + x[..., a] * s) / float(qs)
    table = oracle.fp8_e4m3fn_table()
    mids = np.sort(np.concatenate([(table[:0x7E] + table[1:0x7F]) / 2.0]))
    checked = 0
    for vals, cols in ((ra, a), (rb, b)):
        want = torch_e4m3(vals.astype(np.float32))
        got = q_out[..., 512 + cols]
        m = np.abs(vals)
        near = np.abs(mids[np.clip(np.searchsorted(mids, m), 0, mids.size - 1)] - m) <= 2 ** -20 * m
        near |= np.abs(mids[np.clip(np.searchsorted(mids, m) - 1, 0, mids.size - 1)] - m) <= 2 ** -20 * m
        assert (got[~near] == want[~near]).all()
        checked += int((~near).sum())
    assert checked > 0.99 * 2 * T * H * 32


def test_halves_convention_is_the_interleaved_one_on_permuted_columns():
    """Rotating pairs (i, i+32) equals rotating pairs (2i, 2i+1) after moving column i to
    2i and column i+32 to 2i+1, and moving the result back."""
    T, H = 4, 3
    rng = np.random.default_rng(7)
    th = rng.uniform(-np.pi, np.pi, (16, 32))
    cs = _table(0, 0, 16)
    cs[:, :32], cs[:, 32:] = np.cos(th), np.sin(th)
    inp = _inputs(T, H, 8, max_pos=16)
    perm = np.empty(64, np.int64)              # interleaved column j takes halves column perm[j]
    perm[0::2], perm[1::2] = np.arange(32), np.arange(32) + 32
    inp_i = dict(inp, q_pe=np.ascontiguousarray(inp["q_pe"][..., perm]),
                 k_pe=np.ascontiguousarray(inp["k_pe"][..., perm]))
    slots = np.arange(T, dtype=np.int32)
    q_h, c_h, _ = _run(inp, cs, 1, slots, 0.05, 0.1, np.zeros((T, D), np.uint8))
    q_i, c_i, _ = _run(inp_i, cs, 0, slots, 0.05, 0.1, np.zeros((T, D), np.uint8))
    assert (q_h[..., 512 + perm] == q_i[..., 512:]).all()
    assert (c_h[:, 512 + perm] == c_i[:, 512:]).all()
    assert (q_h[..., :512] == q_i[..., :512]).all()


def test_each_token_uses_its_own_table_row():
    """Identity rows everywhere except row 5 (a quarter turn): only tokens at position 5
    have their pairs swapped."""
    T, H = 6, 2
    cs = _table(1.0, 0.0, 8)
    cs[5, :32], cs[5, 32:] = 0.0, 1.0
    inp = _inputs(T, H, 9, max_pos=8)
    inp["positions"] = np.array([0, 5, 7, 5, 1, 2], np.int32)
    q_out, _, _ = _run(inp, cs, 0, np.full(T, -1, np.int32), 1.0, 1.0, np.zeros((1, D), np.uint8))
    x = bf16_vals(inp["q_pe"])
    a, b = _pairs(0)
    for t in range(T):
        if inp["positions"][t] == 5:
            assert (q_out[t][:, 512 + a] == torch_e4m3(-x[t][:, b])).all()
        else:
            assert (q_out[t, :, 512:] == torch_e4m3(x[t])).all()


def test_paged_cache_rows_land_in_page_and_slot():
    """slot id = page * page_size + slot: checked on the page axis of a (pages, PS, 1, 576)
    cache, with untouched slots keeping their poison."""
    T, H, PS, pages = 5, 2, 16, 6
    inp = _inputs(T, H, 10)
    cache = np.full((pages, PS, 1, D), 0x7F, np.uint8)
    where = [(4, 3), (0, 15), (5, 0), (2, 9), (4, 4)]
    slots = np.array([p * PS + s for p, s in where], np.int32)
    _, new_cache, err = _run(inp, _table(1.0, 0.0), 0, slots, 0.05, 0.1, cache)
    assert err == 0
    rows = np.concatenate([torch_e4m3(bf16_vals(inp["kv_c"]) / np.float32(0.1)),
                           torch_e4m3(bf16_vals(inp["k_pe"]) / np.float32(0.1))], axis=1)
    mask = np.ones((pages, PS), bool)
    for t, (p, s) in enumerate(where):
        assert (new_cache[p, s, 0] == rows[t]).all()
        mask[p, s] = False
    assert (new_cache[mask] == 0x7F).all()


def test_dequantised_entry_is_the_rotated_value_within_half_an_fp8_step():
    """code * scale returns the real rotated value to within e4m3's half-step (2^-4
    relative for normal codes): the scale divides on the way in."""
    T, H, qs, ks = 4, 2, np.float32(0.05), np.float32(0.1)
    rng = np.random.default_rng(11)
    th = rng.uniform(-np.pi, np.pi, (8, 32))
    cs = _table(0, 0, 8)
    cs[:, :32], cs[:, 32:] = np.cos(th), np.sin(th)
    inp = _inputs(T, H, 12, max_pos=8)
    _, cache, _ = _run(inp, cs, 0, np.arange(T, dtype=np.int32), qs, ks, np.zeros((T, D), np.uint8))
    table = oracle.fp8_e4m3fn_table()
    k = bf16_vals(inp["k_pe"]).astype(np.float64)
    rot = cs[inp["positions"]].astype(np.float64)
    real = np.empty((T, 64))
    real[:, 0::2] = k[:, 0::2] * rot[:, :32] - k[:, 1::2] * rot[:, 32:]
    real[:, 1::2] = k[:, 1::2] * rot[:, :32] + k[:, 0::2] * rot[:, 32:]
    back = table[cache[:, 512:]] * float(ks)
    normal = np.abs(real) >= 2 ** -6 * float(ks)
    assert (np.abs(back - real)[normal] <= 2 ** -4 * np.abs(real)[normal] * 1.0001).all()
    lat = table[cache[:, :512]] * float(ks)
    kv = bf16_vals(inp["kv_c"]).astype(np.float64)
    nz = np.abs(kv) >= 2 ** -6 * float(ks)
    assert (np.abs(lat - kv)[nz] <= 2 ** -4 * np.abs(kv)[nz] * 1.0001).all()


def test_errors_leave_the_named_bytes_unwritten():
    T, H = 3, 2
    inp = _inputs(T, H, 13, max_pos=4)
    inp["positions"] = np.array([1, 9, -2], np.int32)   # tokens 1 and 2 outside the table
    cache = np.full((4, D), 0x7F, np.uint8)
    slots = np.array([0, 1, 7], np.int32)                # slot 7 outside the cache
    q_out, new_cache, err = _run(inp, _table(1.0, 0.0, 4), 0, slots, 1.0, 1.0, cache)
    assert err == 3
    assert (q_out[0] != 0x7F).any() and (q_out[1:, :, 512:] == 0x7F).all()
    assert (q_out[1:, :, :512] == torch_e4m3(bf16_vals(inp["q_nope"][1:]))).all()
    assert (new_cache[1, :512] == torch_e4m3(bf16_vals(inp["kv_c"][1]))).all()
    assert (new_cache[1, 512:] == 0x7F).all()
    assert (new_cache[2:] == 0x7F).all()
