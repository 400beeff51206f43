"""Host simulation of the split-KV schedule (CPU only).

tests/native/sched_sim.cpp compiles the library's scheduling header with g++ and runs the
decode kernel's piece iterator for every CTA and the merge kernel's partial lookup for
every unit.  These tests check the properties the GPU path relies on: every attended
position of every (request, row group) is covered exactly once, a unit is written
directly iff one piece covers it, partial slots are unique and inside the workspace, and
the merge finds exactly the slots the decode wrote.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "native", "sched_sim.cpp")
HDR = os.path.join(os.path.dirname(HERE), "paged_mla_latent_gb300", "csrc", "mla_sched.cuh")
LIB = os.path.join(HERE, "native", "_build", "libschedsim.so")


@pytest.fixture(scope="module")
def sim():
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if (not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(SRC),
                                                                  os.path.getmtime(HDR))):
        tmp = LIB + f".{os.getpid()}"
        subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-o", tmp, SRC], check=True)
        os.replace(tmp, LIB)
    lib = ctypes.CDLL(LIB)
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.sched_pieces.restype = ctypes.c_int64
    lib.sched_pieces.argtypes = [i32p, i32p] + [ctypes.c_int] * 6 + [i64p, ctypes.c_int64]
    lib.sched_unit_partials.restype = ctypes.c_int
    lib.sched_unit_partials.argtypes = [i32p, i32p] + [ctypes.c_int] * 8 + [i64p, ctypes.POINTER(ctypes.c_int)]
    lib.sched_pieces_mode.restype = ctypes.c_int64
    lib.sched_pieces_mode.argtypes = [i32p, i32p] + [ctypes.c_int] * 9 + [i64p, ctypes.c_int64]
    lib.sched_unit_partials_mode.restype = ctypes.c_int
    lib.sched_unit_partials_mode.argtypes = ([i32p, i32p] + [ctypes.c_int] * 11 +
                                             [i64p, ctypes.POINTER(ctypes.c_int)])
    lib.sched_pieces_cost.restype = ctypes.c_int64
    lib.sched_pieces_cost.argtypes = [i32p, i32p] + [ctypes.c_int] * 12 + [i64p, ctypes.c_int64]
    lib.sched_unit_partials_cost.restype = ctypes.c_int
    lib.sched_unit_partials_cost.argtypes = ([i32p, i32p] + [ctypes.c_int] * 14 +
                                             [i64p, ctypes.POINTER(ctypes.c_int)])
    ip = ctypes.POINTER(ctypes.c_int)
    lib.sched_host_costs.restype = None
    lib.sched_host_costs.argtypes = [ctypes.c_int] * 3 + [ip, ip, ip]
    lib.sched_pieces_paged.restype = ctypes.c_int64
    lib.sched_pieces_paged.argtypes = ([i32p, i32p] + [ctypes.c_int] * 7 + [i32p] +
                                       [ctypes.c_int] * 2 + [i64p, ctypes.c_int64])
    lib.sched_unit_partials_paged.restype = ctypes.c_int
    lib.sched_unit_partials_paged.argtypes = ([i32p, i32p] + [ctypes.c_int] * 7 + [i32p] +
                                              [ctypes.c_int] * 4 + [i64p, ctypes.POINTER(ctypes.c_int)])
    lib.sched_pieces_full.restype = ctypes.c_int64
    lib.sched_pieces_full.argtypes = ([i32p, i32p] + [ctypes.c_int] * 13 + [i32p] +
                                      [i64p, ctypes.c_int64])
    lib.sched_unit_partials_full.restype = ctypes.c_int
    lib.sched_unit_partials_full.argtypes = ([i32p, i32p] + [ctypes.c_int] * 13 + [i32p] +
                                             [ctypes.c_int] * 2 + [i64p, ctypes.POINTER(ctypes.c_int)])
    lib.sched_request_len.restype = ctypes.c_int
    lib.sched_request_len.argtypes = [i32p, ctypes.c_int, i32p, ctypes.c_int]
    lib.sched_partial_slots.restype = ctypes.c_int64
    lib.sched_partial_slots.argtypes = [ctypes.c_int] * 4
    return lib


def pick_ng(rows):
    return 16 if rows <= 16 else (32 if rows <= 32 else (48 if rows <= 48 else 96))


def cascade_ng(rows, B):
    """The shared-prefix cascade's group rows as the library picks them: 96 when a group of
    at least two requests fits and the batch fills one, else 48."""
    return 96 if rows <= 48 and B >= 96 // rows else 48


def host_costs(sim, mode, NG, rows):
    w, wp, e = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    sim.sched_host_costs(mode, NG, rows, ctypes.byref(w), ctypes.byref(wp), ctypes.byref(e))
    return w.value, wp.value, e.value


# cost-line weights (w_own, w_prefix, piece_cost): none (plain position line), the ones the
# library sets ("host"), and odd ones
COSTS = ["none", "host", (7, 11, 999)]


def resolve_costs(sim, costs, mode, NG, rows):
    if costs == "none":
        return (0, 0, 0)
    if costs == "host":
        return host_costs(sim, mode, NG, rows)
    return costs


def simulate(sim, kv_lens, q_lens, H, splits, grid, costs="none"):
    kvp = np.concatenate([[0], np.cumsum(kv_lens)]).astype(np.int32)
    qop = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    B = len(kv_lens)
    rows = max(q_lens) * H
    NG = pick_ng(rows)
    groups = (rows + NG - 1) // NG
    w, wp, e = resolve_costs(sim, costs, 0, NG, rows)
    i32p = ctypes.POINTER(ctypes.c_int32)
    cap = 8 * (grid + B * groups * max(splits, 1) + 16)
    out = np.zeros(cap * 10, dtype=np.int64)
    n = sim.sched_pieces_cost(kvp.ctypes.data_as(i32p), qop.ctypes.data_as(i32p), B, H, NG, groups,
                              splits, grid, 0, 1, 0, w, wp, e,
                              out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), cap)
    assert n >= 0, f"simulation failed with {n}"
    pieces = out[:10 * n].reshape(n, 10)[:, :8]
    units = {}
    for b in range(B):
        for g in range(groups):
            first = ctypes.c_int64(0)
            count = ctypes.c_int(0)
            need = sim.sched_unit_partials_cost(kvp.ctypes.data_as(i32p), qop.ctypes.data_as(i32p),
                                                B, H, NG, groups, splits, grid, 0, 1, 0, w, wp, e,
                                                b, g, ctypes.byref(first), ctypes.byref(count))
            units[(b, g)] = (need, first.value, count.value)
    slots = sim.sched_partial_slots(B, groups, splits, grid)
    return pieces, units, slots, NG, groups


def check_schedule(sim, kv_lens, q_lens, H, splits, grid, costs="none"):
    pieces, units, n_slots, NG, groups = simulate(sim, kv_lens, q_lens, H, splits, grid, costs)
    B = len(kv_lens)
    by_unit = {}
    for cta, b, g, j0, j1, rows, slot, direct in pieces:
        assert 0 <= b < B and 0 <= g < groups and 0 <= j0 < j1 <= kv_lens[b]
        assert rows == min(NG, q_lens[b] * H - g * NG) and rows > 0
        by_unit.setdefault((b, g), []).append((j0, j1, slot, direct, cta))
    partial_slots = [p[6] for p in pieces if not p[7]]
    assert len(partial_slots) == len(set(partial_slots)), "partial slot written twice"
    assert all(0 <= s < n_slots for s in partial_slots)
    for b in range(B):
        for g in range(groups):
            real = q_lens[b] * H - g * NG > 0
            ps = sorted(by_unit.get((b, g), []))
            need, first, count = units[(b, g)]
            if not real or kv_lens[b] == 0:
                assert not ps
                continue
            # exact cover of [0, L)
            pos = 0
            for j0, j1, *_ in ps:
                assert j0 == pos, f"gap/overlap in unit {(b, g)}"
                pos = j1
            assert pos == kv_lens[b]
            if len(ps) == 1 and ps[0][3]:
                assert need == 0          # written directly, no merge
            else:
                assert need == 1 and not any(p[3] for p in ps)
                expect = set(range(first, first + count))
                got = {p[2] for p in ps}
                assert got <= expect
                if splits <= 0:
                    assert got == expect
                else:   # fixed policy: missing slots are exactly the empty pieces
                    empty = {first + k for k in range(count)
                             if (k + 1) * kv_lens[b] // splits <= k * kv_lens[b] // splits}
                    assert got == expect - empty
    return pieces


CASES = [
    ([1], [1], 12), ([2], [1], 12), ([128], [1], 12), ([300], [1], 12),
    ([256, 300], [1, 1], 12), ([1000, 2500, 130, 1, 257], [1] * 5, 12),
    ([3000, 700, 129], [1, 1, 1], 12), ([0, 400, 0], [1, 1, 1], 12),
    ([4, 130, 1000, 2049], [4] * 4, 12), ([300, 800, 50, 1200], [1, 3, 2, 4], 12),
    ([1500, 333], [1, 1], 96), ([1500, 333], [1, 1], 24), ([142000], [1], 12),
    ([68174] * 16, [1] * 16, 12), ([17750], [1], 96),
]


@pytest.mark.parametrize("kv_lens,q_lens,H", CASES)
@pytest.mark.parametrize("splits,costs", [(0, c) for c in COSTS] + [(k, "none") for k in (1, 2, 7)])
@pytest.mark.parametrize("grid", [1, 5, 152])
def test_schedule_covers_every_position_once(sim, kv_lens, q_lens, H, splits, grid, costs):
    # (the fixed policy has no cost line)
    check_schedule(sim, kv_lens, q_lens, H, splits, grid, costs)


def test_library_costs(sim):
    """The weights the library sets: one per position and 512 per piece on the plain line
    and the 48-row cascade; the cascade in 96-row groups charges 256 positions a piece and a
    prefix position 1.15 own ones (23 : 20)."""
    assert host_costs(sim, 0, 16, 12) == (1, 0, 512)
    assert host_costs(sim, 0, 48, 48) == (1, 0, 512)
    assert host_costs(sim, 0, 96, 96) == (1, 0, 512)
    assert host_costs(sim, 1, 48, 12) == (1, 0, 512)
    assert host_costs(sim, 1, 48, 24) == (1, 0, 512)
    assert host_costs(sim, 1, 96, 12) == (20, 23, 256 * 20)
    assert host_costs(sim, 2, 96, 24) == (20, 23, 256 * 20)


@pytest.mark.parametrize("costs", ["host", (7, 11, 999)])
def test_cost_line_balances_estimated_time(sim, costs):
    """With a piece cost e and weight w, every CTA's estimated time (e per piece it starts
    plus w per position) stays within e + 2w of the line's share W / Gp."""
    rng = np.random.default_rng(5)
    for kv_lens, q_lens, H in [([68174 + i for i in range(16)], [1] * 16, 12),
                               ([int(x) for x in rng.integers(9000, 30000, size=64)], [4] * 64, 12),
                               ([int(x) for x in rng.integers(1, 5000, size=40)], [1] * 40, 12)]:
        pieces = check_schedule(sim, kv_lens, q_lens, H, 0, 152, costs)
        rows = max(q_lens) * H
        NG = pick_ng(rows)
        groups = (rows + NG - 1) // NG
        w, _, e = resolve_costs(sim, costs, 0, NG, rows)
        w = max(w, 1)
        est = np.zeros(152, dtype=np.int64)
        for cta, b, g, j0, j1, *_ in pieces:
            est[cta] += w * (j1 - j0) + (e if j0 == 0 else 0)
        W = groups * sum(e + w * L for L in kv_lens)
        Gp = min(152, max(1, groups * sum(kv_lens) // 256))
        used = est[:Gp]
        assert np.abs(used - W / Gp).max() <= e + 2 * w + 1, (used.min(), used.max(), W / Gp)
        assert (est[Gp:] == 0).all()


def test_auto_policy_balances_rows(sim):
    kv_lens = [68174 + i for i in range(16)]
    pieces = check_schedule(sim, kv_lens, [1] * 16, 12, 0, 152)
    per_cta = np.zeros(152, dtype=np.int64)
    for cta, b, g, j0, j1, *_ in pieces:
        per_cta[cta] += j1 - j0
    W = sum(kv_lens)
    assert per_cta.max() - per_cta.min() <= 1
    assert per_cta.sum() == W


def test_batch1_long_context_fills_every_sm(sim):
    pieces = check_schedule(sim, [142000], [1], 12, 0, 152)
    assert len({p[0] for p in pieces}) == 152


def test_random_batches(sim):
    rng = np.random.default_rng(0)
    for _ in range(40):
        B = int(rng.integers(1, 20))
        T = int(rng.integers(1, 5))
        kv = [int(x) for x in rng.integers(0, 3000, size=B)]
        q = [int(min(t, L)) if L > 0 else 0 for t, L in zip(rng.integers(1, T + 1, size=B), kv)]
        H = int(rng.choice([12, 16, 24, 96]))
        if max(q) == 0:
            continue
        for splits in (0, 1, 3):
            for grid in (1, 7, 152):
                for costs in (COSTS if splits == 0 else ["none"]):
                    check_schedule(sim, kv, q, H, splits, grid, costs)


# ------------------------------------------------------------------ shared-prefix cascade

MIN_SHARED = 1024   # prefixes shorter than this are not split off


def cascade_pieces(sim, kvp, qop, B, H, NG, groups, grid, mode, gsize, shared, costs=(0, 0, 0)):
    i32p = ctypes.POINTER(ctypes.c_int32)
    cap = 8 * (grid + B * groups + 16)
    out = np.zeros(cap * 10, dtype=np.int64)
    n = sim.sched_pieces_cost(kvp.ctypes.data_as(i32p), qop.ctypes.data_as(i32p), B, H, NG, groups,
                              0, grid, mode, gsize, shared, *costs,
                              out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), cap)
    assert n >= 0, f"simulation failed with {n}"
    return out[:10 * n].reshape(n, 10)


def cascade_partials(sim, kvp, qop, B, H, NG, groups, grid, mode, gsize, shared, v, g,
                     costs=(0, 0, 0)):
    i32p = ctypes.POINTER(ctypes.c_int32)
    first = ctypes.c_int64(0)
    count = ctypes.c_int(0)
    need = sim.sched_unit_partials_cost(kvp.ctypes.data_as(i32p), qop.ctypes.data_as(i32p), B, H,
                                        NG, groups, 0, grid, mode, gsize, shared, *costs, v, g,
                                        ctypes.byref(first), ctypes.byref(count))
    return need, first.value, count.value


def check_cascade(sim, kv_lens, q_lens, H, grid, shared, costs="none"):
    """The cascade line (prefix units: groups of gsize requests over [0, P); own units:
    each request over [P, L)) attends every (request, query row, position) exactly once,
    with unique partial slots, each piece's index base at the right entry, causal limits
    only on own units, and the merge's slot ranges matching what the decode wrote."""
    B = len(kv_lens)
    kvp = np.concatenate([[0], np.cumsum(kv_lens)]).astype(np.int32)
    qop = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    rows = max(q_lens) * H
    NG = cascade_ng(rows, B)
    gsize = NG // rows
    P = shared
    VP = (B + gsize - 1) // gsize
    cw = resolve_costs(sim, costs, 1, NG, rows)
    pieces = cascade_pieces(sim, kvp, qop, B, H, NG, 1, grid, 1, gsize, shared, cw)
    n_slots = sim.sched_partial_slots(VP + B, 1, 0, grid)
    cover = {}
    for cta, v, g, j0, j1, prow, slot, direct, kv0, cfrom in pieces:
        assert g == 0 and not direct and 0 <= slot < n_slots
        if v < VP:
            first_b, last_b = v * gsize, min(v * gsize + gsize, B)
            assert kv0 == kvp[first_b] and cfrom == P and j1 <= P
            assert prow == (qop[last_b] - qop[first_b]) * H
        else:
            b = v - VP
            Ls = kv_lens[b] - P
            assert kv0 == kvp[b] + P and cfrom == Ls - q_lens[b] and j1 <= Ls
            assert prow == q_lens[b] * H
        cover.setdefault(v, []).append((j0, j1, slot))
    slots = [p[6] for p in pieces]
    assert len(slots) == len(set(slots)), "partial slot written twice"
    for v in range(VP + B):
        L = P if v < VP else kv_lens[v - VP] - P
        ps = sorted(cover.get(v, []))
        pos = 0
        for j0, j1, _ in ps:
            assert j0 == pos, f"gap/overlap in unit {v}"
            pos = j1
        assert pos == max(L, 0)
        need, first, count = cascade_partials(sim, kvp, qop, B, H, NG, 1, grid, 1, gsize, shared,
                                              v, 0, cw)
        if L <= 0:
            assert need == 0
        else:
            assert need == 1 and {p[2] for p in ps} == set(range(first, first + count))


CASCADE_CASES = [
    # (kv_lens, q_lens, H, shared prefix length the caller declares; >= 1024)
    ([68000] * 16, [1] * 16, 12, 63911),
    ([68000 + 37 * i for i in range(24)], [1] * 24, 12, 63911),
    ([5000, 5000, 7000, 6000, 5500], [1] * 5, 12, 4000),  # two groups (4 + 1)
    ([3000] * 5, [1] * 5, 12, 3000),                      # whole requests shared: no own units
    ([3000, 2500, 4000, 2200, 2600], [1] * 5, 12, 2200),  # one request ends with the prefix
    ([9000] * 4, [2] * 4, 12, 8999),                      # two queries per request
    ([12000] * 7, [1] * 7, 8, 5000),                      # 8 heads: groups of 6 requests
    ([6000, 6100, 5900, 7000, 6500], [4] * 5, 12, 5000),  # 48 rows: 96-row groups of 2
    ([3000 + 11 * i for i in range(9)], [1] * 9, 12, 2048),   # 96-row groups: 8 + 1
]


@pytest.mark.parametrize("kv_lens,q_lens,H,shared", CASCADE_CASES)
@pytest.mark.parametrize("grid", [1, 7, 152])
@pytest.mark.parametrize("costs", COSTS)
def test_cascade_halves_cover_every_position_once(sim, kv_lens, q_lens, H, shared, grid, costs):
    check_cascade(sim, kv_lens, q_lens, H, grid, shared, costs)


# ------------------------------------------------------------------ paged caches

def check_paged(sim, kv_lens, q_lens, H, page_size, splits, grid, costs=(1, 512)):
    """kv_indptr in pages of page_size tokens, last page partly filled: the pieces cover
    each request's real positions [0, L) exactly once, index bases are page bases, causal
    bases use the real length, and the merge's slot ranges match what the decode wrote."""
    B = len(kv_lens)
    counts = [(L + page_size - 1) // page_size for L in kv_lens]
    kvp = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    last = np.array([L - (c - 1) * page_size if c else 1 for L, c in zip(kv_lens, counts)],
                    dtype=np.int32)
    qop = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    rows = max(q_lens) * H
    NG = pick_ng(rows)
    groups = (rows + NG - 1) // NG
    lg = page_size.bit_length() - 1
    i32p = ctypes.POINTER(ctypes.c_int32)
    cap = 8 * (grid + B * groups * max(splits, 1) + 16)
    out = np.zeros(cap * 10, dtype=np.int64)
    w, e = costs
    n = sim.sched_pieces_paged(kvp.ctypes.data_as(i32p), qop.ctypes.data_as(i32p), B, H, NG,
                               groups, splits, grid, lg, last.ctypes.data_as(i32p), w, e,
                               out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), cap)
    assert n >= 0, f"simulation failed with {n}"
    pieces = out[:10 * n].reshape(n, 10)
    by_unit = {}
    for cta, b, g, j0, j1, prow, slot, direct, kv0, cfrom in pieces:
        L, T = kv_lens[b], q_lens[b]
        assert 0 <= j0 < j1 <= L, (b, j0, j1, L)
        assert kv0 == kvp[b] and cfrom == L - T
        by_unit.setdefault((b, g), []).append((j0, j1, slot, direct))
    n_slots = sim.sched_partial_slots(B, groups, splits, grid)
    for b in range(B):
        for g in range(groups):
            real = q_lens[b] * H - g * NG > 0
            ps = sorted(by_unit.get((b, g), []))
            if not real or kv_lens[b] == 0:
                assert not ps
                continue
            pos = 0
            for j0, j1, _, _ in ps:
                assert j0 == pos, f"gap/overlap in unit {(b, g)}"
                pos = j1
            assert pos == kv_lens[b]
            first, count = ctypes.c_int64(0), ctypes.c_int(0)
            need = sim.sched_unit_partials_paged(kvp.ctypes.data_as(i32p), qop.ctypes.data_as(i32p),
                                                 B, H, NG, groups, splits, grid, lg,
                                                 last.ctypes.data_as(i32p), w, e, b, g,
                                                 ctypes.byref(first), ctypes.byref(count))
            if len(ps) == 1 and ps[0][3]:
                assert need == 0
            else:
                assert need == 1 and not any(p[3] for p in ps)
                got = {p[2] for p in ps}
                expect = set(range(first.value, first.value + count.value))
                if splits <= 0:
                    assert got == expect
                else:   # fixed policy over the real length: missing = the empty pieces
                    empty = {first.value + k for k in range(count.value)
                             if (k + 1) * kv_lens[b] // splits <= k * kv_lens[b] // splits}
                    assert got == expect - empty
                assert all(0 <= s < n_slots for s in got)


@pytest.mark.parametrize("page_size", [2, 16, 64, 128])
@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("grid", [1, 7, 152])
def test_paged_schedule_covers_real_positions(sim, page_size, splits, grid):
    check_paged(sim, [1, 2, 127, 128, 129, 3000, 0, 5000], [1, 1, 2, 1, 4, 1, 1, 3], 12,
                page_size, splits, grid)


def test_paged_random_batches(sim):
    rng = np.random.default_rng(7)
    for _ in range(30):
        B = int(rng.integers(1, 12))
        kv = [int(x) for x in rng.integers(0, 9000, size=B)]
        q = [int(min(t, L)) if L > 0 else 0 for t, L in zip(rng.integers(1, 5, size=B), kv)]
        if max(q) == 0:
            continue
        ps = int(rng.choice([2, 8, 32, 64, 256]))
        H = int(rng.choice([12, 16, 96]))
        for grid in (5, 152):
            check_paged(sim, kv, q, H, ps, 0, grid)


def _paged_csr(kv_lens, page_size):
    counts = [(L + page_size - 1) // page_size for L in kv_lens]
    kvp = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    last = np.array([L - (c - 1) * page_size if c else 1 for L, c in zip(kv_lens, counts)],
                    dtype=np.int32)
    return kvp, last


def test_request_len_reads_pages_and_last_fill(sim):
    i32p = ctypes.POINTER(ctypes.c_int32)
    for ps in (1, 2, 64, 1024):
        lens = [0, 1, ps, ps + 1, 3 * ps - 1, 5000]
        kvp, last = _paged_csr(lens, ps)
        lg = ps.bit_length() - 1
        got = [sim.sched_request_len(kvp.ctypes.data_as(i32p), lg, last.ctypes.data_as(i32p), b)
               for b in range(len(lens))]
        assert got == lens
    # out-of-range fills are clamped to [1, page_size] (mla_validate flags them)
    kvp = np.array([0, 2, 4], dtype=np.int32)
    last = np.array([0, 99], dtype=np.int32)
    got = [sim.sched_request_len(kvp.ctypes.data_as(i32p), 4, last.ctypes.data_as(i32p), b)
           for b in range(2)]
    assert got == [17, 32]


def check_cascade_paged(sim, kv_lens, q_lens, H, grid, shared, page_size, costs=(1, 0, 512)):
    """The cascade on a paged cache (P whole pages): prefix units cover [0, P) of their lead
    request's pages, own units [P, L) of each request's real length, with the own units'
    index base P / page_size pages into the request, exactly once each."""
    assert shared % page_size == 0
    B = len(kv_lens)
    kvp, last = _paged_csr(kv_lens, page_size)
    qop = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    rows = max(q_lens) * H
    NG = cascade_ng(rows, B)
    gsize = NG // rows
    P = shared
    VP = (B + gsize - 1) // gsize
    lg = page_size.bit_length() - 1
    i32p = ctypes.POINTER(ctypes.c_int32)
    cap = 8 * (grid + 2 * (VP + B) + 16)
    out = np.zeros(cap * 10, dtype=np.int64)
    # mode 2: the paged cascade the library launches on pages of several tokens
    mode = 2 if page_size > 1 else 1
    args = (kvp.ctypes.data_as(i32p), qop.ctypes.data_as(i32p), B, H, NG, 1, 0, grid, mode, gsize,
            shared, *costs, lg, last.ctypes.data_as(i32p))
    n = sim.sched_pieces_full(*args, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), cap)
    assert n >= 0
    pieces = out[:10 * n].reshape(n, 10)
    n_slots = sim.sched_partial_slots(VP + B, 1, 0, grid)
    cover = {}
    for cta, v, g, j0, j1, prow, slot, direct, kv0, cfrom in pieces:
        assert g == 0 and not direct and 0 <= slot < n_slots and j0 < j1
        if v < VP:
            assert kv0 == kvp[v * gsize] and cfrom == P and j1 <= P
        else:
            b = v - VP
            Ls = kv_lens[b] - P
            assert kv0 == kvp[b] + P // page_size and cfrom == Ls - q_lens[b] and j1 <= Ls
        cover.setdefault(v, []).append((j0, j1, slot))
    slots = [p[6] for p in pieces]
    assert len(slots) == len(set(slots))
    for v in range(VP + B):
        L = P if v < VP else kv_lens[v - VP] - P
        ps = sorted(cover.get(v, []))
        pos = 0
        for j0, j1, _ in ps:
            assert j0 == pos
            pos = j1
        assert pos == max(L, 0)
        first, count = ctypes.c_int64(0), ctypes.c_int(0)
        need = sim.sched_unit_partials_full(*args, v, 0, ctypes.byref(first), ctypes.byref(count))
        if L <= 0:
            assert need == 0
        else:
            assert need == 1 and {p[2] for p in ps} == set(range(first.value, first.value + count.value))


@pytest.mark.parametrize("page_size", [1, 2, 64, 128])
@pytest.mark.parametrize("grid", [1, 7, 152])
def test_paged_cascade_covers_every_position_once(sim, page_size, grid):
    P = (63911 // page_size) * page_size
    check_cascade_paged(sim, [68000 + 37 * i for i in range(16)], [1] * 16, 12, grid, P, page_size)
    check_cascade_paged(sim, [5000, 5000, 7000, 6000, 5500], [1] * 5, 12, grid,
                        (4000 // page_size) * page_size, page_size)
    check_cascade_paged(sim, [9000] * 4, [2] * 4, 12, grid, (8960 // page_size) * page_size,
                        page_size)
    # a request that ends exactly with the prefix (no own positions)
    check_cascade_paged(sim, [2048, 2500, 4000, 2200, 2600], [1] * 5, 12, grid, 2048, page_size)
