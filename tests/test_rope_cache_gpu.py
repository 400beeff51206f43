"""mla_qk_rope_concat_and_cache (the fused step that produces the decode's q and writes the
step's new cache entries, "[Kimi-K3 MLA TP8] MLA performance" §3) against the oracle: the
fp8 bytes of q_out and of the whole cache must be identical (byte work: bit-exact), for
both pair conventions, one-token and paged caches, padding tokens, strided views, scales
that saturate, and the error cases; then the written entries decode like any other."""
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


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _cache(n_pages, page_size, seed):
    """A poisoned pool: every byte 0x7F except some random fp8 rows (so that untouched
    bytes are distinguishable from written ones)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    shape = (n_pages, 576) if page_size == 1 else (n_pages, page_size, 1, 576)
    kv = torch.full(shape, 0x7F, dtype=torch.uint8, device="cuda")
    flat = kv.view(-1, 576)
    some = torch.randperm(flat.shape[0], generator=g, device="cuda")[: flat.shape[0] // 4]
    flat[some] = mla_inputs.fp8_normal_bytes(some.numel() * 576, g, "cuda").view(-1, 576)
    return kv


def _run_both(pm, inp, neox, slots, q_scale, kv_scale, kv, q_pe=None):
    T, H = inp["q_nope"].shape[0], inp["q_nope"].shape[1]
    qs = torch.tensor(q_scale, dtype=torch.float32, device="cuda")
    ks = torch.tensor(kv_scale, dtype=torch.float32, device="cuda")
    q_pe = inp["q_pe"] if q_pe is None else q_pe
    want_q, want_kv, want_err = oracle.rope_concat_cache(
        _bits(inp["q_nope"]), _bits(q_pe), _bits(inp["kv_c"]), _bits(inp["k_pe"]),
        inp["positions"].cpu().numpy(), inp["cos_sin"].cpu().numpy(), neox,
        slots.cpu().numpy(), np.float32(q_scale), np.float32(kv_scale),
        kv.cpu().numpy().reshape(-1, 576))
    q_out = torch.full((T, H, 576), 0x7F, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pm.mla_qk_rope_concat_and_cache(inp["q_nope"], q_pe, inp["kv_c"], inp["k_pe"],
                                    inp["positions"], inp["cos_sin"], neox, slots, qs, ks, q_out,
                                    kv, err)
    torch.cuda.synchronize()
    return (q_out.cpu().numpy(), kv.cpu().numpy().reshape(-1, 576), int(err.item()),
            want_q, want_kv, want_err)


def _assert_exact(got_q, got_kv, want_q, want_kv):
    bad_q = np.argwhere(got_q != want_q)
    assert bad_q.size == 0, f"q_out differs at {bad_q[:5].tolist()}"
    bad_kv = np.argwhere(got_kv != want_kv)
    assert bad_kv.size == 0, f"cache differs at {bad_kv[:5].tolist()}"


@pytest.mark.parametrize("neox", [0, 1])
# 800 tokens x 13 rows x 36 pieces exceed one pass of the grid-stride loop (152 x 8 blocks)
@pytest.mark.parametrize("T,H", [(16, 12), (256, 12), (3, 96), (1, 1), (37, 12), (800, 12)])
def test_bytes_match_oracle(pm, neox, T, H):
    inp = mla_inputs.make_rope_inputs(T, H, max_pos=4096, seed=T * 7 + H + neox, device="cuda")
    kv = _cache(4096, 1, seed=T)
    g = torch.Generator(device="cuda").manual_seed(T + 1)
    slots = torch.randperm(4096, generator=g, device="cuda")[:T].to(torch.int32)
    got_q, got_kv, err, want_q, want_kv, want_err = _run_both(pm, inp, neox, slots, 0.05, 0.1, kv)
    assert err == 0 and want_err == 0
    _assert_exact(got_q, got_kv, want_q, want_kv)


@pytest.mark.parametrize("page_size", [16, 128])
@pytest.mark.parametrize("neox", [0, 1])
def test_paged_cache_and_padding_tokens(pm, page_size, neox):
    T, H = 64, 12
    inp = mla_inputs.make_rope_inputs(T, H, max_pos=2048, seed=page_size + neox, device="cuda")
    kv = _cache(64, page_size, seed=page_size)
    g = torch.Generator(device="cuda").manual_seed(page_size)
    slots = torch.randperm(64 * page_size, generator=g, device="cuda")[:T].to(torch.int32)
    slots[::5] = -1                                    # padding tokens: no entry
    got_q, got_kv, err, want_q, want_kv, want_err = _run_both(pm, inp, neox, slots, 0.05, 0.1, kv)
    assert err == 0 and want_err == 0
    _assert_exact(got_q, got_kv, want_q, want_kv)


def test_strided_views_and_saturating_scales(pm):
    """q_pe as the last 64 columns of a (T, H, 192) projection, kv_c / k_pe as views into
    one (T, 576) buffer, a padded cache row pitch, and scales small enough that many codes
    saturate at +-448."""
    T, H = 24, 12
    inp = mla_inputs.make_rope_inputs(T, H, max_pos=1024, seed=5, device="cuda", value_scale=4.0)
    wide = torch.randn((T, H, 192), device="cuda").to(torch.bfloat16)
    wide[..., 128:] = inp["q_pe"]
    q_pe = wide[..., 128:]
    both = torch.empty((T, 576), dtype=torch.bfloat16, device="cuda")
    both[:, :512], both[:, 512:] = inp["kv_c"], inp["k_pe"]
    inp = dict(inp, kv_c=both[:, :512], k_pe=both[:, 512:])
    pool = torch.full((300, 640), 0x7F, dtype=torch.uint8, device="cuda")
    kv = pool[:, :576]                                 # row pitch 640 bytes
    slots = torch.arange(T, dtype=torch.int32, device="cuda") * 11
    got_q, _, err, want_q, want_kv, want_err = _run_both(pm, inp, 0, slots, 0.004, 0.002, kv,
                                                         q_pe=q_pe)
    assert err == 0 and want_err == 0
    got_kv = kv.cpu().numpy()
    _assert_exact(got_q, got_kv, want_q, want_kv)
    assert (got_q == 0x7E).any() and (got_q == 0xFE).any()   # saturated codes occur
    assert (pool[:, 576:] == 0x7F).all()                      # pitch padding untouched


def test_errors_are_flagged_and_skip_their_bytes(pm):
    T, H = 8, 4
    inp = mla_inputs.make_rope_inputs(T, H, max_pos=128, seed=9, device="cuda")
    inp["positions"][2] = 128          # outside the table
    inp["positions"][5] = -3
    kv = _cache(32, 1, seed=9)
    slots = torch.arange(T, dtype=torch.int32, device="cuda")
    slots[6] = 32                      # outside the cache
    got_q, got_kv, err, want_q, want_kv, want_err = _run_both(pm, inp, 1, slots, 0.05, 0.1, kv)
    assert want_err == 3
    assert err == 1 | 64               # position (bit 1) and slot (bit 64) flagged
    _assert_exact(got_q, got_kv, want_q, want_kv)   # the same bytes written and skipped


def test_no_tokens_is_a_no_op(pm):
    inp = mla_inputs.make_rope_inputs(0, 12, max_pos=16, seed=1, device="cuda")
    kv = _cache(4, 1, seed=1)
    before = kv.clone()
    q_out = torch.empty((0, 12, 576), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    one = torch.tensor(1.0, device="cuda")
    pm.mla_qk_rope_concat_and_cache(inp["q_nope"], inp["q_pe"], inp["kv_c"], inp["k_pe"],
                                    inp["positions"], inp["cos_sin"], 0,
                                    torch.zeros(0, dtype=torch.int32, device="cuda"), one, one,
                                    q_out, kv, err)
    torch.cuda.synchronize()
    assert torch.equal(kv, before) and int(err.item()) == 0


def test_written_entries_decode_like_the_oracle(pm):
    """The step then the decode: 4 requests each append their token's entry at the end of
    its history and decode with the new q; the result equals the oracle decode of the same
    bytes (which the oracle of this step produced identically)."""
    B, H, L = 4, 12, 700
    case = gu.to_device(mla_inputs.make_custom([L] * B, H=H, seed=31, q_scale=1.0, kv_scale=1.0))
    inp = mla_inputs.make_rope_inputs(B, H, max_pos=4096, seed=32, device="cuda")
    # each request's last position is the slot the new entry goes to
    slots = case.kv_indices[case.kv_indptr[1:].long() - 1].clone()
    q_out = torch.empty((B, H, 576), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pm.mla_qk_rope_concat_and_cache(inp["q_nope"], inp["q_pe"], inp["kv_c"], inp["k_pe"],
                                    inp["positions"], inp["cos_sin"], 0, slots, case.q_scale,
                                    case.kv_scale, q_out, case.kv, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    case.q = q_out
    o, lse, st = gu.run_gpu(case)
    assert st == 0
    o_ref, lse_ref = gu.run_oracle(case)
    gu.compare(o, lse, o_ref, lse_ref, what="decode after the cache write")


def test_rejects_bad_arguments_on_host(pm):
    T, H = 4, 12
    inp = mla_inputs.make_rope_inputs(T, H, max_pos=16, seed=2, device="cuda")
    kv = _cache(8, 1, seed=2)
    one = torch.tensor(1.0, device="cuda")
    slots = torch.arange(T, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    good = dict(q_nope=inp["q_nope"], q_pe=inp["q_pe"], kv_c=inp["kv_c"], k_pe=inp["k_pe"],
                positions=inp["positions"], cos_sin=inp["cos_sin"], is_neox=0,
                slot_mapping=slots, q_scale=one, kv_scale=one,
                q_out=torch.empty((T, H, 576), dtype=torch.uint8, device="cuda"), kv_buffer=kv,
                error_word=err)
    for key, bad in (("q_pe", inp["q_pe"].float()), ("kv_c", inp["kv_c"][:, :256]),
                     ("positions", inp["positions"].long()), ("is_neox", 2),
                     ("cos_sin", inp["cos_sin"][:, :32]),
                     ("q_out", torch.empty((T, H, 512), dtype=torch.uint8, device="cuda")),
                     ("slot_mapping", slots[:2])):
        args = dict(good, **{key: bad})
        with pytest.raises((pm.MlaError, TypeError)):
            pm.mla_qk_rope_concat_and_cache(**args)
