"""The C-ABI library loads, exports what include/paged_mla.h declares, and rejects bad
arguments on the host before touching the GPU (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def _declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(mla_[A-Za-z0-9_]+)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    import paged_mla_latent_gb300 as pm
    return pm


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("mla_decode", "mla_merge_partials", "mla_get_workspace_size",
                     "mla_validate", "mla_check_error", "mla_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    path = lib.library_path()
    assert os.path.exists(path)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = _declared_functions() - exported
    assert not missing, f"declared but not exported: {missing}"
    so = ctypes.CDLL(path)
    for name in _declared_functions():
        assert hasattr(so, name)


def test_status_strings(lib):
    assert lib.mla_status_string(0) == "MLA_OK"
    assert lib.mla_status_string(5) == "MLA_ERR_BAD_INDEX"
    assert lib.mla_status_string(6) == "MLA_ERR_TIMEOUT"
    assert lib.mla_status_string(12345) == "MLA_ERR_UNKNOWN"


def test_workspace_size_plan(lib):
    # auto policy: (B*groups + SMs) partial slots of NG rows x (512 + 1) floats + header
    sz = lib.mla_get_workspace_size(16, 12, 1, 0, 152)
    ng, slots = 16, 16 + 152
    plain = 256 + slots * ng * 513 * 4
    assert plain <= sz < plain + 2 * 256
    # 96 heads -> one group of 96 rows
    sz96 = lib.mla_get_workspace_size(1, 96, 1, 0, 152)
    plain96 = 256 + (1 + 152) * 96 * 513 * 4
    assert plain96 <= sz96 < plain96 + 2 * 256
    # 128 heads -> two groups of 96 rows (the second one 32 rows deep)
    sz128 = lib.mla_get_workspace_size(1, 128, 1, 0, 152)
    plain128 = 256 + (2 + 152) * 96 * 513 * 4
    assert plain128 <= sz128 < plain128 + 2 * 256
    # one split per request needs no partials
    assert lib.mla_get_workspace_size(16, 12, 1, 1, 152) == 256
    with pytest.raises(lib.MlaError):
        lib.mla_get_workspace_size(16, 12, 0, 0, 152)     # max_seqlen_q < 1
    with pytest.raises(lib.MlaError):
        lib.mla_get_workspace_size(16, 0, 1, 0, 152)      # no heads


def test_shared_prefix_workspace_size(lib):
    # the cascade's 96-row slots: ceil(B / 8) prefix units + B own units + SMs
    sz = lib.mla_get_shared_prefix_workspace_size(16, 12, 1, 152)
    cascade = 256 + (2 + 16 + 152) * 96 * 513 * 4
    assert cascade <= sz < cascade + 2 * 256
    assert sz > lib.mla_get_workspace_size(16, 12, 1, 0, 152)
    # 48 rows a request: groups of two
    sz48 = lib.mla_get_shared_prefix_workspace_size(64, 12, 4, 152)
    cascade48 = 256 + (32 + 64 + 152) * 96 * 513 * 4
    assert cascade48 <= sz48 < cascade48 + 2 * 256
    # four or more but fewer than eight 12-row requests: the 48-row cascade, groups of four
    sz4 = lib.mla_get_shared_prefix_workspace_size(5, 12, 1, 152)
    cascade4 = 256 + (2 + 5 + 152) * 48 * 513 * 4
    assert cascade4 <= sz4 < cascade4 + 2 * 256
    # batches that never take the shared-prefix path need only the plain workspace
    for B, H, T in [(3, 12, 1), (1, 12, 1), (64, 16, 4), (16, 96, 1)]:
        assert (lib.mla_get_shared_prefix_workspace_size(B, H, T, 152) ==
                lib.mla_get_workspace_size(B, H, T, 0, 152))


def _t(ptr, dtype, shape, stride=None):
    import paged_mla_latent_gb300 as pm
    d = pm.MlaTensor()
    d.ptr = ptr
    d.ndim = len(shape)
    d.dtype = dtype
    if stride is None:
        stride, acc = [], 1
        for s in reversed(shape):
            stride.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, stride)):
        d.shape[i] = s
        d.stride[i] = st
    return d


def _args(**over):
    """Host-side descriptors with fake (never dereferenced) device addresses."""
    F8, BF, F32, I32 = 1, 2, 3, 4
    base = 1 << 40
    a = dict(
        q=_t(base, F8, [2, 12, 576]), kv=_t(base + (1 << 20), F8, [1024, 576]),
        o=_t(base + (2 << 20), BF, [2, 12, 512]), qo=_t(base + (3 << 20), I32, [3]),
        kvp=_t(base + (4 << 20), I32, [3]), idx=_t(base + (5 << 20), I32, [1024]),
        last=_t(base + (6 << 20), I32, [2]), qs=_t(base + (7 << 20), F32, []),
        ks=_t(base + (8 << 20), F32, []), lse=None, mq=1, sm=0.0721, splits=0,
        ws=base + (9 << 20), ws_bytes=1 << 20)
    a.update(over)
    return a


def _call(a):
    import paged_mla_latent_gb300 as pm
    r = lambda d: ctypes.byref(d) if d is not None else None
    return pm._lib.mla_decode(r(a["q"]), r(a["kv"]), r(a["o"]), r(a["qo"]), r(a["kvp"]),
                              r(a["idx"]), r(a["last"]), a["mq"], a["sm"], r(a["qs"]), r(a["ks"]),
                              a["splits"], r(a["lse"]), ctypes.c_void_p(a["ws"]), a["ws_bytes"],
                              None)


@pytest.mark.parametrize("over,expect", [
    (dict(q=None), 1),
    (dict(q=_t(0, 1, [2, 12, 576])), 1),                                   # null pointer
    (dict(q=_t(1 << 40, 3, [2, 12, 576])), 1),                             # q not fp8
    (dict(q=_t(1 << 40, 1, [2, 12, 512])), 2),                             # head dim != 576
    (dict(q=_t((1 << 40) + 8, 1, [2, 12, 576])), 1),                       # q not 16-B aligned
    (dict(kv=_t((1 << 40) + (1 << 20), 1, [1024, 3, 1, 576])), 2),         # page_size not 2^k
    (dict(kv=_t((1 << 40) + (1 << 20), 1, [4, 2048, 1, 576])), 2),         # page_size > 1024
    (dict(kv=_t((1 << 40) + (1 << 20), 1, [512, 2, 1, 576]), last=None), 1),   # no last lens
    (dict(kv=_t((1 << 40) + (1 << 20), 1, [512, 2, 1, 576], [576, 576, 576, 1])), 1),  # overlap
    (dict(kv=_t((1 << 40) + (1 << 20), 1, [1 << 24, 256, 1, 576])), 1),    # rows past int32
    (dict(kv=_t((1 << 40) + (1 << 20), 1, [1024, 576], [584, 1])), 1),    # pitch not 16-B multiple
    (dict(o=_t((1 << 40) + (2 << 20), 2, [2, 12, 256])), 1),               # o width != 512
    (dict(o=_t((1 << 40) + (2 << 20), 4, [2, 12, 512])), 1),               # o int32
    (dict(kvp=_t((1 << 40) + (4 << 20), 4, [4])), 1),                      # indptr size mismatch
    (dict(idx=_t((1 << 40) + (5 << 20), 3, [1024])), 1),                   # indices not int32
    (dict(last=_t((1 << 40) + (6 << 20), 4, [5])), 1),                     # last_page_lens size
    (dict(qs=_t((1 << 40) + (7 << 20), 3, [2])), 1),                       # q_scale not scalar
    (dict(mq=0), 1),
    (dict(mq=65), 1),
    (dict(sm=float("nan")), 1),
    (dict(ws=(1 << 40) + 8), 1),                                           # workspace misaligned
    (dict(lse=_t(1 << 41, 3, [2, 11])), 1),                                # lse shape
])
def test_decode_rejects_bad_arguments_on_host(lib, over, expect):
    assert _call(_args(**over)) == expect


def _call_sp(a, prefix):
    import paged_mla_latent_gb300 as pm
    r = lambda d: ctypes.byref(d) if d is not None else None
    return pm._lib.mla_decode_shared_prefix(
        r(a["q"]), r(a["kv"]), r(a["o"]), r(a["qo"]), r(a["kvp"]), r(a["idx"]), r(a["last"]),
        a["mq"], a["sm"], r(a["qs"]), r(a["ks"]), prefix, r(a["lse"]), ctypes.c_void_p(a["ws"]),
        a["ws_bytes"], None)


@pytest.mark.parametrize("over,prefix,expect", [
    (dict(), -1, 1),                                  # negative shared prefix
    (dict(q=None), 2048, 1),
    (dict(o=_t((1 << 40) + (2 << 20), 2, [2, 12, 256])), 2048, 1),
    (dict(ws=(1 << 40) + 8), 2048, 1),
])
def test_shared_prefix_decode_rejects_bad_arguments_on_host(lib, over, prefix, expect):
    assert _call_sp(_args(**over), prefix) == expect


def test_merge_rejects_bad_arguments_on_host(lib):
    r = lambda d: ctypes.byref(d) if d is not None else None
    F32, I32, BF = 3, 4, 2
    base = 1 << 40
    op = _t(base, F32, [8, 96, 512])
    lp = _t(base + (32 << 20), F32, [8, 96])
    ip = _t(base + (33 << 20), I32, [2])
    ix = _t(base + (34 << 20), I32, [8])
    o = _t(base + (35 << 20), BF, [1, 96, 512])
    bad_o = _t(base + (35 << 20), BF, [1, 95, 512])
    assert lib._lib.mla_merge_partials(r(op), r(lp), r(ip), r(ix), r(bad_o), None, None, None) == 1
    bad_lp = _t(base + (32 << 20), F32, [7, 96])
    assert lib._lib.mla_merge_partials(r(op), r(bad_lp), r(ip), r(ix), r(o), None, None, None) == 1
    odd = _t(base + 4, F32, [8, 96, 512])
    assert lib._lib.mla_merge_partials(r(odd), r(lp), r(ip), r(ix), r(o), None, None, None) == 1


def test_latent_to_v_rejects_bad_arguments_on_host(lib):
    r = lambda d: ctypes.byref(d) if d is not None else None
    BF, F32 = 2, 3
    base = 1 << 40
    o = _t(base, BF, [16, 12, 512])
    w = _t(base + (8 << 20), BF, [12, 512, 128])
    v = _t(base + (16 << 20), BF, [16, 12, 128])
    call = lambda o_, w_, v_: lib._lib.mla_latent_to_v(r(o_), r(w_), r(v_), None)
    assert call(None, w, v) == 1
    assert call(_t(base, F32, [16, 12, 512]), w, v) == 1                     # o not bf16
    assert call(_t(base, BF, [16, 12, 256]), w, v) == 1                      # latent width
    assert call(o, _t(base + (8 << 20), BF, [12, 512, 64]), v) == 1          # v_head_dim
    assert call(o, _t(base + (8 << 20), BF, [11, 512, 128]), v) == 1         # head count
    assert call(o, w, _t(base + (16 << 20), BF, [15, 12, 128])) == 1         # v tokens
    assert call(_t(base + 2, BF, [16, 12, 512]), w, v) == 1                  # o not 16-B aligned
    assert call(_t(base, BF, [16, 12, 512], [6148, 516, 1]), w, v) == 1      # stride not 8k
    assert call(o, _t(base + (8 << 20), BF, [12, 512, 128], [65536, 1, 512]), v) == 1  # w transposed
    # no tokens: nothing to do, nothing enqueued
    assert call(_t(base, BF, [0, 12, 512]), w, _t(base + (16 << 20), BF, [0, 12, 128])) == 0


def test_rope_cache_rejects_bad_arguments_on_host(lib):
    """mla_qk_rope_concat_and_cache: every shape, dtype, stride and alignment check returns
    MLA_ERR_INVALID_ARG (or UNSUPPORTED) before anything touches the device; no tokens is
    a no-op."""
    r = lambda d: ctypes.byref(d) if d is not None else None
    F8, BF, F32, I32 = 1, 2, 3, 4
    b = 1 << 40
    T, H = 4, 12
    good = dict(qn=_t(b, BF, [T, H, 512]), qp=_t(b + (1 << 20), BF, [T, H, 64]),
                kc=_t(b + (2 << 20), BF, [T, 512]), kp=_t(b + (3 << 20), BF, [T, 64]),
                pos=_t(b + (4 << 20), I32, [T]), cs=_t(b + (5 << 20), F32, [128, 64]), neox=0,
                slots=_t(b + (6 << 20), I32, [T]), qs=_t(b + (7 << 20), F32, []),
                ks=_t(b + (8 << 20), F32, []), qo=_t(b + (9 << 20), F8, [T, H, 576]),
                kv=_t(b + (16 << 20), F8, [1024, 576]), err=b + (10 << 20))

    def call(**over):
        a = dict(good, **over)
        return lib._lib.mla_qk_rope_concat_and_cache(
            r(a["qn"]), r(a["qp"]), r(a["kc"]), r(a["kp"]), r(a["pos"]), r(a["cs"]), a["neox"],
            r(a["slots"]), r(a["qs"]), r(a["ks"]), r(a["qo"]), r(a["kv"]),
            ctypes.c_void_p(a["err"]) if a["err"] else None, None)

    assert call(qn=None) == 1
    assert call(qn=_t(b, F32, [T, H, 512])) == 1                          # not bf16
    assert call(qp=_t(b + (1 << 20), BF, [T, H, 32])) == 1                # rope width
    assert call(qp=_t(b + (1 << 20) + 2, BF, [T, H, 64])) == 1            # not 16-B aligned
    assert call(qp=_t(b + (1 << 20), BF, [T, H, 64], [H * 196, 196, 1])) == 1   # stride not 8k
    assert call(kc=_t(b + (2 << 20), BF, [T + 1, 512])) == 1              # token count
    assert call(pos=_t(b + (4 << 20), F32, [T])) == 1                     # positions not int32
    assert call(cs=_t(b + (5 << 20), F32, [128, 32])) == 1                # table width
    assert call(neox=3) == 1
    assert call(slots=_t(b + (6 << 20), I32, [T - 1])) == 1
    assert call(qs=_t(b + (7 << 20), F32, [2])) == 1                      # scale not scalar
    assert call(qo=_t(b + (9 << 20), F8, [T, H, 576], [H * 640, 640, 1])) == 1  # q_out strided
    assert call(kv=_t(b + (16 << 20), F8, [64, 3, 1, 576])) == 2          # page_size not 2^k
    assert call(kv=_t(b + (16 << 20), F8, [1024, 576], [584, 1])) == 1    # pitch not 16-B multiple
    assert call(err=0) == 1                                               # no error word
    # no tokens: nothing to do, nothing enqueued
    assert call(qn=_t(b, BF, [0, H, 512]), qp=_t(b + (1 << 20), BF, [0, H, 64]),
                kc=_t(b + (2 << 20), BF, [0, 512]), kp=_t(b + (3 << 20), BF, [0, 64]),
                pos=_t(b + (4 << 20), I32, [0]), slots=_t(b + (6 << 20), I32, [0]),
                qo=_t(b + (9 << 20), F8, [0, H, 576])) == 0


def test_bounded_wait_selftest_rejects_bad_arguments_on_host(lib):
    """The wait's self-test checks its limit and pointers before launching anything."""
    f = lib._lib.mla_selftest_bounded_wait
    word, res = ctypes.c_void_p(1 << 40), ctypes.c_void_p((1 << 40) + 64)
    assert f(None, res, 1_000_000, None) == 1
    assert f(word, None, 1_000_000, None) == 1
    for bad in (0, 999, 100_000_001):
        assert f(word, res, bad, None) == 1


def test_prefix_expand_rejects_bad_arguments_before_launch(lib):
    """Host-side checks of mla_expand_shared_prefix_indices (fake device addresses: every
    case fails before anything is enqueued)."""
    I32 = 4
    base = 1 << 40
    good = dict(shared=_t(base, I32, [10]), optr=_t(base + 4096, I32, [4]),
                own=_t(base + 8192, I32, [30]), kvp=_t(base + 12288, I32, [4]),
                idx=_t(base + 16384, I32, [60]))
    def call(**kw):
        a = dict(good, **kw)
        return lib._lib.mla_expand_shared_prefix_indices(
            ctypes.byref(a["shared"]), ctypes.byref(a["optr"]), ctypes.byref(a["own"]),
            ctypes.byref(a["kvp"]), ctypes.byref(a["idx"]), None, None)
    assert call(kvp=_t(base + 12288, I32, [5])) == 1          # kv_indptr length != own_indptr
    assert call(optr=_t(base + 4096, 3, [4])) == 1            # own_indptr not int32
    assert call(idx=_t(base + 16384, I32, [29])) == 1         # not even room for B x S shared ids
    assert call(shared=_t(base + 2, I32, [10])) == 1          # misaligned


class _RecordingLib:
    """Stands in for the C library: records each entry point's arguments."""

    def __init__(self, expand_rc=0):
        self.calls = []
        self.expand_rc = expand_rc

    def mla_expand_shared_prefix_indices(self, *args):
        self.calls.append(("expand", args))
        return self.expand_rc

    def mla_decode_shared_prefix(self, *args):
        self.calls.append(("decode", args))
        return 0


def _prepared_with_compact_table(pm):
    import torch
    B, H, n_sh = 2, 12, 5
    own_lens = [3, 4]
    t = {
        "q": torch.zeros(B, H, 576, dtype=torch.uint8),
        "kv": torch.zeros(64, 576, dtype=torch.uint8),
        "o": torch.zeros(B, H, 512, dtype=torch.bfloat16),
        "qo": torch.arange(B + 1, dtype=torch.int32),
        "kvp": torch.zeros(B + 1, dtype=torch.int32),
        "idx": torch.zeros(B * n_sh + sum(own_lens), dtype=torch.int32),
        "last": torch.ones(B, dtype=torch.int32),
        "qs": torch.ones(1, dtype=torch.float32),
        "ks": torch.ones(1, dtype=torch.float32),
        "lse": torch.zeros(B, H, dtype=torch.float32),
        "ws": torch.zeros(4096, dtype=torch.uint8),
        "shared": torch.arange(n_sh, dtype=torch.int32),
        "optr": torch.tensor([0, 3, 7], dtype=torch.int32),
        "own": torch.arange(10, 17, dtype=torch.int32),
    }
    prep = pm.PreparedDecode(t["q"], t["kv"], t["o"], t["qo"], t["kvp"], t["idx"], t["last"], 1,
                             192 ** -0.5, t["qs"], t["ks"], lse_out=t["lse"], workspace=t["ws"],
                             shared_prefix_len=n_sh, stream=0,
                             compact_page_table=(t["shared"], t["optr"], t["own"]))
    return prep, t


def test_prepared_decode_expands_into_the_workspace_error_word(lib, monkeypatch):
    """PreparedDecode with a compact page table: run() enqueues the expansion first, with
    the page-table tensors it was given and the workspace's error word (so mla_check_error
    reports a failed expansion), then the decode, both on the same stream."""
    fake = _RecordingLib()
    monkeypatch.setattr(lib, "_lib", fake)
    prep, t = _prepared_with_compact_table(lib)
    prep.run()
    assert [c[0] for c in fake.calls] == ["expand", "decode"]
    ex, dec = fake.calls[0][1], fake.calls[1][1]
    ptrs = [a._obj.ptr for a in ex[:5]]
    assert ptrs == [t[k].data_ptr() for k in ("shared", "optr", "own", "kvp", "idx")]
    assert ex[5].value == t["ws"].data_ptr()
    assert dec[-3].value == t["ws"].data_ptr()
    assert dec[-2].value == t["ws"].numel()
    assert ex[6].value == dec[-1].value


def test_prepared_decode_stops_when_the_expansion_is_rejected(lib, monkeypatch):
    """A host-side rejection of the expansion raises and enqueues no decode."""
    fake = _RecordingLib(expand_rc=1)
    monkeypatch.setattr(lib, "_lib", fake)
    prep, _ = _prepared_with_compact_table(lib)
    with pytest.raises(lib.MlaError):
        prep.run()
    assert [c[0] for c in fake.calls] == ["expand"]
