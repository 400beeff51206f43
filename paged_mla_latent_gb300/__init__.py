"""Python binding of the GB300 paged latent-MLA decode library (argument marshalling only).

Every function here has the name of the C entry point it calls in
``include/paged_mla.h``; each converts torch tensors to ``mla_tensor_t`` descriptors
(pointer, dtype, shape, strides) and passes the current CUDA stream.  All arithmetic runs
in the library's CUDA kernels; there is no Python or CPU fallback: if the library cannot
be loaded, importing this package raises.

The operation ("[Kimi-K3 MLA TP8] MLA performance", §2-§5; "Scaling Kimi K3 on AMD
Instinct MI355X", §1 and §4): absorbed MLA decode over a paged FP8 cache (one token a
page as captured, or pages of 2..1024 tokens with kv_indptr counting pages and
kv_last_page_lens the last page's fill), each query head scoring every 576-wide latent
row, softmax over the request's positions
(causal within draft tokens), 512-wide BF16 latent output plus optional FP32 lse, and the
softmax-weighted merge of split-KV or context-shard partials.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "MlaError", "mla_decode", "mla_decode_shared_prefix", "mla_decode_noalloc", "mla_merge_partials",
    "mla_validate", "mla_check_error", "mla_get_workspace_size", "mla_get_shared_prefix_workspace_size",
    "mla_status_string", "make_workspace", "library_path", "PreparedDecode", "mla_latent_to_v",
    "mla_selftest_bounded_wait", "mla_qk_rope_concat_and_cache",
]

MLA_DTYPE_FP8_E4M3FN = 1
MLA_DTYPE_BF16 = 2
MLA_DTYPE_FP32 = 3
MLA_DTYPE_INT32 = 4

STATUS_NAMES = {
    0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED",
    3: "MLA_ERR_WORKSPACE_TOO_SMALL", 4: "MLA_ERR_CUDA", 5: "MLA_ERR_BAD_INDEX",
    6: "MLA_ERR_TIMEOUT", 7: "MLA_ERR_BAD_INPUT",
}


class MlaTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("ndim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.status, self.status)}")


def _load() -> ctypes.CDLL:
    path = _build.build()   # no-op when the in-tree library is up to date
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(MlaTensor)
    c_i32, c_sz, vp = ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_get_workspace_size.restype = ctypes.c_int
    lib.mla_get_workspace_size.argtypes = [c_i32, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_sz)]
    lib.mla_decode.restype = ctypes.c_int
    lib.mla_decode.argtypes = [P, P, P, P, P, P, P, c_i32, ctypes.c_float, P, P, c_i32, P, vp, c_sz, vp]
    lib.mla_get_shared_prefix_workspace_size.restype = ctypes.c_int
    lib.mla_get_shared_prefix_workspace_size.argtypes = [c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_sz)]
    lib.mla_decode_shared_prefix.restype = ctypes.c_int
    lib.mla_decode_shared_prefix.argtypes = [P, P, P, P, P, P, P, c_i32, ctypes.c_float, P, P, c_i32, P,
                                             vp, c_sz, vp]
    lib.mla_decode_noalloc.restype = ctypes.c_int
    lib.mla_decode_noalloc.argtypes = [P, P, P, P, P, P, P, c_i32, ctypes.c_float, P, P, c_i32, P, vp, vp]
    lib.mla_merge_partials.restype = ctypes.c_int
    lib.mla_merge_partials.argtypes = [P, P, P, P, P, P, vp, vp]
    lib.mla_expand_shared_prefix_indices.restype = ctypes.c_int
    lib.mla_expand_shared_prefix_indices.argtypes = [P, P, P, P, P, vp, vp]
    lib.mla_validate.restype = ctypes.c_int
    lib.mla_validate.argtypes = [P, P, P, P, P, P, vp, c_sz, vp]
    lib.mla_check_error.restype = ctypes.c_int
    lib.mla_check_error.argtypes = [vp, c_sz, vp]
    lib.mla_latent_to_v.restype = ctypes.c_int
    lib.mla_latent_to_v.argtypes = [P, P, P, vp]
    lib.mla_qk_rope_concat_and_cache.restype = ctypes.c_int
    lib.mla_qk_rope_concat_and_cache.argtypes = [P, P, P, P, P, P, c_i32, P, P, P, P, P, vp, vp]
    lib.mla_selftest_bounded_wait.restype = ctypes.c_int
    lib.mla_selftest_bounded_wait.argtypes = [vp, vp, ctypes.c_int64, vp]
    return lib


_lib = _load()


def library_path() -> str:
    return _build.LIB_PATH


_DTYPES = {
    torch.uint8: MLA_DTYPE_FP8_E4M3FN,           # raw e4m3fn codes
    torch.float8_e4m3fn: MLA_DTYPE_FP8_E4M3FN,
    torch.bfloat16: MLA_DTYPE_BF16,
    torch.float32: MLA_DTYPE_FP32,
    torch.int32: MLA_DTYPE_INT32,
}


_I64x4 = ctypes.c_int64 * 4
_PAD = ((), (0,), (0, 0), (0, 0, 0), (0, 0, 0, 0))


def _desc(t):
    """The mla_tensor_t of a torch tensor: pointer, dtype, shape and strides (elements)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    shape = t.shape
    n = len(shape)
    if n > 4:
        raise ValueError("at most 4 dimensions")
    try:
        code = _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None
    pad = _PAD[4 - n]
    return MlaTensor(t.data_ptr() or None, n, code, _I64x4(*shape, *pad),
                     _I64x4(*t.stride(), *pad))


def _ref(d):
    return ctypes.byref(d) if d is not None else None


def _stream(stream, device):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(rc: int, where: str):
    if rc != 0:
        raise MlaError(rc, where)


def mla_status_string(status: int) -> str:
    return _lib.mla_status_string(int(status)).decode()


def mla_get_workspace_size(batch_size: int, num_heads: int, max_seqlen_q: int = 1,
                           num_kv_splits: int = 0, num_sms: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.mla_get_workspace_size(batch_size, num_heads, max_seqlen_q, num_kv_splits,
                                       num_sms, ctypes.byref(out)), "mla_get_workspace_size")
    return int(out.value)


def mla_get_shared_prefix_workspace_size(batch_size: int, num_heads: int, max_seqlen_q: int = 1,
                                         num_sms: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.mla_get_shared_prefix_workspace_size(batch_size, num_heads, max_seqlen_q, num_sms,
                                                     ctypes.byref(out)),
           "mla_get_shared_prefix_workspace_size")
    return int(out.value)


def make_workspace(batch_size: int, num_heads: int, max_seqlen_q: int = 1,
                   num_kv_splits: int = 0, device=None, shared_prefix: bool = False) -> torch.Tensor:
    """A zero-initialised device workspace large enough for such calls (shared_prefix:
    for mla_decode_shared_prefix)."""
    device = torch.device(device or "cuda")
    with torch.cuda.device(device):
        if shared_prefix:
            n = mla_get_shared_prefix_workspace_size(batch_size, num_heads, max_seqlen_q)
        else:
            n = mla_get_workspace_size(batch_size, num_heads, max_seqlen_q, num_kv_splits)
    return torch.zeros(n, dtype=torch.uint8, device=device)




def mla_decode(q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens,
               max_seqlen_q, sm_scale, q_scale, kv_scale, num_kv_splits=0, lse_out=None,
               workspace=None, stream=None):
    """Enqueue one decode call (see include/paged_mla.h).  Returns the workspace used."""
    if workspace is None:
        workspace = make_workspace(len(kv_indptr) - 1, q.shape[1], max_seqlen_q,
                                   num_kv_splits, q.device)
    descs = [_desc(t) for t in (q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices,
                                kv_last_page_lens, q_scale, kv_scale, lse_out)]
    dq, dkv, do, dqo, dkvp, didx, dlast, dqs, dks, dlse = descs
    rc = _lib.mla_decode(_ref(dq), _ref(dkv), _ref(do), _ref(dqo), _ref(dkvp), _ref(didx),
                         _ref(dlast), int(max_seqlen_q), float(sm_scale), _ref(dqs), _ref(dks),
                         int(num_kv_splits), _ref(dlse), ctypes.c_void_p(workspace.data_ptr()),
                         workspace.numel() * workspace.element_size(), _stream(stream, q.device))
    _check(rc, "mla_decode")
    return workspace


def mla_decode_shared_prefix(q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices,
                             kv_last_page_lens, max_seqlen_q, sm_scale, q_scale, kv_scale,
                             shared_prefix_len, lse_out=None, workspace=None, stream=None):
    """Decode a batch whose requests share their first shared_prefix_len cache positions
    (see include/paged_mla.h).  Returns the workspace used."""
    if workspace is None:
        workspace = make_workspace(len(kv_indptr) - 1, q.shape[1], max_seqlen_q, 0, q.device,
                                   shared_prefix=True)
    descs = [_desc(t) for t in (q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices,
                                kv_last_page_lens, q_scale, kv_scale, lse_out)]
    dq, dkv, do, dqo, dkvp, didx, dlast, dqs, dks, dlse = descs
    rc = _lib.mla_decode_shared_prefix(
        _ref(dq), _ref(dkv), _ref(do), _ref(dqo), _ref(dkvp), _ref(didx), _ref(dlast),
        int(max_seqlen_q), float(sm_scale), _ref(dqs), _ref(dks), int(shared_prefix_len),
        _ref(dlse), ctypes.c_void_p(workspace.data_ptr()),
        workspace.numel() * workspace.element_size(), _stream(stream, q.device))
    _check(rc, "mla_decode_shared_prefix")
    return workspace


class PreparedDecode:
    """One mla_decode (or, with shared_prefix_len, mla_decode_shared_prefix) call whose
    argument descriptors are built once, for a caller that runs the same buffers every step
    (fresh data in the same tensors).  run() enqueues the call through the C ABI with no
    per-call argument marshalling.  The descriptors hold the tensors' addresses, shapes and
    strides as they were here: prepare again after reallocating or reshaping any of them.
    The object keeps the tensors alive.
    """

    def __init__(self, q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens,
                 max_seqlen_q, sm_scale, q_scale, kv_scale, num_kv_splits=0, lse_out=None,
                 workspace=None, shared_prefix_len=None, stream=None, compact_page_table=None):
        """compact_page_table: optional (shared_indices, own_indptr, own_indices) device
        tensors; run() then first rebuilds kv_indptr / kv_indices from them with
        mla_expand_shared_prefix_indices (a caller that uploads its page table every step
        sends the shared pages once).  The expansion's device-side errors (an own_indptr
        that is not monotone, a table longer than kv_indices) go to the workspace's error
        word, where mla_check_error reports them with the decode's own."""
        shared = shared_prefix_len is not None
        if workspace is None:
            workspace = make_workspace(len(kv_indptr) - 1, q.shape[1], max_seqlen_q,
                                       0 if shared else num_kv_splits, q.device,
                                       shared_prefix=shared)
        self.workspace = workspace
        self._keep = (q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens,
                      q_scale, kv_scale, lse_out, workspace)
        self._descs = [_desc(t) for t in self._keep[:10]]
        r = [_ref(d) for d in self._descs]
        tail = (ctypes.c_void_p(workspace.data_ptr()),
                ctypes.c_size_t(workspace.numel() * workspace.element_size()))
        if shared:
            self._fn, self._where = _lib.mla_decode_shared_prefix, "mla_decode_shared_prefix"
            self._args = (r[0], r[1], r[2], r[3], r[4], r[5], r[6], int(max_seqlen_q),
                          float(sm_scale), r[7], r[8], int(shared_prefix_len), r[9]) + tail
        else:
            self._fn, self._where = _lib.mla_decode, "mla_decode"
            self._args = (r[0], r[1], r[2], r[3], r[4], r[5], r[6], int(max_seqlen_q),
                          float(sm_scale), r[7], r[8], int(num_kv_splits), r[9]) + tail
        self._device = q.device
        self._stream = None if stream is None else _stream(stream, q.device)
        self._expand = None
        if compact_page_table is not None:
            sh, optr, own = compact_page_table
            self._expand_keep = (sh, optr, own)
            self._expand_descs = [_desc(t) for t in (sh, optr, own)] + self._descs[4:6]
            self._expand = tuple(_ref(d) for d in self._expand_descs) + (
                ctypes.c_void_p(workspace.data_ptr()),)

    def run(self, stream=None):
        """Enqueue the call on `stream` (default: the stream given when prepared, else
        torch's current stream)."""
        st = _stream(stream, self._device) if stream is not None else (
            self._stream if self._stream is not None else _stream(None, self._device))
        if self._expand is not None:
            rc = _lib.mla_expand_shared_prefix_indices(*self._expand, st)
            if rc != 0:
                raise MlaError(rc, "mla_expand_shared_prefix_indices")
        rc = self._fn(*self._args, st)
        if rc != 0:
            raise MlaError(rc, self._where)
        return self.workspace


def mla_decode_noalloc(q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens,
                       max_seqlen_q, sm_scale, q_scale, kv_scale, num_kv_splits=0, lse_out=None,
                       error_out=None, stream=None):
    """Decode without a workspace: scratch lives in the library's fixed device array.

    For callers that cannot allocate device memory.  error_out: optional int32 device
    tensor receiving the call's raw device error bits.  Raises MlaError on a host-side
    error, including MLA_ERR_WORKSPACE_TOO_SMALL when the call needs more scratch than
    the fixed array holds.
    """
    descs = [_desc(t) for t in (q, kv_buffer, o, qo_indptr, kv_indptr, kv_indices,
                                kv_last_page_lens, q_scale, kv_scale, lse_out)]
    dq, dkv, do, dqo, dkvp, didx, dlast, dqs, dks, dlse = descs
    if error_out is not None:
        # the library copies 4 bytes device-to-device into it after the decode is queued
        if not isinstance(error_out, torch.Tensor) or error_out.dtype != torch.int32 or \
                error_out.numel() < 1 or error_out.device != q.device:
            raise ValueError("error_out must be an int32 tensor of at least one element on "
                             f"{q.device}")
    ew = ctypes.c_void_p(error_out.data_ptr()) if error_out is not None else None
    rc = _lib.mla_decode_noalloc(_ref(dq), _ref(dkv), _ref(do), _ref(dqo), _ref(dkvp), _ref(didx),
                                 _ref(dlast), int(max_seqlen_q), float(sm_scale), _ref(dqs),
                                 _ref(dks), int(num_kv_splits), _ref(dlse), ew,
                                 _stream(stream, q.device))
    _check(rc, "mla_decode_noalloc")


def mla_expand_shared_prefix_indices(shared_indices, own_indptr, own_indices, kv_indptr,
                                     kv_indices, error_word=None, stream=None):
    """Build the full page table of a shared-prefix batch on the device from the shared page
    ids (once) and each request's own ids (see include/paged_mla.h)."""
    descs = [_desc(t) for t in (shared_indices, own_indptr, own_indices, kv_indptr, kv_indices)]
    if error_word is not None and (not isinstance(error_word, torch.Tensor) or
                                   error_word.dtype != torch.int32 or error_word.numel() < 1 or
                                   error_word.device != kv_indices.device):
        raise ValueError("error_word must be an int32 tensor on the page table's device")
    ew = ctypes.c_void_p(error_word.data_ptr()) if error_word is not None else None
    rc = _lib.mla_expand_shared_prefix_indices(*[_ref(d) for d in descs], ew,
                                               _stream(stream, kv_indices.device))
    _check(rc, "mla_expand_shared_prefix_indices")


def mla_merge_partials(o_parts, lse_parts, reduce_indptr, reduce_idx, o, lse_out=None,
                       error_word=None, stream=None):
    """Softmax-weighted merge of partials with a CSR reduce map (see include/paged_mla.h)."""
    descs = [_desc(t) for t in (o_parts, lse_parts, reduce_indptr, reduce_idx, o, lse_out)]
    ew = ctypes.c_void_p(error_word.data_ptr()) if error_word is not None else None
    rc = _lib.mla_merge_partials(*[_ref(d) for d in descs], ew, _stream(stream, o.device))
    _check(rc, "mla_merge_partials")


def mla_latent_to_v(o, w_uv, v, stream=None):
    """v[t, h, :] = o[t, h, :] @ w_uv[h]: the latent o mapped to v_head_dim (see
    include/paged_mla.h)."""
    descs = [_desc(t) for t in (o, w_uv, v)]
    rc = _lib.mla_latent_to_v(*[_ref(d) for d in descs], _stream(stream, v.device))
    _check(rc, "mla_latent_to_v")


def mla_qk_rope_concat_and_cache(q_nope, q_pe, kv_c, k_pe, positions, cos_sin, is_neox,
                                 slot_mapping, q_scale, kv_scale, q_out, kv_buffer,
                                 error_word, stream=None):
    """Rotate q's and the new keys' rope columns, quantise q to the decode's fp8 q_out and
    write each token's new 576-wide entry into kv_buffer at its slot (see
    include/paged_mla.h).  error_word: an int32 device tensor (>= 1 element)."""
    if not isinstance(error_word, torch.Tensor) or error_word.dtype != torch.int32 or \
            error_word.numel() < 1 or error_word.device != q_out.device:
        raise ValueError(f"error_word must be an int32 tensor on {q_out.device}")
    descs = [_desc(t) for t in (q_nope, q_pe, kv_c, k_pe, positions, cos_sin)]
    tail = [_desc(t) for t in (slot_mapping, q_scale, kv_scale, q_out, kv_buffer)]
    rc = _lib.mla_qk_rope_concat_and_cache(*[_ref(d) for d in descs], int(is_neox),
                                           *[_ref(d) for d in tail],
                                           ctypes.c_void_p(error_word.data_ptr()),
                                           _stream(stream, q_out.device))
    _check(rc, "mla_qk_rope_concat_and_cache")


def mla_selftest_bounded_wait(error_word, result, limit_ns, stream=None):
    """Run the library's bounded mbarrier wait on a barrier nothing arrives at (see
    include/paged_mla.h): error_word (1) and result (3) are int32 device tensors."""
    for t, n in ((error_word, 1), (result, 3)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or t.numel() < n or \
                not t.is_cuda:
            raise ValueError(f"expected an int32 CUDA tensor of at least {n} element(s)")
    rc = _lib.mla_selftest_bounded_wait(ctypes.c_void_p(error_word.data_ptr()),
                                        ctypes.c_void_p(result.data_ptr()), int(limit_ns),
                                        _stream(stream, result.device))
    _check(rc, "mla_selftest_bounded_wait")


def mla_validate(q, kv_buffer, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens,
                 workspace, stream=None) -> int:
    """Device-side check of the index inputs; returns the status code (synchronises)."""
    descs = [_desc(t) for t in (q, kv_buffer, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens)]
    return int(_lib.mla_validate(*[_ref(d) for d in descs], ctypes.c_void_p(workspace.data_ptr()),
                                 workspace.numel(), _stream(stream, q.device)))


def mla_check_error(workspace, stream=None) -> int:
    """First device-side error recorded in the workspace since the last check (clears it)."""
    return int(_lib.mla_check_error(ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                    _stream(stream, workspace.device)))
