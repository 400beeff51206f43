"""FP64 CPU oracle for paged latent-MLA decode -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never links, loads or calls it,
and this package imports nothing from the CUDA library: the two share no code.

The arithmetic lives in ``mla_oracle.c`` (plain C, double precision, one (row, head)
at a time, OpenMP across rows); this module only marshals numpy arrays through ctypes
and builds the shared object with gcc on first use.

What it computes ("[Kimi-K3 MLA TP8] MLA performance", §2 geometry, §4.1 argument
table, §5.2 page_size = 1; "Scaling Kimi K3 on AMD Instinct MI355X", §1 DCP merge):

  for request b, query token t < T_b (row r = qo_indptr[b] + t), head h:
    J     = positions 0 .. L_b - T_b + t        (all L_b positions when T_b = 1)
    s_j   = sm_scale * q_scale * kv_scale * sum_{d<576} q[r,h,d] * kv[row_j, d]
    lse   = m + ln sum_j exp(s_j - m),   m = max_j s_j
    o[c]  = kv_scale * sum_j exp(s_j - lse) * kv[row_j, c],   c < 512

  merge of partials (o_i, lse_i):  M = max lse_i, w_i = exp(lse_i - M),
    o = sum w_i o_i / sum w_i,  lse = M + ln sum w_i.

Paged caches (page_size > 1) are reduced to this token view by expand_pages: a request's
positions are its pages' slots in order, the last page holding last_page_lens[b] of them.

The step after the decode (same issue, §2 geometry and §3: the 512-wide latent o is mapped
to v_head_dim = 128 by a separate batched matmul, one 512 x 128 matrix per head):
    v[t, h, n] = sum_{k<512} o[t, h, k] * w_uv[h, k, n]       (latent_to_v)

The step before it (same issue, §3: q's rope part rotated and concatenated after its 512
latent columns, the step's new 576-wide entry written into the cache; rope_concat_cache in
rope_cache.c, fp32 rotation, e4m3 codes of fp32(value / scale), ties to even, saturating):
    q_out[t, h] = e4m3([q_nope[t, h] / q_scale, rot(q_pe[t, h], pos_t) / q_scale])
    cache[slot_t] = e4m3([kv_c[t] / kv_scale, rot(k_pe[t], pos_t) / kv_scale])

Every function has a pin in ``tests/test_oracle_pins.py`` (brute force, closed forms,
invariants); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "rope_cache.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmlaoracle.so")
_lock = threading.Lock()
_lib = None

D = 576
DV = 512

_u8p = ctypes.POINTER(ctypes.c_uint8)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile mla_oracle.c into oracle/_build/libmlaoracle.so (portable C, no ISA flags)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(p) for p in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-adds, every float operation rounds on its own
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, *_SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.mlao_fp8_e4m3fn.restype = ctypes.c_double
        lib.mlao_fp8_e4m3fn.argtypes = [ctypes.c_uint]
        lib.mlao_fp8_table.restype = None
        lib.mlao_fp8_table.argtypes = [_f64p]
        lib.mlao_attend_one.restype = ctypes.c_int
        lib.mlao_attend_one.argtypes = [_u8p, _u8p, ctypes.c_int64, _i32p, ctypes.c_int64,
                                        ctypes.c_double, ctypes.c_double, _f64p, _f64p]
        lib.mlao_decode.restype = ctypes.c_int
        lib.mlao_decode.argtypes = [_u8p, ctypes.c_int, _u8p, ctypes.c_int64, _i32p, _i32p,
                                    _i32p, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                    ctypes.c_double, _f64p, _f64p, ctypes.c_int]
        lib.mlao_merge.restype = None
        lib.mlao_merge.argtypes = [_f64p, _f64p, ctypes.c_int, ctypes.c_int64, _f64p, _f64p]
        lib.mlao_max_threads.restype = ctypes.c_int
        lib.mlao_max_threads.argtypes = []
        lib.mlao_e4m3_encode.restype = ctypes.c_uint
        lib.mlao_e4m3_encode.argtypes = [ctypes.c_double]
        _u16p = ctypes.POINTER(ctypes.c_uint16)
        _f32p = ctypes.POINTER(ctypes.c_float)
        lib.mlao_rope_concat_cache.restype = ctypes.c_int
        lib.mlao_rope_concat_cache.argtypes = [_u16p, _u16p, _u16p, _u16p, _i32p, _f32p,
                                               ctypes.c_int64, ctypes.c_int, _i32p,
                                               ctypes.c_float, ctypes.c_float, ctypes.c_int64,
                                               ctypes.c_int, _u8p, _u8p, ctypes.c_int64]
        _lib = lib
        return lib


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def _u8(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint8:
        raise TypeError("fp8 operands are passed as their raw uint8 bytes")
    return np.ascontiguousarray(a)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def fp8_e4m3fn_table() -> np.ndarray:
    """The 256 float8 e4m3fn codes decoded from the format definition (fp64)."""
    lib = _load()
    out = np.empty(256, dtype=np.float64)
    lib.mlao_fp8_table(_ptr(out, _f64p))
    return out


def max_threads() -> int:
    return int(_load().mlao_max_threads())


def attend_one(qvec, kv, rows, sm_scale, q_scale, kv_scale):
    """One (query row, head): qvec (576,) u8, kv (N, 576) u8, rows (n_att,) int32.

    Returns (o (512,) fp64, lse float).  Scales are taken as given (pass the float32
    values the kernel sees, converted exactly to Python floats).
    """
    lib = _load()
    qvec = _u8(qvec).reshape(-1)
    kv = _u8(kv)
    rows = _i32(rows).reshape(-1)
    if qvec.size != D or kv.ndim != 2 or kv.shape[1] != D:
        raise ValueError("qvec must be (576,), kv (N, 576)")
    o = np.empty(DV, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    c = float(sm_scale) * float(q_scale) * float(kv_scale)
    rc = lib.mlao_attend_one(_ptr(qvec, _u8p), _ptr(kv, _u8p), kv.shape[0],
                             _ptr(rows, _i32p), rows.size, c, float(kv_scale),
                             _ptr(o, _f64p), _ptr(lse, _f64p))
    if rc != 0:
        raise ValueError(f"oracle attend_one failed with status {rc}")
    return o, float(lse[0])


def decode(q, kv, qo_indptr, kv_indptr, kv_indices, sm_scale, q_scale, kv_scale,
           n_threads: int = 0):
    """Whole decode call on host arrays.

    q (sum_T, H, 576) u8; kv (N, 576) u8 (or (N,1,1,576)); indptrs (B+1,) int32;
    kv_indices (>= kv_indptr[B],) int32.  Returns (o (sum_T, H, 512) fp64,
    lse (sum_T, H) fp64).
    """
    lib = _load()
    q = _u8(q)
    if q.ndim != 3 or q.shape[2] != D:
        raise ValueError("q must be (sum_T, H, 576)")
    kv = _u8(kv).reshape(-1, D)
    qo = _i32(qo_indptr)
    kvp = _i32(kv_indptr)
    idx = _i32(kv_indices)
    B = qo.size - 1
    if kvp.size != B + 1:
        raise ValueError("qo_indptr and kv_indptr must both have B+1 entries")
    if idx.size < int(kvp[-1]):
        raise ValueError("kv_indices shorter than kv_indptr[B]")
    if int(qo[-1]) != q.shape[0]:
        raise ValueError("qo_indptr[B] must equal q.shape[0]")
    n_tok, H = q.shape[0], q.shape[1]
    o = np.zeros((n_tok, H, DV), dtype=np.float64)
    lse = np.zeros((n_tok, H), dtype=np.float64)
    if idx.size == 0:
        idx = np.zeros(1, dtype=np.int32)
    rc = lib.mlao_decode(_ptr(q, _u8p), H, _ptr(kv, _u8p), kv.shape[0], _ptr(qo, _i32p),
                         _ptr(kvp, _i32p), _ptr(idx, _i32p), B, float(sm_scale),
                         float(q_scale), float(kv_scale), _ptr(o, _f64p), _ptr(lse, _f64p),
                         int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle decode failed with status {rc}")
    return o, lse


def expand_pages(kv_indptr, kv_indices, last_page_lens, page_size: int):
    """Token view of a paged cache: request b holds pages kv_indices[kv_indptr[b] ..
    kv_indptr[b+1]) in order; every page but the last contributes its page_size slots,
    the last one its first last_page_lens[b] slots; slot s of page p is cache row
    p * page_size + s.  Returns (token indptr (B+1,), row ids) as int32 arrays.

    ("[Kimi-K3 MLA TP8] MLA performance" §5.2: page-granular addressing of the same cache,
    page_size = the allocator's block size; a request's length is
    (pages - 1) * page_size + last_page_len.)
    """
    kvp = np.asarray(kv_indptr, dtype=np.int64)
    idx = np.asarray(kv_indices, dtype=np.int64)
    last = np.asarray(last_page_lens, dtype=np.int64)
    B = kvp.size - 1
    ptr = [0]
    rows = []
    for b in range(B):
        pages = idx[kvp[b]:kvp[b + 1]]
        n = 0
        for i, pg in enumerate(pages):
            used = page_size if i + 1 < pages.size else int(last[b])
            if not 1 <= used <= page_size:
                raise ValueError("last_page_lens must lie in [1, page_size]")
            rows.extend(int(pg) * page_size + s for s in range(used))
            n += used
        ptr.append(ptr[-1] + n)
    return (np.asarray(ptr, dtype=np.int32),
            np.asarray(rows if rows else [0], dtype=np.int32))


def decode_paged(q, kv_pages, qo_indptr, kv_indptr, kv_indices, last_page_lens, page_size,
                 sm_scale, q_scale, kv_scale, n_threads: int = 0):
    """decode() of a paged cache: kv_pages (N_pages, page_size, 576) (or with a head axis),
    kv_indptr in pages, kv_indices page ids, last_page_lens the last page's valid slots."""
    tok_ptr, rows = expand_pages(kv_indptr, kv_indices, last_page_lens, page_size)
    kv = _u8(kv_pages).reshape(-1, D)
    return decode(q, kv, qo_indptr, tok_ptr, rows, sm_scale, q_scale, kv_scale, n_threads)


def merge(o_parts, lse_parts):
    """Merge partials of one output: o_parts (P, W) fp64, lse_parts (P,) fp64."""
    lib = _load()
    o_parts = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    lse_parts = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64)).reshape(-1)
    P = lse_parts.size
    W = o_parts.size // max(P, 1) if P else 0
    o = np.empty(max(W, 1), dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    if P == 0:
        return np.zeros(0), float("-inf")
    lib.mlao_merge(_ptr(o_parts, _f64p), _ptr(lse_parts, _f64p), P, W, _ptr(o, _f64p),
                   _ptr(lse, _f64p))
    return o[:W].copy(), float(lse[0])


def merge_rows(o_parts, lse_parts):
    """Merge along axis 0 for every trailing row: o_parts (P, R, W), lse_parts (P, R)."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    P, R, W = o_parts.shape
    o = np.empty((R, W))
    lse = np.empty(R)
    for r in range(R):
        o[r], lse[r] = merge(o_parts[:, r, :], lse_parts[:, r])
    return o, lse


def bf16_to_f64(a) -> np.ndarray:
    """Exact float64 values of bfloat16 bit patterns (uint16 / int16 array): the bf16 word
    is the high half of a float32."""
    u = np.asarray(a).view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def latent_to_v(o, w_uv) -> np.ndarray:
    """v[t, h, :] = o[t, h, :] @ w_uv[h] in float64: o (T, H, K) and w_uv (H, K, N) real
    arrays (K = kv_lora_rank 512, N = v_head_dim 128 for the model; any sizes here).

    ("[Kimi-K3 MLA TP8] MLA performance" §2: kv_lora_rank 512, v_head_dim 128, 12 heads a
    GPU; §3: the decode's latent o goes through a separate per-head matmul to v_head_dim.)
    """
    o = np.asarray(o, dtype=np.float64)
    w = np.asarray(w_uv, dtype=np.float64)
    if o.ndim != 3 or w.ndim != 3 or o.shape[1] != w.shape[0] or o.shape[2] != w.shape[1]:
        raise ValueError("o (T, H, K) and w_uv (H, K, N) must agree in H and K")
    out = np.empty((o.shape[0], o.shape[1], w.shape[2]), dtype=np.float64)
    for h in range(o.shape[1]):
        out[:, h, :] = o[:, h, :] @ w[h]
    return out


def e4m3_encode(x) -> int:
    """e4m3fn code of the finite value nearest to x (ties to the even code, saturating at
    +-448, NaN -> 0x7F): the format's round-to-nearest-even, by search over its table."""
    return int(_load().mlao_e4m3_encode(float(x)))


def rope_concat_cache(q_nope, q_pe, kv_c, k_pe, positions, cos_sin, neox, slot_mapping,
                      q_scale, kv_scale, cache):
    """The fused step before the decode (rope_cache.c).

    q_nope (T, H, 512), q_pe (T, H, 64), kv_c (T, 512), k_pe (T, 64): bf16 bit patterns
    (uint16 arrays); positions, slot_mapping (T,) int32; cos_sin (max_pos, 64) float32;
    cache: uint8 array whose slots are its rows of 576 bytes in slot order (a paged cache
    (N_pages, PS, [1,] 576) reshaped to (N_pages * PS, 576)).  Returns (q_out (T, H, 576)
    uint8, new cache (same shape as `cache`), error bits: 1 position outside the table,
    2 slot outside the cache).  q_out bytes that are not written are 0x7F (fp8 NaN).
    """
    lib = _load()
    _u16p = ctypes.POINTER(ctypes.c_uint16)
    _f32p = ctypes.POINTER(ctypes.c_float)

    def u16(a):
        a = np.asarray(a)
        if a.dtype not in (np.uint16, np.int16):
            raise TypeError("bf16 operands are passed as their uint16 bit patterns")
        return np.ascontiguousarray(a.view(np.uint16))

    qn, qp, kc, kp = u16(q_nope), u16(q_pe), u16(kv_c), u16(k_pe)
    T, H = qn.shape[0], qn.shape[1]
    if qn.shape != (T, H, 512) or qp.shape != (T, H, 64) or kc.shape != (T, 512) or \
            kp.shape != (T, 64):
        raise ValueError("shapes: q_nope (T,H,512), q_pe (T,H,64), kv_c (T,512), k_pe (T,64)")
    pos = _i32(positions).reshape(-1)
    slots = _i32(slot_mapping).reshape(-1)
    cs = np.ascontiguousarray(np.asarray(cos_sin, dtype=np.float32))
    if pos.size != T or slots.size != T or cs.ndim != 2 or cs.shape[1] != 64:
        raise ValueError("positions/slot_mapping (T,), cos_sin (max_pos, 64)")
    out_cache = _u8(cache).copy()
    flat = out_cache.reshape(-1, D)
    q_out = np.full((T, H, D), 0x7F, dtype=np.uint8)
    err = lib.mlao_rope_concat_cache(
        _ptr(qn, _u16p), _ptr(qp, _u16p), _ptr(kc, _u16p), _ptr(kp, _u16p), _ptr(pos, _i32p),
        _ptr(cs, _f32p), cs.shape[0], int(bool(neox)), _ptr(slots, _i32p),
        float(np.float32(q_scale)), float(np.float32(kv_scale)), T, H, _ptr(q_out, _u8p),
        _ptr(flat, _u8p), flat.shape[0])
    return q_out, out_cache, int(err)
