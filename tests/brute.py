"""Independent brute-force reference used to pin the oracle (tests only).

It shares nothing with ``oracle/``: FP8 bytes are decoded by torch's own
float8_e4m3fn -> float64 cast, and the softmax is evaluated with numpy float64 array
operations over a dense gathered matrix (no streaming, no per-row loops over d).
"""
import numpy as np
import torch


def fp8_decode(u8) -> np.ndarray:
    """Decode e4m3fn bytes with torch's cast (an implementation independent of the oracle)."""
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(u8, dtype=np.uint8)))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def attend(qvec_u8, rows_u8, logit_scale, kv_scale):
    """Dense softmax attention of one query over the given (n, 576) rows, float64."""
    qf = fp8_decode(qvec_u8).reshape(576)
    K = fp8_decode(rows_u8).reshape(-1, 576)
    if K.shape[0] == 0:
        return np.zeros(512), -np.inf
    s = logit_scale * (K @ qf)
    m = s.max()
    e = np.exp(s - m)
    z = e.sum()
    o = kv_scale * (e[:, None] * K[:, :512]).sum(axis=0) / z
    return o, float(m + np.log(z))


def decode(q_u8, kv_u8, qo_indptr, kv_indptr, kv_indices, sm_scale, q_scale, kv_scale):
    q_u8 = np.asarray(q_u8)
    kv_u8 = np.asarray(kv_u8).reshape(-1, 576)
    n_tok, H = q_u8.shape[0], q_u8.shape[1]
    o = np.zeros((n_tok, H, 512))
    lse = np.zeros((n_tok, H))
    c = sm_scale * q_scale * kv_scale
    for b in range(len(qo_indptr) - 1):
        T = qo_indptr[b + 1] - qo_indptr[b]
        L = kv_indptr[b + 1] - kv_indptr[b]
        rows = np.asarray(kv_indices[kv_indptr[b]:kv_indptr[b + 1]])
        for t in range(T):
            r = qo_indptr[b] + t
            n_att = L - T + t + 1
            for h in range(H):
                o[r, h], lse[r, h] = attend(q_u8[r, h], kv_u8[rows[:max(n_att, 0)]], c, kv_scale)
    return o, lse
