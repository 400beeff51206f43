"""Helpers shared by the GPU tests: run the CUDA path on a workload, run the oracle on the
same bytes, compare with the tolerance the decode must meet."""
import math

import numpy as np
import torch

import mla_inputs
import oracle

# max|o - o_ref| <= O_ATOL + O_RTOL * |o_ref| elementwise, and |lse - lse_ref| <= LSE_ATOL.
O_ATOL = 1e-2
O_RTOL = 1e-2
LSE_ATOL = 1e-3


def to_device(case, device="cuda"):
    for f in ("q", "kv", "qo_indptr", "kv_indptr", "kv_indices", "kv_last_page_lens", "q_scale",
              "kv_scale"):
        setattr(case, f, getattr(case, f).to(device))
    return case


def run_gpu(case, num_kv_splits=0, o_dtype=torch.bfloat16, with_lse=True, workspace=None,
            kv_view=None, q_override=None, shared_prefix=None):
    """shared_prefix: None -> mla_decode; an int P -> mla_decode_shared_prefix(P)."""
    import paged_mla_latent_gb300 as pm
    q = case.q if q_override is None else q_override
    n_tok, H = q.shape[0], q.shape[1]
    o = torch.full((n_tok, H, 512), float("nan"), dtype=o_dtype, device=q.device)
    lse = torch.full((n_tok, H), float("nan"), dtype=torch.float32, device=q.device) if with_lse else None
    if workspace is None:
        workspace = pm.make_workspace(case.B, H, case.max_seqlen_q, num_kv_splits, q.device,
                                      shared_prefix=shared_prefix is not None)
    kv = case.kv if kv_view is None else kv_view
    if shared_prefix is None:
        pm.mla_decode(q, kv, o, case.qo_indptr, case.kv_indptr, case.kv_indices,
                      case.kv_last_page_lens, case.max_seqlen_q, case.sm_scale, case.q_scale,
                      case.kv_scale, num_kv_splits=num_kv_splits, lse_out=lse, workspace=workspace)
    else:
        pm.mla_decode_shared_prefix(q, kv, o, case.qo_indptr, case.kv_indptr, case.kv_indices,
                                    case.kv_last_page_lens, case.max_seqlen_q, case.sm_scale,
                                    case.q_scale, case.kv_scale, shared_prefix, lse_out=lse,
                                    workspace=workspace)
    torch.cuda.synchronize()
    status = pm.mla_check_error(workspace)
    return o, lse, status


def run_oracle(case, q_override=None):
    sm, qs, ks = case.scales()
    q = (case.q if q_override is None else q_override).cpu().numpy()
    ps = int(case.meta.get("page_size", 1))
    if ps > 1:
        return oracle.decode_paged(q, case.kv.cpu().numpy(), case.qo_indptr.cpu().numpy(),
                                   case.kv_indptr.cpu().numpy(), case.kv_indices.cpu().numpy(),
                                   case.kv_last_page_lens.cpu().numpy(), ps, sm, qs, ks)
    return oracle.decode(q, case.kv.cpu().numpy(), case.qo_indptr.cpu().numpy(),
                         case.kv_indptr.cpu().numpy(), case.kv_indices.cpu().numpy(), sm, qs, ks)


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what="", rows_mask=None):
    """Assert the tolerance; returns a dict of error statistics."""
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    d = np.abs(o - o_ref)
    bound = O_ATOL + O_RTOL * np.abs(o_ref)
    stats = dict(max_abs=float(d.max()) if d.size else 0.0,
                 worst_ratio=float((d / bound).max()) if d.size else 0.0,
                 err_over_std=float(d.max() / max(o_ref.std(), 1e-30)) if d.size else 0.0)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    assert (d <= bound).all(), f"{what}: o error {stats}"
    if lse_gpu is not None:
        l = lse_gpu.cpu().numpy().astype(np.float64)
        both_inf = np.isneginf(l) & np.isneginf(lse_ref)
        dl = np.where(both_inf, 0.0, np.abs(l - lse_ref))
        stats["lse_max_abs"] = float(dl.max()) if dl.size else 0.0
        assert (dl <= LSE_ATOL).all(), f"{what}: lse error {stats}"
    return stats


def gather_rows(case, b):
    """Host copy of the cache rows request b attends, in position order."""
    s, e = int(case.kv_indptr[b]), int(case.kv_indptr[b + 1])
    idx = case.kv_indices[s:e].long()
    return case.kv.index_select(0, idx).cpu().numpy()


def oracle_sampled(case, samples):
    """Oracle for a few (request, token-within-request, head) triples of a large case."""
    sm, qs, ks = case.scales()
    out = []
    q_host = {}
    for b, t, h in samples:
        rows = gather_rows(case, b)
        L = rows.shape[0]
        T = case.q_lens[b]
        r = int(case.qo_indptr[b]) + t
        if r not in q_host:
            q_host[r] = case.q[r].cpu().numpy()
        n_att = L - T + t + 1
        o, lse = oracle.attend_one(q_host[r][h], rows, np.arange(n_att, dtype=np.int32), sm, qs, ks)
        out.append((r, h, o, lse))
    return out


def oracle_requests(case, reqs):
    """Oracle for every query token and head of the requests `reqs` of a large case (one-
    token pages): {b: (o_ref (T_b, H, 512), lse_ref (T_b, H))}.  Each request's rows are
    gathered once on the device, copied to the host and decoded by the oracle as a batch
    of one (all its heads and drafts at once, OpenMP across them)."""
    sm, qs, ks = case.scales()
    out = {}
    for b in reqs:
        rows = gather_rows(case, b)
        L = rows.shape[0]
        t0, t1 = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        q = case.q[t0:t1].cpu().numpy()
        o_ref, lse_ref = oracle.decode(q, rows, np.array([0, t1 - t0], np.int32),
                                       np.array([0, L], np.int32), np.arange(L, dtype=np.int32),
                                       sm, qs, ks)
        out[b] = (o_ref, lse_ref)
    return out


def compare_requests(case, o, lse, refs, what=""):
    """Assert the tolerance on every (token, head) of the requests in `refs`."""
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    worst = 0.0
    for b, (o_ref, lse_ref) in refs.items():
        t0, t1 = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        d = np.abs(og[t0:t1] - o_ref)
        bound = O_ATOL + O_RTOL * np.abs(o_ref)
        assert (d <= bound).all(), (what, b, float(d.max()))
        dl = np.abs(lg[t0:t1] - lse_ref)
        assert (dl <= LSE_ATOL).all(), (what, b, float(dl.max()))
        worst = max(worst, float((d / bound).max()))
    return worst
