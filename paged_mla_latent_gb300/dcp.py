"""Decode context parallelism (DCP): the exchange around the decode when every GPU holds
only a share of each request's cached positions.

"Scaling Kimi K3 on AMD Instinct MI355X", §1 "Cache": with eight-way DCP each GPU stores
one eighth of the cached positions; every GPU then attends eight times as many heads over
its eighth of the history, and the partial answers, which carry their normalisation
(log-sum-exp), are merged exactly.  The steps, per decode step:

  1. all-gather q: rank r holds q for its H_l heads; afterwards every rank holds all
     world * H_l heads (head r * H_l + h is rank r's head h);
  2. local decode of all heads over the rank's positions -> partial (o fp32, lse);
  3. all-to-all: the partials of rank r's heads go back to rank r;
  4. LSE merge of the world partials of each (token, head) -> o (and lse).

Steps 2 and 4 are this library's mla_decode and mla_merge_partials (CUDA kernels); steps
1 and 3 are torch.distributed collectives (NCCL between GPUs).  Nothing here computes
attention: this module moves tensors and builds index maps.

Partition (how positions are spread, the caller's cache layout): contiguous blocks of each
request's page order, with the last rank holding the request's last q_len positions, so
that only it sees the draft tokens of a multi-token verification step.  There the decode's
own causal rule (query t sees positions <= kv_len - q_len + t) is the global rule.  Every
other rank holds history only, which every query sees: it decodes each request's q_len
tokens as one token with q_len * heads heads (a reshape of q), so no mask applies.  A batch
whose requests have different q_len > 1 is not supported on those ranks.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch


def partition_positions(kv_indptr, kv_indices, kv_last_page_lens, q_lens: Sequence[int],
                        world: int, page_size: int = 1):
    """Split every request's pages into `world` contiguous blocks, the last block holding
    at least the pages of the request's last q_len positions.

    kv_indptr (B+1,), kv_indices, kv_last_page_lens (B,) int32 (any device; read on the
    host).  Returns a list over ranks of (kv_indptr_r (B+1,), kv_indices_r, last_r (B,))
    int32 tensors on kv_indices' device.  A rank with no positions of request b gets an
    empty range there (and last_r[b] = page_size).
    """
    ip = [int(x) for x in kv_indptr.cpu().tolist()]
    last = [int(x) for x in kv_last_page_lens.cpu().tolist()] if kv_last_page_lens is not None \
        else [1] * (len(ip) - 1)
    dev = kv_indices.device
    B = len(ip) - 1
    ranks_ptr = [[0] for _ in range(world)]
    ranks_idx: List[List[torch.Tensor]] = [[] for _ in range(world)]
    ranks_last = [[] for _ in range(world)]
    for b in range(B):
        n = ip[b + 1] - ip[b]                      # pages
        L = (n - 1) * page_size + last[b] if n > 0 else 0
        T = int(q_lens[b])
        # pages holding the last T positions start at page (L - T) // page_size
        tail_first = max(0, (L - T) // page_size) if n > 0 else 0
        cuts = [min(r * n // world, tail_first) for r in range(world)] + [n]
        for r in range(world):
            a, e = cuts[r], cuts[r + 1]
            ranks_idx[r].append(kv_indices[ip[b] + a: ip[b] + e])
            ranks_ptr[r].append(ranks_ptr[r][-1] + (e - a))
            ranks_last[r].append(last[b] if (e == n and e > a) else page_size)
    out = []
    for r in range(world):
        idx = torch.cat(ranks_idx[r]) if ranks_idx[r] else torch.zeros(0, dtype=torch.int32, device=dev)
        if idx.numel() == 0:
            idx = torch.zeros(1, dtype=torch.int32, device=dev)   # never read (all ranges empty)
        out.append((torch.tensor(ranks_ptr[r], dtype=torch.int32, device=dev),
                    idx.to(torch.int32).contiguous(),
                    torch.tensor(ranks_last[r], dtype=torch.int32, device=dev)))
    return out


def merge_map(n_tok: int, world: int, device) -> Tuple[torch.Tensor, torch.Tensor]:
    """Reduce map of step 4 for partials laid out (world, n_tok, H_l, 512) -> rows
    s * n_tok + t: output row t merges rows {s * n_tok + t : s < world}."""
    t = torch.arange(n_tok, dtype=torch.int64)
    idx = (torch.arange(world, dtype=torch.int64)[None, :] * n_tok + t[:, None]).reshape(-1)
    indptr = torch.arange(0, (n_tok + 1) * world, world, dtype=torch.int64)
    return indptr.to(torch.int32).to(device), idx.to(torch.int32).to(device)


def _default_attend(q, kv, o, qo_indptr, kv_indptr, kv_indices, last, max_seqlen_q, sm_scale,
                    q_scale, kv_scale, lse_out, num_kv_splits=0, workspace=None):
    from . import mla_decode
    mla_decode(q, kv, o, qo_indptr, kv_indptr, kv_indices, last, max_seqlen_q, sm_scale,
               q_scale, kv_scale, num_kv_splits=num_kv_splits, lse_out=lse_out,
               workspace=workspace)


def _default_merge(o_parts, lse_parts, reduce_indptr, reduce_idx, o, lse_out):
    from . import mla_merge_partials
    mla_merge_partials(o_parts, lse_parts, reduce_indptr, reduce_idx, o, lse_out)


def local_partials(q_all, kv_buffer, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens,
                   q_lens: Sequence[int], max_seqlen_q: int, sm_scale, q_scale, kv_scale,
                   holds_drafts: bool, attend: Optional[Callable] = None, num_kv_splits=0,
                   workspace=None):
    """Step 2: all heads of q_all (n_tok, H_all, 576) over this rank's positions.  Returns
    (o (n_tok, H_all, 512) fp32, lse (n_tok, H_all) fp32).  holds_drafts: this rank holds
    every request's last q_len positions (the decode's causal rule applies as is); else
    each request's q_len tokens are decoded as one token of q_len * H_all heads."""
    attend = attend or _default_attend
    n_tok, H_all = q_all.shape[0], q_all.shape[1]
    dev = q_all.device
    o = torch.empty((n_tok, H_all, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((n_tok, H_all), dtype=torch.float32, device=dev)
    if holds_drafts or max_seqlen_q == 1:
        attend(q_all, kv_buffer, o, qo_indptr, kv_indptr, kv_indices, kv_last_page_lens,
               max_seqlen_q, sm_scale, q_scale, kv_scale, lse, num_kv_splits, workspace)
        return o, lse
    T = int(q_lens[0])
    if any(int(t) != T for t in q_lens):
        raise ValueError("context-parallel decode of draft tokens needs one q_len per batch")
    B = len(q_lens)
    qo1 = torch.arange(B + 1, dtype=torch.int32, device=qo_indptr.device)
    attend(q_all.view(B, T * H_all, q_all.shape[2]), kv_buffer, o.view(B, T * H_all, 512), qo1,
           kv_indptr, kv_indices, kv_last_page_lens, 1, sm_scale, q_scale, kv_scale,
           lse.view(B, T * H_all), num_kv_splits, workspace)
    return o, lse


def dcp_decode(q_local, kv_buffer, o_local, qo_indptr, kv_indptr, kv_indices,
               kv_last_page_lens, max_seqlen_q: int, sm_scale, q_scale, kv_scale,
               lse_local=None, group=None, holds_drafts: Optional[bool] = None,
               attend: Optional[Callable] = None, merge: Optional[Callable] = None,
               num_kv_splits: int = 0, workspace=None):
    """One context-parallel decode step on this rank.

    q_local (n_tok, H_l, 576) fp8: this rank's heads; kv_buffer / kv_indptr / kv_indices /
    kv_last_page_lens: this rank's share of the cache (partition_positions); qo_indptr the
    batch's query CSR (the same on every rank); o_local (n_tok, H_l, 512) (and lse_local
    (n_tok, H_l)) receive the merged result for this rank's heads.  holds_drafts defaults
    to "this is the last rank of the group" (partition_positions puts the drafts there).
    attend / merge replace mla_decode / mla_merge_partials (same arguments), e.g. to run the
    layer's data movement on CPU tensors.
    """
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if holds_drafts is None:
        holds_drafts = rank == world - 1
    n_tok, H_l, D = q_local.shape
    q_lens = (qo_indptr[1:] - qo_indptr[:-1]).cpu().tolist()
    # 1. all-gather q (as bytes: collectives move fp8 codes unchanged)
    gathered = torch.empty((world * n_tok, H_l, D), dtype=torch.uint8, device=q_local.device)
    dist.all_gather_into_tensor(gathered, q_local.contiguous().view(torch.uint8), group=group)
    q_all = gathered.view(world, n_tok, H_l, D).permute(1, 0, 2, 3).reshape(n_tok, world * H_l, D)
    if q_local.dtype != torch.uint8:
        q_all = q_all.view(q_local.dtype)
    # 2. local partials of all heads
    o_part, lse_part = local_partials(q_all, kv_buffer, qo_indptr, kv_indptr, kv_indices,
                                      kv_last_page_lens, q_lens, max_seqlen_q, sm_scale, q_scale,
                                      kv_scale, holds_drafts, attend, num_kv_splits, workspace)
    # 3. all-to-all: rank r receives every rank's partials of r's heads
    send_o = o_part.view(n_tok, world, H_l, 512).permute(1, 0, 2, 3).contiguous()
    send_l = lse_part.view(n_tok, world, H_l).permute(1, 0, 2).contiguous()
    recv_o = torch.empty_like(send_o)
    recv_l = torch.empty_like(send_l)
    dist.all_to_all_single(recv_o, send_o, group=group)
    dist.all_to_all_single(recv_l, send_l, group=group)
    # 4. merge the world partials of each (token, head)
    ip, idx = merge_map(n_tok, world, q_local.device)
    (merge or _default_merge)(recv_o.view(world * n_tok, H_l, 512), recv_l.view(world * n_tok, H_l),
                              ip, idx, o_local, lse_local)


def emulate_ranks(q_locals: List[torch.Tensor], kv_buffer, shares, qo_indptr,
                  max_seqlen_q: int, sm_scale, q_scale, kv_scale, o_dtype=torch.bfloat16,
                  attend: Optional[Callable] = None, merge: Optional[Callable] = None):
    """All ranks of a DCP group played by one process (one device): the collectives become
    a concatenation (step 1) and slicing (step 3); steps 2 and 4 run as in dcp_decode.
    For checking the layer's data movement on one GPU.  shares: partition_positions' list.
    Returns [(o_r, lse_r)] per rank."""
    world = len(q_locals)
    n_tok, H_l, D = q_locals[0].shape
    q_lens = (qo_indptr[1:] - qo_indptr[:-1]).cpu().tolist()
    q_all = torch.stack([q.contiguous() for q in q_locals], dim=1).reshape(n_tok, world * H_l, D)
    parts = []
    for r, (kvp, idx, last) in enumerate(shares):
        parts.append(local_partials(q_all, kv_buffer, qo_indptr, kvp, idx, last, q_lens,
                                    max_seqlen_q, sm_scale, q_scale, kv_scale, r == world - 1,
                                    attend))
    out = []
    ip, idx = merge_map(n_tok, world, q_all.device)
    for r in range(world):
        o_parts = torch.stack([p[0].view(n_tok, world, H_l, 512)[:, r] for p in parts])
        l_parts = torch.stack([p[1].view(n_tok, world, H_l)[:, r] for p in parts])
        o = torch.empty((n_tok, H_l, 512), dtype=o_dtype, device=q_all.device)
        lse = torch.empty((n_tok, H_l), dtype=torch.float32, device=q_all.device)
        (merge or _default_merge)(o_parts.reshape(world * n_tok, H_l, 512),
                                  l_parts.reshape(world * n_tok, H_l), ip, idx, o, lse)
        out.append((o, lse))
    return out
