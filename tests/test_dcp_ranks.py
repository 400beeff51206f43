"""Decode context parallelism ("Scaling Kimi K3 on AMD Instinct MI355X" §1 "Cache"): the
exchange layer (all-gather of q, local decode of all heads over a rank's share of the
positions, all-to-all of the partials back to the head owners, LSE merge) run as 2 and 4
gloo ranks on CPU.  Each rank's local decode and the merge are the oracle's (injected in
place of the CUDA calls), so what is tested is the layer's data movement: the partition,
the head order of the all-gather, the causal handling of draft tokens on ranks without
them, the routing of the all-to-all and the merge map.  The merged result of every rank
must equal the oracle's unsplit decode of that rank's heads."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import mla_inputs
import oracle


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def oracle_attend(q, kv, o, qo_indptr, kv_indptr, kv_indices, last, max_seqlen_q, sm_scale,
                  q_scale, kv_scale, lse_out, num_kv_splits=0, workspace=None):
    """The oracle in place of mla_decode (same arguments), writing fp32 o and lse."""
    qs, ks = float(q_scale.item()), float(kv_scale.item())
    ps = kv.shape[1] if kv.dim() == 4 else 1
    args = (q.cpu().numpy().view(np.uint8), kv.cpu().numpy().view(np.uint8),
            qo_indptr.cpu().numpy(), kv_indptr.cpu().numpy(), kv_indices.cpu().numpy())
    if ps > 1:
        o_ref, l_ref = oracle.decode_paged(*args, last.cpu().numpy(), ps, sm_scale, qs, ks)
    else:
        o_ref, l_ref = oracle.decode(*args, sm_scale, qs, ks)
    o.copy_(torch.from_numpy(o_ref).to(o.dtype))
    lse_out.copy_(torch.from_numpy(l_ref).to(lse_out.dtype))


def oracle_merge(o_parts, lse_parts, reduce_indptr, reduce_idx, o, lse_out):
    """The oracle's LSE merge in place of mla_merge_partials, following the reduce map."""
    ip, idx = reduce_indptr.tolist(), reduce_idx.tolist()
    op = o_parts.double().numpy()
    lp = lse_parts.double().numpy()
    for r in range(len(ip) - 1):
        rows = idx[ip[r]:ip[r + 1]]
        for h in range(o.shape[1]):
            m, l = oracle.merge(op[rows, h, :], lp[rows, h])
            o[r, h] = torch.from_numpy(m).to(o.dtype)
            if lse_out is not None:
                lse_out[r, h] = l


def _case(kv_lens, q_len, H, page_size, seed):
    if page_size == 1:
        return mla_inputs.make_custom(kv_lens, q_lens=[q_len] * len(kv_lens), H=H, seed=seed,
                                      q_scale=1.0, kv_scale=1.0)
    return mla_inputs.make_paged(kv_lens, q_lens=[q_len] * len(kv_lens), H=H,
                                 page_size=page_size, seed=seed, q_scale=1.0, kv_scale=1.0)


def _rank_main(rank, world, port, kv_lens, q_len, H_l, page_size, seed):
    import torch.distributed as dist
    from paged_mla_latent_gb300 import dcp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case = _case(kv_lens, q_len, H_l * world, page_size, seed)
        shares = dcp.partition_positions(case.kv_indptr, case.kv_indices, case.kv_last_page_lens,
                                         case.q_lens, world, page_size)
        kvp, idx, last = shares[rank]
        q_local = case.q[:, rank * H_l:(rank + 1) * H_l].contiguous()
        n_tok = case.q.shape[0]
        o = torch.zeros((n_tok, H_l, 512), dtype=torch.float32)
        lse = torch.zeros((n_tok, H_l), dtype=torch.float32)
        dcp.dcp_decode(q_local, case.kv, o, case.qo_indptr, kvp, idx, last, case.max_seqlen_q,
                       case.sm_scale, case.q_scale, case.kv_scale, lse_local=lse,
                       attend=oracle_attend, merge=oracle_merge)
        # the unsplit oracle decode of the whole request, this rank's heads
        full = torch.zeros((n_tok, H_l * world, 512))
        full_l = torch.zeros((n_tok, H_l * world))
        oracle_attend(case.q, case.kv, full, case.qo_indptr, case.kv_indptr, case.kv_indices,
                      case.kv_last_page_lens, case.max_seqlen_q, case.sm_scale, case.q_scale,
                      case.kv_scale, full_l)
        ref = full[:, rank * H_l:(rank + 1) * H_l]
        ref_l = full_l[:, rank * H_l:(rank + 1) * H_l]
        assert torch.allclose(o, ref, rtol=1e-5, atol=1e-6), float((o - ref).abs().max())
        assert torch.allclose(lse, ref_l, rtol=0, atol=1e-5), float((lse - ref_l).abs().max())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,kv_lens,q_len,H_l,page_size", [
    (2, [300, 77, 1000], 1, 3, 1),
    (2, [300, 77, 1000], 4, 3, 1),     # draft tokens: causal on the last rank only
    (4, [513, 9, 260], 4, 2, 1),       # a request shorter than the ranks
    (4, [700, 130, 64], 2, 2, 16),     # pages of 16 tokens, ragged last pages
])
def test_dcp_exchange_equals_unsplit_decode(world, kv_lens, q_len, H_l, page_size):
    mp.start_processes(_rank_main, args=(world, _free_port(), kv_lens, q_len, H_l, page_size, 5),
                       nprocs=world, join=True, start_method="spawn")


@pytest.mark.parametrize("world,page_size", [(2, 1), (4, 1), (8, 1), (3, 16), (8, 64)])
@pytest.mark.parametrize("q_len", [1, 4])
def test_partition_covers_every_position_once_with_drafts_on_the_last_rank(world, page_size, q_len):
    from paged_mla_latent_gb300 import dcp
    kv_lens = [1, 5, 64, 65, 1000, 17750, 3]
    case = _case(kv_lens, q_len, 2, page_size, 7) if page_size > 1 else \
        mla_inputs.make_custom(kv_lens, q_lens=[q_len] * len(kv_lens), H=2, seed=7)
    kvp = case.kv_indptr.tolist()
    ids = case.kv_indices.tolist()
    last = case.kv_last_page_lens.tolist()
    shares = dcp.partition_positions(case.kv_indptr, case.kv_indices, case.kv_last_page_lens,
                                     case.q_lens, world, page_size)
    for b, L in enumerate(kv_lens):
        pages, got_len = [], 0
        for r, (ip, idx, lst) in enumerate(shares):
            ip = ip.tolist()
            p = idx.tolist()[ip[b]:ip[b + 1]]
            pages += p
            n = len(p)
            length = (n - 1) * page_size + lst[b] if n else 0
            if n and r < world - 1:
                assert lst[b] == page_size          # whole pages before the last rank
            got_len += length
            if r == world - 1:
                assert length >= min(q_len, L)      # the drafts are all on the last rank
        assert pages == ids[kvp[b]:kvp[b + 1]]      # every page once, in order
        assert got_len == L


def test_merge_map_routes_every_rank_once():
    from paged_mla_latent_gb300 import dcp
    ip, idx = dcp.merge_map(5, 3, "cpu")
    assert ip.tolist() == [0, 3, 6, 9, 12, 15]
    for t in range(5):
        assert sorted(idx[ip[t]:ip[t + 1]].tolist()) == [t, 5 + t, 10 + t]
