"""The context-parallel decode layer on one GPU with the CUDA kernels: emulate_ranks plays
every rank of the group in one process (the collectives become a concatenation and
slicing), so the partition, the head order, the draft-token handling and the merge map run
with mla_decode and mla_merge_partials.  Each rank's merged heads must match the oracle's
unsplit decode ("Scaling Kimi K3 on AMD Instinct MI355X" §1 "Cache": eight ranks, each
attending all heads over an eighth of the history)."""
import pytest
import torch

import mla_inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world,kv_lens,q_len,H_l,page_size", [
    (8, [17750 * 8], 1, 12, 1),              # the 142K request over 8 ranks, 96 heads
    (8, [3000, 700, 41], 4, 12, 1),          # draft tokens (causal on the last rank only)
    (4, [2500, 513], 2, 12, 64),             # pages of 64 tokens
    (2, [1200, 90, 5000], 1, 16, 1),
])
def test_emulated_ranks_match_oracle(world, kv_lens, q_len, H_l, page_size):
    from paged_mla_latent_gb300 import dcp
    H = H_l * world
    if page_size == 1:
        host = mla_inputs.make_custom(kv_lens, q_lens=[q_len] * len(kv_lens), H=H, seed=41,
                                      q_scale=1.0, kv_scale=1.0)
    else:
        host = mla_inputs.make_paged(kv_lens, q_lens=[q_len] * len(kv_lens), H=H,
                                     page_size=page_size, seed=41, q_scale=1.0, kv_scale=1.0)
    o_ref, lse_ref = gu.run_oracle(host)
    case = gu.to_device(host)
    shares = dcp.partition_positions(case.kv_indptr, case.kv_indices, case.kv_last_page_lens,
                                     case.q_lens, world, page_size)
    q_locals = [case.q[:, r * H_l:(r + 1) * H_l] for r in range(world)]
    outs = dcp.emulate_ranks(q_locals, case.kv, shares, case.qo_indptr, case.max_seqlen_q,
                             case.sm_scale, case.q_scale, case.kv_scale)
    torch.cuda.synchronize()
    for r, (o, lse) in enumerate(outs):
        gu.compare(o, lse, o_ref[:, r * H_l:(r + 1) * H_l], lse_ref[:, r * H_l:(r + 1) * H_l],
                   what=f"rank {r}")
