"""Parity of mla_latent_to_v (the latent o mapped to v_head_dim = 128 by each head's
512 x 128 matrix, "[Kimi-K3 MLA TP8] MLA performance" §2 geometry and §3) with the FP64
oracle, through the C ABI.

Bound: the products of two bf16 values are exact in fp32; the kernel sums 512 of them in
two fp32 chains and rounds the total to bf16.  So |v - v_ref| <= 2^-8 |v_ref| (the final
rounding, half a bf16 ulp) + 512 * 2^-24 * sum_k |o_k w_kn| (the fp32 sums).
"""
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


def _bf16_host(t):
    return oracle.bf16_to_f64(t.detach().cpu().contiguous().view(torch.int16).numpy())


def _check(o, w, v):
    o64, w64 = _bf16_host(o), _bf16_host(w)
    ref = oracle.latent_to_v(o64, w64)
    mag = oracle.latent_to_v(np.abs(o64), np.abs(w64))
    got = _bf16_host(v)
    bound = 2.0 ** -8 * np.abs(ref) + 512 * 2.0 ** -24 * mag + 1e-30
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert (err <= bound).all(), f"worst err/bound {(err / bound).max():.3f}"
    return float((err / bound).max())


# token tiles: 16 (c16, 96-head shard, ragged), 32 (mtp), 128 (1,061 tokens: nine tiles, six
# stages cycling), 256 (4,096 tokens: a ring of four stages), one head
@pytest.mark.parametrize("n_tok,H", [(16, 12), (1, 96), (37, 12), (256, 12), (1061, 12), (3, 16),
                                     (4096, 12), (200, 1)])
def test_latent_to_v_matches_oracle(pm, n_tok, H):
    o, w = mla_inputs.make_vproj(n_tok, H, seed=n_tok + H, device="cuda")
    v = torch.full((n_tok, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    pm.mla_latent_to_v(o, w, v)
    torch.cuda.synchronize()
    _check(o, w, v)


def test_latent_to_v_strided_views(pm):
    """o and v as views of wider buffers (token and head strides not those of a dense
    tensor); columns outside the views stay untouched."""
    n_tok, H = 21, 12
    o_full = torch.randn((n_tok, H, 520), device="cuda").to(torch.bfloat16)
    o = o_full[:, :, :512]
    _, w = mla_inputs.make_vproj(1, H, seed=5, device="cuda")
    v_full = torch.full((n_tok, H, 136), 3.0, dtype=torch.bfloat16, device="cuda")
    v = v_full[:, :, :128]
    pm.mla_latent_to_v(o, w, v)
    torch.cuda.synchronize()
    _check(o, w, v)
    assert (v_full[:, :, 128:] == 3.0).all()


def test_latent_to_v_after_decode(pm):
    """The decode's own bf16 o (its real layout and values) through the projection."""
    case = gu.to_device(mla_inputs.make_custom([900, 2100, 64], q_lens=[1, 2, 1], H=12, seed=31,
                                               q_scale=1.0, kv_scale=1.0, name="vproj-chain"))
    o, lse, st = gu.run_gpu(case)
    assert st == 0
    _, w = mla_inputs.make_vproj(1, 12, seed=32, device="cuda")
    v = torch.empty((o.shape[0], 12, 128), dtype=torch.bfloat16, device="cuda")
    pm.mla_latent_to_v(o, w, v)
    torch.cuda.synchronize()
    _check(o, w, v)
    # and the chain against the oracle's decode: o within the decode's tolerance carries
    # through a matrix of column norm ~1
    o_ref, _ = gu.run_oracle(case)
    v_chain = oracle.latent_to_v(o_ref, _bf16_host(w))
    got = _bf16_host(v)
    colsum = np.abs(_bf16_host(w)).sum(axis=1)                  # (H, 128)
    tol = (gu.O_ATOL + gu.O_RTOL * np.abs(o_ref).max(axis=2, keepdims=True)) * colsum[None] \
        + 2.0 ** -8 * np.abs(v_chain) + 1e-6
    assert (np.abs(got - v_chain) <= tol).all()
