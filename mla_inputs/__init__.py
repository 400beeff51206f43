"""Seeded synthetic workloads for paged latent-MLA decode.

This module only *makes inputs*: FP8 bytes, index lists and lengths.  It holds none of
the attention arithmetic, so both the CUDA path and the CPU oracle may use it.  The
shapes follow the argument capture in "[Kimi-K3 MLA TP8] MLA performance" (ROCm/aiter
issue 4541):

  * §2: 12 query heads per GPU at TP8 (96 globally), one 576-byte latent entry per token.
  * §4.1 / §4.2: concurrency 16 and 24, kv_buffer of 5,283,840 rows x 576 fp8,
    kv_indices buffer of 4,718,592 int32 (longer than the attended total),
    kv_len ~68.4K per request, q_len 1.
  * §1 "Environment": the workload is a 63,911-token shared prefix + 4,089 unique input
    tokens + up to 350 generated tokens per request.
  * §5.2: page_size = 1 as captured (kv_indptr holds token counts, kv_last_page_lens is
    all ones), and the block-granular layout it proposes: make_paged builds caches of
    page_size-token pages (128 = the allocator's block), kv_indptr counting pages.

and the long-context / shard figures of "Scaling Kimi K3 on AMD Instinct MI355X",
§1 "Cache" (142,000-token conversation, DCP8 -> 8 shards, 96 heads per shard call).
make_vproj draws the inputs of the step after the decode (latent o and one 512 x 128
matrix per head, §2 of the issue: kv_lora_rank 512, v_head_dim 128).

Values are N(0, 1) draws, clamped to +-448 (the e4m3fn range) and rounded to
float8_e4m3fn by torch's cast; only the resulting bytes matter.  Lengths and jitter come
from numpy's PCG64 (platform independent); bulk values and permutations from a seeded
torch generator on the target device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

D = 576          # latent entry width (512 latent + 64 rope)
DV = 512         # value width
SM_SCALE = 192.0 ** -0.5             # 0.07216878364870322 as printed in issue §2
POISON_FP8 = 0x7F                    # an e4m3fn NaN code
DEFAULT_Q_SCALE = 0.05
DEFAULT_KV_SCALE = 0.1


@dataclass
class Case:
    """One decode call's inputs (all tensors on one device)."""
    name: str
    q: torch.Tensor              # (sum_T, H, 576) uint8 (fp8 e4m3fn bytes)
    kv: torch.Tensor             # (N_rows, 576) uint8
    qo_indptr: torch.Tensor      # (B+1,) int32
    kv_indptr: torch.Tensor      # (B+1,) int32
    kv_indices: torch.Tensor     # (>= kv_indptr[B],) int32
    kv_last_page_lens: torch.Tensor  # (B,) int32, all ones
    q_scale: torch.Tensor        # 0-dim float32
    kv_scale: torch.Tensor       # 0-dim float32
    sm_scale: float
    kv_lens: list
    q_lens: list
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return len(self.kv_lens)

    @property
    def H(self) -> int:
        return int(self.q.shape[1])

    @property
    def max_seqlen_q(self) -> int:
        return max(self.q_lens) if self.q_lens else 1

    @property
    def total_kv(self) -> int:
        return int(sum(self.kv_lens))

    def scales(self):
        """(sm_scale, q_scale, kv_scale) as Python floats equal to the float32 values."""
        return (float(np.float32(self.sm_scale)), float(self.q_scale.item()),
                float(self.kv_scale.item()))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def fp8_normal_bytes(n: int, gen: torch.Generator, device, chunk: int = 1 << 26) -> torch.Tensor:
    """n float8_e4m3fn bytes from N(0,1), clamped to +-448 (the cast rounds to nearest even)."""
    out = torch.empty(n, dtype=torch.uint8, device=device)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        x = torch.randn(m, generator=gen, device=device, dtype=torch.float32)
        x.clamp_(-448.0, 448.0)
        out[s:s + m] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        del x
    return out


def make_vproj(n_tok: int, H: int = 12, seed: int = 0, device="cpu", o_scale: float = 1.0):
    """Inputs of the latent -> v_head_dim step: o (n_tok, H, 512) bf16 from N(0, o_scale^2)
    and w_uv (H, 512, 128) bf16 from N(0, 1/512), the scale of a random-init projection."""
    gen = _gen(seed, device)
    o = (torch.randn((n_tok, H, DV), generator=gen, device=device) * o_scale).to(torch.bfloat16)
    w = (torch.randn((H, DV, 128), generator=gen, device=device) * DV ** -0.5).to(torch.bfloat16)
    return o, w


def make_rope_inputs(n_tok: int, H: int = 12, max_pos: int = 73728, seed: int = 0,
                     device="cpu", value_scale: float = 1.0, rope_base: float = 10000.0):
    """Inputs of the step before the decode (q rope + concat + cache write): bf16 q_nope
    (n_tok, H, 512), q_pe (n_tok, H, 64), kv_c (n_tok, 512), k_pe (n_tok, 64) from
    N(0, value_scale^2); positions uniform in [0, max_pos); a float32 rotary table
    (max_pos, 64) of cos then sin of p * rope_base^(-i/32), i < 32 (the caller's table: the
    pages give neither base nor scaling, any table is valid input).  max_pos 73,728 is the
    captured deployment's max model length (issue §1)."""
    gen = _gen(seed, device)

    def normal(*shape):
        return (torch.randn(shape, generator=gen, device=device) * value_scale).to(torch.bfloat16)

    q_nope, q_pe = normal(n_tok, H, DV), normal(n_tok, H, 64)
    kv_c, k_pe = normal(n_tok, DV), normal(n_tok, 64)
    positions = torch.randint(0, max_pos, (n_tok,), generator=gen, device=device,
                              dtype=torch.int64).to(torch.int32)
    inv = rope_base ** (-np.arange(32, dtype=np.float64) / 32.0)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    table = torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32))
    return dict(q_nope=q_nope, q_pe=q_pe, kv_c=kv_c, k_pe=k_pe, positions=positions,
                cos_sin=table.to(device))


def _finish(name, q, kv, kv_lens, q_lens, indices, index_buffer, pool_rows, device,
            q_scale, kv_scale, poison, gen, meta):
    B = len(kv_lens)
    kv_indptr = torch.tensor(np.concatenate([[0], np.cumsum(kv_lens)]).astype(np.int32),
                             device=device)
    qo_indptr = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32),
                             device=device)
    total = int(sum(kv_lens))
    n_buf = max(int(index_buffer or 0), total)
    idx = torch.empty(n_buf, dtype=torch.int32, device=device)
    idx[:total] = indices
    if n_buf > total:
        if poison:
            # entries past kv_indptr[B] point outside the pool: a stray read is detectable
            idx[total:] = pool_rows + 7
        else:
            idx[total:] = torch.randint(0, pool_rows, (n_buf - total,), generator=gen,
                                        device=device, dtype=torch.int64).to(torch.int32)
    if poison:
        attended = torch.zeros(pool_rows, dtype=torch.bool, device=device)
        for b in range(B):
            T, L = q_lens[b], kv_lens[b]
            if L > 0:
                attended[idx[int(kv_indptr[b]):int(kv_indptr[b]) + L].long()] = True
        kv[~attended] = POISON_FP8
    return Case(name=name, q=q, kv=kv, qo_indptr=qo_indptr, kv_indptr=kv_indptr,
                kv_indices=idx, kv_last_page_lens=torch.ones(B, dtype=torch.int32, device=device),
                q_scale=torch.tensor(q_scale, dtype=torch.float32, device=device),
                kv_scale=torch.tensor(kv_scale, dtype=torch.float32, device=device),
                sm_scale=SM_SCALE, kv_lens=list(map(int, kv_lens)), q_lens=list(map(int, q_lens)),
                meta=meta)


def make_custom(kv_lens, q_lens=None, H: int = 12, pool_rows: Optional[int] = None,
                seed: int = 0, device="cpu", q_scale: float = DEFAULT_Q_SCALE,
                kv_scale: float = DEFAULT_KV_SCALE, poison: bool = False,
                shared_prefix: int = 0, index_buffer: int = 0, name: str = "custom") -> Case:
    """Requests with the given kv_lens / q_lens; rows drawn from a seeded permutation.

    The first ``shared_prefix`` positions of every request point at the same rows (the
    prefix-cache pattern of the captured workload); the rest are distinct per request.
    """
    kv_lens = [int(x) for x in kv_lens]
    B = len(kv_lens)
    q_lens = [1] * B if q_lens is None else [int(x) for x in q_lens]
    need = shared_prefix + sum(max(L - shared_prefix, 0) for L in kv_lens)
    if pool_rows is None:
        pool_rows = max(need, 1) + 64
    if need > pool_rows:
        raise ValueError("pool too small for the requested lengths")
    gen = _gen(seed, device)
    kv = fp8_normal_bytes(pool_rows * D, gen, device).view(pool_rows, D)
    q = fp8_normal_bytes(sum(q_lens) * H * D, gen, device).view(sum(q_lens), H, D)
    perm = torch.randperm(pool_rows, generator=gen, device=device).to(torch.int32)
    prefix = perm[:shared_prefix]
    off = shared_prefix
    parts = []
    for L in kv_lens:
        p = min(L, shared_prefix)
        u = L - p
        parts.append(prefix[:p])
        parts.append(perm[off:off + u])
        off += u
    indices = torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int32, device=device)
    return _finish(name, q, kv, kv_lens, q_lens, indices, index_buffer, pool_rows, device,
                   q_scale, kv_scale, poison, gen,
                   dict(shared_prefix=shared_prefix, pool_rows=pool_rows))


def make_paged(kv_lens, q_lens=None, H: int = 12, page_size: int = 64,
               pool_pages: Optional[int] = None, seed: int = 0, device="cpu",
               q_scale: float = DEFAULT_Q_SCALE, kv_scale: float = DEFAULT_KV_SCALE,
               poison: bool = False, shared_prefix: int = 0, index_buffer: int = 0,
               name: str = "paged") -> Case:
    """Requests over a cache of page_size-token pages (kv (pool_pages, page_size, 1, 576)).

    kv_indptr counts pages, kv_indices are page ids from a seeded permutation, and
    kv_last_page_lens[b] = the valid slots of request b's last page, so that
    kv_lens[b] = (pages_b - 1) * page_size + last_b.  The first shared_prefix tokens (a
    multiple of page_size) are the same pages in every request.  poison: every slot no
    request attends, the unused tails of last pages included, holds an e4m3 NaN.
    """
    kv_lens = [int(x) for x in kv_lens]
    B = len(kv_lens)
    q_lens = [1] * B if q_lens is None else [int(x) for x in q_lens]
    if shared_prefix % page_size:
        raise ValueError("a shared prefix of whole pages only")
    sp = shared_prefix // page_size
    counts = [(L + page_size - 1) // page_size for L in kv_lens]
    need = sp + sum(max(c - sp, 0) for c in counts)
    if pool_pages is None:
        pool_pages = max(need, 1) + 8
    if need > pool_pages:
        raise ValueError("pool too small for the requested lengths")
    gen = _gen(seed, device)
    kv = fp8_normal_bytes(pool_pages * page_size * D, gen, device).view(pool_pages, page_size, 1, D)
    q = fp8_normal_bytes(sum(q_lens) * H * D, gen, device).view(sum(q_lens), H, D)
    perm = torch.randperm(pool_pages, generator=gen, device=device).to(torch.int32)
    off = sp
    parts = []
    for c in counts:
        p = min(c, sp)
        parts.append(perm[:p])
        parts.append(perm[off:off + c - p])
        off += c - p
    pages = torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int32, device=device)
    kv_indptr = torch.tensor(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32),
                             device=device)
    qo_indptr = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32),
                             device=device)
    last = torch.tensor([L - (c - 1) * page_size if c > 0 else 1
                         for L, c in zip(kv_lens, counts)], dtype=torch.int32, device=device)
    n_buf = max(int(index_buffer or 0), int(pages.numel()))
    idx = torch.empty(max(n_buf, 1), dtype=torch.int32, device=device)
    idx[:pages.numel()] = pages
    if n_buf > pages.numel():
        idx[pages.numel():] = (pool_pages + 7) if poison else 0
    if poison:
        used = torch.zeros(pool_pages, page_size, dtype=torch.bool, device=device)
        for b in range(B):
            pg = idx[int(kv_indptr[b]):int(kv_indptr[b + 1])].long()
            if pg.numel() == 0:
                continue
            used[pg[:-1]] = True
            used[pg[-1], :int(last[b])] = True
        kv[~used] = POISON_FP8
    return Case(name=name, q=q, kv=kv, qo_indptr=qo_indptr, kv_indptr=kv_indptr,
                kv_indices=idx, kv_last_page_lens=last,
                q_scale=torch.tensor(q_scale, dtype=torch.float32, device=device),
                kv_scale=torch.tensor(kv_scale, dtype=torch.float32, device=device),
                sm_scale=SM_SCALE, kv_lens=kv_lens, q_lens=q_lens,
                meta=dict(page_size=page_size, shared_prefix=shared_prefix,
                          pool_pages=pool_pages))


def _shared_prefix_lens(B: int, seed: int):
    """kv_len = 63,911 shared + 4,089 unique + U[0, 350) generated (issue §1, §4.1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return [63911 + 4089 + int(u) for u in rng.integers(0, 350, size=B)]


def _mtp_lens(B: int, seed: int):
    """kv_len log-uniform in [2,048, 65,536] (multi-token verification workload)."""
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    u = rng.uniform(math.log(2048.0), math.log(65536.0), size=B)
    return [int(min(65536, max(2048, round(math.exp(x))))) for x in u]


# name -> (description, builder kwargs).  Sizes are the captured / stated ones.
CONFIGS = {
    "tiny": "batch 2, 12 heads, q_len 1, kv_lens {256, 300}, 1,024-row pool, "
            "kv_indices = seeded permutation of the pool",
    "c16": "batch 16, 12 heads, q_len 1, 63,911 shared-prefix + 4,089 unique + U[0,350) "
           "positions per request, 5,283,840-row pool, 4,718,592-entry index buffer",
    "c24": "batch 24, otherwise as c16",
    "long": "batch 1, 12 heads, q_len 1, kv_len 142,000, 2^18-row pool, random page order",
    "long96": "batch 1, 96 heads, q_len 1, kv_len 142,000 (the unsplit 96-head reference "
              "for the 8-shard context-parallel merge)",
    "mtp": "batch 64, 12 heads, q_len 4 (causal within the drafts), kv_len log-uniform "
           "[2,048, 65,536], 2^22-row pool",
    "c16p128": "c16's lengths on 128-token pages (the allocator's block size): 41,280-page "
               "pool (c16's 5,283,840 rows), the shared prefix's 499 whole pages shared, the "
               "rest of each request on its own pages, 36,864-entry page-index buffer",
    "longp128": "long's 142,000 positions on 128-token pages (1,110 pages, the last holding "
                "48), 2,048-page pool in random page order",
}


def make_case(name: str, seed: int = 0, device="cpu", q_scale: float = DEFAULT_Q_SCALE,
              kv_scale: float = DEFAULT_KV_SCALE, poison: bool = False) -> Case:
    """Build one of the named workloads (see CONFIGS)."""
    if name == "tiny":
        gen = _gen(seed, device)
        pool = 1024
        kv = fp8_normal_bytes(pool * D, gen, device).view(pool, D)
        q = fp8_normal_bytes(2 * 12 * D, gen, device).view(2, 12, D)
        perm = torch.randperm(pool, generator=gen, device=device).to(torch.int32)
        kv_lens = [256, 300]
        case = _finish("tiny", q, kv, kv_lens, [1, 1], perm[:556], 0, pool, device,
                       q_scale, kv_scale, poison, gen, dict(pool_rows=pool))
        # the whole permutation is the index buffer; positions >= 556 are never attended
        full = perm.clone()
        if poison:
            full[556:] = pool + 7
        case.kv_indices = full
        return case
    if name in ("c16", "c24"):
        B = 16 if name == "c16" else 24
        return make_custom(_shared_prefix_lens(B, seed), H=12, pool_rows=5_283_840,
                           seed=seed, device=device, q_scale=q_scale, kv_scale=kv_scale,
                           poison=poison, shared_prefix=63911, index_buffer=4_718_592,
                           name=name)
    if name == "long":
        return make_custom([142000], H=12, pool_rows=1 << 18, seed=seed, device=device,
                           q_scale=q_scale, kv_scale=kv_scale, poison=poison, name=name)
    if name == "long96":
        return make_custom([142000], H=96, pool_rows=1 << 18, seed=seed, device=device,
                           q_scale=q_scale, kv_scale=kv_scale, poison=poison, name=name)
    if name == "mtp":
        lens = _mtp_lens(64, seed)
        return make_custom(lens, q_lens=[4] * 64, H=12, pool_rows=1 << 22, seed=seed,
                           device=device, q_scale=q_scale, kv_scale=kv_scale, poison=poison,
                           name=name)
    if name == "c16p128":
        return make_paged(_shared_prefix_lens(16, seed), H=12, page_size=128, pool_pages=41_280,
                          seed=seed, device=device, q_scale=q_scale, kv_scale=kv_scale,
                          poison=poison, shared_prefix=63_872, index_buffer=36_864, name=name)
    if name == "longp128":
        return make_paged([142000], H=12, page_size=128, pool_pages=2048, seed=seed,
                          device=device, q_scale=q_scale, kv_scale=kv_scale, poison=poison,
                          name=name)
    raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS)}")


def shard_views(case: Case, n_shards: int):
    """Split every request's positions into n_shards contiguous blocks (context shards).

    Returns a list of (kv_indptr, kv_indices) pairs, one per shard, on case's device.
    Shard s of request b covers positions [s*L_b//n, (s+1)*L_b//n) in page order.
    """
    out = []
    dev = case.kv_indices.device
    for s in range(n_shards):
        lens, parts = [], []
        for b, L in enumerate(case.kv_lens):
            lo, hi = s * L // n_shards, (s + 1) * L // n_shards
            base = int(case.kv_indptr[b])
            parts.append(case.kv_indices[base + lo: base + hi])
            lens.append(hi - lo)
        ip = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), device=dev)
        out.append((ip, torch.cat(parts).contiguous(), lens))
    return out


# ---- accounting (bytes and flops the path must move / do; used for reporting) ----

def gathered_kv_bytes(kv_lens) -> int:
    """576 bytes of cache per attended position (the gathered-bytes convention)."""
    return D * int(sum(kv_lens))


def algorithmic_bytes(case: Case, shared_prefix: int = 0) -> int:
    """Cache rows + 4-byte indices + q in + o out (bf16) + lse out (fp32).

    With ``shared_prefix`` = P > 0 the first P positions of every request name the same
    rows, so a call that is told so needs each of those rows (and its index) once.
    """
    n_rows = int(sum(case.q_lens)) * case.H
    positions = case.total_kv - (case.B - 1) * shared_prefix if shared_prefix > 0 else case.total_kv
    if int(case.meta.get("page_size", 1)) > 1:
        # 576 B per distinct cache row (shared pages once) and 4 B per page id of every
        # request (each request names its pages, shared ones included)
        return (D * positions + 4 * int(case.kv_indptr[-1]) + n_rows * D
                + n_rows * DV * 2 + n_rows * 4)
    return (580 * positions + n_rows * D + n_rows * DV * 2 + n_rows * 4)


def useful_flops(kv_lens, q_lens, H: int) -> int:
    """2 * (576 + 512) multiply-adds per (query row, head, attended position).

    Causal drafts attend L - T + t + 1 positions.
    """
    total = 0
    for L, T in zip(kv_lens, q_lens):
        for t in range(T):
            total += max(L - T + t + 1, 0)
    return 2 * (D + DV) * H * total
