"""A seeded sweep of random call shapes against the oracle: batch sizes, head counts whose
rows fill 16-, 32- and 48-row groups to different depths, draft counts, ragged and tiny
histories, pages of 1 to 128 tokens, the split policies, sharp and flat softmax scales and
both entry points.  Each shape draws its own lengths, so the causal cut, the padding rows,
the last partial tile and the piece boundaries land at many alignments that the targeted
tests do not pick.  Tolerances are the suite's (tests/gpu_util.py)."""
import random

import pytest

import mla_inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

N_CASES = 120


def _shape(i):
    r = random.Random(1000 + i)
    H = r.choice([8, 12, 16, 20, 24, 40, 48, 96])
    T = r.choice([1, 1, 1, 2, 3, 4])
    B = r.randint(1, 9)
    page = r.choice([1, 1, 1, 2, 16, 128])
    lens = []
    for _ in range(B):
        kind = r.random()
        if kind < 0.15:
            L = T                            # exactly the drafts
        elif kind < 0.35:
            L = r.randint(T, 40)             # shorter than one tile
        elif kind < 0.85:
            L = r.randint(100, 2500)
        else:
            L = r.randint(3000, 9000)        # several pieces under the automatic split
        lens.append(max(L, T))
    splits = r.choice([0, 0, 0, 1, 3])
    sharp = r.random() < 0.5
    shared = 0
    if i % 4 == 3:
        # the shared-prefix entry: one-token pages, q_len 1, and at least one full group of
        # 48 rows, the prefix below every length
        H, T, page, splits = r.choice([8, 12, 16, 20, 24]), 1, 1, 0
        B = max(B, 48 // H + r.randint(0, 3))
        shared = r.choice([1024, 1100, 2500])   # at least the cascade's 1,024-position minimum
        lens = [max(L, shared + r.randint(1, 400)) for L in lens]
        lens += [shared + r.randint(1, 3000) for _ in range(B - len(lens))]
    return dict(H=H, T=T, lens=lens, page=page, splits=splits, sharp=sharp, shared=shared,
                seed=2000 + i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_matches_oracle(i):
    s = _shape(i)
    scales = dict(q_scale=1.0, kv_scale=1.0) if s["sharp"] else {}
    q_lens = [s["T"]] * len(s["lens"])
    if s["page"] == 1:
        case = mla_inputs.make_custom(s["lens"], q_lens=q_lens, H=s["H"], seed=s["seed"],
                                      shared_prefix=s["shared"], name=f"sweep{i}", **scales)
    else:
        case = mla_inputs.make_paged(s["lens"], q_lens=q_lens, H=s["H"], page_size=s["page"],
                                     seed=s["seed"], poison=True, name=f"sweep{i}", **scales)
    case = gu.to_device(case)
    kw = dict(num_kv_splits=s["splits"])
    if s["shared"]:
        kw = dict(shared_prefix=s["shared"])
    o, lse, status = gu.run_gpu(case, **kw)
    assert status == 0, f"device error {status} for {s}"
    o_ref, lse_ref = gu.run_oracle(case)
    gu.compare(o, lse, o_ref, lse_ref, what=f"{case.name} {s}")
