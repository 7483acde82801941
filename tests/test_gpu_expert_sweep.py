"""A seeded sweep of random expert-stage shapes, bf16 and fp8, against the oracle.

Each case draws ranks, tokens, experts, top-k, hidden size H and expert width I
(multiples of 128), and the router (softmax, or Zipf with hot and empty experts).
The packed rows per expert then range from a few, where the fp8 kernel streams its
weights with direct stores, past one 128-row tile, where it stages its output, to
several hundred, where the bf16 linear 2 takes the CTA-pair kernel. Rows are
checked within the bars of the fixed-shape expert tests: every third packed row
and the first and last row of every expert.
"""
from __future__ import annotations

import numpy as np
import pytest

from combine_moe_layout_gb300 import workloads as wl
from gpu_common import free_gpu, require_gpu
from test_gpu_expert import check_expert_stage
from test_gpu_expert_fp8 import check_fp8_stage

pytestmark = pytest.mark.gpu


def _cases(dtype: str, n: int, seed: int):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        R = int(rng.choice([1, 2, 4]))
        E = R * int(rng.integers(1, 9))
        k = int(rng.integers(1, min(E, 4) + 1))
        T = int(rng.choice([8, 40, 128, 300, 600]))
        if R * T * k > 3000:
            continue
        case = dict(num_ranks=R, tokens_per_rank=T, hidden=128 * int(rng.integers(1, 6)), num_experts=E, topk=k,
                    max_m=T, router=str(rng.choice(["softmax", "zipf"])), x_dist="normal",
                    intermediate=128 * int(rng.integers(1, 4)))
        if dtype == "fp8":
            case.update(dtype="fp8", expert="scale")
        out.append((f"{dtype}_{len(out)}", case))
    return out


def _rows(n: int, off: np.ndarray, E: int, R: int) -> list:
    """Every third packed row and the first and last row of each expert."""
    ends = {int(off[e * R]) for e in range(E)} | {int(off[(e + 1) * R]) - 1 for e in range(E)}
    return sorted(set(range(0, n, 3)) | {p for p in ends if 0 <= p < n})


# plus two shapes of >= 512 rows per expert, where the bf16 linear 2 takes the CTA-pair kernel
BF16 = _cases("bf16", 12, 31) + [
    ("bf16_pair_a", dict(num_ranks=2, tokens_per_rank=600, hidden=384, num_experts=2, topk=2, max_m=600,
                         x_dist="normal", intermediate=256)),
    ("bf16_pair_b", dict(num_ranks=1, tokens_per_rank=600, hidden=256, num_experts=2, topk=2, max_m=600,
                         router="zipf", x_dist="normal", intermediate=384)),
]
FP8 = _cases("fp8", 12, 32)


@pytest.mark.parametrize("name,case", BF16, ids=[c[0] for c in BF16])
def test_bf16_expert_shape_matches_the_oracle(name, case):
    require_gpu()
    w = wl.custom(name, **case)
    check_expert_stage(w)
    free_gpu()


@pytest.mark.parametrize("name,case", FP8, ids=[c[0] for c in FP8])
def test_fp8_expert_shape_matches_the_oracle(name, case):
    require_gpu()
    w = wl.custom(name, **case)
    check_fp8_stage(w, lambda n, off: _rows(n, off, w.num_experts, w.num_ranks))
    free_gpu()
