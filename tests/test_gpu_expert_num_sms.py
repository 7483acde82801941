"""The expert stage with the SM count limited (moe_desc.num_sms): each persistent
CTA (or CTA pair) then walks many tiles, and the pair kernel gets fewer clusters
than SMs. A tile's result does not depend on which CTA computes it, so h and y
must be bit-identical to the run on all SMs."""
from __future__ import annotations

import pytest
import torch

from combine_moe_layout_gb300 import _binding as B
from combine_moe_layout_gb300 import pipeline as P
from combine_moe_layout_gb300 import workloads as wl
from gpu_common import free_gpu, require_gpu

pytestmark = pytest.mark.gpu

CASES = {
    # bf16, 1200 rows per expert: linear 2 takes the CTA-pair kernel
    "bf16_pair": wl.custom("sms_bf16_pair", num_ranks=4, tokens_per_rank=600, hidden=256, num_experts=4, topk=2,
                           max_m=600, x_dist="normal", intermediate=384),
    # bf16, Zipf routing: hot and cold experts, the one-CTA kernel for both linears
    "bf16_zipf": wl.custom("sms_bf16_zipf", num_ranks=4, tokens_per_rank=128, hidden=384, num_experts=32, topk=4,
                           max_m=128, router="zipf", x_dist="normal", intermediate=256),
    # fp8, 200 rows per expert: the staged form
    "fp8_staged": wl.custom("sms_fp8_staged", num_ranks=4, tokens_per_rank=200, hidden=256, num_experts=8, topk=2,
                            max_m=200, dtype="fp8", expert="scale", x_dist="normal", intermediate=384),
    # fp8, 64 rows per expert: the weight-streaming form
    "fp8_streaming": wl.custom("sms_fp8_stream", num_ranks=4, tokens_per_rank=128, hidden=384, num_experts=32,
                               topk=4, max_m=128, dtype="fp8", expert="scale", x_dist="normal", intermediate=256),
}


def _stage(w, num_sms, inp):
    step = P.MoeStep(w, "cuda:0", num_sms)
    d = P.to_device(inp, "cuda:0")
    step.reset()
    step.layout(d)
    step.dispatch(d)
    packed = B.allocate_packed(step.desc, "cuda:0")
    step.recv(packed)
    rows, H, I = w.num_tokens * w.topk, w.hidden, w.intermediate
    y = torch.zeros((rows, H), dtype=torch.bfloat16, device="cuda:0")
    if w.dtype == "fp8":
        wts = wl.expert_weights_fp8(w, "cuda:0")
        h = torch.zeros((rows, I), dtype=torch.uint8, device="cuda:0")
        hs = torch.zeros((rows, I // 128), dtype=torch.float32, device="cuda:0")
        step.expert_mlp_fp8(wts, packed, h, hs, y)
        out = (h, hs, y)
    else:
        wts = wl.expert_weights(w, "cuda:0")
        h = torch.zeros((rows, I), dtype=torch.bfloat16, device="cuda:0")
        step.expert_mlp(wts, packed, h, y)
        out = (h, y)
    assert step.error() == B.MOE_OK
    n = int(packed.region_offsets[-1].item())
    return [t[:n].clone() for t in out]


@pytest.mark.parametrize("name", list(CASES))
def test_expert_stage_is_independent_of_the_sm_count(name):
    require_gpu()
    w = CASES[name]
    inp = wl.make_inputs(w)
    want = _stage(w, 0, inp)
    for sms in (1, 3, 8):
        got = _stage(w, sms, inp)
        for a, b in zip(got, want):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (name, sms)
    free_gpu()
