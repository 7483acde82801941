"""Layers chained on one stream: each layer's x is the previous layer's combine
output, written by the kernel immediately before that layer's dispatch.

Under programmatic dependent launch the dispatch of layer l + 1 may be
scheduled while the combine of layer l is still running (combine lets its
dependents launch early for decode-sized batches). Every kernel reads its
inputs only after its dependency wait, so each layer must still see the
finished output of the one before. Each layer is checked against the oracle
run on that layer's own input (the GPU output of the previous layer, itself
checked), with no host synchronisation between the layers.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_gb300 import _binding as B
from combine_moe_layout_gb300 import pipeline as P
from combine_moe_layout_gb300 import workloads as wl
from gpu_common import assert_combine_close, free_gpu, require_gpu

pytestmark = pytest.mark.gpu

LAYERS = 6

# 1024 tokens: at most the early-trigger batch size, so each combine lets the
# next layer's first kernel launch before it has finished. Weights are the raw
# top-k softmax probabilities (not renormalised), so each layer changes x.
CHAINS = {
    "bf16": wl.custom("chain_bf16", num_ranks=8, tokens_per_rank=128, hidden=1024, num_experts=64, topk=4,
                      max_m=128, dtype="bf16", renormalize=False, x_dist="normal"),
    "bf16q": wl.custom("chain_bf16q", num_ranks=8, tokens_per_rank=128, hidden=1024, num_experts=64, topk=4,
                       max_m=128, dtype="bf16q", renormalize=False, expert="scale", x_dist="normal"),
}


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()
    yield
    free_gpu()


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "separate"])
@pytest.mark.parametrize("name", list(CHAINS))
def test_layers_chained_through_combine_output(name, fused):
    w = CHAINS[name]
    dev = torch.device("cuda:0")
    if fused:
        assert B.moe_layout_dispatch_kernels(B.MoeDesc.of(w)) == 1
    step = P.MoeStep(w, dev)
    R, T, H, k = w.num_ranks, w.tokens_per_rank, w.hidden, w.topk
    # every layer's routing and output buffer exist before the first launch, so
    # the layers' kernels follow each other with nothing in between
    routes = [wl.make_inputs(w, seed=100 + layer) for layer in range(LAYERS)]
    idx = [torch.from_numpy(r.topk_idx).to(dev) for r in routes]
    wts = [torch.from_numpy(r.topk_weights).to(dev) for r in routes]
    x0 = torch.from_numpy(routes[0].x.view(np.int16)).to(dev).view(torch.bfloat16)
    outs = [torch.empty(R, T, H, dtype=torch.bfloat16, device=dev) for _ in range(LAYERS)]
    step.reset()
    torch.cuda.synchronize()

    x = x0
    for layer in range(LAYERS):
        d = P.DeviceInputs(idx[layer], wts[layer], x, None)
        if fused:
            step.layout_dispatch(d)
        else:
            step.layout(d)
            step.dispatch(d)
        step.experts()
        step.combine(d, out=outs[layer])
        x = outs[layer]
    assert step.error() == B.MOE_OK

    prev = routes[0].x
    for layer in range(LAYERS):
        inp = wl.Inputs(routes[layer].topk_idx, routes[layer].topk_weights, prev, None)
        ref = oracle.run(w, inp)
        got = outs[layer].view(torch.int16).cpu().numpy().view(np.uint16).reshape(w.num_tokens, H)
        assert_combine_close(got, ref.out)
        prev = got.reshape(R, T, H)
