"""The C-ABI calls inside a captured CUDA graph: they allocate nothing and launch on
the caller's stream, so a step captured once replays on new inputs copied into the
captured input buffers.

- The dispatch -> experts -> combine step (separate and fused layout+dispatch) on
  the DeepSeek decode shape, replayed on three new input sets, each checked against
  the oracle.
- The whole MoE step with the fp8 expert stage (layout+dispatch, receive hook,
  linear 1 + SwiGLU + quantise h, linear 2, packed combine), replayed on new inputs
  and checked bit for bit against the same calls made eagerly on those inputs.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_gb300 import _binding as B
from combine_moe_layout_gb300 import pipeline as P
from combine_moe_layout_gb300 import workloads as wl
from gpu_common import assert_combine_close, free_gpu, require_gpu

pytestmark = pytest.mark.gpu


def _load(d: P.DeviceInputs, inp: wl.Inputs):
    """Copy a new input set into the captured device input buffers."""
    d.topk_idx.copy_(torch.from_numpy(inp.topk_idx))
    d.topk_weights.copy_(torch.from_numpy(inp.topk_weights))
    d.x.copy_(torch.from_numpy(inp.x).view(d.x.dtype))
    if d.x_scales is not None:
        d.x_scales.copy_(torch.from_numpy(inp.x_scales))


@pytest.mark.parametrize("fused", [False, True], ids=["separate", "fused"])
def test_step_replays_from_a_cuda_graph(fused):
    require_gpu()
    w = wl.WORKLOADS["ds_decode"]
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(wl.make_inputs(w, seed=1), "cuda:0")
    step.reset()
    step.run(d, fused=fused)  # eager once (kernel attributes set before capture)
    torch.cuda.synchronize()
    assert step.error() == B.MOE_OK
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step.run(d, fused=fused)
    for seed in (11, 12, 13):
        inp = wl.make_inputs(w, seed=seed)
        ref = oracle.run(w, inp)
        _load(d, inp)
        step.buf.out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert step.error() == B.MOE_OK
        assert np.array_equal(step.buf.tok_slot.cpu().numpy(), ref.tok_slot)
        out = step.buf.out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert_combine_close(out.ravel(), ref.out.ravel())
    free_gpu()


def test_fp8_moe_step_with_experts_replays_from_a_cuda_graph():
    require_gpu()
    w = wl.custom("graph_fp8", num_ranks=4, tokens_per_rank=200, hidden=256, num_experts=8, topk=2, max_m=200,
                  dtype="fp8", expert="scale", x_dist="normal", intermediate=384)
    rows, H, I = w.num_tokens * w.topk, w.hidden, w.intermediate
    step = P.MoeStep(w, "cuda:0")
    packed = B.allocate_packed(step.desc, "cuda:0")
    wts = wl.expert_weights_fp8(w, "cuda:0")
    h = torch.empty((rows, I), dtype=torch.uint8, device="cuda:0")
    hs = torch.empty((rows, I // 128), dtype=torch.float32, device="cuda:0")
    y = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda:0")
    d = P.to_device(wl.make_inputs(w, seed=1), "cuda:0")

    def moe_step():
        step.layout_dispatch(d)
        step.recv(packed)
        step.expert_mlp_fp8(wts, packed, h, hs, y)
        step.combine_packed(d, y, packed)

    step.reset()
    moe_step()  # eager once
    torch.cuda.synchronize()
    assert step.error() == B.MOE_OK
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        moe_step()
    for seed in (21, 22):
        inp = wl.make_inputs(w, seed=seed)
        _load(d, inp)
        moe_step()  # eager on the new inputs
        torch.cuda.synchronize()
        assert step.error() == B.MOE_OK
        want_out, want_h = step.buf.out.clone(), h.clone()
        ref = oracle.run(w, inp, sel=np.zeros(0, np.int64))   # layout only
        assert np.array_equal(packed.region_offsets.cpu().numpy(), oracle.region_offsets(ref.counts, w.max_m))
        step.buf.out.fill_(float("nan"))
        h.fill_(0x7F)
        graph.replay()
        torch.cuda.synchronize()
        assert step.error() == B.MOE_OK
        assert torch.equal(h, want_h)
        assert torch.equal(step.buf.out.view(torch.int16), want_out.view(torch.int16))
    free_gpu()
