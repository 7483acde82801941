"""The allocation-free expert stage (moe_expert_mlp_noalloc and its fp8 form) against the two-call
stage with a caller buffer for h: bit-identical outputs on two calls in a row,
and the size limit of its fixed scratch array."""
from __future__ import annotations

import pytest
import torch

from combine_moe_layout_gb300 import _binding as B
from combine_moe_layout_gb300 import pipeline as P
from combine_moe_layout_gb300 import workloads as wl
from gpu_common import free_gpu, require_gpu

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": wl.custom("noalloc_ragged", num_ranks=4, tokens_per_rank=200, hidden=256, num_experts=8, topk=2,
                        max_m=200, intermediate=384),
    "tiny": wl.WORKLOADS["tiny"],
}


def _packed(w):
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(wl.make_inputs(w), "cuda:0")
    step.reset()
    step.layout(d)
    step.dispatch(d)
    packed = B.allocate_packed(step.desc, "cuda:0")
    step.recv(packed)
    assert step.error() == B.MOE_OK
    return step, packed


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_the_two_call_stage_twice(name):
    require_gpu()
    w = CASES[name]
    step, packed = _packed(w)
    rows, H, I = w.num_tokens * w.topk, w.hidden, w.intermediate
    wts = wl.expert_weights(w, "cuda:0")
    h = torch.empty((rows, I), dtype=torch.bfloat16, device="cuda:0")
    y_ref = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda:0")
    step.expert_mlp(wts, packed, h, y_ref)
    assert step.error() == B.MOE_OK
    for _ in range(2):
        y = torch.full((rows, H), float("nan"), dtype=torch.bfloat16, device="cuda:0")
        B.moe_expert_mlp_noalloc(step.desc, I, packed.region_offsets, packed.packed_x, wts.w_gate, wts.w_up,
                                 wts.w_down, y, step.buf.err)
        assert step.error() == B.MOE_OK
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    free_gpu()


def test_noalloc_replays_from_a_cuda_graph():
    """Captured once into a CUDA graph (no allocation happens inside the capture)
    and replayed twice: bit-identical to the two-call stage each time."""
    require_gpu()
    w = CASES["ragged"]
    step, packed = _packed(w)
    rows, H, I = w.num_tokens * w.topk, w.hidden, w.intermediate
    wts = wl.expert_weights(w, "cuda:0")
    h = torch.empty((rows, I), dtype=torch.bfloat16, device="cuda:0")
    y_ref = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda:0")
    step.expert_mlp(wts, packed, h, y_ref)
    assert step.error() == B.MOE_OK
    y = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda:0")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        B.moe_expert_mlp_noalloc(step.desc, I, packed.region_offsets, packed.packed_x, wts.w_gate, wts.w_up,
                                 wts.w_down, y, step.buf.err)
    for _ in range(2):
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert step.error() == B.MOE_OK
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    free_gpu()


def test_noalloc_rejects_a_stage_above_its_scratch():
    """The Mixtral shape needs 1.9 GB for h, above the 32 MiB array: MOE_ENOMEM, nothing launched."""
    require_gpu()
    w = wl.WORKLOADS["mixtral"]
    desc = B.MoeDesc.of(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    off = torch.zeros(w.num_experts * w.num_ranks + 1, dtype=torch.int32, device="cuda:0")
    with pytest.raises(B.MoeError) as e:
        B.moe_expert_mlp_noalloc(desc, w.intermediate, off, None, None, None, None, None, err)
    assert e.value.status == B.MOE_ENOMEM
    assert int(err.item()) == 0


FP8_CASES = {
    # 200 rows per expert (the staged form of the fp8 kernel)
    "ragged": wl.custom("noalloc_fp8_ragged", num_ranks=4, tokens_per_rank=200, hidden=256, num_experts=8, topk=2,
                        max_m=200, dtype="fp8", expert="scale", x_dist="normal", intermediate=384),
    # 8 rows per expert (the weight-streaming form)
    "tiny": wl.custom("noalloc_fp8_tiny", num_ranks=2, tokens_per_rank=16, hidden=128, num_experts=8, topk=2,
                      max_m=16, dtype="fp8", expert="scale", x_dist="normal", intermediate=256),
}


def _fp8_reference(w):
    step, packed = _packed(w)
    rows, H, I = w.num_tokens * w.topk, w.hidden, w.intermediate
    wts = wl.expert_weights_fp8(w, "cuda:0")
    h = torch.empty((rows, I), dtype=torch.uint8, device="cuda:0")
    hs = torch.empty((rows, I // 128), dtype=torch.float32, device="cuda:0")
    y_ref = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda:0")
    step.expert_mlp_fp8(wts, packed, h, hs, y_ref)
    assert step.error() == B.MOE_OK
    return step, packed, wts, y_ref


def _noalloc_fp8(step, packed, wts, w, y):
    B.moe_expert_mlp_noalloc_fp8(step.desc, w.intermediate, packed.region_offsets, packed.packed_x,
                                 packed.packed_scales, wts.w_gate, wts.w_gate_scales, wts.w_up, wts.w_up_scales,
                                 wts.w_down, wts.w_down_scales, y, step.buf.err)


@pytest.mark.parametrize("name", list(FP8_CASES))
def test_noalloc_fp8_matches_the_two_call_stage_twice(name):
    require_gpu()
    w = FP8_CASES[name]
    step, packed, wts, y_ref = _fp8_reference(w)
    for _ in range(2):
        y = torch.full_like(y_ref, float("nan"))
        _noalloc_fp8(step, packed, wts, w, y)
        assert step.error() == B.MOE_OK
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    free_gpu()


def test_noalloc_fp8_replays_from_a_cuda_graph():
    require_gpu()
    w = FP8_CASES["ragged"]
    step, packed, wts, y_ref = _fp8_reference(w)
    y = torch.empty_like(y_ref)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        _noalloc_fp8(step, packed, wts, w, y)
    for _ in range(2):
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert step.error() == B.MOE_OK
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    free_gpu()


def test_noalloc_fp8_rejects_a_stage_above_its_scratch():
    """The DeepSeek prefill shape needs 512 MiB of e4m3 h: MOE_ENOMEM, nothing launched."""
    require_gpu()
    w = wl.WORKLOADS["ds_prefill"]
    desc = B.MoeDesc.of(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    off = torch.zeros(w.num_experts * w.num_ranks + 1, dtype=torch.int32, device="cuda:0")
    with pytest.raises(B.MoeError) as e:
        B.moe_expert_mlp_noalloc_fp8(desc, w.intermediate, off, None, None, None, None, None, None, None, None, None,
                                     err)
    assert e.value.status == B.MOE_ENOMEM
    assert int(err.item()) == 0
