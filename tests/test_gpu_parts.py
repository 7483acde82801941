"""The receive side in G parts, each a separate allocation between poisoned
guard bands, through the C ABI: the layout+dispatch call puts each slot's row,
scales and header into its part and each count + 1 flag into its part, the
synthetic experts and combine read the parts, and combine clears every part's
flags. Checked against the oracle (dispatch bit-exact per (source rank,
token, choice) at the part and local slot the partition rule gives; combine
within 2^-7 with exact zeros) and against the single-buffer step (identical
output), for G = 1, 2, 4 and 8, on the fused kernel and on the two-kernel path, and with combine's
bulk-TMA form (16384 tokens, k = 4).
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_gb300 import _binding as B
from combine_moe_layout_gb300 import parts as PL
from combine_moe_layout_gb300 import pipeline as P
from combine_moe_layout_gb300 import workloads as wl
from gpu_common import Guarded, assert_combine_close, free_gpu, require_gpu

pytestmark = pytest.mark.gpu

CASES = {
    # fused layout+dispatch kernel, fp8 rows + scales, scaling experts
    "fused_fp8": wl.custom("parts_fp8", num_ranks=8, tokens_per_rank=128, hidden=1024, num_experts=64, topk=8,
                           max_m=128, dtype="fp8", expert="scale", x_dist="normal", renormalize=False),
    # bf16 rows quantised on dispatch
    "fused_bf16q": wl.custom("parts_bf16q", num_ranks=4, tokens_per_rank=100, hidden=512, num_experts=32, topk=4,
                             max_m=100, dtype="bf16q", expert="scale", x_dist="normal", renormalize=False),
    # 1500 tokens per rank: the cluster layout kernel, then the dispatch kernel (bf16, identity experts)
    "two_kernels_bf16": wl.custom("parts_bf16", num_ranks=4, tokens_per_rank=1500, hidden=256, num_experts=16,
                                  topk=4, max_m=1500, x_dist="normal"),
    # 16384 tokens with k = 4: combine stages its pieces with bulk TMA, reading y from the parts
    "tma_combine_fp8": wl.custom("parts_tma", num_ranks=8, tokens_per_rank=2048, hidden=256, num_experts=32, topk=4,
                                 max_m=2048, dtype="fp8", expert="scale", x_dist="normal", renormalize=False),
}
TWO_KERNELS = ("two_kernels_bf16", "tma_combine_fp8")


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()
    yield
    free_gpu()


def _run_parts(w, inp, G, dev):
    desc = B.MoeDesc.of(w)
    guards = []

    def alloc(shape, dtype):
        g = Guarded(shape, dtype, dev)
        guards.append(g)
        return g.t

    pb = B.allocate_parts(desc, G, dev, alloc=alloc)
    if pb.expert_out is None:  # identity experts: combine reads the dispatched rows themselves
        pb.expert_out = [r.view(torch.bfloat16) for r in pb.recv_x]
    d = P.to_device(inp, dev)
    R, T, k, H = w.num_ranks, w.tokens_per_rank, w.topk, w.hidden
    counts = torch.zeros((w.num_experts, R), dtype=torch.int32, device=dev)
    tok_slot = torch.empty((R, T, k), dtype=torch.int32, device=dev)
    out = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    B.moe_reset_parts(desc, pb, err)
    B.moe_layout_dispatch_parts(desc, d.topk_idx, d.x, d.x_scales, counts, tok_slot, pb, err)
    flags = [f.clone() for f in pb.flags]
    if w.dtype != "bf16":
        B.moe_expert_stub_parts(desc, pb, counts, err)
    B.moe_combine_parts(desc, pb, d.topk_weights, tok_slot, out, err)
    status = B.moe_get_error(err)
    return pb, guards, counts, tok_slot, flags, out, status


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("name", list(CASES))
def test_parts_match_the_oracle_and_the_single_buffer(name, G):
    w = CASES[name]
    if w.num_ranks % G:
        pytest.skip("the parts must divide the ranks")
    dev = torch.device("cuda:0")
    inp = wl.make_inputs(w, seed=11)
    ref = oracle.run(w, inp)
    pb, guards, counts, tok_slot, flags, out, status = _run_parts(w, inp, G, dev)
    assert status == B.MOE_OK, B.moe_status_string(status)
    assert B.moe_layout_dispatch_kernels(B.MoeDesc.of(w)) == (2 if name in TWO_KERNELS else 1)

    assert np.array_equal(counts.cpu().numpy(), ref.counts)
    ts = tok_slot.cpu().numpy()
    assert np.array_equal(ts, ref.tok_slot)
    per_regions = w.num_experts * w.num_ranks // G
    for g in range(G):
        want = ref.flags.reshape(-1)[g * per_regions:(g + 1) * per_regions]
        assert np.array_equal(flags[g].cpu().numpy().astype(np.uint64), want), f"flags of part {g}"
        assert not pb.flags[g].any().item(), "combine clears every part's flags"

    # every (source rank, token, choice) in the part and at the local slot the partition rule gives
    Pn = PL.slots_per_part(w.num_ranks, w.num_experts, w.max_m, G)
    part, local = PL.part_of_slot(ref.slots.slot_id, Pn)
    rows = np.empty_like(ref.slots.rows)
    meta = np.empty_like(ref.slots.meta)
    sc = np.empty_like(ref.slots.scales)
    for g in range(G):
        sel = np.nonzero(part == g)[0]
        idx = torch.from_numpy(local[sel]).to(dev)
        rows[sel] = pb.recv_x[g].index_select(0, idx).cpu().numpy()
        meta[sel] = pb.recv_meta[g].index_select(0, idx).cpu().numpy()
        if pb.recv_scales is not None:
            sc[sel] = pb.recv_scales[g].index_select(0, idx).cpu().numpy()
    assert np.array_equal(rows, ref.slots.rows)
    assert np.array_equal(meta, ref.slots.meta)
    if pb.recv_scales is not None:
        assert np.array_equal(sc.view(np.uint32), ref.slots.scales.view(np.uint32))

    got = out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(w.num_tokens, w.hidden)
    assert_combine_close(got, ref.out)
    assert all(g.guards_intact() for g in guards), "a write left its part"

    # the same step on the single buffer gives the same bits
    step = P.MoeStep(w, dev)
    step.reset()
    step.run(P.to_device(inp, dev), fused=True)
    assert step.error() == B.MOE_OK
    assert torch.equal(step.buf.out.view(torch.int16), out.view(torch.int16))


def test_invalid_part_tables_are_rejected():
    w = CASES["fused_fp8"]
    dev = torch.device("cuda:0")
    desc = B.MoeDesc.of(w)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pb = B.allocate_parts(desc, 2, dev)
    t = pb.table()
    for bad in (0, 3, B.MOE_MAX_PARTS + 1):  # 3 does not divide 8 ranks
        t.num_parts = bad
        st = B.load().moe_reset_parts(B.ctypes.byref(desc), B.ctypes.byref(t), B._ptr(err), B._stream(None))
        assert st == B.MOE_EINVAL
    t.num_parts = 2
    t.flags[1] = None
    st = B.load().moe_reset_parts(B.ctypes.byref(desc), B.ctypes.byref(t), B._ptr(err), B._stream(None))
    assert st == B.MOE_EINVAL
