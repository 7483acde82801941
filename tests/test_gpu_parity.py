"""GPU path vs the CPU oracle, through the C ABI.

Dispatch must agree bit-exactly (slot contents, scales, counts, headers),
compared per (source rank, token); combine within 2^-7 relative per element,
with exact zeros. Every config is compared in full, the large ones (32768
tokens) in chunks of tokens, and also through properties that hold at any size
(identity experts return the input; scaling experts follow their closed form).
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_gb300 import _binding as B
from combine_moe_layout_gb300 import pipeline as P
from combine_moe_layout_gb300 import workloads as wl
from gpu_common import (TOL, assert_combine_close, check_dispatch, check_layout, check_region_sets,
                        check_touched_slots_gpu, free_gpu, gather_slots, require_gpu, run_step)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()
    yield
    free_gpu()


def _full_parity(w, inp, num_sms=0, region_sets=True, fused=False):
    ref = oracle.run(w, inp)
    step, d, flags, err, _ = run_step(w, inp, num_sms=num_sms, fused=fused)
    assert err == B.MOE_OK, B.moe_status_string(err)
    ts = check_layout(step, flags, ref, w)
    check_dispatch(step, w, ts, ref)
    if region_sets:
        check_region_sets(step, w, ts, ref)
    else:
        check_touched_slots_gpu(step, w, ref.counts)
    out = step.buf.out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(w.num_tokens, w.hidden)
    assert_combine_close(out, ref.out)
    assert not step.buf.flags.any().item(), "combine must clear the count+1 flags"
    return step, d, ref, out


FUSED = [False, True]
FUSED_IDS = ["separate", "fused"]


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
def test_tiny(fused):
    w = wl.WORKLOADS["tiny"]
    inp = wl.make_inputs(w)
    step, d, ref, out = _full_parity(w, inp, fused=fused)
    # identity experts, renormalised weights: combine returns the input
    assert np.array_equal(out, inp.x.reshape(w.num_tokens, w.hidden))


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
def test_ds_decode(fused):
    w = wl.WORKLOADS["ds_decode"]
    if fused:
        assert B.moe_layout_dispatch_kernels(B.MoeDesc.of(w)) == 1
    _full_parity(w, wl.make_inputs(w), region_sets=False, fused=fused)


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
def test_skewed(fused):
    w = wl.WORKLOADS["skewed"]
    inp = wl.make_inputs(w)
    step, d, ref, out = _full_parity(w, inp, region_sets=False, fused=fused)
    assert np.array_equal(out, inp.x.reshape(w.num_tokens, w.hidden))
    # the hot expert fills nearly all of rank 0's slots for it
    assert ref.counts[0].max() > 0.9 * w.tokens_per_rank


def _large_parity(w, chunk_tokens, fused=False):
    """Every token of a large config against the oracle, in chunks of tokens: full
    layout; every (source rank, token, choice)'s row, scales and header at the
    GPU's slot; every combine row."""
    inp = wl.make_inputs(w)
    counts, flags, tok_slot = oracle.layout(inp.topk_idx, w.num_experts, w.max_m)
    dt = w.dtype_code
    step, d, fl, err, _ = run_step(w, inp, fused=fused)
    assert err == B.MOE_OK, B.moe_status_string(err)
    out_t = step.buf.out.view(w.num_tokens, w.hidden)
    ts = None
    for t0 in range(0, w.num_tokens, chunk_tokens):
        sel = np.arange(t0, min(w.num_tokens, t0 + chunk_tokens), dtype=np.int64)
        slots = oracle.dispatch(inp.x, inp.x_scales, tok_slot, w.num_experts, w.max_m, dt, sel)
        y = oracle.expert_stub(slots, w.num_ranks, w.hidden, w.num_experts, w.max_m, dt)
        out_ref = oracle.combine(tok_slot, inp.topk_weights, slots.slot_id, y, w.num_experts, w.max_m, sel)
        ref = oracle.OracleResult(counts, flags, tok_slot, slots, y, out_ref, sel)
        if ts is None:
            ts = check_layout(step, fl, ref, w)
        check_dispatch(step, w, ts, ref)
        got = out_t[t0:t0 + sel.size].view(torch.int16).cpu().numpy().view(np.uint16)
        assert_combine_close(got, out_ref)
        del slots, y, out_ref, ref
    check_touched_slots_gpu(step, w, counts)
    return step, d, inp


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
def test_mixtral(fused):
    w = wl.WORKLOADS["mixtral"]
    if fused:  # 4096 tokens per rank: the fused call runs the two kernels
        assert B.moe_layout_dispatch_kernels(B.MoeDesc.of(w)) == 2
    step, d, inp = _large_parity(w, 4096, fused=fused)
    # every token: identity experts with renormalised weights give back x exactly
    assert torch.equal(step.buf.out.view(torch.int16), d.x.view(torch.int16))


def _scaled_closed_form_all_tokens(step, d, w, chunk=2048):
    """out ~= x_deq * sum_j w_j (1 + e_j/256) within 2^-7 for every token (on the device)."""
    out = step.buf.out.view(w.num_tokens, w.hidden)
    x = d.x.view(w.num_tokens, w.hidden)
    sc = d.x_scales.view(w.num_tokens, -1)
    c = (d.topk_weights.double() * (1 + d.topk_idx.double() / 256)).sum(-1).view(-1)
    for t0 in range(0, w.num_tokens, chunk):
        t1 = min(w.num_tokens, t0 + chunk)
        deq = x[t0:t1].view(torch.float8_e4m3fn).float().double() * sc[t0:t1].double().repeat_interleave(128, dim=1)
        ref = deq * c[t0:t1, None]
        got = out[t0:t1].double()
        assert bool(((got - ref).abs() <= TOL * ref.abs()).all())
        assert bool((got[ref == 0] == 0).all())


def test_ds_decode_closed_form():
    w = wl.WORKLOADS["ds_decode"]
    inp = wl.make_inputs(w)
    step, d, flags, err, _ = run_step(w, inp)
    assert err == B.MOE_OK
    _scaled_closed_form_all_tokens(step, d, w)


def test_ds_prefill():
    w = wl.WORKLOADS["ds_prefill"]
    free = torch.cuda.mem_get_info()[0]
    need = sum(B.moe_buffer_sizes(B.MoeDesc.of(w)).values()) + (2 << 30)
    assert free > need, f"ds_prefill needs {need / 2**30:.1f} GiB of device memory, {free / 2**30:.1f} free"
    step, d, inp = _large_parity(w, 2048)
    _scaled_closed_form_all_tokens(step, d, w)
    # group-limited routing: each token reaches at most 4 logical ranks
    ranks = (d.topk_idx.long() // w.local_experts)
    per_tok = torch.stack([(ranks == r).any(-1) for r in range(w.num_ranks)], -1).sum(-1)
    assert int(per_tok.max()) <= 4


# --- edge cases ------------------------------------------------------------------

EDGE = {
    "minimal": dict(num_ranks=1, tokens_per_rank=1, hidden=8, num_experts=1, topk=1, max_m=1),
    "ragged_chunks_k3": dict(num_ranks=3, tokens_per_rank=300, hidden=256, num_experts=12, topk=3, max_m=300),
    "k16_fp8_one_scale": dict(num_ranks=2, tokens_per_rank=130, hidden=128, num_experts=32, topk=16, max_m=200,
                              dtype="fp8", expert="scale", x_dist="normal"),
    "two_pieces_per_row": dict(num_ranks=4, tokens_per_rank=64, hidden=16384, num_experts=8, topk=2, max_m=64,
                               x_dist="normal"),
    "decode_plus_one": dict(num_ranks=8, tokens_per_rank=129, hidden=7168, num_experts=256, topk=8, max_m=129,
                            dtype="fp8", expert="scale", x_dist="normal", renormalize=False),
    "slots_exceed_tokens": dict(num_ranks=2, tokens_per_rank=20, hidden=64, num_experts=4, topk=4, max_m=33),
    "k6_bf16": dict(num_ranks=4, tokens_per_rank=77, hidden=1024, num_experts=16, topk=6, max_m=80),
    # layout on a cluster of 3 CTAs per rank, the last slice ragged
    "cluster3_ragged": dict(num_ranks=2, tokens_per_rank=1500, hidden=64, num_experts=32, topk=4, max_m=1500),
    # 16384 tokens and k >= 4: combine stages its pieces with bulk TMA; hidden 256 leaves a partial chunk
    "tma_combine_k6_bf16": dict(num_ranks=4, tokens_per_rank=4096, hidden=256, num_experts=16, topk=6,
                                max_m=4096, x_dist="normal"),
    "tma_combine_k4_fp8": dict(num_ranks=8, tokens_per_rank=2048, hidden=1024, num_experts=32, topk=4,
                               max_m=2048, dtype="fp8", expert="scale", x_dist="normal", renormalize=False),
    # bf16 rows quantised to fp8 on dispatch: rows of two 16 KiB pieces, and one scale per row with k = 16
    "quant_two_pieces": dict(num_ranks=2, tokens_per_rank=40, hidden=16384, num_experts=8, topk=2, max_m=40,
                             dtype="bf16q", expert="scale", x_dist="normal"),
    "quant_k16_one_scale": dict(num_ranks=2, tokens_per_rank=130, hidden=128, num_experts=32, topk=16, max_m=200,
                                dtype="bf16q", expert="scale", x_dist="normal"),
    # 4096 experts: the cluster's bitmaps do not fit, the chunked layout kernel runs
    "many_experts_chunked": dict(num_ranks=1, tokens_per_rank=1024, hidden=64, num_experts=4096, topk=2,
                                 max_m=1024),
}


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
@pytest.mark.parametrize("name", list(EDGE))
def test_edge_shapes(name, fused):
    w = wl.custom(name, **EDGE[name])
    small = w.num_experts * w.num_ranks * w.max_m * w.row_bytes < (1 << 28)
    _full_parity(w, wl.make_inputs(w, seed=3), region_sets=small, fused=fused)


# Input rows, or slot rows, at 16-byte but not 32-byte alignment: the fused
# kernel then takes its 16-byte vector forms (for quantised rows, and for plain
# rows longer than 8 KiB, its generic form). Rows are offset inside larger
# buffers; the results must equal the oracle's.
MISALIGNED = {
    "quant_x": (wl.custom("mis_quant", num_ranks=4, tokens_per_rank=64, hidden=1024, num_experts=32, topk=4,
                          max_m=64, dtype="bf16q", expert="scale", x_dist="normal"), "x"),
    "long_rows_recv": (wl.custom("mis_long", num_ranks=2, tokens_per_rank=48, hidden=6144, num_experts=8, topk=2,
                                 max_m=48, x_dist="normal"), "recv_x"),
    "fp8_k16_both": (wl.custom("mis_k16", num_ranks=2, tokens_per_rank=40, hidden=1024, num_experts=32, topk=16,
                               max_m=40, dtype="fp8", expert="scale", x_dist="normal"), "both"),
}


def _offset16(t: torch.Tensor) -> torch.Tensor:
    """A copy of t whose storage starts 16 bytes past a 256-byte boundary."""
    nb = t.numel() * t.element_size()
    raw = torch.empty(nb + 16, dtype=torch.uint8, device=t.device)
    v = raw[16:16 + nb].view(t.dtype).view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("name", list(MISALIGNED))
def test_fused_with_16_byte_aligned_rows(name):
    w, which = MISALIGNED[name]
    inp = wl.make_inputs(w, seed=9)
    ref = oracle.run(w, inp)
    desc = B.MoeDesc.of(w)
    assert B.moe_layout_dispatch_kernels(desc) == 1
    bufs = B.allocate_buffers(desc, "cuda:0")
    if which in ("recv_x", "both"):
        bufs.recv_x = _offset16(bufs.recv_x)
    step = P.MoeStep(w, "cuda:0", buffers=bufs)
    d = P.to_device(inp, "cuda:0")
    if which in ("x", "both"):
        d = P.DeviceInputs(d.topk_idx, d.topk_weights, _offset16(d.x), d.x_scales)
    assert (d.x.data_ptr() % 32 != 0) == (which in ("x", "both"))
    assert (step.buf.recv_x.data_ptr() % 32 != 0) == (which in ("recv_x", "both"))
    step.reset()
    step.layout_dispatch(d)
    flags = step.buf.flags.clone()
    step.experts()
    step.combine(d)
    assert step.error() == B.MOE_OK
    ts = check_layout(step, flags, ref, w)
    check_dispatch(step, w, ts, ref)
    out = step.buf.out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(w.num_tokens, w.hidden)
    assert_combine_close(out, ref.out)


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
@pytest.mark.parametrize("num_sms", [1, 3])
def test_few_sms_deep_pipeline(num_sms, fused):
    """With one or three SMs every dispatch CTA streams many rows through its stages."""
    w = wl.custom("deep", num_ranks=4, tokens_per_rank=200, hidden=2048, num_experts=16, topk=4, max_m=200,
                  x_dist="normal")
    if fused:
        assert B.moe_layout_dispatch_kernels(B.MoeDesc.of(w, num_sms)) == 1
    _full_parity(w, wl.make_inputs(w, seed=5), num_sms=num_sms, region_sets=False, fused=fused)


def test_fused_max_tokens_per_rank():
    """1024 tokens per rank: the largest batch the fused kernel takes, with several rows per CTA."""
    w = wl.custom("fused_max", num_ranks=4, tokens_per_rank=1024, hidden=1024, num_experts=64, topk=8, max_m=1024,
                  dtype="fp8", expert="scale", x_dist="normal", renormalize=False)
    assert B.moe_layout_dispatch_kernels(B.MoeDesc.of(w)) == 1
    _full_parity(w, wl.make_inputs(w, seed=9), region_sets=False, fused=True)


def test_empty_batch():
    w = wl.custom("empty", num_ranks=2, tokens_per_rank=0, hidden=128, num_experts=4, topk=2, max_m=4)
    inp = wl.make_inputs(w)
    step, d, flags, err, guards = run_step(w, inp, guards=True)
    assert err == B.MOE_OK
    assert not step.buf.counts.any().item()
    assert bool((flags == 1).all()), "an empty batch still signals count + 1 = 1"
    assert all(g.guards_intact() for g in guards)


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
def test_repeated_steps_reuse_buffers(fused):
    """Combine clears the flags, so the same buffers serve the next step."""
    w = wl.custom("rep", num_ranks=4, tokens_per_rank=50, hidden=512, num_experts=16, topk=4, max_m=64,
                  dtype="fp8", expert="scale", x_dist="normal")
    step = P.MoeStep(w, "cuda:0")
    step.reset()
    for seed in (1, 2, 3):
        inp = wl.make_inputs(w, seed=seed)
        ref = oracle.run(w, inp)
        d = P.to_device(inp, "cuda:0")
        step.run(d, fused=fused)
        assert step.error() == B.MOE_OK
        out = step.buf.out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(w.num_tokens, w.hidden)
        assert_combine_close(out, ref.out)
        assert np.array_equal(step.buf.tok_slot.cpu().numpy(), ref.tok_slot)


def test_layout_is_deterministic():
    w = wl.WORKLOADS["ds_decode"]
    inp = wl.make_inputs(w)
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(inp, "cuda:0")
    step.reset()
    seen = []
    for _ in range(3):
        step.layout(d)
        seen.append(step.buf.tok_slot.clone())
        step.reset()
    assert all(torch.equal(seen[0], s) for s in seen[1:])


# --- error paths (no fault, no trap: the kernels latch a status and skip) ----------

def _guarded_run(w, topk_idx, reset_before_dispatch=False, fused=False):
    inp = wl.make_inputs(w)
    inp.topk_idx[...] = topk_idx
    step, d, flags, err, guards = None, None, None, None, None
    desc = B.MoeDesc.of(w)
    from gpu_common import guarded_buffers
    bufs, guards = guarded_buffers(desc, "cuda:0")
    step = P.MoeStep(w, "cuda:0", buffers=bufs)
    d = P.to_device(inp, "cuda:0")
    step.reset()
    if fused:
        step.layout_dispatch(d)
    else:
        step.layout(d)
        if reset_before_dispatch:
            step.reset()
        step.dispatch(d)
    step.experts()
    step.combine(d)
    return step, step.error(), guards


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
def test_duplicate_expert_is_rejected_without_stray_writes(fused):
    w = wl.custom("dup", num_ranks=2, tokens_per_rank=8, hidden=128, num_experts=8, topk=2, max_m=8)
    idx = wl.make_inputs(w).topk_idx.copy()
    idx[1, 3, 1] = idx[1, 3, 0]
    step, err, guards = _guarded_run(w, idx, fused=fused)
    assert err == B.MOE_EINVAL
    assert all(g.guards_intact() for g in guards)


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
@pytest.mark.parametrize("bad", [8, -2, 1 << 30, -(1 << 30)])
def test_out_of_range_expert_is_rejected(bad, fused):
    w = wl.custom("oor", num_ranks=2, tokens_per_rank=8, hidden=128, num_experts=8, topk=2, max_m=8)
    idx = wl.make_inputs(w).topk_idx.copy()
    idx[0, 5, 0] = bad
    step, err, guards = _guarded_run(w, idx, fused=fused)
    assert err == B.MOE_EINVAL
    assert int(step.buf.tok_slot[0, 5, 0]) == -1
    assert all(g.guards_intact() for g in guards)


def test_dispatch_without_layout_times_out():
    """Zeroed count+1 flags: the bounded wait gives up, latches a timeout and writes nothing."""
    w = wl.custom("noflags", num_ranks=2, tokens_per_rank=8, hidden=128, num_experts=8, topk=2, max_m=8)
    idx = wl.make_inputs(w).topk_idx
    step, err, guards = _guarded_run(w, idx, reset_before_dispatch=True)
    assert err == B.MOE_ETIMEOUT
    assert bool((step.buf.recv_meta == -7).all()), "no slot may be written without its count"
    assert all(g.guards_intact() for g in guards)
    # the context is still usable: a normal step succeeds afterwards
    inp = wl.make_inputs(w)
    step.reset()
    step.run(P.to_device(inp, "cuda:0"))
    assert step.error() == B.MOE_OK


def test_host_validation():
    w = wl.WORKLOADS["tiny"]
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(wl.make_inputs(w), "cuda:0")
    bad = B.MoeDesc.of(w)
    bad.tokens_per_rank = bad.max_m + 1
    with pytest.raises(B.MoeError) as e:
        B.moe_layout(bad, d.topk_idx, step.buf.counts, step.buf.flags, step.buf.tok_slot, step.buf.err)
    assert e.value.status == B.MOE_EINVAL
    # rows must start on a 16-byte boundary
    xs = torch.empty(d.x.numel() * 2 + 8, dtype=torch.uint8, device="cuda:0")[2:2 + d.x.numel() * 2]
    with pytest.raises(B.MoeError):
        B.moe_dispatch(B.MoeDesc.of(w), xs, None, step.buf.tok_slot, step.buf.flags, step.buf.recv_x, None,
                       step.buf.recv_meta, step.buf.err)


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
@pytest.mark.parametrize("name", ["tiny", "ds_decode", "skewed"])
def test_pinned_host_inputs_and_output(name, fused):
    """Inputs and output in pinned host memory, read and written by the kernels
    directly: the same bits as the all-device step."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(inp, "cuda:0")
    step.reset()
    step.buf.recv_meta.fill_(-7)
    step.run(d, fused=fused)
    assert step.error() == B.MOE_OK
    ref = step.buf.out.clone()
    ref_meta = step.buf.recv_meta.clone()
    h = P.to_pinned_host(inp)
    hout = torch.empty((w.num_ranks, w.tokens_per_rank, w.hidden), dtype=torch.bfloat16).pin_memory()
    step.buf.recv_meta.fill_(-7)
    if fused:
        step.layout_dispatch(h)
    else:
        step.layout(h)
        step.dispatch(h)
    step.experts()
    step.combine(h, out=hout)
    assert step.error() == B.MOE_OK
    torch.cuda.synchronize()
    assert torch.equal(hout.view(torch.int16), ref.cpu().view(torch.int16))
    assert torch.equal(step.buf.recv_meta, ref_meta)


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
def test_ds_decode_bf16_rows_quantised_on_dispatch(fused):
    """bf16 input rows: the slots hold the oracle's E4M3 codes and scales bit for bit."""
    w = wl.WORKLOADS["ds_decode_bf16in"]
    if fused:
        assert B.moe_layout_dispatch_kernels(B.MoeDesc.of(w)) == 1
    inp = wl.make_inputs(w)
    step, d, ref, out = _full_parity(w, inp, region_sets=False, fused=fused)
    # the dispatched rows are half the input bytes
    assert step.buf.recv_x.shape[1] == w.hidden


def _e4m3_boundary_rows(R, T, H, seed=9):
    """bf16 rows whose 128-element blocks have amax = 448 * 2^e (so the scale is 2^e exactly) and whose other
    elements are e4m3 rounding boundaries times 2^e (exact ties, the subnormal midpoints and 2^-10), their bf16
    neighbours and negatives: x / scale lands on or next to a boundary, where the quotient decides the code."""
    rng = np.random.default_rng(seed)
    mids = [(1 + (2 * m + 1) / 16) * 2.0 ** e for e in range(-6, 9) for m in range(8)]
    mids += [(j + 0.5) * 2.0 ** -9 for j in range(7)] + [2.0 ** -10, 2.0 ** -7]
    mids = np.array(mids, dtype=np.float32)
    bits = mids.view(np.uint32) >> 16  # exact in bf16: at most 5 significant bits
    cand = np.concatenate([bits, bits + 1, bits - 1]).astype(np.uint32)
    cand = cand[(cand << 16).view(np.float32) < 448.0]  # below the block's amax
    nblk = R * T * H // 128
    e = rng.integers(-20, 21, size=nblk)
    vals = rng.choice(cand, size=(nblk, 128)).astype(np.uint32)
    vals[:, 0] = np.float32(448.0).view(np.uint32) >> 16
    # scale by 2^e: add e to the bf16 exponent field (every value stays normal)
    vals = (vals + (e[:, None] << 7).astype(np.int64)).astype(np.uint32)
    vals |= (rng.integers(0, 2, size=(nblk, 128)) << 15).astype(np.uint32)  # random signs
    vals[:, 0] &= 0x7FFF
    return vals.astype(np.uint16).reshape(R, T, H)


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
def test_quantised_dispatch_at_e4m3_rounding_boundaries(fused):
    """Quotients x / scale exactly on e4m3 rounding boundaries (ties to even, the subnormal midpoints, 2^-10) and
    one bf16 step either side: the slot codes and scales equal the oracle's, which divides in fp32."""
    w = wl.custom("qties", num_ranks=2, tokens_per_rank=100, hidden=1024, num_experts=8, topk=2, max_m=100,
                  dtype="bf16q", expert="scale", renormalize=False)
    inp = wl.make_inputs(w)
    inp.x = _e4m3_boundary_rows(w.num_ranks, w.tokens_per_rank, w.hidden)
    # the inputs do put quotients on boundaries: every block's scale is a power of two
    xf = (inp.x.astype(np.uint32) << 16).view(np.float32).reshape(-1, 128)
    q = np.abs(xf) / (np.abs(xf).max(axis=1, keepdims=True) / np.float32(448))
    m = (q.view(np.uint32) & 0xFFFFF) == 0x80000
    assert m.mean() > 0.2, "most quotients sit exactly on a tie"
    _full_parity(w, inp, fused=fused)


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
@pytest.mark.parametrize("num_sms", [1, 4])
def test_quantised_dispatch_deep_pipeline(num_sms, fused):
    w = wl.custom("qdeep", num_ranks=4, tokens_per_rank=300, hidden=1024, num_experts=16, topk=4, max_m=300,
                  dtype="bf16q", expert="scale", x_dist="normal", renormalize=False)
    _full_parity(w, wl.make_inputs(w, seed=12), num_sms=num_sms, region_sets=False, fused=fused)


def test_quantised_dispatch_rejects_input_scales():
    w = wl.custom("qrej", num_ranks=2, tokens_per_rank=8, hidden=256, num_experts=4, topk=2, max_m=8,
                  dtype="bf16q", expert="scale", x_dist="normal")
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(wl.make_inputs(w), "cuda:0")
    bogus = torch.ones((2, 8, 2), dtype=torch.float32, device="cuda:0")
    step.reset()
    step.layout(d)
    with pytest.raises(B.MoeError):
        B.moe_dispatch(step.desc, d.x, bogus, step.buf.tok_slot, step.buf.flags, step.buf.recv_x,
                       step.buf.recv_scales, step.buf.recv_meta, step.buf.err)


# --- receive hook: compaction into expert-major buffers, and the packed combine ----

def _slot_of_packed(offsets: np.ndarray, counts: np.ndarray, max_m: int) -> np.ndarray:
    """Slot id of every packed row, from the offsets (host side, for the checks)."""
    c = counts.ravel()
    return np.concatenate([r * max_m + np.arange(c[r]) for r in range(c.size)]).astype(np.int64) \
        if c.sum() else np.zeros(0, np.int64)


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
@pytest.mark.parametrize("name", ["tiny", "ds_decode", "skewed", "ds_decode_bf16in"])
def test_recv_packs_expert_major_and_combine_reads_it(name, fused):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    ref = oracle.run(w, inp)
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(inp, "cuda:0")
    step.reset()
    step.run(d, fused=fused)                      # slot-layout combine, the reference for the packed one
    assert step.error() == B.MOE_OK
    out_slots = step.buf.out.clone()
    packed = B.allocate_packed(step.desc, "cuda:0")
    packed.packed_meta.fill_(-7)
    # the flags were cleared by combine: signal again and receive
    if fused:
        step.layout_dispatch(d)
    else:
        step.layout(d)
        step.dispatch(d)
    step.recv(packed)
    assert step.error() == B.MOE_OK
    off = oracle.region_offsets(ref.counts, w.max_m)
    assert np.array_equal(packed.region_offsets.cpu().numpy(), off)
    opk = oracle.compact(ref.slots, off, w.num_ranks, w.num_experts, w.max_m, w.num_tokens * w.topk)
    n = int(off[-1])
    assert n == w.num_tokens * w.topk
    assert np.array_equal(packed.packed_meta[:n].cpu().numpy(), opk.meta)
    assert np.array_equal(packed.packed_x[:n].cpu().numpy(), opk.rows)
    if packed.packed_scales is not None:
        assert np.array_equal(packed.packed_scales[:n].cpu().numpy().view(np.uint32), opk.scales.view(np.uint32))
    # the forward map: choice j of token t of rank src sits at packed row offsets[slot / max_m] + slot % max_m
    ts = ref.tok_slot.astype(np.int64)
    assert np.array_equal(packed.tok_packed.cpu().numpy(), off[ts // w.max_m] + ts % w.max_m)
    # expert outputs in packed order, then the packed combine
    y = step.y
    sop = torch.from_numpy(_slot_of_packed(off, ref.counts, w.max_m)).cuda()
    packed_y = y.index_select(0, sop).contiguous()
    step.combine_packed(d, packed_y, packed)
    assert step.error() == B.MOE_OK
    assert torch.equal(step.buf.out.view(torch.int16), out_slots.view(torch.int16))
    assert not step.buf.flags.any().item()


RECV_REGIONS = {
    # E * R = 8192 regions: the largest count scan the one-kernel receive hook holds in shared memory
    "8192_regions": wl.custom("recv8192", num_ranks=32, tokens_per_rank=6, hidden=128, num_experts=256, topk=8,
                              max_m=6, dtype="fp8", expert="scale", x_dist="normal"),
    # E * R = 16384 regions: the two-kernel form (one-CTA scan, then compaction)
    "16384_regions": wl.custom("recv16384", num_ranks=64, tokens_per_rank=5, hidden=128, num_experts=256, topk=8,
                               max_m=5, dtype="fp8", expert="scale", x_dist="normal"),
    # E * R = 8196 regions, bf16 rows: just past the one-kernel limit
    "8196_regions": wl.custom("recv8196", num_ranks=2, tokens_per_rank=40, hidden=64, num_experts=4098, topk=3,
                              max_m=40),
    # an empty batch on each form: offsets all zero, nothing packed
    "empty_one_kernel": wl.custom("recv_empty1", num_ranks=4, tokens_per_rank=0, hidden=128, num_experts=64,
                                  topk=4, max_m=4),
    "empty_two_kernels": wl.custom("recv_empty2", num_ranks=2, tokens_per_rank=0, hidden=64, num_experts=4098,
                                   topk=3, max_m=4),
}


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
@pytest.mark.parametrize("masked", [0.0, 0.3], ids=["all", "masked"])
@pytest.mark.parametrize("name", list(RECV_REGIONS))
def test_recv_on_both_sides_of_the_one_kernel_region_limit(name, masked, fused):
    """The receive hook with region counts at and past what its one-kernel form scans
    in shared memory: offsets, packed rows, scales and headers and the forward map
    equal the oracle's, and the packed combine equals the slot combine bit for bit."""
    w = RECV_REGIONS[name]
    inp = wl.make_inputs(w, seed=3)
    if masked:
        inp = wl.mask_choices(inp, masked, seed=4)
    ref = oracle.run(w, inp)
    step, d, _, err, _ = run_step(w, inp, fused=fused)
    assert err == B.MOE_OK, B.moe_status_string(err)
    out_slots = step.buf.out.clone()
    packed = B.allocate_packed(step.desc, "cuda:0")
    packed.packed_meta.fill_(-7)
    packed.tok_packed.fill_(12345)
    packed.region_offsets.fill_(-9)
    if fused:
        step.layout_dispatch(d)
    else:
        step.layout(d)
        step.dispatch(d)
    step.recv(packed)
    assert step.error() == B.MOE_OK
    off = oracle.region_offsets(ref.counts, w.max_m)
    assert np.array_equal(packed.region_offsets.cpu().numpy(), off)
    n = int(off[-1])
    opk = oracle.compact(ref.slots, off, w.num_ranks, w.num_experts, w.max_m, n)
    assert np.array_equal(packed.packed_meta[:n].cpu().numpy(), opk.meta)
    assert np.array_equal(packed.packed_x[:n].cpu().numpy(), opk.rows)
    if packed.packed_scales is not None:
        assert np.array_equal(packed.packed_scales[:n].cpu().numpy().view(np.uint32), opk.scales.view(np.uint32))
    t64 = ref.tok_slot.astype(np.int64)
    want_tp = np.where(t64 >= 0, off[np.maximum(t64, 0) // w.max_m] + np.maximum(t64, 0) % w.max_m, -1)
    assert np.array_equal(packed.tok_packed.cpu().numpy(), want_tp)
    sop = torch.from_numpy(np.sort(t64[t64 >= 0].ravel())).cuda()   # slots in packed order
    step.combine_packed(d, step.y.index_select(0, sop).contiguous(), packed)
    assert step.error() == B.MOE_OK
    assert torch.equal(step.buf.out.view(torch.int16), out_slots.view(torch.int16))


def test_recv_without_counts_times_out():
    w = wl.WORKLOADS["tiny"]
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(wl.make_inputs(w), "cuda:0")
    step.reset()
    step.layout(d)
    step.dispatch(d)
    step.reset()                                  # the count + 1 signals never arrive
    packed = B.allocate_packed(step.desc, "cuda:0")
    step.recv(packed)
    assert step.error() == B.MOE_ETIMEOUT



# --- cross-node traffic accounting ---------------------------------------------------

@pytest.mark.parametrize("name,rpn", [("ds_prefill", 2), ("ds_decode", 4), ("skewed", 4), ("tiny", 1)])
def test_route_stats_match_the_oracle(name, rpn):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    ref = oracle.route_stats(inp.topk_idx, w.num_experts, rpn)
    desc = B.MoeDesc.of(w)
    stats = torch.zeros((w.num_ranks, 4), dtype=torch.int64, device="cuda:0")
    err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    B.moe_route_stats(desc, torch.from_numpy(inp.topk_idx).cuda(), rpn, stats, err)
    assert B.moe_get_error(err) == B.MOE_OK
    assert np.array_equal(stats.cpu().numpy(), ref)


@pytest.mark.parametrize("limited,key", [(False, "unlimited"), (True, "node_limited")])
def test_route_stats_reproduce_the_printed_copies_on_the_gpu(limited, key):
    import json
    import os
    import test_workloads as tw
    want = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "node_limited_routing.json")))
    want = want["printed"][key]
    idx, R, gpn, E, k = tw._page_routing(limited)
    full = np.repeat(idx[None], R, axis=0)
    desc = B.MoeDesc(R, idx.shape[0], 128, E, k, idx.shape[0], B.MOE_BF16, 0)
    stats = torch.zeros((R, 4), dtype=torch.int64, device="cuda:0")
    err = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    B.moe_route_stats(desc, torch.from_numpy(full).cuda(), gpn, stats, err)
    assert B.moe_get_error(err) == B.MOE_OK
    st = stats[0].cpu().numpy()
    assert f"{st[1] / st[0]:.2f}" == want["per_expert"]
    assert f"{st[2] / st[0]:.2f}" == want["per_gpu_dedup"]
    assert f"{st[3] / st[0]:.2f}" == want["per_node_dedup"]


# --- masked choices (expert -1: the choice names no expert) -------------------------

MASKED = {
    # the chunk layout (T <= 128 is one chunk per rank; T = 100 here), bf16 identity experts
    "chunk": wl.custom("masked_chunk", num_ranks=2, tokens_per_rank=100, hidden=256, num_experts=16, topk=4,
                       max_m=100, x_dist="normal"),
    # the cluster layout (T > 128) and, fused, the fused kernel
    "cluster": wl.custom("masked_cluster", num_ranks=3, tokens_per_rank=700, hidden=128, num_experts=24, topk=3,
                         max_m=700),
    # fp8 rows with scales and the scaling experts
    "fp8": wl.custom("masked_fp8", num_ranks=4, tokens_per_rank=64, hidden=512, num_experts=32, topk=8, max_m=64,
                     dtype="fp8", expert="scale", x_dist="normal"),
}


@pytest.mark.parametrize("fused", FUSED, ids=FUSED_IDS)
@pytest.mark.parametrize("name", list(MASKED))
def test_masked_choices_are_skipped_everywhere(name, fused):
    """About a quarter of the choices, and every choice of some tokens, are -1: no
    error; layout, slots, combine, the receive hook and the route stats all equal
    the oracle's, a fully masked token combines to +0, and its forward-map
    entries read -1."""
    require_gpu()
    w = MASKED[name]
    inp = wl.mask_choices(wl.make_inputs(w), 0.25)
    ref = oracle.run(w, inp)
    step, d, flags, err, _ = run_step(w, inp, fused=fused)
    assert err == B.MOE_OK
    assert np.array_equal(step.buf.counts.cpu().numpy(), ref.counts)
    assert np.array_equal(flags.cpu().numpy().astype(np.uint64), ref.flags)
    ts = step.buf.tok_slot.cpu().numpy()
    assert np.array_equal(ts, ref.tok_slot)
    assert (ts[inp.topk_idx == -1] == -1).all()
    valid = ts.ravel() >= 0
    rows, meta, sc = gather_slots(step, w, ts.ravel()[valid])
    assert np.array_equal(meta, ref.slots.meta) and np.array_equal(rows, ref.slots.rows)
    if sc is not None:
        assert np.array_equal(sc.view(np.uint32), ref.slots.scales.view(np.uint32))
    check_region_sets(step, w, ts, ref)
    out = step.buf.out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert_combine_close(out.ravel(), ref.out.ravel())
    dead = (inp.topk_idx.reshape(-1, w.topk) < 0).all(axis=1)
    assert dead.any() and (out.reshape(-1, w.hidden)[dead] == 0).all()
    out_slots = step.buf.out.clone()
    # the receive hook and the packed combine (the flags were cleared by combine: signal again)
    packed = B.allocate_packed(step.desc, "cuda:0")
    packed.tok_packed.fill_(12345)
    if fused:
        step.layout_dispatch(d)
    else:
        step.layout(d)
        step.dispatch(d)
    step.recv(packed)
    assert step.error() == B.MOE_OK
    off = oracle.region_offsets(ref.counts, w.max_m)
    t64 = ts.astype(np.int64)
    want_tp = np.where(t64 >= 0, off[np.maximum(t64, 0) // w.max_m] + np.maximum(t64, 0) % w.max_m, -1)
    assert np.array_equal(packed.tok_packed.cpu().numpy(), want_tp)
    n = int(off[-1])
    sop = torch.from_numpy(np.sort(t64[t64 >= 0].ravel())).cuda()   # slots in packed order
    packed_y = step.y.index_select(0, sop).contiguous()
    assert packed_y.shape[0] == n
    step.combine_packed(d, packed_y, packed)
    assert step.error() == B.MOE_OK
    assert torch.equal(step.buf.out.view(torch.int16), out_slots.view(torch.int16))
    # route stats
    stats = torch.zeros((w.num_ranks, 4), dtype=torch.int64, device="cuda:0")
    B.moe_route_stats(step.desc, d.topk_idx, 2 if w.num_ranks % 2 == 0 else 1, stats, step.buf.err)
    assert step.error() == B.MOE_OK
    assert np.array_equal(stats.cpu().numpy(),
                          oracle.route_stats(inp.topk_idx, w.num_experts, 2 if w.num_ranks % 2 == 0 else 1))
    free_gpu()


def test_recv_with_a_count_above_max_m_overflows_without_stray_writes():
    """A forged count of max_m + 5 (its flag consistent with it): the receive hook
    latches MOE_EOVERFLOW, clamps the region to max_m slots and writes nothing
    outside its buffers; the context stays usable."""
    require_gpu()
    from gpu_common import Guarded
    w = wl.custom("overflow", num_ranks=2, tokens_per_rank=16, hidden=128, num_experts=8, topk=2, max_m=16)
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(wl.make_inputs(w), "cuda:0")
    step.reset()
    step.layout(d)
    step.dispatch(d)
    assert step.error() == B.MOE_OK
    r = int(torch.argmax(step.buf.counts.view(-1)).item())
    forged = w.max_m + 5
    step.buf.counts.view(-1)[r] = forged
    step.buf.flags.view(-1)[r] = forged + 1
    R, T, H, E, k = w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk
    n = R * T * k
    g = {"region_offsets": Guarded((E * R + 1,), torch.int32, "cuda:0"),
         "packed_x": Guarded((n, 2 * H), torch.uint8, "cuda:0"),
         "packed_meta": Guarded((n, 4), torch.int32, "cuda:0"),
         "tok_packed": Guarded((R, T, k), torch.int32, "cuda:0")}
    packed = B.PackedBuffers(g["region_offsets"].t, g["packed_x"].t, None, g["packed_meta"].t, g["tok_packed"].t)
    step.recv(packed)
    assert step.error() == B.MOE_EOVERFLOW
    assert all(v.guards_intact() for v in g.values())
    off = packed.region_offsets.cpu().numpy()
    assert int(off[r + 1] - off[r]) == w.max_m          # clamped
    # the context is still usable: a clean step afterwards
    step.reset()
    step.run(d)
    assert step.error() == B.MOE_OK
    free_gpu()
