"""Helpers of the GPU tests: running a step, guard bands, and the parity checks
against the CPU oracle (dispatch bit-exact per (source rank, token), combine
within 2^-7 relative with exact zeros)."""
from __future__ import annotations

import gc

import numpy as np
import torch

import oracle
from combine_moe_layout_gb300 import _binding as B
from combine_moe_layout_gb300 import pipeline as P

TOL = 2.0 ** -7          # one bf16 ulp, relative: the combine bar
POISON_BYTE = 0xA5
POISON_META = -7
GUARD = 4096             # guard elements on each side of a guarded buffer


def require_gpu():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    B.load()


def free_gpu():
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


class Guarded:
    """A device buffer with poisoned guard bands before and after it."""

    def __init__(self, shape, dtype, device, fill=None):
        n = int(np.prod(shape)) if len(shape) else 1
        self.full = torch.empty(n + 2 * GUARD, dtype=dtype, device=device)
        self.full.view(torch.uint8).fill_(POISON_BYTE)
        self.t = self.full[GUARD:GUARD + n].view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def guards_intact(self) -> bool:
        g = self.full.view(torch.uint8)
        nb = GUARD * self.full.element_size()
        return bool((g[:nb] == POISON_BYTE).all()) and bool((g[-nb:] == POISON_BYTE).all())


def guarded_buffers(desc, device):
    """MoeBuffers whose every tensor sits between guard bands."""
    R, T, H, E, k, M = desc.num_ranks, desc.tokens_per_rank, desc.hidden, desc.num_experts, desc.topk, desc.max_m
    slots = E * R * M
    fp8 = desc.dtype != B.MOE_BF16  # slots hold e4m3 rows + scales
    row = H if fp8 else 2 * H
    g = {
        "counts": Guarded((E, R), torch.int32, device, 0),
        "flags": Guarded((E, R), torch.int64, device, 0),
        "tok_slot": Guarded((R, T, k), torch.int32, device),
        "recv_x": Guarded((slots, row), torch.uint8, device),
        "recv_scales": Guarded((slots, H // 128), torch.float32, device) if fp8 else None,
        "recv_meta": Guarded((slots, 4), torch.int32, device, POISON_META),
        "expert_out": Guarded((slots, H), torch.bfloat16, device) if fp8 else None,
        "out": Guarded((R, T, H), torch.bfloat16, device),
        "err": Guarded((1,), torch.int32, device, 0),
    }
    bufs = B.MoeBuffers(**{name: (v.t if v is not None else None) for name, v in g.items()})
    return bufs, [v for v in g.values() if v is not None]


def run_step(w, inp, device="cuda:0", num_sms=0, guards=False, fused=False):
    """layout -> dispatch (or the fused call) -> experts -> combine; returns
    (step, device inputs, flags after layout, error, guard list)."""
    desc = B.MoeDesc.of(w, num_sms)
    glist = []
    if guards:
        bufs, glist = guarded_buffers(desc, device)
    else:
        bufs = B.allocate_buffers(desc, device)
        bufs.recv_meta.fill_(POISON_META)
    step = P.MoeStep(w, device, num_sms, buffers=bufs)
    small = step.slots * w.row_bytes <= (1 << 30)
    if small:
        step.buf.recv_x.fill_(POISON_BYTE)
    d = P.to_device(inp, device)
    step.reset()
    if fused:
        step.layout_dispatch(d)
        flags = step.buf.flags.clone()
    else:
        step.layout(d)
        flags = step.buf.flags.clone()
        step.dispatch(d)
    step.experts()
    step.combine(d)
    err = step.error()
    return step, d, flags, err, glist


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def assert_combine_close(got_bits: np.ndarray, ref_bits: np.ndarray):
    g, r = bf16_bits_to_f64(got_bits), bf16_bits_to_f64(ref_bits)
    assert not np.isnan(g).any()
    assert (g[r == 0] == 0).all(), "where the oracle gives 0 the kernel must give exactly 0"
    err = np.abs(g - r)
    bad = err > TOL * np.abs(r)
    assert not bad.any(), f"{bad.sum()} elements beyond 2^-7 relative; worst {err[bad].max()}"


def check_layout(step, flags_after_layout, ref, w):
    counts = step.buf.counts.cpu().numpy()
    assert np.array_equal(counts, ref.counts), "counts differ from the oracle"
    assert np.array_equal(flags_after_layout.cpu().numpy().astype(np.uint64), ref.flags), "count+1 flags differ"
    ts = step.buf.tok_slot.cpu().numpy().astype(np.int64)
    R, T, k, M = w.num_ranks, w.tokens_per_rank, w.topk, w.max_m
    s = ts.ravel()
    # slot-set semantics: distinct slots, each in its (expert, source) region below the count
    assert (s >= 0).all() and np.unique(s).size == s.size
    src = np.repeat(np.arange(R), T * k)
    region = s // M
    assert np.array_equal(region, ref.tok_slot.ravel().astype(np.int64) // M)
    assert np.array_equal(region % R, src)
    assert (s % M < counts.ravel()[region]).all()
    # design property: positions are the token order, the same as the oracle's
    assert np.array_equal(ts, ref.tok_slot.astype(np.int64))
    return ts


def gather_slots(step, w, slots: np.ndarray):
    idx = torch.from_numpy(slots.astype(np.int64)).to(step.buf.recv_x.device)
    rows = step.buf.recv_x.index_select(0, idx).cpu().numpy()
    meta = step.buf.recv_meta.index_select(0, idx).cpu().numpy()
    sc = step.buf.recv_scales.index_select(0, idx).cpu().numpy() if step.buf.recv_scales is not None else None
    return rows, meta, sc


def check_dispatch(step, w, ts_gpu, ref):
    """Every (source rank, token, choice) finds its own row, scales and header
    in the slot the GPU gave it: the per-expert set compare keyed by (source rank, token)."""
    k = w.topk
    sel = ref.sel
    slots = ts_gpu.reshape(-1, k)[sel].ravel()
    rows, meta, sc = gather_slots(step, w, slots)
    assert np.array_equal(meta, ref.slots.meta), "slot headers differ"
    assert np.array_equal(rows, ref.slots.rows), "slot rows differ"
    if sc is not None:
        assert np.array_equal(sc.view(np.uint32), ref.slots.scales.view(np.uint32)), "slot scales differ"


def check_region_sets(step, w, ts_gpu, ref):
    """Per (expert, source) region: the filled slots are exactly 0..count-1 and hold
    exactly the tokens the oracle routed there; the rest of the region is untouched."""
    M, R, E = w.max_m, w.num_ranks, w.num_experts
    meta = step.buf.recv_meta.cpu().numpy().reshape(E * R, M, 4)
    counts = ref.counts.reshape(E * R)
    filled = np.arange(M)[None, :] < counts[:, None]
    assert (meta[~filled] == POISON_META).all(), "a slot at or above its count was written"
    src_ok = meta[..., 0][filled] == np.repeat(np.arange(E * R) % R, counts)
    assert src_ok.all()
    got = sorted(map(tuple, meta[filled][:, :2].tolist()))
    ref_keys = sorted(map(tuple, ref.slots.meta[:, :2].tolist()))
    assert got == ref_keys
    rows = step.buf.recv_x.cpu().numpy().reshape(E * R, M, -1)
    assert (rows[~filled] == POISON_BYTE).all(), "payload written outside the filled slots"


def check_touched_slots_gpu(step, w, counts: np.ndarray, chunk_regions: int = 256):
    """On the device: a slot's payload and header differ from the poison exactly
    when the slot is below its region's count."""
    M, R, E = w.max_m, w.num_ranks, w.num_experts
    dev = step.buf.recv_x.device
    rows = step.buf.recv_x.view(E * R, M, -1)
    meta = step.buf.recv_meta.view(E * R, M, 4)
    cnt = torch.from_numpy(counts.reshape(E * R).astype(np.int64)).to(dev)
    pos = torch.arange(M, device=dev)
    for r0 in range(0, E * R, chunk_regions):
        r1 = min(E * R, r0 + chunk_regions)
        filled = pos[None, :] < cnt[r0:r1, None]
        touched_meta = (meta[r0:r1] != POISON_META).any(dim=-1)
        assert torch.equal(touched_meta, filled), "slot headers written outside 0..count-1"
        if step.slots * w.row_bytes <= (1 << 30):
            # rows hold random data; a filled row could by chance be all-poison only with negligible probability
            touched_rows = (rows[r0:r1] != POISON_BYTE).any(dim=-1)
            assert torch.equal(touched_rows, filled), "payload written outside 0..count-1"
