"""GPU parity of the expert stage (linear 1 with SwiGLU, linear 2) against the oracle.

The tensor cores multiply bf16 exactly and accumulate in fp32 in an order of
their own; the oracle sums in fp64. Both round h and y to bf16 once. So the
bars, derived from that arithmetic and written out below, are:

  h:  |h_gpu - h_orc| <= 2^-7 |h_orc| + 1.01 eta,
      eta = |silu'(g)| dg + |silu(g)| du + dg du + 2^-20 |h|,
      dg = (K + 2) 2^-22 sum_c |x_c w_gate[i][c]|  (du alike), K = H:
      the fp32 sums g and u differ from the exact ones by at most dg, du; silu
      and the product in fp32 add a few ulp; the two bf16 roundings of values
      that differ by eta are at most 2^-7 |h| + eta apart.
  y (down alone, on a generator-made h):
      |y_gpu - y_orc| <= 2^-7 |y_orc| + (I + 2) 2^-22 sum_i |h_i w_down[j][i]|.
  y (the chain): the same plus sum_i tol_h[i] |w_down[j][i]|, the h
      differences the chain may carry into linear 2.

A mistake in the kernel (a wrong K block, swizzle, expert or row) moves values
by about their own size, far outside these bars.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_gb300 import _binding as B
from combine_moe_layout_gb300 import pipeline as P
from combine_moe_layout_gb300 import workloads as wl
from gpu_common import free_gpu, require_gpu

pytestmark = pytest.mark.gpu

CASES = {
    # several m-tiles per expert with ragged tails, three gate/up n-tiles, one 256-wide down tile
    "ragged": wl.custom("expert_ragged", num_ranks=4, tokens_per_rank=200, hidden=256, num_experts=8, topk=2,
                        max_m=200, intermediate=384),
    # fewer packed rows than one tile; down tiles 128 wide (H = 128)
    "tiny": wl.WORKLOADS["tiny"],
    # Zipf routing: hot experts with many tiles, empty experts; H = 384 gives three 128-wide down tiles
    "zipf": wl.custom("expert_zipf", num_ranks=4, tokens_per_rank=256, hidden=384, num_experts=32, topk=4,
                      max_m=256, router="zipf", x_dist="normal", intermediate=256),
    # 1200 rows per expert on average: the default build takes the CTA-pair kernel
    # (five 256-row pair tiles per expert, the last one ragged)
    "pair_default": wl.custom("expert_pair", num_ranks=4, tokens_per_rank=600, hidden=256, num_experts=4, topk=2,
                              max_m=600, x_dist="normal", intermediate=256),
}


def _val(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _silu(g):
    return g / (1.0 + np.exp(-g))


def _dsilu(g):
    s = 1.0 / (1.0 + np.exp(-g))
    return s * (1.0 + g * (1.0 - s))


def h_tolerance(x: np.ndarray, wg: np.ndarray, wu: np.ndarray, h_orc: np.ndarray, awg=None, awu=None) -> np.ndarray:
    """Per-element bar for h of one row (x [H] and weights as fp64 values; awg,
    awu: their absolute values when the caller has them already)."""
    K = x.size
    g, u = wg @ x, wu @ x
    awg = np.abs(wg) if awg is None else awg
    awu = np.abs(wu) if awu is None else awu
    dg = (K + 2) * 2.0 ** -22 * (awg @ np.abs(x))
    du = (K + 2) * 2.0 ** -22 * (awu @ np.abs(x))
    eta = np.abs(_dsilu(g)) * dg + np.abs(_silu(g)) * du + dg * du + 2.0 ** -20 * np.abs(_silu(g) * u)
    return 2.0 ** -7 * np.abs(h_orc) + 1.01 * eta


def y_tolerance(h: np.ndarray, wd: np.ndarray, y_orc: np.ndarray, tol_h: np.ndarray | None = None) -> np.ndarray:
    """Per-element bar for y of one row (h [I] and w_down [H][I] as fp64 values)."""
    K = h.size
    tol = 2.0 ** -7 * np.abs(y_orc) + (K + 2) * 2.0 ** -22 * (np.abs(wd) @ np.abs(h))
    if tol_h is not None:
        tol = tol + np.abs(wd) @ tol_h
    return tol


def _packed_step(w):
    """Layout, dispatch and the receive hook on the GPU; the oracle's packed rows
    (bit-identical to the GPU's, which is checked) and region offsets."""
    inp = wl.make_inputs(w)
    ref = oracle.run(w, inp)
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(inp, "cuda:0")
    step.reset()
    step.layout(d)
    step.dispatch(d)
    packed = B.allocate_packed(step.desc, "cuda:0")
    step.recv(packed)
    assert step.error() == B.MOE_OK
    off = oracle.region_offsets(ref.counts, w.max_m)
    n = int(off[-1])
    opk = oracle.compact(ref.slots, off, w.num_ranks, w.num_experts, w.max_m, w.num_tokens * w.topk)
    assert np.array_equal(packed.region_offsets.cpu().numpy(), off)
    assert np.array_equal(packed.packed_x[:n].cpu().numpy(), opk.rows)
    return step, d, packed, off, opk, n


def _expert_of_rows(off: np.ndarray, E: int, R: int, n: int) -> np.ndarray:
    starts = off[np.arange(E) * R]
    return (np.searchsorted(starts, np.arange(n), side="right") - 1).astype(np.int64)


def _guarded_rows(rows: int, cols: int, extra: int = 64):
    """A bf16 [rows][cols] view with poisoned rows after it."""
    full = torch.empty((rows + extra, cols), dtype=torch.bfloat16, device="cuda:0")
    full.view(torch.int16).fill_(0x7FA5)
    return full, full[:rows]


def check_expert_stage(w, sample=None):
    """Run the bf16 expert stage on w's packed rows and check every packed row (or
    the rows in `sample`) against the oracle within the bars above; rows past the
    packed buffer stay untouched."""
    step, d, packed, off, opk, n = _packed_step(w)
    E, R, H, I = w.num_experts, w.num_ranks, w.hidden, w.intermediate
    rows = w.num_tokens * w.topk
    wts = wl.expert_weights(w, "cpu")
    dev = wl.ExpertWeights(I, wts.w_gate.cuda(), wts.w_up.cuda(), wts.w_down.cuda())
    h_full, h = _guarded_rows(rows, I)
    y_full, y = _guarded_rows(rows, H)
    step.expert_mlp(dev, packed, h, y)
    assert step.error() == B.MOE_OK
    assert bool((h_full[rows:].view(torch.int16) == 0x7FA5).all()) and bool((y_full[rows:].view(torch.int16) == 0x7FA5).all())
    hb, yb = _bits(h[:n]), _bits(y[:n])
    wg, wu, wd = (_bits(t).reshape(t.shape) for t in (wts.w_gate, wts.w_up, wts.w_down))
    ex = _expert_of_rows(off, E, R, n)
    vals = {}
    bad_h = bad_y = 0
    for p in (range(n) if sample is None else sample):
        e = int(ex[p])
        if e not in vals:
            vals[e] = (_val(wg[e]).reshape(I, H), _val(wu[e]).reshape(I, H), _val(wd[e]).reshape(H, I))
        wgv, wuv, wdv = vals[e]
        xr = opk.rows[p].view(np.uint16)
        ho, yo = oracle.expert_mlp_row(xr, wg[e], wu[e], wd[e])
        th = h_tolerance(_val(xr), wgv, wuv, _val(ho))
        ty = y_tolerance(_val(ho), wdv, _val(yo), th)
        bad_h += int((np.abs(_val(hb[p]) - _val(ho)) > th).sum())
        bad_y += int((np.abs(_val(yb[p]) - _val(yo)) > ty).sum())
    assert bad_h == 0 and bad_y == 0, (bad_h, bad_y)
    return n


@pytest.mark.parametrize("name", list(CASES))
def test_expert_stage_matches_oracle(name):
    require_gpu()
    check_expert_stage(CASES[name])
    free_gpu()


@pytest.mark.parametrize("name", ["ragged", "zipf"])
def test_expert_down_alone_on_generated_h(name):
    """Linear 2 on an h drawn by the seeded generator: the tight bar for y."""
    require_gpu()
    w = CASES[name]
    step, d, packed, off, opk, n = _packed_step(w)
    E, R, H, I = w.num_experts, w.num_ranks, w.hidden, w.intermediate
    rows = w.num_tokens * w.topk
    rng = np.random.default_rng(11)
    h_host = torch.from_numpy(rng.standard_normal((rows, I)).astype(np.float32)).to(torch.bfloat16)
    wts = wl.expert_weights(w, "cpu", seed=5)
    y_full, y = _guarded_rows(rows, H)
    B.moe_expert_down(step.desc, I, packed.region_offsets, h_host.cuda(), wts.w_down.cuda(), y, step.buf.err)
    assert step.error() == B.MOE_OK
    yb = _bits(y[:n])
    hb = _bits(h_host)
    wd = _bits(wts.w_down).reshape(E, H, I)
    ex = _expert_of_rows(off, E, R, n)
    bad = 0
    for p in range(n):
        e = ex[p]
        yo = oracle.linear_row(hb[p], wd[e])
        ty = y_tolerance(_val(hb[p]), _val(wd[e]).reshape(H, I), _val(yo))
        bad += int((np.abs(_val(yb[p]) - _val(yo)) > ty).sum())
    assert bad == 0
    free_gpu()


def test_expert_stage_feeds_the_packed_combine():
    """The chain layout -> dispatch -> recv -> experts -> packed combine gives
    the oracle's combine of the oracle's expert outputs, within the combine bar
    widened by the expert-output bar."""
    require_gpu()
    w = CASES["ragged"]
    step, d, packed, off, opk, n = _packed_step(w)
    E, R, H, I, k = w.num_experts, w.num_ranks, w.hidden, w.intermediate, w.topk
    wts = wl.expert_weights(w, "cpu")
    dev = wl.ExpertWeights(I, wts.w_gate.cuda(), wts.w_up.cuda(), wts.w_down.cuda())
    rows = w.num_tokens * k
    h = torch.empty((rows, I), dtype=torch.bfloat16, device="cuda:0")
    y = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda:0")
    step.expert_mlp(dev, packed, h, y)
    step.combine_packed(d, y, packed)
    assert step.error() == B.MOE_OK
    out = _val(_bits(step.buf.out)).reshape(R * w.tokens_per_rank, H)
    # oracle expert outputs per packed row, then the weighted sum per token
    wg, wu, wd = (_bits(t).reshape(t.shape) for t in (wts.w_gate, wts.w_up, wts.w_down))
    ex = _expert_of_rows(off, E, R, n)
    y_o = np.zeros((n, H))
    ty = np.zeros((n, H))
    for p in range(n):
        e = ex[p]
        xr = opk.rows[p].view(np.uint16)
        ho, yo = oracle.expert_mlp_row(xr, wg[e], wu[e], wd[e])
        th = h_tolerance(_val(xr), _val(wg[e]).reshape(I, H), _val(wu[e]).reshape(I, H), _val(ho))
        y_o[p] = _val(yo)
        ty[p] = y_tolerance(_val(ho), _val(wd[e]).reshape(H, I), y_o[p], th)
    inp = wl.make_inputs(w)
    ref = oracle.run(w, inp)
    ts = ref.tok_slot.astype(np.int64).reshape(-1, k)
    prow = off[ts // w.max_m] + ts % w.max_m
    wt = inp.topk_weights.reshape(-1, k).astype(np.float64)
    exact = np.einsum("tj,tjh->th", wt, y_o[prow])
    # combine's own bar (fp32 sum of k terms, one bf16 rounding) plus the expert-output bars carried through
    tol = 2.0 ** -7 * np.abs(exact) + np.einsum("tj,tjh->th", np.abs(wt), ty[prow] + 2.0 ** -20 * np.abs(y_o[prow]))
    assert int((np.abs(out - exact) > tol).sum()) == 0
    free_gpu()


def _with_variant(flags, name, cases):
    import os

    from combine_moe_layout_gb300 import _build
    path = os.path.join(os.path.dirname(_build.LIB), name)
    variant = B._open(_build.build(extra_flags=flags, lib_path=path))
    real = B.load()
    try:
        B._lib = variant
        for c in cases:
            test_expert_stage_matches_oracle(c)
    finally:
        B._lib = real


def test_expert_stage_with_narrow_tile_groups():
    """A build with n-tile groups two wide: two gate/up n-tiles out of three then a
    narrower last group (ragged), two down n-tiles out of three (Zipf); the same
    results within the same bars."""
    require_gpu()
    _with_variant(["-DMOE_GEMM_GROUP_N=2"], "libmoe_layout_group2.so", ("ragged", "zipf"))


def test_expert_stage_pair_kernel_single_accumulator():
    """The CTA-pair kernel forced on (the default build takes it only for experts
    of 512 rows or more on average, as in the Mixtral-shape test), with one
    256-column accumulator per CTA: the same results within the same bars."""
    require_gpu()
    _with_variant(["-DMOE_GEMM_PAIR=2", "-DMOE_GEMM_PAIR_TMEM_COLS=256"], "libmoe_layout_pair256.so",
                  ("ragged", "tiny", "zipf"))


def test_expert_stage_pair_kernel_double_accumulator():
    """The CTA-pair kernel forced on, with two 256-column accumulators per CTA."""
    require_gpu()
    _with_variant(["-DMOE_GEMM_PAIR=2"], "libmoe_layout_pair512.so", ("ragged", "tiny", "zipf"))


def test_expert_stage_rejects_what_it_cannot_run():
    require_gpu()
    w = CASES["tiny"]
    step = P.MoeStep(w, "cuda:0")
    packed = B.allocate_packed(step.desc, "cuda:0")
    rows, H, I = w.num_tokens * w.topk, w.hidden, w.intermediate
    x = torch.zeros((rows, H), dtype=torch.bfloat16, device="cuda:0")
    wg = torch.zeros((w.num_experts, I, H), dtype=torch.bfloat16, device="cuda:0")
    h = torch.zeros((rows, I), dtype=torch.bfloat16, device="cuda:0")
    for bad_inter in (0, 64, 200):
        with pytest.raises(B.MoeError) as e:
            B.moe_expert_gate_up(step.desc, bad_inter, packed.region_offsets, x, wg, wg, h, step.buf.err)
        assert e.value.status == B.MOE_EINVAL
    fp8 = B.MoeDesc.of(wl.WORKLOADS["ds_decode"])
    with pytest.raises(B.MoeError) as e:
        B.moe_expert_down(fp8, 2048, packed.region_offsets, h, wg, x, step.buf.err)
    assert e.value.status == B.MOE_EINVAL
    # more experts than the kernels' shared memory holds (offsets and tile prefixes, 12 bytes per expert):
    # rejected on the host before any tensor map or launch
    many = B.MoeDesc(1, 4, 128, 3000, 2, 4, 0, 0)
    off = torch.zeros(3001, dtype=torch.int32, device="cuda:0")
    for fn in (lambda: B.moe_expert_gate_up(many, 256, off, x, wg, wg, h, step.buf.err),
               lambda: B.moe_expert_down(many, 256, off, h, wg, x, step.buf.err)):
        with pytest.raises(B.MoeError) as e:
            fn()
        assert e.value.status == B.MOE_EINVAL
    free_gpu()


def test_expert_stage_on_the_mixtral_shape_sampled_rows():
    """The full Mixtral 8x7B expert shape (H 4096, I 14336, 8 experts, 65536
    packed rows; the CTA-pair kernel), checked on sampled rows of two experts:
    the first and last row of each expert's range and rows in between."""
    require_gpu()
    w = wl.WORKLOADS["mixtral"]
    inp = wl.make_inputs(w)
    ref = oracle.run(w, inp, sel=np.zeros(0, np.int64))   # layout only
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(inp, "cuda:0")
    step.reset()
    step.layout(d)
    step.dispatch(d)
    packed = B.allocate_packed(step.desc, "cuda:0")
    step.recv(packed)
    E, R, H, I, k, T = w.num_experts, w.num_ranks, w.hidden, w.intermediate, w.topk, w.tokens_per_rank
    off = oracle.region_offsets(ref.counts, w.max_m)
    assert np.array_equal(packed.region_offsets.cpu().numpy(), off)
    wts = wl.expert_weights(w, "cuda:0")
    rows = w.num_tokens * k
    h = torch.empty((rows, I), dtype=torch.bfloat16, device="cuda:0")
    y = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda:0")
    step.expert_mlp(wts, packed, h, y)
    assert step.error() == B.MOE_OK
    # packed row of every (source rank, token, choice) from the oracle's layout
    ts = ref.tok_slot.astype(np.int64).reshape(-1)
    prow = off[ts // w.max_m] + ts % w.max_m
    owner = np.empty(rows, np.int64)
    owner[prow] = np.arange(rows)
    x_bits = inp.x.reshape(R * T, H)
    rng = np.random.default_rng(3)
    for e in (0, E - 1):
        lo, hi = int(off[e * R]), int(off[(e + 1) * R])
        assert hi > lo
        sample = sorted({lo, hi - 1, *rng.integers(lo, hi, 3).tolist()})
        wg, wu, wd = (_bits(t[e]) for t in (wts.w_gate, wts.w_up, wts.w_down))
        wgv, wuv, wdv = _val(wg).reshape(I, H), _val(wu).reshape(I, H), _val(wd).reshape(H, I)
        awg, awu = np.abs(wgv), np.abs(wuv)
        for p in sample:
            tok = owner[p] // k
            assert inp.topk_idx.reshape(-1, k)[tok, owner[p] % k] == e
            xr = x_bits[tok]
            ho, yo = oracle.expert_mlp_row(xr, wg.reshape(I, H), wu.reshape(I, H), wd.reshape(H, I))
            th = h_tolerance(_val(xr), wgv, wuv, _val(ho), awg, awu)
            ty = y_tolerance(_val(ho), wdv, _val(yo), th)
            assert int((np.abs(_val(_bits(h[p])) - _val(ho)) > th).sum()) == 0, p
            assert int((np.abs(_val(_bits(y[p])) - _val(yo)) > ty).sum()) == 0, p
    del wts, h, y
    free_gpu()
