"""GPU parity of the fp8 expert stage against the oracle.

Rows are e4m3 codes with one fp32 scale per 128 elements; weights are e4m3 with
one fp32 scale per 128 x 128 block. The tensor cores sum code products per
128-wide K block in fp32 and the kernel adds each block, times its two scales,
in fp32; the oracle sums the dequantised values in fp64. The bars follow:

  accumulation: a dot product of length K differs from the exact one by at most
      d = (K + 2) 2^-22 sum |x w|  (sum over dequantised values).
  h (linear 1 + SwiGLU, then block-quantised): hv_gpu is within
      eta = |silu'(g)| dg + |silu(g)| du + dg du + 2^-20 |hv|
  of the exact hv. The block scale is amax / 448 in fp32 of the kernel's own
  values, so |s_gpu - amax_exact / 448| <= max(eta over the block) / 448
  + 2^-22 amax / 448. Each code is the nearest e4m3 value of hv_gpu / s_gpu,
  so the dequantised h is within half an e4m3 ulp (at (|hv| + eta) / s_gpu)
  times s_gpu, plus eta, of the exact hv.
  y (linear 2 alone, on an fp8 h drawn by the seeded generator):
      |y_gpu - y_orc| <= 2^-7 |y_orc| + d.
  y (the chain): the same plus sum_i |w_down[j][i]| (2 tol_h[i]), the two
      sides' quantisations of h carried through linear 2.
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
    # three m-tiles per expert with ragged tails, three gate/up n-tiles, one 256-wide down tile
    "ragged": wl.custom("fp8_ragged", num_ranks=4, tokens_per_rank=200, hidden=256, num_experts=8, topk=2,
                        max_m=200, dtype="fp8", expert="scale", x_dist="normal", intermediate=384),
    # fewer rows than one tile, one 128-wide down tile
    "tiny": wl.custom("fp8_tiny", num_ranks=2, tokens_per_rank=16, hidden=128, num_experts=8, topk=2, max_m=16,
                      dtype="fp8", expert="scale", x_dist="normal", intermediate=256),
    # Zipf routing (hot and empty experts), three 128-wide down tiles; rows checked on a sample
    "zipf": wl.custom("fp8_zipf", num_ranks=4, tokens_per_rank=128, hidden=384, num_experts=32, topk=4,
                      max_m=128, dtype="fp8", expert="scale", router="zipf", x_dist="normal", intermediate=256),
    # 1200 rows per expert on average (ten m-tiles each, all in the hot class, the
    # last one ragged), three h blocks, one 256-wide down tile; rows checked on a sample
    "many_rows": wl.custom("fp8_many", num_ranks=4, tokens_per_rank=600, hidden=256, num_experts=4, topk=2,
                           max_m=600, dtype="fp8", expert="scale", x_dist="normal", intermediate=384),
}


def _e4m3(codes) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def _val(bits) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _deq_row(codes, scales) -> np.ndarray:
    return _e4m3(codes) * np.repeat(np.asarray(scales, np.float64), 128)


def _deq_mat(codes, scales) -> np.ndarray:
    N, K = codes.shape
    return _e4m3(codes) * np.repeat(np.repeat(np.asarray(scales, np.float64), 128, 0), 128, 1)


def _halfulp_e4m3(v: np.ndarray) -> np.ndarray:
    """Half the spacing of e4m3 values at magnitude v (subnormal spacing 2^-9, top binade capped at 256)."""
    v = np.minimum(np.abs(v), 448.0)
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
    return np.where(v < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))


def _silu(g):
    return g / (1.0 + np.exp(-g))


def _dsilu(g):
    s = 1.0 / (1.0 + np.exp(-g))
    return s * (1.0 + g * (1.0 - s))


def h_bars(x, Wg, Wu, aWg, aWu, hv):
    """eta per element of hv for one row (x and weights dequantised, fp64)."""
    K = x.size
    g, u = Wg @ x, Wu @ x
    dg = (K + 2) * 2.0 ** -22 * (aWg @ np.abs(x))
    du = (K + 2) * 2.0 ** -22 * (aWu @ np.abs(x))
    return np.abs(_dsilu(g)) * dg + np.abs(_silu(g)) * du + dg * du + 2.0 ** -20 * np.abs(hv)


def check_h_row(hv, eta, hq_gpu, hs_gpu):
    """Number of scale and value violations of one GPU h row against the exact hv."""
    I = hv.size
    bad = 0
    tol = np.zeros(I)
    for b in range(I // 128):
        sl = slice(128 * b, 128 * b + 128)
        amax = np.abs(hv[sl]).max()
        s_exact = amax / 448.0 if amax > 0 else 1.0
        s = float(hs_gpu[b])
        if abs(s - s_exact) > eta[sl].max() / 448.0 + 2.0 ** -22 * s_exact:
            bad += 1
        t = _halfulp_e4m3((np.abs(hv[sl]) + eta[sl]) / s) * s + eta[sl] + 2.0 ** -22 * np.abs(hv[sl])
        tol[sl] = t
        bad += int((np.abs(_e4m3(hq_gpu[sl]) * s - hv[sl]) > t).sum())
    return bad, tol


def _packed_step(w):
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
    assert np.array_equal(packed.packed_x[:n].cpu().numpy(), opk.rows)
    assert np.array_equal(packed.packed_scales[:n].cpu().numpy().view(np.uint32), opk.scales.view(np.uint32))
    return step, d, packed, off, opk, n, inp, ref


def _expert_of_rows(off, E, R, n):
    starts = off[np.arange(E) * R]
    return (np.searchsorted(starts, np.arange(n), side="right") - 1).astype(np.int64)


def _sample(name, n, off, E, R):
    if name not in ("zipf", "many_rows"):
        return range(n)
    firsts = {int(off[e * R]) for e in range(E) if off[(e + 1) * R] > off[e * R]}
    lasts = {int(off[(e + 1) * R]) - 1 for e in range(E) if off[(e + 1) * R] > off[e * R]}
    return sorted(set(range(0, n, 5)) | firsts | lasts)


def _host(t):
    return t.cpu().numpy()


class _Experts:
    """Host copies of the fp8 weights, dequantised once per expert."""

    def __init__(self, wts):
        self.q = {k: _host(getattr(wts, k)) for k in ("w_gate", "w_up", "w_down")}
        self.s = {k: _host(getattr(wts, k + "_scales")) for k in ("w_gate", "w_up", "w_down")}
        self.cache = {}

    def deq(self, name, e):
        key = (name, e)
        if key not in self.cache:
            W = _deq_mat(self.q[name][e], self.s[name][e])
            self.cache[key] = (W, np.abs(W))
        return self.cache[key]


def _run_stage(w, step, packed):
    E, H, I = w.num_experts, w.hidden, w.intermediate
    rows = w.num_tokens * w.topk
    wts = wl.expert_weights_fp8(w, "cuda:0")
    h = torch.full((rows + 64, I), 0x7F, dtype=torch.uint8, device="cuda:0")
    hs = torch.full((rows + 64, I // 128), -1.0, dtype=torch.float32, device="cuda:0")
    y = torch.empty((rows + 64, H), dtype=torch.bfloat16, device="cuda:0")
    y.view(torch.int16).fill_(0x7FA5)
    step.expert_mlp_fp8(wts, packed, h[:rows], hs[:rows], y[:rows])
    assert step.error() == B.MOE_OK
    # rows past the packed buffer stay untouched
    assert bool((h[rows:] == 0x7F).all()) and bool((hs[rows:] == -1.0).all())
    assert bool((y[rows:].view(torch.int16) == 0x7FA5).all())
    return wts, h[:rows], hs[:rows], y[:rows]


def check_fp8_stage(w, sample=None):
    """Run the fp8 expert stage on w's packed rows and check every packed row (or
    the rows sample(n, off) picks) against the oracle within the bars above."""
    step, d, packed, off, opk, n, inp, ref = _packed_step(w)
    E, R, H, I = w.num_experts, w.num_ranks, w.hidden, w.intermediate
    wts, h, hs, y = _run_stage(w, step, packed)
    X = _Experts(wts)
    hq_g, hs_g, y_g = _host(h[:n]), _host(hs[:n]), y[:n].view(torch.int16).cpu().numpy().view(np.uint16)
    ex = _expert_of_rows(off, E, R, n)
    bad_h = bad_y = 0
    for p in (range(n) if sample is None else sample(n, off)):
        e = int(ex[p])
        xq, xs = opk.rows[p], opk.scales[p]
        hv, hq_o, hs_o = oracle.gate_up_row_fp8(xq, xs, X.q["w_gate"][e], X.s["w_gate"][e], X.q["w_up"][e],
                                                X.s["w_up"][e])
        Wg, aWg = X.deq("w_gate", e)
        Wu, aWu = X.deq("w_up", e)
        eta = h_bars(_deq_row(xq, xs), Wg, Wu, aWg, aWu, hv)
        b, tol_h = check_h_row(hv, eta, hq_g[p], hs_g[p])
        bad_h += b
        # y through the oracle's own h
        y_o = oracle.linear_row_fp8(hq_o, hs_o, X.q["w_down"][e], X.s["w_down"][e])
        Wd, aWd = X.deq("w_down", e)
        ho = _deq_row(hq_o, hs_o)
        ty = 2.0 ** -7 * np.abs(_val(y_o)) + (I + 2) * 2.0 ** -22 * (aWd @ np.abs(ho)) + aWd @ (2.0 * tol_h)
        bad_y += int((np.abs(_val(y_g[p]) - _val(y_o)) > ty).sum())
    assert bad_h == 0 and bad_y == 0, (bad_h, bad_y)
    return n


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_expert_stage_matches_oracle(name):
    require_gpu()
    w = CASES[name]
    check_fp8_stage(w, None if name not in ("zipf", "many_rows") else
                    (lambda n, off: _sample(name, n, off, w.num_experts, w.num_ranks)))
    free_gpu()


@pytest.mark.parametrize("name", ["ragged", "tiny"])
def test_fp8_expert_down_alone_on_generated_h(name):
    """Linear 2 on an fp8 h drawn by the seeded generator: the tight bar for y."""
    require_gpu()
    w = CASES[name]
    step, d, packed, off, opk, n, inp, ref = _packed_step(w)
    E, R, H, I = w.num_experts, w.num_ranks, w.hidden, w.intermediate
    rows = w.num_tokens * w.topk
    rng = np.random.default_rng(12)
    hq = rng.integers(0, 256, (rows, I), dtype=np.uint8)
    hq[(hq & 0x7F) == 0x7F] = 0x38
    hs = rng.uniform(0.25, 4.0, (rows, I // 128)).astype(np.float32) * 2.0 ** -7
    wts = wl.expert_weights_fp8(w, "cuda:0", seed=9)
    y = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda:0")
    B.moe_expert_down_fp8(step.desc, I, packed.region_offsets, torch.from_numpy(hq).cuda(),
                          torch.from_numpy(hs).cuda(), wts.w_down, wts.w_down_scales, y, step.buf.err)
    assert step.error() == B.MOE_OK
    X = _Experts(wts)
    y_g = y[:n].view(torch.int16).cpu().numpy().view(np.uint16)
    ex = _expert_of_rows(off, E, R, n)
    bad = 0
    for p in range(n):
        e = int(ex[p])
        y_o = oracle.linear_row_fp8(hq[p], hs[p], X.q["w_down"][e], X.s["w_down"][e])
        Wd, aWd = X.deq("w_down", e)
        ty = 2.0 ** -7 * np.abs(_val(y_o)) + (I + 2) * 2.0 ** -22 * (aWd @ np.abs(_deq_row(hq[p], hs[p])))
        bad += int((np.abs(_val(y_g[p]) - _val(y_o)) > ty).sum())
    assert bad == 0
    free_gpu()


def test_fp8_expert_stage_rejects_bf16_rows():
    require_gpu()
    w = wl.WORKLOADS["tiny"]
    step = P.MoeStep(w, "cuda:0")
    packed = B.allocate_packed(step.desc, "cuda:0")
    z = torch.zeros(16, dtype=torch.uint8, device="cuda:0")
    zs = torch.zeros(16, dtype=torch.float32, device="cuda:0")
    with pytest.raises(B.MoeError) as e:
        B.moe_expert_gate_up_fp8(step.desc, 256, packed.region_offsets, z, zs, z, zs, z, zs, z, zs, step.buf.err)
    assert e.value.status == B.MOE_EINVAL
    # more experts than either form of the kernel holds in shared memory: rejected on the host
    many = B.MoeDesc(1, 4, 128, 3000, 2, 4, 1, 0)
    off = torch.zeros(3001, dtype=torch.int32, device="cuda:0")
    for fn in (lambda: B.moe_expert_gate_up_fp8(many, 256, off, z, zs, z, zs, z, zs, z, zs, step.buf.err),
               lambda: B.moe_expert_down_fp8(many, 256, off, z, zs, z, zs, z, step.buf.err)):
        with pytest.raises(B.MoeError) as e:
            fn()
        assert e.value.status == B.MOE_EINVAL
    free_gpu()


@pytest.mark.parametrize("name", ["ds_decode", "ds_prefill"])
def test_fp8_expert_stage_on_the_deepseek_shapes_sampled_rows(name):
    """The full DeepSeek shapes (top-8 of 256 experts, H 7168, I 2048, 11.3 GB of
    fp8 weights): decode, 8 x 128 tokens, about 32 rows per expert; prefill,
    8 x 4096 tokens, about 1024 rows per expert. Checked on sampled rows of two
    experts: the first and last row of each expert's range and one between."""
    require_gpu()
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    ref = oracle.run(w, inp, sel=np.zeros(0, np.int64))     # layout only
    step = P.MoeStep(w, "cuda:0")
    d = P.to_device(inp, "cuda:0")
    step.reset()
    step.layout(d)
    step.dispatch(d)
    packed = B.allocate_packed(step.desc, "cuda:0")
    step.recv(packed)
    assert step.error() == B.MOE_OK
    E, R, H, I, k, T = w.num_experts, w.num_ranks, w.hidden, w.intermediate, w.topk, w.tokens_per_rank
    off = oracle.region_offsets(ref.counts, w.max_m)
    assert np.array_equal(packed.region_offsets.cpu().numpy(), off)
    rows = w.num_tokens * k
    wts = wl.expert_weights_fp8(w, "cuda:0")
    h = torch.empty((rows, I), dtype=torch.uint8, device="cuda:0")
    hs = torch.empty((rows, I // 128), dtype=torch.float32, device="cuda:0")
    y = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda:0")
    step.expert_mlp_fp8(wts, packed, h, hs, y)
    assert step.error() == B.MOE_OK
    ts = ref.tok_slot.astype(np.int64).reshape(-1)
    prow = off[ts // w.max_m] + ts % w.max_m
    owner = np.empty(rows, np.int64)
    owner[prow] = np.arange(rows)
    xq = inp.x.reshape(R * T, H)
    xs = inp.x_scales.reshape(R * T, H // 128)
    counts = off[(np.arange(E) + 1) * R] - off[np.arange(E) * R]
    experts = [int(np.argmax(counts)), int(np.nonzero(counts)[0][0])]
    for e in experts:
        lo, hi = int(off[e * R]), int(off[(e + 1) * R])
        sample = sorted({lo, hi - 1, (lo + hi) // 2})
        q = {n: getattr(wts, n)[e].cpu().numpy() for n in ("w_gate", "w_up", "w_down")}
        sc = {n: getattr(wts, n + "_scales")[e].cpu().numpy() for n in ("w_gate", "w_up", "w_down")}
        Wg, Wu, Wd = (_deq_mat(q[n], sc[n]) for n in ("w_gate", "w_up", "w_down"))
        aWg, aWu, aWd = np.abs(Wg), np.abs(Wu), np.abs(Wd)
        for p in sample:
            tok = owner[p] // k
            assert inp.topk_idx.reshape(-1, k)[tok, owner[p] % k] == e
            hv, hq_o, hs_o = oracle.gate_up_row_fp8(xq[tok], xs[tok], q["w_gate"], sc["w_gate"], q["w_up"],
                                                    sc["w_up"])
            eta = h_bars(_deq_row(xq[tok], xs[tok]), Wg, Wu, aWg, aWu, hv)
            bad, tol_h = check_h_row(hv, eta, h[p].cpu().numpy(), hs[p].cpu().numpy())
            assert bad == 0, p
            y_o = oracle.linear_row_fp8(hq_o, hs_o, q["w_down"], sc["w_down"])
            ty = 2.0 ** -7 * np.abs(_val(y_o)) + (I + 2) * 2.0 ** -22 * (aWd @ np.abs(_deq_row(hq_o, hs_o))) + \
                aWd @ (2.0 * tol_h)
            y_g = y[p].view(torch.int16).cpu().numpy().view(np.uint16)
            assert int((np.abs(_val(y_g) - _val(y_o)) > ty).sum()) == 0, p
    del wts, h, hs, y
    free_gpu()
