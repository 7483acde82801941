"""Pins of the CPU oracle to facts outside itself (runs without a GPU).

Each check rests on something the oracle cannot influence: library conversions
(torch's float32->bf16 and e4m3->float), numbers the pages print, brute force
by a different enumeration, counting invariants (numpy bincount), and closed
forms of the combine for identity and scaling experts.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_bf16_bits(vals32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(vals32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# --- number formats ---------------------------------------------------------

def test_bf16_rounding_matches_torch_on_float32_inputs(oracle_lib):
    """On float32 inputs, round-to-nearest-even to bf16 is torch's conversion."""
    rng = np.random.default_rng(11)
    normal = rng.standard_normal(4000).astype(np.float32) * np.float32(3.0)
    # exact ties: a bf16 pattern with only the rounding bit set below it
    hi = rng.integers(0, 0x7F7F, 2000, dtype=np.uint32)
    ties = ((hi << 16) | 0x8000).view(np.float32)
    tiny = (rng.integers(1, 1 << 23, 1000, dtype=np.uint32)).view(np.float32)  # float32 subnormals
    near_max = np.array([3.3895314e38, 3.39e38, -3.3961e38, 1e-45, 2 ** -126, -(2 ** -130)], dtype=np.float32)
    vals = np.concatenate([normal, ties, -ties, tiny, near_max]).astype(np.float32)
    ref = _torch_bf16_bits(vals)
    got = np.array([oracle.bf16_from_double(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_ties_go_to_even(oracle_lib):
    # spacing of bf16 in [1, 2) is 2^-7: 1 + 2^-8 is halfway between 1 and 1 + 2^-7
    assert oracle.bf16_from_double(1 + 2 ** -8) == 0x3F80
    assert oracle.bf16_from_double(1 + 3 * 2 ** -8) == 0x3F82
    assert oracle.bf16_from_double(1 + 2 ** -8 + 2 ** -40) == 0x3F81  # just above the tie
    assert oracle.bf16_from_double(-0.0) == 0x8000


def test_bf16_value_roundtrips_every_finite_pattern(oracle_lib):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    for b, r in zip(bits[::7], ref[::7]):
        v = oracle.bf16_value(int(b))
        if np.isnan(r):
            assert np.isnan(v)
            continue
        assert v == float(r)
        assert oracle.bf16_from_double(v) == int(b)


def test_e4m3_decode_matches_torch(oracle_lib):
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for code in range(256):
        v = oracle.e4m3_value(code)
        if np.isnan(ref[code]):
            assert np.isnan(v) and (code & 0x7F) == 0x7F
        else:
            assert v == ref[code], hex(code)
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9


# --- buffer sizes: the pages' printed numbers --------------------------------

def test_buffer_sizes_reproduce_the_printed_estimates(oracle_lib):
    g = json.load(open(os.path.join(GOLDEN, "fixed_slot_buffer_sizes.json")))
    c0, c1, c2 = g["cases"]
    sizes = {}
    for c in (c0, c1, c2):
        R, E, M, H = c["ranks"], c["experts"], c["max_tokens"], c["hidden"]
        s = oracle.buffer_sizes(R, M, H, E, 8, M, oracle.FP8_E4M3)
        per_rank = (s["recv_x"] + s["recv_scales"] + s["recv_meta"]) / R
        L = E // R
        assert L == c["printed"]["local_experts"]
        sizes[id(c)] = (per_rank, per_rank / (L * R * M))
    per_rank, message = sizes[id(c0)]
    assert message == c0["printed"]["message_bytes"]
    assert f"{per_rank / 2 ** 20:.0f}" == c0["printed"]["reserved_MiB_rounded"]
    per_rank1, message1 = sizes[id(c1)]
    assert round(per_rank1 / 1e6) == c1["printed"]["approx_MB"]
    assert round(message1 / 1e3, 1) == c1["printed"]["message_approx_KB"]
    per_rank2, _ = sizes[id(c2)]
    assert round(per_rank2 / 1e6) == c2["printed"]["approx_MB"]
    assert per_rank2 / per_rank1 == c2["printed"]["ratio_to_batch_64"]


def test_used_slots_match_the_printed_fill(oracle_lib):
    """Each token fills k slots, so a rank receives N*k/R messages on average:
    7.2 MiB of the 232 MiB estimate at 64 ranks x 128 tokens, top-8 of 256."""
    g = json.load(open(os.path.join(GOLDEN, "fixed_slot_buffer_sizes.json")))["cases"][0]
    R, E, M = g["ranks"], g["experts"], g["max_tokens"]
    rng = np.random.default_rng(3)
    idx = np.argsort(rng.random((R * M, E)), axis=1)[:, :8].astype(np.int32).reshape(R, M, 8)
    counts, _, _ = oracle.layout(idx, E, M)
    used_per_rank = counts.sum() * g["printed"]["message_bytes"] / R
    assert f"{used_per_rank / 2 ** 20:.1f}" == g["printed"]["used_MiB_rounded_1dp"]


# --- layout -------------------------------------------------------------------

def _brute_layout(idx, E, max_m):
    """Region by region: collect the (token, choice) pairs of each (expert, source)."""
    R, T, k = idx.shape
    counts = np.zeros((E, R), np.int64)
    slot = np.full((R, T, k), -1, np.int64)
    for e in range(E):
        for src in range(R):
            hits = [(t, j) for t in range(T) for j in range(k) if idx[src, t, j] == e]
            counts[e, src] = len(hits)
            for pos, (t, j) in enumerate(hits):
                slot[src, t, j] = (e * R + src) * max_m + pos
    return counts, slot


@pytest.mark.parametrize("R,T,E,k,max_m,seed", [
    (2, 16, 8, 2, 16, 0), (3, 7, 6, 3, 9, 1), (1, 5, 4, 4, 5, 2), (4, 33, 16, 8, 40, 3), (2, 0, 4, 1, 3, 4),
])
def test_layout_matches_brute_force(oracle_lib, R, T, E, k, max_m, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(R * T)]).astype(np.int32).reshape(R, T, k) \
        if R * T else np.zeros((R, T, k), np.int32)
    counts, flags, tok_slot = oracle.layout(idx, E, max_m)
    bc, bs = _brute_layout(idx, E, max_m)
    assert np.array_equal(counts, bc)
    assert np.array_equal(tok_slot, bs)
    assert np.array_equal(flags, bc.astype(np.uint64) + 1)


def test_layout_tiny_matches_brute_force(oracle_lib):
    w = wl.WORKLOADS["tiny"]
    inp = wl.make_inputs(w)
    counts, _, tok_slot = oracle.layout(inp.topk_idx, w.num_experts, w.max_m)
    bc, bs = _brute_layout(inp.topk_idx, w.num_experts, w.max_m)
    assert np.array_equal(counts, bc) and np.array_equal(tok_slot, bs)


@pytest.mark.parametrize("name", ["ds_decode", "skewed"])
def test_layout_invariants(oracle_lib, name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    idx = inp.topk_idx
    R, T, k, E, M = w.num_ranks, w.tokens_per_rank, w.topk, w.num_experts, w.max_m
    counts, flags, tok_slot = oracle.layout(idx, E, M)
    for src in range(R):  # counts are the per-source routing histogram
        assert np.array_equal(counts[:, src], np.bincount(idx[src].ravel(), minlength=E))
    assert counts.sum() == R * T * k
    assert np.array_equal(flags, counts.astype(np.uint64) + 1)  # count + 1: non-zero means arrived
    s = tok_slot.ravel().astype(np.int64)
    assert np.unique(s).size == s.size  # every (src, t, j) has its own slot
    region, pos = s // M, s % M
    src_of = np.repeat(np.arange(R), T * k)
    assert np.array_equal(region, idx.ravel().astype(np.int64) * R + src_of)
    assert (pos < counts.ravel()[region]).all()
    # the filled slots of a region are exactly 0..count-1
    filled = np.zeros(E * R * M, bool)
    filled[s] = True
    want = np.arange(M)[None, :] < counts.reshape(E * R, 1)
    assert np.array_equal(filled.reshape(E * R, M), want)


def test_layout_rejects_bad_routing(oracle_lib):
    idx = np.array([[[0, 1], [2, 2]]], np.int32)  # duplicate expert in one token
    with pytest.raises(oracle.OracleError) as e:
        oracle.layout(idx, 4, 2)
    assert e.value.code == oracle.EINVAL
    for bad in (4, -2):   # -1 is a masked choice, not an error
        with pytest.raises(oracle.OracleError) as e:
            oracle.layout(np.array([[[0, bad]]], np.int32), 4, 2)
        assert e.value.code == oracle.EINVAL


def test_layout_overflow_errors_out(oracle_lib):
    """Slots smaller than the batch: the implementation errors out."""
    idx = np.zeros((1, 3, 1), np.int32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.layout(idx, 2, 2)
    assert e.value.code == oracle.EOVERFLOW


def test_validate(oracle_lib):
    v = oracle.validate
    assert v(2, 16, 128, 8, 2, 16, 0) == 0
    assert v(3, 16, 128, 8, 2, 16, 0) == oracle.EINVAL   # E % R
    assert v(2, 17, 128, 8, 2, 16, 0) == oracle.EINVAL   # T > max_m
    assert v(2, 16, 130, 8, 2, 16, 0) == oracle.EINVAL   # bf16 rows of whole 16-byte vectors
    assert v(2, 16, 192, 8, 2, 16, 1) == oracle.EINVAL   # fp8 needs whole 128-element blocks
    assert v(2, 16, 128, 8, 9, 16, 0) == oracle.EINVAL   # k > E
    assert v(2, 0, 128, 8, 2, 16, 0) == 0                # empty batch is valid


# --- dispatch -----------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny"])
def test_dispatch_slots_hold_source_rows(oracle_lib, name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    counts, _, tok_slot = oracle.layout(inp.topk_idx, w.num_experts, w.max_m)
    sl = oracle.dispatch(inp.x, inp.x_scales, tok_slot, w.num_experts, w.max_m, w.dtype_code)
    R, T, k = tok_slot.shape
    rows = inp.x.reshape(R * T, -1).view(np.uint8)
    for i in range(R * T):
        src, t = divmod(i, T)
        for j in range(k):
            n = i * k + j
            assert sl.slot_id[n] == tok_slot[src, t, j]
            assert np.array_equal(sl.rows[n], rows[i])
            assert list(sl.meta[n]) == [src, t, inp.topk_idx[src, t, j], j]


def test_dispatch_fp8_carries_scales(oracle_lib):
    w = wl.custom("fp8s", num_ranks=2, tokens_per_rank=5, hidden=256, num_experts=4, topk=2, max_m=6,
                  dtype="fp8", expert="scale", x_dist="normal")
    inp = wl.make_inputs(w)
    _, _, tok_slot = oracle.layout(inp.topk_idx, 4, 6)
    sl = oracle.dispatch(inp.x, inp.x_scales, tok_slot, 4, 6, 1)
    assert np.array_equal(sl.rows, np.repeat(inp.x.reshape(10, 256), 2, axis=0))
    assert np.array_equal(sl.scales, np.repeat(inp.x_scales.reshape(10, 2), 2, axis=0))


# --- synthetic experts ----------------------------------------------------------

def test_expert_stub_is_the_nearest_bf16(oracle_lib):
    """y is the bf16 nearest to q*scale*(1+e/256) (exact in fp64), ties to even."""
    w = wl.custom("fp8s", num_ranks=2, tokens_per_rank=6, hidden=256, num_experts=8, topk=3, max_m=6,
                  dtype="fp8", expert="scale", x_dist="normal")
    inp = wl.make_inputs(w)
    _, _, tok_slot = oracle.layout(inp.topk_idx, 8, 6)
    sl = oracle.dispatch(inp.x, inp.x_scales, tok_slot, 8, 6, 1)
    y = oracle.expert_stub(sl, 2, 256, 8, 6, 1)
    q = torch.from_numpy(sl.rows).view(torch.float8_e4m3fn).double().numpy()
    e = sl.meta[:, 2].astype(np.float64)
    v = q * np.repeat(sl.scales.astype(np.float64), 128, axis=1) * (1 + e / 256)[:, None]

    def val(bits):
        return torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()

    yv = val(y)
    up, dn = val(y.astype(np.int32) + 1), val(y.astype(np.int32) - 1)
    err = np.abs(yv - v)
    nz = v != 0
    assert (err[nz] <= np.abs(up - v)[nz]).all() and (err[nz] <= np.abs(dn - v)[nz]).all()
    tie = nz & ((err == np.abs(up - v)) | (err == np.abs(dn - v)))
    assert ((y[tie] & 1) == 0).all()
    assert (yv[~nz] == 0).all()


# --- combine --------------------------------------------------------------------

def _deq(inp, w):
    q = torch.from_numpy(inp.x).view(torch.float8_e4m3fn).double().numpy()
    return q * np.repeat(inp.x_scales.astype(np.float64), 128, axis=-1)


def _bf16_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_combine_identity_experts_return_the_input(oracle_lib):
    """Identity experts with weights that sum to 1 give back x exactly, signed zeros included."""
    for w in (wl.WORKLOADS["tiny"],
              wl.custom("mix_small", num_ranks=4, tokens_per_rank=64, hidden=512, num_experts=8, topk=2,
                        max_m=64, x_dist="normal")):
        inp = wl.make_inputs(w)
        inp.x.reshape(-1)[[3, 77, 500]] = 0x8000  # -0.0
        inp.x.reshape(-1)[[5, 90]] = 0x0000       # +0.0
        res = oracle.run(w, inp)
        assert np.array_equal(res.out, inp.x.reshape(w.num_tokens, w.hidden))


def test_combine_scaling_experts_closed_form(oracle_lib):
    """y_e = x * (1 + e/256) gives out = x * sum_j w_j (1 + e_j/256), up to the bf16 roundings."""
    w = wl.custom("ds_small", num_ranks=4, tokens_per_rank=24, hidden=512, num_experts=32, topk=8, max_m=24,
                  dtype="fp8", expert="scale", x_dist="normal", renormalize=False)
    inp = wl.make_inputs(w)
    res = oracle.run(w, inp)
    c = (inp.topk_weights.astype(np.float64) * (1 + inp.topk_idx / 256.0)).sum(-1)
    ref = _deq(inp, w) * c[..., None]
    got = _bf16_to_f64(res.out).reshape(ref.shape)
    assert (np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref)).all()
    assert ((got == 0) == (ref == 0)).all()


def test_combine_single_unit_weight_is_exact(oracle_lib):
    w = wl.custom("k1", num_ranks=2, tokens_per_rank=8, hidden=256, num_experts=4, topk=1, max_m=8,
                  dtype="fp8", expert="scale", x_dist="normal")
    inp = wl.make_inputs(w)
    inp.topk_weights[:] = 1.0
    res = oracle.run(w, inp)
    # with one expert and weight 1 the output is that expert's bf16 row
    order = np.argsort(res.slots.slot_id)
    by_slot = dict(zip(res.slots.slot_id[order], res.y[order]))
    want = np.stack([by_slot[s] for s in res.tok_slot.reshape(-1)])
    assert np.array_equal(res.out, want)


def test_combine_is_linear_in_the_weights(oracle_lib):
    """Doubling every weight doubles the output exactly; a zero weight drops that expert."""
    w = wl.custom("lin", num_ranks=2, tokens_per_rank=12, hidden=256, num_experts=8, topk=3, max_m=12,
                  dtype="fp8", expert="scale", x_dist="normal", renormalize=False)
    inp = wl.make_inputs(w)
    base = oracle.run(w, inp)
    inp2 = wl.Inputs(inp.topk_idx, inp.topk_weights * 2, inp.x, inp.x_scales)
    dbl = oracle.run(w, inp2)
    assert np.array_equal(_bf16_to_f64(dbl.out), 2 * _bf16_to_f64(base.out))
    # zero weight on choice 2 equals a top-2 combine of the same rows
    wz = inp.topk_weights.copy()
    wz[..., 2] = 0
    zero = oracle.combine(base.tok_slot, wz, base.slots.slot_id, base.y, 8, 12)
    two = oracle.combine(base.tok_slot[..., :2].copy(), inp.topk_weights[..., :2].copy(), base.slots.slot_id,
                         base.y, 8, 12)
    assert np.array_equal(zero, two)
    assert not np.array_equal(zero, base.out)


def test_combine_order_of_tokens_is_the_input_order(oracle_lib):
    """Selecting a subset of tokens gives the same rows as the full run."""
    w = wl.WORKLOADS["tiny"]
    inp = wl.make_inputs(w)
    full = oracle.run(w, inp)
    sel = np.array([31, 0, 17, 5], np.int64)
    part = oracle.run(w, inp, sel)
    assert np.array_equal(part.out, full.out[sel])


# --- quantise-on-dispatch (bf16 rows to E4M3 + 128-element scales) --------------

def _e4m3_torch(vals32):
    return torch.from_numpy(np.asarray(vals32, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encoder_matches_torch(oracle_lib):
    """Within the finite range, the nearest-even E4M3 code is torch's conversion."""
    rng = np.random.default_rng(21)
    finite = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    finite = finite[np.isfinite(finite)]
    mags = np.unique(np.abs(finite))
    ties = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)           # exact midpoints
    near = np.concatenate([ties * (1 + 2.0 ** -20), ties * (1 - 2.0 ** -20)]).astype(np.float32)
    rand = (rng.standard_normal(20000) * 30).astype(np.float32)
    tiny = (rng.random(2000) * 2.0 ** -6).astype(np.float32)           # the subnormal range
    vals = np.concatenate([finite, ties, -ties, near, rand, tiny, -tiny])
    vals = vals[np.abs(vals) <= 448]
    got = np.array([oracle.e4m3_from_float(float(v)) for v in vals], np.uint8)
    assert np.array_equal(got, _e4m3_torch(vals))


def test_e4m3_encoder_saturates_and_round_trips(oracle_lib):
    for v in (448.0, 449.0, 463.9, 464.0, 470.0, 479.0, 1e6, float("inf")):
        assert oracle.e4m3_from_float(v) == 0x7E
        assert oracle.e4m3_from_float(-v) == 0xFE
    assert oracle.e4m3_from_float(2.0 ** -10) == 0x00     # halfway to the smallest subnormal: to even (0)
    assert oracle.e4m3_from_float(3 * 2.0 ** -10) == 0x02  # halfway between m=1 and m=2: to even
    for code in range(256):
        v = oracle.e4m3_value(code)
        if np.isfinite(v):
            assert oracle.e4m3_from_float(v) == code


def test_quantize_row_properties(oracle_lib):
    rng = np.random.default_rng(8)
    xf = rng.standard_normal(1024).astype(np.float32)
    xf[256:384] = 0.0                                      # an all-zero block
    bits = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q, sc = oracle.quantize_row(bits)
    xv = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert sc[2] == 1.0 and (q[256:384] == 0).all()
    for b in range(8):
        blk = slice(128 * b, 128 * (b + 1))
        amax = np.abs(xv[blk]).max()
        if amax == 0:
            continue
        assert sc[b] == np.float32(amax) / np.float32(448.0)
        # the largest element maps to +-448 exactly
        i = np.abs(xv[blk]).argmax() + 128 * b
        assert (q[i] & 0x7F) == 0x7E
        # each code is the torch conversion of x / scale taken in fp32
        assert np.array_equal(q[blk], _e4m3_torch(xv[blk] / sc[b]))
        deq = torch.from_numpy(q[blk]).view(torch.float8_e4m3fn).double().numpy() * sc[b]
        assert (np.abs(deq - xv[blk]) <= 2 ** -4 * np.abs(xv[blk]) + sc[b] * 2 ** -9).all()


def test_dispatch_quantises_each_token_once(oracle_lib):
    w = wl.WORKLOADS["ds_decode_bf16in"]
    w = wl.custom("q_small", num_ranks=2, tokens_per_rank=6, hidden=256, num_experts=8, topk=3, max_m=6,
                  dtype="bf16q", expert="scale", x_dist="normal")
    inp = wl.make_inputs(w)
    assert inp.x.dtype == np.uint16 and inp.x_scales is None
    _, _, tok_slot = oracle.layout(inp.topk_idx, 8, 6)
    sl = oracle.dispatch(inp.x, None, tok_slot, 8, 6, oracle.BF16_TO_FP8)
    assert sl.rows.shape == (12 * 3, 256) and sl.scales.shape == (12 * 3, 2)
    for i in range(12):
        q, sc = oracle.quantize_row(inp.x.reshape(12, 256)[i])
        for j in range(3):
            assert np.array_equal(sl.rows[i * 3 + j], q) and np.array_equal(sl.scales[i * 3 + j], sc)


# --- receive side: compaction into expert-major buffers ----------------------------

def test_compaction_groups_each_expert_by_source_then_token(oracle_lib):
    """Packed rows of expert e are exactly its tokens, source rank by source rank,
    each source's tokens in increasing order; offsets are the cumulative counts."""
    w = wl.custom("cmp", num_ranks=3, tokens_per_rank=20, hidden=64, num_experts=6, topk=2, max_m=20)
    inp = wl.make_inputs(w, seed=4)
    counts, _, tok_slot = oracle.layout(inp.topk_idx, 6, 20)
    off = oracle.region_offsets(counts, 20)
    assert np.array_equal(off[1:], np.cumsum(counts.ravel()))             # counts in (expert, source) order
    sl = oracle.dispatch(inp.x, None, tok_slot, 6, 20, oracle.BF16)
    pk = oracle.compact(sl, off, 3, 6, 20, 3 * 20 * 2)
    rows = inp.x.reshape(60, -1).view(np.uint8)
    p = 0
    for e in range(6):                                                      # brute force enumeration
        for src in range(3):
            for t in range(20):
                if e in inp.topk_idx[src, t]:
                    j = list(inp.topk_idx[src, t]).index(e)
                    assert list(pk.meta[p]) == [src, t, e, j]
                    assert np.array_equal(pk.rows[p], rows[src * 20 + t])
                    p += 1
    assert p == 120


# --- the expert stage: SwiGLU MLP of one row ------------------------------------

def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _val(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_expert_mlp_row_matches_a_library_matmul(oracle_lib):
    """h and y agree with numpy's fp64 matmuls and torch's silu, with the same two bf16 roundings."""
    rng = np.random.default_rng(30)
    H, I = 64, 96
    x = _bf16(rng.standard_normal(H))
    wg, wu, wd = (_bf16(rng.standard_normal(sh) * 0.1) for sh in ((I, H), (I, H), (H, I)))
    h, y = oracle.expert_mlp_row(x, wg, wu, wd)
    g = _val(wg).reshape(I, H) @ _val(x)
    u = _val(wu).reshape(I, H) @ _val(x)
    hf = torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u
    hb = torch.from_numpy(hf.astype(np.float32)).to(torch.bfloat16).double().numpy()   # float32 first: see below
    # the oracle rounds the fp64 value once; compare values, allowing the float32 step of the library route
    assert (np.abs(_val(h) - hf) <= np.abs(hf) * 2.0 ** -8 * 1.0001).all()
    assert (np.abs(_val(h) - hb) <= np.abs(hb) * 2.0 ** -7).all()
    yf = _val(wd).reshape(H, I) @ _val(h)
    assert (np.abs(_val(y) - yf) <= np.abs(yf) * 2.0 ** -8 * 1.0001).all()


def test_expert_mlp_row_is_zero_for_zero_gate(oracle_lib):
    """silu(0) = 0: a zero gate weight matrix gives h = 0 and y = 0 exactly."""
    rng = np.random.default_rng(31)
    H, I = 32, 48
    x = _bf16(rng.standard_normal(H))
    h, y = oracle.expert_mlp_row(x, np.zeros((I, H), np.uint16), _bf16(rng.standard_normal((I, H))),
                                 _bf16(rng.standard_normal((H, I))))
    assert ((h & 0x7FFF) == 0).all()                     # silu(0) * u is -0 where u < 0
    assert ((y & 0x7FFF) == 0).all()


def test_linear_row_matches_a_library_matmul_and_an_identity(oracle_lib):
    """y = x W^T within one bf16 rounding of numpy's fp64 product; the identity matrix returns x."""
    rng = np.random.default_rng(32)
    K, N = 80, 48
    x = _bf16(rng.standard_normal(K))
    w = _bf16(rng.standard_normal((N, K)) * 0.1)
    y = oracle.linear_row(x, w)
    yf = _val(w).reshape(N, K) @ _val(x)
    assert (np.abs(_val(y) - yf) <= np.abs(yf) * 2.0 ** -8 * 1.0001).all()
    eye = _bf16(np.eye(K))
    assert (oracle.linear_row(x, eye) == x).all()
    # a permutation matrix permutes
    perm = rng.permutation(K)
    assert (oracle.linear_row(x, _bf16(np.eye(K)[perm])) == x[perm]).all()


# --- the fp8 expert stage ------------------------------------------------------

def _e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def _fp8_case(rng, K, N):
    xq = rng.integers(0, 256, K, dtype=np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0x38                           # no NaN codes
    wq = rng.integers(0, 256, (N, K), dtype=np.uint8)
    wq[(wq & 0x7F) == 0x7F] = 0x30
    xs = rng.uniform(0.5, 2.0, K // 128).astype(np.float32) * 2.0 ** -6
    ws = rng.uniform(0.5, 2.0, (N // 128, K // 128)).astype(np.float32) * 2.0 ** -7
    return xq, xs, wq, ws


def _dequant_rows(wq, ws):
    N, K = wq.shape
    return _e4m3(wq) * np.repeat(np.repeat(ws.astype(np.float64), 128, 0), 128, 1)[:N, :K]


def test_linear_row_fp8_matches_a_library_matmul(oracle_lib):
    """y = bf16((x * xs) . (w * ws)) within one bf16 rounding of numpy's fp64 product over
    torch's e4m3 decode; block scales indexed [n / 128][k / 128]."""
    rng = np.random.default_rng(40)
    K, N = 256, 384
    xq, xs, wq, ws = _fp8_case(rng, K, N)
    y = oracle.linear_row_fp8(xq, xs, wq, ws)
    x = _e4m3(xq) * np.repeat(xs.astype(np.float64), 128)
    yf = _dequant_rows(wq, ws) @ x
    assert (np.abs(_val(y) - yf) <= np.abs(yf) * 2.0 ** -8 * 1.0001).all()


def test_linear_row_fp8_unit_scales_identity(oracle_lib):
    """Identity codes (1.0 = 0x38) with unit scales return the row's values, rounded to bf16 (exact for e4m3)."""
    rng = np.random.default_rng(41)
    K = 256
    xq = rng.integers(0, 256, K, dtype=np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0
    wq = np.where(np.eye(K, dtype=bool), np.uint8(0x38), np.uint8(0)).astype(np.uint8)
    y = oracle.linear_row_fp8(xq, np.ones(K // 128, np.float32), wq, np.ones((K // 128, K // 128), np.float32))
    x = _e4m3(xq)
    assert np.array_equal(_val(y), x)      # every e4m3 value is a bf16 value (signed zeros compare equal)


def test_gate_up_row_fp8_matches_library_ops(oracle_lib):
    """hv = silu(g) u from numpy fp64 products and torch's silu; the h codes equal torch's
    float8_e4m3fn cast of fp32(hv) / (amax / 448) in fp32, per 128-block."""
    rng = np.random.default_rng(42)
    H, I = 256, 384
    xq, xs, wgq, wgs = _fp8_case(rng, H, I)
    _, _, wuq, wus = _fp8_case(rng, H, I)
    hv, hq, hs = oracle.gate_up_row_fp8(xq, xs, wgq, wgs, wuq, wus)
    x = _e4m3(xq) * np.repeat(xs.astype(np.float64), 128)
    g, u = _dequant_rows(wgq, wgs) @ x, _dequant_rows(wuq, wus) @ x
    want = torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u
    assert np.allclose(hv, want, rtol=1e-12, atol=1e-300)
    hf = torch.from_numpy(hv.astype(np.float32)).view(I // 128, 128)
    amax = hf.abs().amax(dim=1)
    sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    assert np.array_equal(hs, sc.numpy())
    codes = (hf / sc[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy().ravel()
    assert np.array_equal(hq, codes)


# --- masked choices (expert -1) --------------------------------------------------

@pytest.mark.parametrize("R,T,E,k,max_m,seed", [(2, 16, 8, 2, 16, 5), (3, 33, 16, 8, 40, 6)])
def test_layout_with_masked_choices_matches_brute_force(oracle_lib, R, T, E, k, max_m, seed):
    """A masked choice gets no slot and is not counted; the others keep token order."""
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(R * T)]).astype(np.int32).reshape(R, T, k)
    idx[rng.random(idx.shape) < 0.3] = -1
    idx[:, 0, :] = -1                                   # a token with every choice masked
    counts, flags, tok_slot = oracle.layout(idx, E, max_m)
    bc, bs = _brute_layout(idx, E, max_m)
    assert np.array_equal(counts, bc) and np.array_equal(tok_slot, bs)
    assert (tok_slot[idx == -1] == -1).all()
    assert counts.sum() == int((idx >= 0).sum())


def test_combine_with_masked_choices_sums_only_the_others(oracle_lib):
    """Identity experts: out = bf16(x * sum of the unmasked weights); a token with
    every choice masked is exactly +0."""
    w = wl.WORKLOADS["tiny"]
    inp = wl.mask_choices(wl.make_inputs(w), 0.3)
    ref = oracle.run(w, inp)
    x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).double().numpy().reshape(-1, w.hidden)
    wsum = np.where(inp.topk_idx >= 0, inp.topk_weights.astype(np.float64), 0.0).reshape(-1, w.topk).sum(axis=1)
    got = torch.from_numpy(ref.out.view(np.int16)).view(torch.bfloat16).double().numpy().reshape(-1, w.hidden)
    want = x * wsum[:, None]
    assert (np.abs(got - want) <= np.abs(want) * 2.0 ** -8 * 1.0001).all()
    dead = (inp.topk_idx.reshape(-1, w.topk) < 0).all(axis=1)
    assert dead.any()
    assert (ref.out.reshape(-1, w.hidden)[dead] == 0).all()   # +0 bits
    # the masked choices send nothing: one slot per unmasked choice
    assert ref.slots.slot_id.size == int((inp.topk_idx >= 0).sum())


def test_route_stats_skip_masked_choices(oracle_lib):
    """Counting with masked choices equals counting the same routing with those choices removed."""
    rng = np.random.default_rng(7)
    R, T, E, k, per_node = 8, 64, 64, 4, 2
    idx = np.stack([rng.permutation(E)[:k] for _ in range(R * T)]).astype(np.int32).reshape(R, T, k)
    idx[rng.random(idx.shape) < 0.25] = -1
    got = oracle.route_stats(idx, E, per_node)
    L = E // R
    want = np.zeros((R, 4), np.int64)
    for src in range(R):
        want[src, 0] = T
        for t in range(T):
            ranks = [e // L for e in idx[src, t] if e >= 0]
            off = [r for r in ranks if r // per_node != src // per_node]
            want[src, 1] += len(off)
            want[src, 2] += len(set(off))
            want[src, 3] += len({r // per_node for r in off})
    assert np.array_equal(got, want)
