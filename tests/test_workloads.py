"""The seeded input generators (runs without a GPU)."""
import json
import os

import numpy as np
import pytest
import torch

from combine_moe_layout_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SMALL = ["tiny", "ds_decode", "skewed"]


@pytest.mark.parametrize("name", SMALL)
def test_shapes_and_routing_validity(name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    R, T, H, E, k = w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk
    assert inp.topk_idx.shape == (R, T, k) and inp.topk_idx.dtype == np.int32
    assert inp.topk_weights.shape == (R, T, k) and inp.topk_weights.dtype == np.float32
    assert inp.x.shape == (R, T, H)
    assert inp.x.dtype == (np.uint8 if w.dtype == "fp8" else np.uint16)
    idx = inp.topk_idx.reshape(-1, k)
    assert (idx >= 0).all() and (idx < E).all()
    srt = np.sort(idx, axis=1)
    assert (np.diff(srt, axis=1) > 0).all(), "a token picks k distinct experts"
    assert (inp.topk_weights > 0).all()
    if w.renormalize or w.router == "zipf":
        assert np.allclose(inp.topk_weights.sum(-1), 1.0, atol=1e-6)


def test_seeded_generation_is_deterministic():
    a = wl.make_inputs(wl.WORKLOADS["ds_decode"])
    b = wl.make_inputs(wl.WORKLOADS["ds_decode"])
    for f in ("topk_idx", "topk_weights", "x", "x_scales"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    c = wl.make_inputs(wl.WORKLOADS["ds_decode"], seed=1)
    assert not np.array_equal(a.topk_idx, c.topk_idx)


def test_fp8_block_quantisation():
    w = wl.WORKLOADS["ds_decode"]
    rng = np.random.default_rng(5)
    xf = rng.standard_normal((64, w.hidden), dtype=np.float32)
    codes, scales = wl.quantize_e4m3_blocks(xf)
    assert codes.dtype == np.uint8 and scales.shape == (64, w.hidden // 128)
    assert not np.isin(codes & 0x7F, [0x7F]).any(), "no NaN codes"
    deq = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy() * np.repeat(scales, 128, axis=1)
    blk_amax = np.abs(xf.reshape(64, -1, 128)).max(-1)
    # each block's largest element maps to +-448 and the rest keep 3 mantissa bits
    assert np.allclose(np.abs(deq.reshape(64, -1, 128)).max(-1), blk_amax, rtol=2 ** -4)
    err = np.abs(deq - xf)
    assert (err <= 2 ** -4 * np.abs(xf) + np.repeat(scales, 128, axis=1) * 2 ** -9).all()


def test_zipf_router_is_skewed_toward_low_experts():
    w = wl.WORKLOADS["skewed"]
    inp = wl.make_inputs(w)
    freq = np.bincount(inp.topk_idx.ravel(), minlength=w.num_experts)
    assert freq.argmax() == 0
    # expert 0 is in nearly every token's top-8; popularity falls with the index
    assert freq[0] > 0.9 * w.num_tokens
    assert freq[:16].sum() > freq[16:64].sum() > freq[192:].sum()


def test_group_router_keeps_four_groups():
    w = wl.WORKLOADS["ds_prefill"]
    rng = np.random.default_rng(0)
    idx, wts = wl.route_group_limited(rng, 2048, w.num_experts, w.topk, groups=8, keep_groups=4,
                                      per_group_top=2)
    groups_per_token = np.array([len(set(r)) for r in (idx // 32)])
    assert groups_per_token.max() <= 4
    assert np.allclose(wts.sum(1), 1.0, atol=1e-6)


def test_group_router_reproduces_the_printed_simulation():
    """The node-limited choice, fed the page's score construction, gives the
    printed nodes per token and cross-node copies per token."""
    g = json.load(open(os.path.join(GOLDEN, "node_limited_routing.json")))
    s = g["setup"]
    nodes, gpn, E, k, keep, tokens = s["nodes"], s["gpus_per_node"], s["experts"], s["topk"], s["max_nodes"], \
        s["tokens"]
    rng = np.random.default_rng(0)
    base = rng.random((tokens, E))
    scores = base + rng.random(E) * 0.5
    per_gpu = E // (nodes * gpn)
    for limited, key in ((False, "unlimited"), (True, "node_limited")):
        if limited:
            idx = wl.group_limited_choice(scores, k, groups=nodes, keep_groups=keep, per_group_top=k // keep)
        else:
            idx = np.argsort(-scores, axis=1)[:, :k]
        gpu = idx // per_gpu
        node = gpu // gpn
        want = g["printed"][key]
        assert f"{np.mean([len(set(r)) for r in node]):.2f}" == want["nodes_per_token"]
        copies = {
            "per_expert": (node != 0).sum(1).mean(),
            "per_gpu_dedup": np.mean([len({x for x in r if x // gpn != 0}) for r in gpu]),
            "per_node_dedup": np.mean([len(set(r) - {0}) for r in node]),
        }
        for name, c in copies.items():
            assert f"{c:.2f}" == want[name], (key, name, c)
            ms = tokens * c * s["token_bytes"] / (s["link_GBps"] * 1e9) * 1e3
            assert f"{ms:.2f}" == want["ms"][name], (key, name, ms)


def test_algorithmic_bytes_of_the_decode_step():
    """Bytes each step must move (read once, write once, untouched slots excluded)."""
    b = wl.WORKLOADS["ds_decode"].algorithmic_bytes()
    N, k, H = 1024, 8, 7168
    row = H + 56 * 4
    assert b["dispatch"] == N * row + N * k * (row + 16) + N * k * 4
    assert b["combine"] == N * k * 2 * H + N * 2 * H + N * k * 8
    assert 195e6 < b["total"] < 205e6


# The per-config algorithmic bytes the step is measured against (MB): layout (bytes), dispatch, combine, total.
# Those count a 4-byte source-token index per slot; the dispatch here writes a 16-byte header {src, t, e, j} per
# slot instead, so its dispatch bytes are 12 bytes per dispatched choice above them.
CONTRACT_BYTES = {
    "tiny": (704, 0.025, 0.025, 0.051),
    "ds_decode": (90112, 68.19, 132.19, 200.47),
    "mixtral": (525056, 805.83, 805.83, 1612.19),
    "skewed": (311296, 528.74, 528.74, 1057.80),
    "ds_prefill": (2121728, 2182.09, 4229.96, 6414.16),
}


@pytest.mark.parametrize("name", list(CONTRACT_BYTES))
def test_algorithmic_bytes_match_the_contract(name):
    w = wl.WORKLOADS[name]
    b = w.algorithmic_bytes()
    lay, dis, com, tot = CONTRACT_BYTES[name]
    header_extra = w.num_tokens * w.topk * 12
    assert b["layout"] == lay
    assert abs(b["combine"] / 1e6 - com) < 0.006
    assert abs((b["dispatch"] - header_extra) / 1e6 - dis) < 0.006
    assert abs((b["total"] - header_extra) / 1e6 - tot) < 0.006


def _page_routing(limited: bool):
    """The page's simulation as a routing of 64 ranks (8 nodes of 8): rank 0 holds the page's 4096 tokens."""
    g = json.load(open(os.path.join(GOLDEN, "node_limited_routing.json")))["setup"]
    nodes, gpn, E, k, keep, tokens = g["nodes"], g["gpus_per_node"], g["experts"], g["topk"], g["max_nodes"], \
        g["tokens"]
    rng = np.random.default_rng(0)
    scores = rng.random((tokens, E)) + rng.random(E) * 0.5
    if limited:
        idx = wl.group_limited_choice(scores, k, groups=nodes, keep_groups=keep, per_group_top=k // keep)
    else:
        idx = np.argsort(-scores, axis=1)[:, :k]
    return idx.astype(np.int32), nodes * gpn, gpn, E, k


@pytest.mark.parametrize("limited,key", [(False, "unlimited"), (True, "node_limited")])
def test_oracle_route_stats_reproduce_the_printed_copies(limited, key):
    """The oracle's per-node deduplication accounting gives the page's copies per token."""
    import oracle
    want = json.load(open(os.path.join(GOLDEN, "node_limited_routing.json")))["printed"][key]
    idx, R, gpn, E, k = _page_routing(limited)
    # a 64-rank job (E/R = 4 experts per rank); rank 0 holds the page's tokens
    full = np.zeros((R, idx.shape[0], k), np.int32)
    full[0] = idx
    full[1:] = idx[None]                                    # other ranks: same choices (only rank 0 is read)
    st = oracle.route_stats(full, E, gpn)[0]
    n = st[0]
    assert f"{st[1] / n:.2f}" == want["per_expert"]
    assert f"{st[2] / n:.2f}" == want["per_gpu_dedup"]
    assert f"{st[3] / n:.2f}" == want["per_node_dedup"]
