"""Seeded synthetic workloads for MoE expert-parallel dispatch and combine.

This module only generates inputs: router choices and weights, token
activations, and the fp8 block quantisation of those activations. It holds none
of the dispatch/combine arithmetic, so the CUDA path and the CPU oracle can both
consume what it makes without sharing any of the method.

The shapes stand in for the models the pages name: DeepSeek-V3 (hidden 7168,
256 experts, top-8, fp8 with one fp32 scale per 128 elements; "NVSHMEM and
DeepEP: GPU-initiated communication", high-throughput and low-latency sections)
and Mixtral 8x7B (8 experts, top-2; Perplexity, "Efficient and portable
mixture-of-experts communication", introduction). No dataset is involved.

Draw order for one workload, from ``numpy.random.default_rng(seed)``: the
routing randomness, then the activations, then (Zipf router only) the weight
logits.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch

E4M3_MAX = 448.0  # largest finite FP8 E4M3 ("e4m3fn") value
SCALE_BLOCK = 128  # elements per fp32 scale


@dataclass(frozen=True)
class Workload:
    name: str
    num_ranks: int          # R logical EP ranks
    tokens_per_rank: int    # T
    hidden: int             # H
    num_experts: int        # E
    topk: int               # k
    max_m: int              # slots per (expert, source rank)
    dtype: str              # "bf16", "fp8", or "bf16q" (bf16 rows quantised to fp8 on dispatch)
    router: str             # "softmax", "zipf" or "group"
    renormalize: bool       # softmax router: renormalise the k weights to sum 1
    expert: str             # "identity" or "scale" (y = x * (1 + e/256))
    x_dist: str             # "uniform" (U(-1,1)) or "normal" (N(0,1))
    seed: int = 0
    intermediate: int = 0   # I of the expert MLP (linear 1: H -> 2I with SwiGLU, linear 2: I -> H)

    @property
    def local_experts(self) -> int:
        return self.num_experts // self.num_ranks

    @property
    def num_tokens(self) -> int:
        return self.num_ranks * self.tokens_per_rank

    @property
    def row_bytes(self) -> int:
        """Bytes of a dispatched row (what a slot holds)."""
        return 2 * self.hidden if self.dtype == "bf16" else self.hidden

    @property
    def in_row_bytes(self) -> int:
        """Bytes of a caller's input row."""
        return self.hidden if self.dtype == "fp8" else 2 * self.hidden

    @property
    def scales_per_row(self) -> int:
        return 0 if self.dtype == "bf16" else self.hidden // SCALE_BLOCK

    @property
    def dtype_code(self) -> int:
        return {"bf16": 0, "fp8": 1, "bf16q": 2}[self.dtype]

    def algorithmic_bytes(self) -> dict:
        """Bytes each step must move at least once (slots never touched are not counted).

        layout: read topk_idx, write tok_slot, write counts and flags.
        dispatch: read every input row (+ its scales) once, write the dispatched
        row (+ scales + 16-byte header) into k slots, read tok_slot.
        combine: read k bf16 expert rows per token, write one bf16 row, read
        weights and tok_slot.
        """
        N, k, H, E, R = self.num_tokens, self.topk, self.hidden, self.num_experts, self.num_ranks
        sc = self.scales_per_row * 4
        lay = N * k * 4 + N * k * 4 + E * R * (4 + 8)
        in_sc = sc if self.dtype == "fp8" else 0
        dis = N * (self.in_row_bytes + in_sc) + N * k * (self.row_bytes + sc + 16) + N * k * 4
        com = N * k * 2 * H + N * 2 * H + N * k * 4 + N * k * 4
        # receive hook: read counts and flags, write the offsets, move each filled slot (row + scales + header)
        # once into its packed row; the packed combine also reads one offset per choice
        rcv = E * R * (4 + 8 + 4) + 2 * N * k * (self.row_bytes + sc + 16)
        return {"layout": lay, "dispatch": dis, "combine": com, "recv": rcv, "combine_packed": com + N * k * 4,
                "total": lay + dis + com, "total_packed": lay + dis + rcv + com + N * k * 4}


# Expert MLP widths I: DeepSeek-V3 experts 2048, Mixtral 8x7B experts 14336 (the
# models' published configurations; the pages give hidden sizes, not these).
WORKLOADS = {
    "tiny": Workload("tiny", 2, 16, 128, 8, 2, 16, "bf16", "softmax", True, "identity", "uniform",
                     intermediate=256),
    "ds_decode": Workload("ds_decode", 8, 128, 7168, 256, 8, 128, "fp8", "softmax", False, "scale", "normal",
                          intermediate=2048),
    "mixtral": Workload("mixtral", 8, 4096, 4096, 8, 2, 4096, "bf16", "softmax", True, "identity", "normal",
                        intermediate=14336),
    "skewed": Workload("skewed", 16, 256, 7168, 256, 8, 256, "bf16", "zipf", True, "identity", "normal",
                       intermediate=2048),
    "ds_prefill": Workload("ds_prefill", 8, 4096, 7168, 256, 8, 4096, "fp8", "group", True, "scale", "normal",
                           intermediate=2048),
    # the Mixtral shape with fp8 rows (the fp8 expert stage at 8192 rows per expert)
    "mixtral_fp8": Workload("mixtral_fp8", 8, 4096, 4096, 8, 2, 4096, "fp8", "softmax", True, "scale", "normal",
                            intermediate=14336),
    # the decode shape with bf16 rows quantised to fp8 + scales on dispatch
    "ds_decode_bf16in": Workload("ds_decode_bf16in", 8, 128, 7168, 256, 8, 128, "bf16q", "softmax", False, "scale",
                                 "normal", intermediate=2048),
}

DESCRIPTIONS = {
    "tiny": "2 ranks x 16 tokens, hidden 128 bf16 U(-1,1), 8 experts, top-2 renormalised softmax, max_m 16",
    "ds_decode": "DeepSeek-shape decode: 8 ranks x 128 tokens, hidden 7168 fp8 e4m3 + 128-elt fp32 scales, "
                 "256 experts, top-8 of softmax, max_m 128",
    "mixtral": "Mixtral-shape prefill: 8 ranks x 4096 tokens, hidden 4096 bf16, 8 experts, top-2 renormalised, "
               "max_m 4096",
    "skewed": "Zipf(1.2) routing: 16 ranks x 256 tokens, hidden 7168 bf16, 256 experts, top-8, max_m 256",
    "ds_prefill": "DeepSeek-shape prefill: 8 ranks x 4096 tokens, hidden 7168 fp8 e4m3 + scales, 256 experts in "
                  "8 groups, top-4 groups then top-8 of sigmoid scores, max_m 4096",
    "mixtral_fp8": "Mixtral-shape prefill with fp8 rows: 8 ranks x 4096 tokens, hidden 4096 e4m3 + 128-elt fp32 "
                   "scales, 8 experts, top-2 renormalised, max_m 4096",
    "ds_decode_bf16in": "DeepSeek-shape decode with bf16 input rows quantised on dispatch to fp8 e4m3 + 128-elt "
                        "fp32 scales: 8 ranks x 128 tokens, hidden 7168, 256 experts, top-8 of softmax, max_m 128",
}


def custom(name="custom", **kw) -> Workload:
    """A workload with the given sizes; defaults are the tiny case."""
    return replace(WORKLOADS["tiny"], name=name, **kw)


@dataclass
class Inputs:
    topk_idx: np.ndarray      # [R][T][k] int32
    topk_weights: np.ndarray  # [R][T][k] float32
    x: np.ndarray             # [R][T][H] uint16 bf16 bits (bf16, bf16q), or uint8 e4m3 codes (fp8)
    x_scales: np.ndarray | None  # [R][T][H/128] float32 (fp8 input only)


# --- routers (input generation only) -----------------------------------------

def _topk_desc(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores per row, largest first; ties go to the lower index."""
    order = np.argsort(-scores, axis=1, kind="stable")
    return order[:, :k]


def _softmax(logits: np.ndarray) -> np.ndarray:
    z = logits.astype(np.float64)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    return p / p.sum(axis=1, keepdims=True)


def route_softmax(rng, n: int, E: int, k: int, renormalize: bool):
    """Top-k of a softmax over N(0,1) router logits; weights are the k probabilities."""
    p = _softmax(rng.standard_normal((n, E), dtype=np.float32))
    idx = _topk_desc(p, k)
    w = np.take_along_axis(p, idx, axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return idx.astype(np.int32), w.astype(np.float32)


def route_zipf_choices(rng, n: int, E: int, k: int, s: float = 1.2) -> np.ndarray:
    """k distinct experts per token drawn without replacement from p(e) ~ (e+1)^-s.

    Sequential draws without replacement with renormalised probabilities have
    the same distribution as the k largest of log p(e) + Gumbel noise
    (the Gumbel-top-k construction), which is what is drawn here. Expert 0 is
    the most popular, so the hot experts all live on rank 0.
    """
    logp = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    g = rng.gumbel(size=(n, E))
    return _topk_desc(logp[None, :] + g, k).astype(np.int32)


def group_limited_choice(scores: np.ndarray, k: int, groups: int, keep_groups: int, per_group_top: int):
    """k best experts among the keep_groups best groups of contiguous experts.

    A group's score is the sum of its per_group_top best expert scores
    (DeepSeek-V3 node-limited routing as "NVSHMEM and DeepEP: GPU-initiated
    communication", high-throughput section, describes it: score each node by its
    top-2 experts, keep 4 nodes, pick 8 experts inside them).
    """
    n, E = scores.shape
    per = scores.reshape(n, groups, E // groups)
    group_score = (-np.sort(-per, axis=2)[:, :, :per_group_top]).sum(axis=2)
    kept = _topk_desc(group_score, keep_groups)
    allowed = np.zeros((n, groups), dtype=bool)
    np.put_along_axis(allowed, kept, True, axis=1)
    masked = np.where(np.repeat(allowed, E // groups, axis=1), scores, -np.inf)
    return _topk_desc(masked, k)


def route_group_limited(rng, n: int, E: int, k: int, groups: int, keep_groups: int, per_group_top: int):
    """Group-limited routing on sigmoid(N(0,1)) scores; weights are the chosen
    scores renormalised to sum 1 (no bias term). Group g = logical rank g."""
    logits = rng.standard_normal((n, E), dtype=np.float32).astype(np.float64)
    scores = 1.0 / (1.0 + np.exp(-logits))
    idx = group_limited_choice(scores, k, groups, keep_groups, per_group_top)
    w = np.take_along_axis(scores, idx, axis=1)
    w = w / w.sum(axis=1, keepdims=True)
    return idx.astype(np.int32), w.astype(np.float32)


# --- activations (input generation only) -------------------------------------

def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def quantize_e4m3_blocks(a: np.ndarray):
    """E4M3 codes and fp32 scales, one scale per 128 contiguous elements of a row.

    scale = amax(block) / 448 (1 for an all-zero block); code = e4m3(x / scale)
    rounded to nearest even and clamped to +-448 (torch's conversion).
    """
    shape = a.shape
    H = shape[-1]
    blocks = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).reshape(-1, H // SCALE_BLOCK, SCALE_BLOCK)
    amax = blocks.abs().amax(dim=2)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (blocks / scale.unsqueeze(2)).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    codes = q.view(torch.uint8).reshape(shape).numpy()
    return codes, scale.reshape(shape[:-1] + (H // SCALE_BLOCK,)).numpy().astype(np.float32)


def make_inputs(w: Workload, seed: int | None = None) -> Inputs:
    rng = np.random.default_rng(w.seed if seed is None else seed)
    R, T, H, E, k = w.num_ranks, w.tokens_per_rank, w.hidden, w.num_experts, w.topk
    n = R * T
    if w.router == "softmax":
        idx, wts = route_softmax(rng, n, E, k, w.renormalize)
    elif w.router == "zipf":
        idx, wts = route_zipf_choices(rng, n, E, k), None
    elif w.router == "group":
        idx, wts = route_group_limited(rng, n, E, k, groups=R, keep_groups=min(4, R),
                                       per_group_top=max(1, k // min(4, R)))
    else:
        raise ValueError(f"unknown router {w.router}")
    if w.x_dist == "uniform":
        xf = rng.uniform(-1.0, 1.0, size=(n, H)).astype(np.float32)
    else:
        xf = rng.standard_normal((n, H), dtype=np.float32)
    if wts is None:  # Zipf router: softmax of N(0,1) logits over the chosen experts
        wts = _softmax(rng.standard_normal((n, k), dtype=np.float32)).astype(np.float32)
    if w.dtype == "fp8":
        x, sc = quantize_e4m3_blocks(xf)
        x = x.reshape(R, T, H)
        sc = sc.reshape(R, T, H // SCALE_BLOCK)
    else:
        x, sc = _to_bf16_bits(xf).reshape(R, T, H), None
    return Inputs(idx.reshape(R, T, k), wts.reshape(R, T, k), x, sc)


def mask_choices(inputs: Inputs, frac: float, seed: int = 1) -> Inputs:
    """A copy of the inputs with about `frac` of the routing choices masked
    (expert -1: the choice names no expert) and, in every rank, every choice of
    about one token in 16 masked."""
    rng = np.random.default_rng(seed)
    idx = inputs.topk_idx.copy()
    idx[rng.random(idx.shape) < frac] = -1
    R, T, k = idx.shape
    if T:
        idx[:, rng.integers(0, T, size=max(1, T // 16)), :] = -1
    return replace(inputs, topk_idx=idx)


# --- expert weights (input generation only) ----------------------------------

@dataclass
class ExpertWeights:
    inter: int
    w_gate: torch.Tensor  # [E][I][H] bf16
    w_up: torch.Tensor    # [E][I][H] bf16
    w_down: torch.Tensor  # [E][H][I] bf16


def expert_weights(w: Workload, device="cpu", seed: int | None = None, inter: int | None = None) -> ExpertWeights:
    """Synthetic bf16 expert weights: N(0, 1/K) entries (K the input width of
    each linear map), drawn with torch's generator on `device` in the order
    gate, up, down. No trained weights are involved."""
    I = w.intermediate if inter is None else inter
    E, H = w.num_experts, w.hidden
    g = torch.Generator(device=device)
    g.manual_seed((w.seed if seed is None else seed) + 7919)

    def draw(shape, fan_in):
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        return t.mul_(fan_in ** -0.5).to(torch.bfloat16)

    return ExpertWeights(I, draw((E, I, H), H), draw((E, I, H), H), draw((E, H, I), I))


@dataclass
class ExpertWeightsFp8:
    inter: int
    w_gate: torch.Tensor         # [E][I][H] uint8 e4m3 codes
    w_gate_scales: torch.Tensor  # [E][I/128][H/128] float32
    w_up: torch.Tensor
    w_up_scales: torch.Tensor
    w_down: torch.Tensor         # [E][H][I] uint8
    w_down_scales: torch.Tensor  # [E][H/128][I/128] float32


def _block_quantize_e4m3(v: torch.Tensor):
    """e4m3 codes and one fp32 scale per 128 x 128 block of [n][N][K] values
    (scale = block amax / 448, 1 for an all-zero block; torch's nearest-even cast)."""
    n, N, K = v.shape
    b = v.view(n, N // 128, 128, K // 128, 128)
    amax = b.abs().amax(dim=(2, 4))
    sc = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (b / sc[:, :, None, :, None]).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).view(n, N, K), sc.float()


def expert_weights_fp8(w: Workload, device="cpu", seed: int | None = None, inter: int | None = None,
                       chunk: int = 16) -> ExpertWeightsFp8:
    """Synthetic fp8 expert weights: N(0, 1/K) draws (torch's generator on
    `device`, gate then up then down, `chunk` experts at a time) block-quantised
    to e4m3 with one fp32 scale per 128 x 128 block."""
    I = w.intermediate if inter is None else inter
    E, H = w.num_experts, w.hidden
    g = torch.Generator(device=device)
    g.manual_seed((w.seed if seed is None else seed) + 104729)

    def draw(N, K):
        q = torch.empty((E, N, K), dtype=torch.uint8, device=device)
        s = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=device)
        for e0 in range(0, E, chunk):
            e1 = min(E, e0 + chunk)
            v = torch.randn((e1 - e0, N, K), generator=g, device=device, dtype=torch.float32).mul_(K ** -0.5)
            q[e0:e1], s[e0:e1] = _block_quantize_e4m3(v)
            del v
        return q, s

    wg, sg = draw(I, H)
    wu, su = draw(I, H)
    wd, sd = draw(H, I)
    return ExpertWeightsFp8(I, wg, sg, wu, su, wd, sd)
