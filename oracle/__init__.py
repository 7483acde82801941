"""CPU oracle for MoE expert-parallel dispatch and combine.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm may
import this package. The library in ``combine_moe_layout_gb300`` never does,
and the two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain single-threaded C, fp64); this
module only compiles it with gcc and marshals numpy arrays. Each wrapper names
the passage its C routine follows:

* "How GPUs Talk to Each Other During LLM Inference", section 7 (Expert
  Parallelism): dispatch sends a token to the ranks of its k experts; combine
  sums the router-weighted expert outputs at the token's home.
* Perplexity, "Efficient and portable mixture-of-experts communication",
  sections Portable kernels / Dispatch / Combine: count + 1 signals, private
  per-(expert, sender) regions, back-indices, weighted sum at the receiver.
* "NVSHMEM and DeepEP: GPU-initiated communication", low-latency section and
  Exercise 2: fixed slots per (local expert, source rank), the per-slot message
  of hidden + hidden/128*4 + 16 bytes, FP8 dispatch with 128-element scales,
  BF16 combine.

Parity of ``expert_stub`` is not a property of the pages (it is the synthetic
expert of the workloads); it is pinned by a nearest-bf16 property test.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_STAMP = os.path.join(_LIBDIR, "liboracle.stamp")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]

OK, EINVAL, EOVERFLOW = 0, -1, -2
BF16, FP8_E4M3, BF16_TO_FP8 = 0, 1, 2

_lib = None


def _source_hash() -> str:
    h = hashlib.sha256()
    with open(_SRC, "rb") as f:
        h.update(f.read())
    h.update(" ".join(_CFLAGS).encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_lib/liboracle.so (cached by source hash)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    want = _source_hash()
    if not force and os.path.exists(_LIB) and os.path.exists(_STAMP):
        with open(_STAMP) as f:
            if f.read().strip() == want:
                return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    with open(_STAMP, "w") as f:
        f.write(want)
    return _LIB


def _bind(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i32, i64, vp, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
    lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_value.restype = dbl
    lib.orc_bf16_from_double.argtypes = [dbl]
    lib.orc_bf16_from_double.restype = ctypes.c_uint16
    lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_value.restype = dbl
    lib.orc_e4m3_from_float.argtypes = [ctypes.c_float]
    lib.orc_e4m3_from_float.restype = ctypes.c_uint8
    lib.orc_quantize_row.argtypes = [vp, i32, vp, vp]
    lib.orc_quantize_row.restype = None
    lib.orc_region_offsets.argtypes = [i32, i32, i32, vp, vp]
    lib.orc_region_offsets.restype = i32
    lib.orc_compact.argtypes = [i32, i32, i32, i64, i32, vp, i64, vp, vp, vp, vp, i64, vp, vp, vp]
    lib.orc_compact.restype = i32
    lib.orc_route_stats.argtypes = [i32] * 5 + [vp, vp]
    lib.orc_route_stats.restype = i32
    lib.orc_expert_mlp_row.argtypes = [i32, i32] + [vp] * 6
    lib.orc_expert_mlp_row.restype = None
    lib.orc_linear_row.argtypes = [i32, i32, vp, vp, vp]
    lib.orc_linear_row.restype = None
    lib.orc_linear_row_fp8.argtypes = [i32, i32] + [vp] * 5
    lib.orc_linear_row_fp8.restype = None
    lib.orc_gate_up_row_fp8.argtypes = [i32, i32] + [vp] * 9
    lib.orc_gate_up_row_fp8.restype = None
    lib.orc_validate.argtypes = [i32] * 7
    lib.orc_validate.restype = i32
    lib.orc_buffer_sizes.argtypes = [i32] * 7 + [vp]
    lib.orc_buffer_sizes.restype = i32
    lib.orc_layout.argtypes = [i32] * 5 + [vp] * 4
    lib.orc_layout.restype = i32
    lib.orc_dispatch.argtypes = [i32] * 7 + [vp] * 3 + [i64] + [vp] * 5
    lib.orc_dispatch.restype = i32
    lib.orc_expert_stub.argtypes = [i32] * 5 + [i64] + [vp] * 4
    lib.orc_expert_stub.restype = i32
    lib.orc_combine.argtypes = [i32] * 6 + [i64] + [vp] * 3 + [i64] + [vp] * 3
    lib.orc_combine.restype = i32
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def compile_variant(source: str, out_path: str) -> str:
    """Compile another copy of the oracle source with the same flags (used by the
    tests that plant mistakes in the oracle to show the pins catch them)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source)
    subprocess.run(["gcc", *_CFLAGS, "-o", out_path, src, "-lm"], check=True)
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


def _check(code: int, what: str):
    if code != OK:
        raise OracleError(code, what)


# --- number formats ---------------------------------------------------------

def bf16_value(bits: int) -> float:
    return _load().orc_bf16_value(int(bits))


def bf16_from_double(v: float) -> int:
    return int(_load().orc_bf16_from_double(float(v)))


def e4m3_value(code: int) -> float:
    return _load().orc_e4m3_value(int(code))


def e4m3_from_float(v: float) -> int:
    return int(_load().orc_e4m3_from_float(float(v)))


def quantize_row(x_bits: np.ndarray):
    """E4M3 codes and 128-element fp32 scales of one bf16 row (uint16 bits)."""
    xb = np.ascontiguousarray(x_bits, dtype=np.uint16)
    H = xb.size
    q = np.zeros(H, np.uint8)
    sc = np.zeros(H // 128, np.float32)
    _load().orc_quantize_row(_p(xb), H, _p(q), _p(sc))
    return q, sc


# --- problem description ----------------------------------------------------

def validate(R, T, H, E, k, max_m, dtype) -> int:
    return int(_load().orc_validate(R, T, H, E, k, max_m, dtype))


SIZE_NAMES = ("recv_x", "recv_scales", "recv_meta", "counts", "flags", "tok_slot", "expert_out")


def buffer_sizes(R, T, H, E, k, max_m, dtype) -> dict:
    """Bytes of every buffer for all R logical ranks (the [NVDE] receive-buffer estimate)."""
    out = np.zeros(7, dtype=np.int64)
    _check(_load().orc_buffer_sizes(R, T, H, E, k, max_m, dtype, _p(out)), "buffer_sizes")
    return dict(zip(SIZE_NAMES, (int(v) for v in out)))


# --- the path -----------------------------------------------------------------

def layout(topk_idx: np.ndarray, num_experts: int, max_m: int):
    """Counts [E][R], count+1 flags [E][R] and slot ids [R][T][k] (sequential definition)."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    R, T, k = idx.shape
    counts = np.zeros((num_experts, R), dtype=np.int32)
    flags = np.zeros((num_experts, R), dtype=np.uint64)
    tok_slot = np.full((R, T, k), -1, dtype=np.int32)
    _check(_load().orc_layout(R, T, num_experts, k, max_m, _p(idx), _p(counts), _p(flags), _p(tok_slot)),
           "layout")
    return counts, flags, tok_slot


@dataclass
class SparseSlots:
    """The filled part of the fixed-slot buffer, one entry per (selected token, choice j)."""
    slot_id: np.ndarray   # [n*k] int64
    rows: np.ndarray      # [n*k, row_bytes] uint8
    scales: np.ndarray    # [n*k, H/128] float32 (empty for bf16)
    meta: np.ndarray      # [n*k, 4] int32: source rank, token, expert, choice


def dispatch(x: np.ndarray, x_scales, tok_slot: np.ndarray, num_experts: int, max_m: int,
             dtype: int, sel: np.ndarray | None = None) -> SparseSlots:
    """Slots written for the selected tokens (flat ids src*T+t; all tokens when None)."""
    R, T, k = tok_slot.shape
    H = x.shape[-1]  # x is [R][T][H] of uint8 codes (fp8) or uint16 bits (bf16)
    row_bytes = 2 * H if dtype == BF16 else H  # bytes of a dispatched row
    in_row_bytes = H if dtype == FP8_E4M3 else 2 * H
    xb = np.ascontiguousarray(x).view(np.uint8).reshape(R * T, in_row_bytes)
    nsc = 0 if dtype == BF16 else H // 128
    sc = None
    if dtype == FP8_E4M3:
        sc = np.ascontiguousarray(x_scales, dtype=np.float32).reshape(R * T, nsc)
    if sel is None:
        sel = np.arange(R * T, dtype=np.int64)
    sel = np.ascontiguousarray(sel, dtype=np.int64)
    n = sel.size * k
    out = SparseSlots(np.zeros(n, np.int64), np.zeros((n, row_bytes), np.uint8),
                      np.zeros((n, nsc), np.float32), np.zeros((n, 4), np.int32))
    ts = np.ascontiguousarray(tok_slot, dtype=np.int32)
    _check(_load().orc_dispatch(R, T, H, num_experts, k, max_m, dtype, _p(xb), _p(sc), _p(ts),
                                sel.size, _p(sel), _p(out.slot_id), _p(out.rows), _p(out.scales),
                                _p(out.meta)), "dispatch")
    keep = out.slot_id >= 0                   # masked choices (-1) send nothing
    if not keep.all():
        out = SparseSlots(out.slot_id[keep], out.rows[keep], out.scales[keep], out.meta[keep])
    return out


def expert_stub(slots: SparseSlots, R: int, H: int, num_experts: int, max_m: int, dtype: int) -> np.ndarray:
    """Synthetic expert outputs (bf16 bits) for the given slots."""
    n = slots.slot_id.size
    y = np.zeros((n, H), dtype=np.uint16)
    _check(_load().orc_expert_stub(R, H, num_experts, max_m, dtype, n, _p(slots.slot_id), _p(slots.rows),
                                   _p(slots.scales), _p(y)), "expert_stub")
    return y


def combine(tok_slot: np.ndarray, topk_weights: np.ndarray, slot_id: np.ndarray, y: np.ndarray,
            num_experts: int, max_m: int, sel: np.ndarray | None = None) -> np.ndarray:
    """bf16 bits [n_sel, H] of sum_j w_j * Y[tok_slot[tok][j]] for the selected tokens."""
    R, T, k = tok_slot.shape
    H = y.shape[1]
    if sel is None:
        sel = np.arange(R * T, dtype=np.int64)
    sel = np.ascontiguousarray(sel, dtype=np.int64)
    out = np.zeros((sel.size, H), dtype=np.uint16)
    ts = np.ascontiguousarray(tok_slot, dtype=np.int32)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    sid = np.ascontiguousarray(slot_id, dtype=np.int64)
    yy = np.ascontiguousarray(y, dtype=np.uint16)
    _check(_load().orc_combine(R, T, H, num_experts, k, max_m, sel.size, _p(sel), _p(ts), _p(w), sid.size,
                               _p(sid), _p(yy), _p(out)), "combine")
    return out


def region_offsets(counts: np.ndarray, max_m: int) -> np.ndarray:
    """Exclusive prefix of the counts in (expert, source rank) order, plus the total: int32 [E*R + 1]."""
    c = np.ascontiguousarray(counts, dtype=np.int32)
    E, R = c.shape
    out = np.zeros(E * R + 1, np.int32)
    _check(_load().orc_region_offsets(R, E, max_m, _p(c), _p(out)), "region_offsets")
    return out


def route_stats(topk_idx: np.ndarray, num_experts: int, ranks_per_node: int) -> np.ndarray:
    """int64 [R][4]: tokens and cross-node copies per expert / per destination rank / per destination node."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    R, T, k = idx.shape
    out = np.zeros((R, 4), np.int64)
    _check(_load().orc_route_stats(R, T, num_experts, k, ranks_per_node, _p(idx), _p(out)), "route_stats")
    return out


def expert_mlp_row(x_bits: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray):
    """bf16 bits of h [I] and y [H] of one row through one expert (SwiGLU MLP, fp64 sums)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    wg = np.ascontiguousarray(w_gate, dtype=np.uint16)
    wu = np.ascontiguousarray(w_up, dtype=np.uint16)
    wd = np.ascontiguousarray(w_down, dtype=np.uint16)
    I, H = wg.shape
    h = np.zeros(I, np.uint16)
    y = np.zeros(H, np.uint16)
    _load().orc_expert_mlp_row(H, I, _p(x), _p(wg), _p(wu), _p(wd), _p(h), _p(y))
    return h, y


def linear_row(x_bits: np.ndarray, w: np.ndarray) -> np.ndarray:
    """bf16 bits of y [N] = x [K] through the bf16 weight matrix w [N][K] (fp64 sum, one rounding)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    wm = np.ascontiguousarray(w, dtype=np.uint16)
    N, K = wm.shape
    y = np.zeros(N, np.uint16)
    _load().orc_linear_row(K, N, _p(x), _p(wm), _p(y))
    return y


def linear_row_fp8(xq: np.ndarray, xs: np.ndarray, wq: np.ndarray, ws: np.ndarray) -> np.ndarray:
    """bf16 bits of y [N] for an fp8 row (codes [K], scales [K/128]) through fp8 weights
    (codes [N][K], block scales [N/128][K/128])."""
    x = np.ascontiguousarray(xq, dtype=np.uint8)
    s = np.ascontiguousarray(xs, dtype=np.float32)
    w = np.ascontiguousarray(wq, dtype=np.uint8)
    sw = np.ascontiguousarray(ws, dtype=np.float32)
    N, K = w.shape
    y = np.zeros(N, np.uint16)
    _load().orc_linear_row_fp8(K, N, _p(x), _p(s), _p(w), _p(sw), _p(y))
    return y


def gate_up_row_fp8(xq, xs, wgq, wgs, wuq, wus):
    """(hv fp64 [I], h codes [I], h scales [I/128]) of linear 1 + SwiGLU for one fp8 row."""
    x = np.ascontiguousarray(xq, dtype=np.uint8)
    s = np.ascontiguousarray(xs, dtype=np.float32)
    wg = np.ascontiguousarray(wgq, dtype=np.uint8)
    sg = np.ascontiguousarray(wgs, dtype=np.float32)
    wu = np.ascontiguousarray(wuq, dtype=np.uint8)
    su = np.ascontiguousarray(wus, dtype=np.float32)
    I, H = wg.shape
    hv = np.zeros(I, np.float64)
    hq = np.zeros(I, np.uint8)
    hs = np.zeros(I // 128, np.float32)
    _load().orc_gate_up_row_fp8(H, I, _p(x), _p(s), _p(wg), _p(sg), _p(wu), _p(su), _p(hv), _p(hq), _p(hs))
    return hv, hq, hs


@dataclass
class Packed:
    rows: np.ndarray     # [n, row_bytes] uint8
    scales: np.ndarray   # [n, H/128] float32
    meta: np.ndarray     # [n, 4] int32


def compact(slots: SparseSlots, offsets: np.ndarray, R: int, E: int, max_m: int, n_packed: int) -> Packed:
    """Packed (expert, source rank, position) rows of the given sparse slots."""
    n = slots.slot_id.size
    rb = slots.rows.shape[1]
    nsc = slots.scales.shape[1]
    out = Packed(np.zeros((n_packed, rb), np.uint8), np.zeros((n_packed, nsc), np.float32),
                 np.zeros((n_packed, 4), np.int32))
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    _check(_load().orc_compact(R, E, max_m, rb, nsc, _p(off), n, _p(slots.slot_id), _p(slots.rows),
                               _p(slots.scales), _p(slots.meta), n_packed, _p(out.rows), _p(out.scales),
                               _p(out.meta)), "compact")
    return out


@dataclass
class OracleResult:
    counts: np.ndarray
    flags: np.ndarray
    tok_slot: np.ndarray
    slots: SparseSlots
    y: np.ndarray
    out: np.ndarray
    sel: np.ndarray


def run(workload, inputs, sel: np.ndarray | None = None) -> OracleResult:
    """Layout (all tokens), then dispatch, synthetic experts and combine for the selected tokens."""
    w = workload
    dt = w.dtype_code
    counts, flags, tok_slot = layout(inputs.topk_idx, w.num_experts, w.max_m)
    if sel is None:
        sel = np.arange(w.num_ranks * w.tokens_per_rank, dtype=np.int64)
    slots = dispatch(inputs.x, inputs.x_scales, tok_slot, w.num_experts, w.max_m, dt, sel)
    y = expert_stub(slots, w.num_ranks, w.hidden, w.num_experts, w.max_m, dt)
    out = combine(tok_slot, inputs.topk_weights, slots.slot_id, y, w.num_experts, w.max_m, sel)
    return OracleResult(counts, flags, tok_slot, slots, y, out, sel)
