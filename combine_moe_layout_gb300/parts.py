"""Host-side plan of a receive side split into parts (numpy only, no GPU).

The EP group's fixed-slot buffers split the way its GPUs would hold them
(Perplexity, "Efficient and portable mixture-of-experts communication",
section "NVSHMEM": every rank owns private receive buffers that senders put
into and signal; include/moe_layout.h, moe_parts): with G parts, part g holds
the regions of ranks [g*R/G, (g+1)*R/G), i.e. global slots [g*P, (g+1)*P) with
P = E*R*max_m / G at local slot s - g*P, and regions [g*E*R/G, (g+1)*E*R/G) of
the count + 1 flags. The plan says, for one part, which (source rank, token,
choice) entries it receives, at which local slots, and which flags it waits on.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def slots_per_part(num_ranks: int, num_experts: int, max_m: int, num_parts: int) -> int:
    if num_parts < 1 or num_ranks % num_parts:
        raise ValueError("the number of parts must divide the number of ranks")
    return num_experts * num_ranks * max_m // num_parts


def part_of_slot(slot, per_part: int):
    """(part, local slot) of global slot ids."""
    slot = np.asarray(slot, dtype=np.int64)
    return slot // per_part, slot % per_part


@dataclass
class ReceivePlan:
    part: int
    entries: np.ndarray      # [n, 3] int64: source rank, token, choice (in that order)
    local_slots: np.ndarray  # [n] int64: where each entry lands in this part
    regions: np.ndarray      # global regions (e*R + src) whose count + 1 flags this part holds


def receive_plan(tok_slot: np.ndarray, num_experts: int, max_m: int, num_parts: int, part: int) -> ReceivePlan:
    """What part `part` receives, from the global slot ids tok_slot [R][T][k]
    (-1: no slot)."""
    R, T, k = tok_slot.shape
    P = slots_per_part(R, num_experts, max_m, num_parts)
    s = tok_slot.reshape(-1).astype(np.int64)
    g, local = part_of_slot(np.where(s >= 0, s, 0), P)
    mine = (s >= 0) & (g == part)
    flat = np.nonzero(mine)[0]
    entries = np.stack([flat // (T * k), (flat // k) % T, flat % k], axis=1)
    per = num_experts * R // num_parts
    return ReceivePlan(part, entries, local[mine], np.arange(part * per, (part + 1) * per, dtype=np.int64))
