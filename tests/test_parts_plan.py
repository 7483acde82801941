"""The receive side split into parts, planned on the host by two processes (gloo,
no GPU): each process plays one GPU of an EP group holding one part, computes
from the shared routing which entries it receives, at which local slots, and
which count + 1 flags it waits on; rank 0 gathers the plans and checks them
against the oracle's layout: every entry lands in exactly one part at its
global slot, the parts' flags are disjoint and cover every region, and each
region's entries in its part are exactly its count.
"""
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    from combine_moe_layout_gb300 import workloads as wl
    w = wl.custom("plan", num_ranks=4, tokens_per_rank=96, hidden=128, num_experts=16, topk=4, max_m=96)
    inp = wl.mask_choices(wl.make_inputs(w, seed=5), 0.2, seed=6)
    return w, inp


def _worker(rank, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(WORLD), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    import torch.distributed as dist

    import oracle
    from combine_moe_layout_gb300 import parts

    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    w, inp = _case()
    _, _, tok_slot = oracle.layout(inp.topk_idx, w.num_experts, w.max_m)
    plan = parts.receive_plan(tok_slot, w.num_experts, w.max_m, WORLD, rank)
    got = [None] * WORLD
    dist.all_gather_object(got, (plan.entries.tolist(), plan.local_slots.tolist(), plan.regions.tolist()))
    dist.destroy_process_group()
    q.put((rank, got))


def test_receive_plans_of_two_parts_cover_every_entry_once():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in range(WORLD))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0

    sys.path.insert(0, ROOT)
    import oracle
    from combine_moe_layout_gb300 import parts
    w, inp = _case()
    counts, _, tok_slot = oracle.layout(inp.topk_idx, w.num_experts, w.max_m)
    plans = res[0]
    assert plans == res[1], "every rank gathered the same plans"
    P = parts.slots_per_part(w.num_ranks, w.num_experts, w.max_m, WORLD)
    seen = {}
    all_regions = []
    for g, (entries, local, regions) in enumerate(plans):
        local = np.asarray(local, dtype=np.int64)
        assert local.size == np.unique(local).size and (local >= 0).all() and (local < P).all()
        all_regions += regions
        per_region = np.zeros(w.num_experts * w.num_ranks, dtype=np.int64)
        for (src, t, j), l in zip(entries, local.tolist()):
            key = (src, t, j)
            assert key not in seen, f"{key} received twice"
            seen[key] = g
            s = int(tok_slot[src, t, j])
            assert s == g * P + l, "the local slot is the global slot's place in its part"
            assert s // w.max_m in regions, "an entry's flag lives in its own part"
            per_region[s // w.max_m] += 1
        assert (per_region[regions] == counts.reshape(-1)[regions]).all()
    assert sorted(all_regions) == list(range(w.num_experts * w.num_ranks)), "flags split without overlap"
    valid = {(s, t, j) for s, t, j in zip(*np.nonzero(tok_slot >= 0))}
    assert set(seen) == valid, "every routed entry lands in exactly one part; masked ones in none"
    assert len(valid) < tok_slot.size, "the case includes masked choices"


def test_part_rule_on_the_host():
    """The host rule, single process: the parts must divide the ranks; part g holds global slots
    [g P, (g + 1) P) at local slot s - g P; G = 1 is the whole buffer; every plan's entries and local slots
    agree with the rule, and the union of the G plans is every routed entry exactly once."""
    import pytest
    sys.path.insert(0, ROOT)
    import oracle
    from combine_moe_layout_gb300 import parts

    with pytest.raises(ValueError):
        parts.slots_per_part(4, 16, 8, 3)
    with pytest.raises(ValueError):
        parts.slots_per_part(4, 16, 8, 0)
    assert parts.slots_per_part(4, 16, 8, 1) == 16 * 4 * 8
    g, loc = parts.part_of_slot(np.array([0, 127, 128, 511]), 128)
    assert g.tolist() == [0, 0, 1, 3] and loc.tolist() == [0, 127, 0, 127]
    w, inp = _case()
    _, _, tok_slot = oracle.layout(inp.topk_idx, w.num_experts, w.max_m)
    for G in (1, 2, 4):
        P = parts.slots_per_part(w.num_ranks, w.num_experts, w.max_m, G)
        seen = 0
        for g in range(G):
            plan = parts.receive_plan(tok_slot, w.num_experts, w.max_m, G, g)
            src, t, j = plan.entries.T
            s = tok_slot[src, t, j].astype(np.int64)
            assert (s // P == g).all() and np.array_equal(s % P, plan.local_slots)
            assert plan.regions.size == w.num_experts * w.num_ranks // G
            seen += plan.entries.shape[0]
        assert seen == int((tok_slot >= 0).sum())
