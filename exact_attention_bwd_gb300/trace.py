"""Per-role event traces of the trace build (FA_TRACE=1; csrc/trace.cuh): reading and summary.

In a trace build the first CTAS CTAs of a tensor-core launch record, per role (0 the TMA
producer, 1 the MMA issuer, 2 and 3 the compute warp groups: the softmax groups of the
forward's two query tiles, or the backward's first compute group and its dQ group), a
sequence of (time, event, argument) records: the start of a work item, the two ends of
every wait on a named barrier, and marks.  The records sit at the end of the call's
workspace (the planner appends the region), zeroed by the call before the launch.

    import os; os.environ["FA_TRACE"] = "1"        # before the binding loads the library
    o, lse, ws = binding.forward(q, k, v, ...)
    recs = trace.read(ws, binding.fa_fwd_workspace_size(params))
    print(trace.format_summary(trace.summarise(recs), "fwd"))
"""
from __future__ import annotations

import collections

import numpy as np

CTAS, ROLES, SLOTS = 16, 4, 8192
REGION_BYTES = CTAS * ROLES * SLOTS * 16

EV_ITEM, EV_WAIT, EV_GOT, EV_MARK = 1, 2, 3, 4
BARRIERS = ["q_full", "q_empty", "k_full", "k_empty", "v_full", "v_empty", "s_full", "p_full", "o_full", "o_free",
            "do_full", "do_empty", "kv_full", "dp_full", "ds_full", "ds_free", "dq_full", "dq_free", "dkv_full",
            "q_tmem", "pv_done", "pds_full", "pds_free", "dkv_free"]
MARKS = ["issue_s", "issue_pv", "issue_dp", "issue_dv", "issue_dq", "issue_dk", "softmax_done", "epilogue",
         "epilogue_done", "dq_reduced", "step_done"]
ROLE_NAMES = {"fwd": ["producer", "mma", "softmax tile 0", "softmax tile 1"],
              "bwd": ["producer", "mma", "compute group 0", "dq group"]}


def barrier_name(i: int) -> str:
    return BARRIERS[i - 1] if 1 <= i <= len(BARRIERS) else f"barrier{i}"


def mark_name(i: int) -> str:
    return MARKS[i - 1] if 1 <= i <= len(MARKS) else f"mark{i}"


def parse(region: np.ndarray) -> dict:
    """{(cta, role): [(t_ns, event, argument), ...]} from the raw trace region (uint64 words
    or bytes); a role's records end at the first zero timestamp."""
    words = np.ascontiguousarray(region).view(np.uint64).reshape(CTAS, ROLES, SLOTS, 2)
    out = {}
    for c in range(CTAS):
        for r in range(ROLES):
            w = words[c, r]
            n = int(np.argmax(w[:, 0] == 0)) if np.any(w[:, 0] == 0) else SLOTS
            if n == 0:
                continue
            t = w[:n, 0].astype(np.int64)
            ev = (w[:n, 1] >> np.uint64(32)).astype(np.int64)
            arg = (w[:n, 1] & np.uint64(0xFFFFFFFF)).astype(np.int64)
            out[(c, r)] = list(zip(t.tolist(), ev.tolist(), arg.tolist()))
    return out


def read(workspace, ws_size: int) -> dict:
    """Records of a finished call from its workspace tensor (the device is synchronised by
    the copy); ws_size is the fa_*_workspace_size of the call's parameters."""
    raw = workspace[ws_size - REGION_BYTES:ws_size].cpu().numpy()
    return parse(raw)


def summarise(recs: dict) -> dict:
    """Per role, over the recording CTAs: total span, time waiting per barrier, the number
    of work items and marks, and the first-to-last span of each CTA."""
    roles = collections.defaultdict(lambda: dict(span=0, waits=collections.Counter(), n_waits=collections.Counter(),
                                                  items=0, marks=collections.Counter(), ctas=0))
    for (cta, role), rs in recs.items():
        r = roles[role]
        r["ctas"] += 1
        r["span"] += rs[-1][0] - rs[0][0]
        open_wait = {}
        for t, ev, arg in rs:
            if ev == EV_ITEM:
                r["items"] += 1
            elif ev == EV_WAIT:
                open_wait[arg] = t
            elif ev == EV_GOT and arg in open_wait:
                r["waits"][barrier_name(arg)] += t - open_wait.pop(arg)
                r["n_waits"][barrier_name(arg)] += 1
            elif ev == EV_MARK:
                r["marks"][mark_name(arg)] += 1
    return dict(roles)


def format_summary(summ: dict, kind: str = "fwd") -> str:
    names = ROLE_NAMES.get(kind, [f"role{i}" for i in range(ROLES)])
    lines = []
    for role in sorted(summ):
        r = summ[role]
        span = max(r["span"], 1)
        waited = sum(r["waits"].values())
        parts = ", ".join(f"{b} {100.0 * v / span:.1f}% ({r['n_waits'][b]})" for b, v in r["waits"].most_common())
        lines.append(f"{names[role] if role < len(names) else role}: {r['ctas']} CTAs, span {span / 1e3:.1f} us, "
                     f"items {r['items']}, waiting {100.0 * waited / span:.1f}%: {parts}")
    return "\n".join(lines)
