"""The trace reader (exact_attention_bwd_gb300/trace.py) on synthetic records: layout of
the region, the end of a role's records, wait pairing and the per-role summary."""
import numpy as np

from exact_attention_bwd_gb300 import trace


def _region(recs):
    """recs: {(cta, role): [(t, event, arg), ...]} -> raw uint64 region."""
    w = np.zeros((trace.CTAS, trace.ROLES, trace.SLOTS, 2), np.uint64)
    for (c, r), rs in recs.items():
        for n, (t, ev, arg) in enumerate(rs):
            w[c, r, n, 0] = t
            w[c, r, n, 1] = (ev << 32) | arg
    return w.reshape(-1)


def test_parse_and_summarise():
    b_sfull = trace.BARRIERS.index("s_full") + 1
    b_ofull = trace.BARRIERS.index("o_full") + 1
    recs = {
        (0, 2): [(1000, trace.EV_ITEM, 5), (1100, trace.EV_WAIT, b_sfull), (1400, trace.EV_GOT, b_sfull),
                 (1500, trace.EV_MARK, trace.MARKS.index("softmax_done") + 1), (1600, trace.EV_WAIT, b_ofull),
                 (1700, trace.EV_GOT, b_ofull), (2000, trace.EV_ITEM, 9)],
        (3, 1): [(50, trace.EV_ITEM, 1), (60, trace.EV_WAIT, 1), (90, trace.EV_GOT, 1)],
    }
    region = _region(recs)
    assert region.nbytes == trace.REGION_BYTES
    got = trace.parse(region)
    assert set(got) == {(0, 2), (3, 1)}
    assert got[(0, 2)][0] == (1000, trace.EV_ITEM, 5)
    assert len(got[(0, 2)]) == 7                     # records end at the first zero stamp
    summ = trace.summarise(got)
    r2 = summ[2]
    assert r2["span"] == 1000 and r2["items"] == 2 and r2["ctas"] == 1
    assert r2["waits"]["s_full"] == 300 and r2["waits"]["o_full"] == 100
    assert r2["marks"]["softmax_done"] == 1
    assert summ[1]["waits"]["q_full"] == 30
    text = trace.format_summary(summ, "fwd")
    assert "softmax tile 0" in text and "s_full 30.0%" in text


def test_names_match_the_device_enums():
    """The name tables follow the enum order of csrc/trace.cuh (values from 1)."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(trace.__file__), "csrc", "trace.cuh")).read()
    bar = re.search(r"enum TraceBarrier : uint32_t \{(.*?)\};", src, re.S).group(1)
    names = [re.sub(r"=.*", "", x).strip() for x in bar.replace("\n", " ").split(",") if x.strip()]
    assert len(names) == len(trace.BARRIERS)
    for n, py in zip(names, trace.BARRIERS):
        assert n[2:].lower() == py.replace("_", ""), (n, py)
    mk = re.search(r"enum TraceMark : uint32_t \{(.*?)\};", src, re.S).group(1)
    marks = [re.sub(r"=.*", "", x).strip() for x in mk.replace("\n", " ").split(",") if x.strip()]
    assert len(marks) == len(trace.MARKS)
    for n, py in zip(marks, trace.MARKS):
        assert n[2:].lower() == py.replace("_", ""), (n, py)
