"""The per-task trace's host side (moe_expert_forward_gb300/trace.py): record
layout, decoding of a raw buffer (unwritten slots dropped) and the phase
summary, on hand-made records."""
import numpy as np

from moe_expert_forward_gb300 import trace as TR


def _rec(cta, task, typ, e, n, b, t0, t1, t2, mode=3):
    r = np.zeros(1, dtype=TR.RECORD)
    r["cta"], r["task"], r["type"], r["expert"], r["tile"], r["block"] = cta, task, typ, e, n, b
    r["valid"], r["mode"] = 128, mode
    r["t_issue"], r["t_mma_done"], r["t_epi_done"] = t0, t1, t2
    return r


def test_record_layout_and_decode():
    assert TR.RECORD.itemsize == 64 and TR.buffer_bytes(152, 10, 2) == 64 * 152 * 10 * 2
    buf = np.zeros(4, dtype=TR.RECORD)                 # two CTAs x two slots, one slot unwritten
    buf[0] = _rec(0, 0, 1, 3, 0, 5, 1000, 3000, 4000)[0]
    buf[1] = _rec(0, 1, 2, 3, 1, 5, 5000, 7000, 9000)[0]
    buf[2] = _rec(1, 0, 1, 4, 0, 6, 1500, 2500, 6000)[0]
    raw = np.frombuffer(buf.tobytes(), dtype=np.uint8)
    rec = TR.records(raw)
    assert rec.size == 3 and list(rec["expert"]) == [3, 3, 4]


def test_summary_phases_overlap_and_tail():
    rec = np.concatenate([_rec(0, 0, 1, 3, 0, 5, 1000, 3000, 4000), _rec(0, 1, 2, 3, 1, 5, 5000, 7000, 9000),
                          _rec(1, 0, 1, 4, 0, 6, 1500, 2500, 6000)])
    s = TR.summary(rec)["fused"]
    assert s["tasks"] == 3 and s["span_us"] == 8.0                    # 1000 -> 9000 ns
    assert s["l1"]["tasks"] == 2 and s["l1"]["last_done_us"] == 5.0
    assert s["l2"]["first_issue_us"] == 4.0 and s["l1_l2_overlap_us"] == 1.0
    assert s["l1"]["mean_task_us"] == ((4000 - 1000) + (6000 - 1500)) / 2 / 1e3
    assert s["tail_us"]["max"] == 3.0 and s["tail_us"]["mean"] == 1.5  # CTA 1 ends at 6000, the launch at 9000
    assert TR.summary(rec[:0]) == {}
