"""Host side of the per-task trace (Options.trace_buf in include/mm_moe.h): the
record layout, decoding, and a phase summary: when each phase of the stream
starts and ends, and how long the tasks take.  DeepGEMM PR #440 ("Why the order
and not the pool size, and the lag ladder") reads event traces of an
instrumented build the same way, timing the end of the dispatch pull against the
lag."""
from __future__ import annotations

import numpy as np

# one 64-byte record per task (TraceRec in csrc/internal.h)
RECORD = np.dtype([("cta", "<u4"), ("task", "<u4"), ("type", "<u4"), ("expert", "<u4"), ("tile", "<u4"),
                   ("block", "<u4"), ("valid", "<u4"), ("mode", "<u4"), ("t_issue", "<u8"),
                   ("t_mma_done", "<u8"), ("t_epi_done", "<u8"), ("reserved", "<u8")])
assert RECORD.itemsize == 64


def buffer_bytes(grid: int, tasks_per_cta: int, launches: int = 1) -> int:
    """Bytes of a trace buffer holding `tasks_per_cta` records per CTA and launch."""
    return RECORD.itemsize * grid * tasks_per_cta * launches


def records(raw) -> np.ndarray:
    """The written records of a trace buffer (bytes, a uint8 numpy array or a
    uint8 torch tensor), in buffer order; unwritten slots (type 0) are dropped."""
    if hasattr(raw, "cpu"):
        raw = raw.cpu().numpy()
    a = np.frombuffer(np.ascontiguousarray(raw).tobytes(), dtype=RECORD)
    return a[a["type"] != 0]


def summary(rec: np.ndarray) -> dict:
    """Per task type: count, the first issue and the last completion (µs after
    the launch's first issue), the mean task time from first issue to stored
    output, and the MMA share of it; plus the overlap of the L1 and L2 phases and
    the idle tail (µs from each CTA's last task to the launch's last)."""
    if rec.size == 0:
        return {}
    out = {}
    for mode in np.unique(rec["mode"]):
        r = rec[rec["mode"] == mode]
        t0 = int(r["t_issue"].min())
        end = int(r["t_epi_done"].max())
        m = {"tasks": int(r.size), "span_us": (end - t0) / 1e3}
        for typ, name in ((1, "l1"), (2, "l2")):
            q = r[r["type"] == typ]
            if q.size == 0:
                continue
            dur = (q["t_epi_done"].astype(np.int64) - q["t_issue"].astype(np.int64)) / 1e3
            mma = (q["t_mma_done"].astype(np.int64) - q["t_issue"].astype(np.int64)) / 1e3
            m[name] = {"tasks": int(q.size), "first_issue_us": (int(q["t_issue"].min()) - t0) / 1e3,
                       "last_done_us": (int(q["t_epi_done"].max()) - t0) / 1e3,
                       "mean_task_us": float(dur.mean()), "mean_issue_to_mma_done_us": float(mma.mean())}
        if "l1" in m and "l2" in m:
            m["l1_l2_overlap_us"] = max(0.0, m["l1"]["last_done_us"] - m["l2"]["first_issue_us"])
        last = np.array([int(r[r["cta"] == c]["t_epi_done"].max()) for c in np.unique(r["cta"])])
        tail = (end - last) / 1e3
        m["tail_us"] = {"mean": float(tail.mean()), "max": float(tail.max())}
        out[{1: "l1_launch", 2: "l2_launch", 3: "fused"}.get(int(mode), str(int(mode)))] = m
    return out
