"""Decoding of the per-tile GEMM timeline (hmm_set_trace).

Each record is 8 uint64: packed (sm, problem, expert, K blocks), then the
globaltimer stamps of: scheduler publish, first / last TMA load issued, first
MMA issued / last MMA committed, epilogue saw the accumulator, epilogue done.
"""
from __future__ import annotations

import numpy as np

FIELDS = ("sched", "load0", "load1", "mma0", "mma1", "epi0", "epi1")


def decode(raw: np.ndarray, grid: int):
    """raw: uint64 array of the whole trace buffer.  Returns a structured
    array with one row per recorded tile (cta, slot, sm, prob, e, kb, times)."""
    raw = np.asarray(raw, dtype=np.uint64)
    cap = raw.size // (8 * grid)
    rec = raw[: grid * cap * 8].reshape(grid, cap, 8)
    rows = []
    for cta in range(grid):
        for i in range(cap):
            r = rec[cta, i]
            if r[1] == 0:
                break
            pk = int(r[0])
            rows.append((cta, i, pk >> 48, (pk >> 40) & 0xFF, (pk >> 20) & 0xFFFFF, pk & 0xFFFFF,
                         *[int(v) for v in r[1:]]))
    dt = [("cta", "i4"), ("slot", "i4"), ("sm", "i4"), ("prob", "i4"), ("e", "i4"), ("kb", "i4")]
    dt += [(f, "i8") for f in FIELDS]
    return np.array(rows, dtype=dt)


def summarize(t) -> dict:
    """Per-problem tile statistics (microseconds) and the fraction of the
    launch each CTA's MMA issuer spent between the first MMA and the
    epilogue's view of the accumulator (tensor work in flight)."""
    if t.size == 0:
        return {}
    t0 = int(t["sched"].min())
    t1 = int(np.max(np.where(t["epi1"] > 0, t["epi1"], t["mma1"])))
    out = {"span_us": (t1 - t0) / 1e3, "tiles": int(t.size)}
    done = t["epi0"] > 0
    for p in np.unique(t["prob"]):
        s = t[(t["prob"] == p) & done]
        if s.size == 0:
            continue
        out[f"prob{p}"] = {
            "tiles": int(s.size),
            "kb": float(s["kb"].mean()),
            "load_span_us": float(np.mean(s["load1"] - s["load0"]) / 1e3),
            "mma_issue_span_us": float(np.mean(s["mma1"] - s["mma0"]) / 1e3),
            "mma_to_acc_us": float(np.mean(s["epi0"] - s["mma0"]) / 1e3),
            "epilogue_us": float(np.mean(s["epi1"] - s["epi0"]) / 1e3),
            "sched_lead_us": float(np.mean(s["load0"] - s["sched"]) / 1e3),
        }
    busy, gaps = [], []
    for c in np.unique(t["cta"]):
        s = np.sort(t[(t["cta"] == c) & done], order="slot")
        if s.size == 0:
            continue
        busy.append(np.sum(s["epi0"] - s["mma0"]) / max(1, t1 - t0))
        if s.size > 1:
            gaps.append(np.mean(s["mma0"][1:] - s["mma1"][:-1]) / 1e3)
    out["mma_busy_frac_mean"] = float(np.mean(busy))
    out["mma_gap_between_tiles_us"] = float(np.mean(gaps)) if gaps else 0.0
    return out
