"""Reports on the decode kernel's trace (``Engine.trace_decode``).

The trace holds %globaltimer stamps (ns) per (step, phase, event, CTA):
  event 0  phase start (after the step's grid barrier for the first phase)
  event 1  activations staged (GEMV phases) / attention started
  event 2  GEMV or attention done (the eager epilogues included)
  event 3  phase done (the remaining epilogue: the LM argmax)
  event 4  producer issued the phase's first slot (attention: q arrived)
  event 5  producer issued its last slot (attention: warp 0 done with the ring)
and a ring trace of CTA 0 with stamps per global slot index:
  0 copy issued, 1 data seen by its consumer warp, 2 released.

``phase_table`` summarises where a step's time goes per phase type;
``stream_report`` shows how continuously CTA 0's producer kept HBM busy.
Run as ``python -m autoregressive_decode_gb300.trace_report stamps.npy
[ring.npy [nslot]]`` on arrays saved from ``trace_decode`` (nslot: the
engine's ring slots, 11 for the 1.8B model).
"""
from __future__ import annotations

import sys

import numpy as np

PHASES = ("QKV", "ATT", "O", "GU", "D")


def phase_name(phi: int, n_phases: int) -> str:
    return "LM" if phi == n_phases - 1 else PHASES[phi % 5]


def token_times_us(stamps: np.ndarray) -> np.ndarray:
    """Per step: first phase start (earliest CTA) to last phase end (latest CTA)."""
    st = stamps.astype(np.int64)
    return np.array([(st[t, -1, 3].max() - st[t, 0, 0].min()) / 1e3 for t in range(st.shape[0])])


def phase_table(stamps: np.ndarray, skip_steps: int = 1) -> dict:
    """Mean over steps (after the first skip_steps) and layers, per phase type,
    in microseconds:
      span       earliest start to latest end over the CTAs
      start_skew latest minus earliest start
      act        staging (mean over CTAs): the wait for the input activations
      work       GEMV / attention (mean over CTAs)
      epi        the rest of the phase (mean over CTAs)
      end_skew   latest minus earliest end
      gap        next phase's earliest start minus this phase's latest end
                 (negative: the phases overlap across CTAs)"""
    st = stamps.astype(np.int64)
    n, n_ph = st.shape[0], st.shape[1]
    rows: dict[str, list] = {}
    for t in range(skip_steps, n):
        for ph in range(n_ph):
            s = st[t, ph]
            if s[0].max() == 0:          # phase not run in this step (e.g. no LM head)
                continue
            if ph + 1 < n_ph:
                nxt = st[t, ph + 1, 0].min()
            elif t + 1 < n:
                nxt = st[t + 1, 0, 0].min()
            else:
                nxt = None
            row = [s[3].max() - s[0].min(), s[0].max() - s[0].min(), (s[1] - s[0]).mean(),
                   (s[2] - s[1]).mean(), (s[3] - s[2]).mean(), s[3].max() - s[3].min(),
                   (nxt - s[3].max()) if nxt is not None else np.nan]
            rows.setdefault(phase_name(ph, n_ph), []).append(row)
    keys = ("span", "start_skew", "act", "work", "epi", "end_skew", "gap")
    out = {}
    for name, vals in rows.items():
        a = np.array(vals, dtype=np.float64) / 1e3
        out[name] = {k: float(np.nanmean(a[:, i])) if np.isfinite(a[:, i]).any() else float("nan")
                     for i, k in enumerate(keys)}
        out[name]["count"] = len(vals)
    return out


def stream_report(stamps: np.ndarray, ring: np.ndarray, step: int, nslot: int, stall_us: float = 1.0,
                  wake_us: float = 0.5) -> dict:
    """CTA 0's producer during one step: slots issued, median time between
    consecutive copies, the time in gaps longer than stall_us (the stream
    stopped), and how often a copy was issued within wake_us of the release of
    the ring slot it reuses (the ring was full and the producer waited)."""
    st = stamps.astype(np.int64)
    sl = ring.astype(np.int64)
    n = int((sl[:, 0] > 0).sum())
    sl = sl[:n]
    start, end = st[step, 0, 0, 0], st[step, -1, 3, 0]
    sel = np.flatnonzero((sl[:, 0] >= start) & (sl[:, 0] <= end))
    if len(sel) < 2:
        return {"slots": int(len(sel))}
    issue = sl[sel, 0]
    gaps = np.diff(issue) / 1e3
    ring_full = 0
    for g in sel:
        if g >= nslot and sl[g - nslot, 2] > 0 and (sl[g, 0] - sl[g - nslot, 2]) < wake_us * 1e3:
            ring_full += 1
    return {"slots": int(len(sel)), "window_us": float((end - start) / 1e3),
            "median_issue_gap_us": float(np.median(gaps)),
            "stalled_us": float(gaps[gaps > stall_us].sum()),
            "issued_right_after_release": int(ring_full)}


def format_table(table: dict) -> str:
    cols = ("span", "start_skew", "act", "work", "epi", "end_skew", "gap")
    lines = [f"{'phase':6s}" + "".join(f"{c:>11s}" for c in cols) + "   (us, mean)"]
    for name in ("QKV", "ATT", "O", "GU", "D", "LM"):
        if name in table:
            r = table[name]
            lines.append(f"{name:6s}" + "".join(f"{r[c]:11.2f}" for c in cols) + f"   x{r['count']}")
    return "\n".join(lines)


def main(argv: list[str]) -> int:
    if not argv:
        print(__doc__)
        return 2
    stamps = np.load(argv[0])
    print("per-step us:", np.round(token_times_us(stamps), 1))
    print(format_table(phase_table(stamps)))
    if len(argv) > 1:
        ring = np.load(argv[1])
        nslot = int(argv[2]) if len(argv) > 2 else 11
        print("CTA 0 stream, step", min(1, stamps.shape[0] - 1), ":",
              stream_report(stamps, ring, min(1, stamps.shape[0] - 1), nslot))
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
