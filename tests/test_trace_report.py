"""The trace report on synthetic stamps with a known schedule (no GPU)."""
import numpy as np

from autoregressive_decode_gb300 import trace_report as TR


def synthetic_trace(n_steps=3, L=2, G=4):
    """Each phase: CTA i starts at base + i*100 ns, stages for 1,000 ns, works
    for 2,000 ns, finishes its epilogue 500 ns later; the next phase starts
    3,000 ns after the previous one's earliest start."""
    P = 5 * L + 1
    st = np.zeros((n_steps, P, 6, G), np.uint64)
    t0 = 1_000_000
    for t in range(n_steps):
        for ph in range(P):
            base = t0 + (t * P + ph) * 3000
            for i in range(G):
                s = base + i * 100
                st[t, ph, 0, i] = s
                st[t, ph, 1, i] = s + 1000
                st[t, ph, 2, i] = s + 3000
                st[t, ph, 3, i] = s + 3500
    return st


def test_phase_table_known_schedule():
    st = synthetic_trace()
    tab = TR.phase_table(st)
    for name in ("QKV", "ATT", "O", "GU", "D", "LM"):
        r = tab[name]
        assert abs(r["act"] - 1.0) < 1e-9 and abs(r["work"] - 2.0) < 1e-9 and abs(r["epi"] - 0.5) < 1e-9
        assert abs(r["start_skew"] - 0.3) < 1e-9 and abs(r["end_skew"] - 0.3) < 1e-9
        assert abs(r["span"] - 3.8) < 1e-9
    # consecutive phases overlap: next earliest start is 3.0 us after this earliest start,
    # this latest end is 3.8 us after it
    assert abs(tab["QKV"]["gap"] + 0.8) < 1e-9
    assert tab["QKV"]["count"] == 2 * 2      # 2 steps after the skipped one, 2 layers


def test_token_times_and_stream_report():
    st = synthetic_trace()
    tt = TR.token_times_us(st)
    assert np.allclose(tt, (10 * 3000 + 300 + 3500) / 1e3)
    ring = np.zeros((32768, 4), np.uint64)
    step_start = int(st[1, 0, 0, 0])
    # 20 slots issued every 400 ns, one 2,000 ns stall after slot 9; each released 300 ns after issue
    t = step_start
    for g in range(20):
        t += 400 if g != 10 else 2000
        ring[g] = (t, t + 100, t + 300, 0)
    rep = TR.stream_report(st, ring, step=1, nslot=4)
    assert rep["slots"] == 20
    assert abs(rep["median_issue_gap_us"] - 0.4) < 1e-9
    assert abs(rep["stalled_us"] - 2.0) < 1e-9
    assert rep["issued_right_after_release"] == 0
    assert "QKV" in TR.format_table(TR.phase_table(st))
