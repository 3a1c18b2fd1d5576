"""The timeline tool's host arithmetic on a synthetic trace with known answers.

Three calls of three CTAs each, every CTA's SM clock at exactly 2 cycles per
ns.  Calls start 8000 ns apart; in each, CTA i enters at +10 i ns, is released
at +1000 ns and exits at +5000 + 100 i ns.  Stamps: quant_done 1.5 us after
the release (clock only), the issuer's issue time 4000 cycles (2 us), the
gather's re-poll count 3.  The tool must give the period, the release and
entry offsets, the phase times, the duration and the count exactly."""

import numpy as np

from fp8_block_scale_x128_gb300 import timeline as tl

GHZ = 2  # cycles per ns
CALLS, CTAS = 3, 3


def _trace():
    tr = np.zeros((4, CTAS, 64, 2), dtype=np.uint64)
    P = tl.POINTS.index
    for e in range(1, CALLS + 1):
        base = 100_000 + 8000 * e
        for i in range(CTAS):
            def stamp(name, gt, ck=None):
                tr[e, i, P(name), 0] = gt
                tr[e, i, P(name), 1] = GHZ * gt if ck is None else ck
            entry, wait, ex = base + 10 * i, base + 1000, base + 5000 + 100 * i
            stamp("entry", entry)
            stamp("wait", wait)
            stamp("exit", ex)
            stamp("quant_done", 1, GHZ * (wait + 1500))  # clock-only stamp
            stamp("iss_issue", 1, 4000)                  # a duration in cycles
            stamp("gather_polls", 1, 3)                  # a count
    return tr


def test_analyse_and_report_give_the_known_times():
    calls = tl.analyse(_trace(), range(1, CALLS + 1), CTAS)
    assert calls is not None and len(calls) == CALLS
    for c in calls:
        assert abs(c["ghz"] - GHZ) < 1e-9
        assert c["phases"]["quant_done"][:2] == (1.5, 1.5)
        assert c["phases"]["iss_issue"][:2] == (2.0, 2.0)
        assert c["phases"]["gather_polls"][:2] == (3.0, 3.0)
        assert c["last"]["quant_done"] == 1.5  # the last CTA to exit (CTA 2)
    text = tl.report(1, 5120, 4096, CTAS, calls).splitlines()

    def row(label):
        return [ln for ln in text if label in ln][0].split()

    def field(words, key):  # the value after the key's last occurrence (labels hold "last" too)
        return words[len(words) - 1 - words[::-1].index(key) + 1]

    assert row("period between last exits")[-2] == "8.00"
    # the previous call's last exit was at its start + 5200 ns, i.e. 2800 ns
    # before this call's start: releases at +1000 ns are 3.80 us after it, and
    # entries at +0 / +10 / +20 ns 2.80 / 2.81 / 2.82 us after it
    rel = row("release after previous last exit")
    assert (field(rel, "first"), field(rel, "median"), field(rel, "last")) == ("3.80", "3.80", "3.80")
    ent = row("entry after previous last exit")
    assert (field(ent, "first"), field(ent, "median"), field(ent, "last")) == ("2.80", "2.81", "2.82")
    assert row("quant_done")[1:3] == ["1.50", "1.50"]
    assert row("iss_issue")[1:3] == ["2.00", "2.00"]
    assert row("gather_polls")[1:3] == ["3.00", "3.00"]


def test_missing_required_stamps_give_none():
    tr = _trace()
    tr[2, 1, tl.POINTS.index("wait"), 0] = 0  # one CTA of one call lost its release stamp
    assert tl.analyse(tr, range(1, CALLS + 1), CTAS) is None
