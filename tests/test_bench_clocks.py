"""bench.py's clock record: parsing of nvidia-smi samples and the rule that
voids a timing (hardware or thermal slowdown, or clocks stuck low with no
reason; a power cap is kept)."""
import bench

ROW = "0, {sm}, 2070, 600.0, 0x0, {hw}, {hwt}, {swt}, {cap}"


def _sampler(rows, t=100.0):
    s = bench.ClockSampler("0")
    for i, r in enumerate(rows):
        s.samples.append((t + 0.1 * i, [x.strip() for x in r.split(",")]))
    return s


def _row(sm=2070, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return ROW.format(sm=sm, hw=hw, hwt=hwt, swt=swt, cap=cap)


def test_summary_median_window_and_reasons():
    s = _sampler([_row(1000), _row(2070), _row(2070, cap="Active"), _row(1980)])
    c = s.summary(100.05, 100.35)   # the last three samples
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070 and c["samples"] == 3 and c["in_window"]
    assert c["reasons"] == ["sw_power_cap"]
    # no sample inside the window: all samples, flagged
    c = s.summary(200.0, 201.0)
    assert not c["in_window"] and c["samples"] == 4
    assert bench.ClockSampler("0").summary(0, 1) == {"error": "no nvidia-smi samples"}


def test_rejection_rule():
    ok = _sampler([_row(2070)] * 5).summary(0, 1e9)
    assert not bench.clocks_rejected(ok)
    for kw in (dict(hw="Active"), dict(hwt="Active"), dict(swt="Active")):
        assert bench.clocks_rejected(_sampler([_row(2070, **kw)] * 3).summary(0, 1e9)), kw
    # a power cap is kept, even with lower clocks
    assert not bench.clocks_rejected(_sampler([_row(1500, cap="Active")] * 3).summary(0, 1e9))
    # clocks well below the maximum with no reason: a leftover lock
    assert bench.clocks_rejected(_sampler([_row(1200)] * 3).summary(0, 1e9))
    assert not bench.clocks_rejected({"error": "no nvidia-smi samples"})
