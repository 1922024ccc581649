"""bench.py's decode roofline: which launch time it divides the algorithmic
bytes by (host logic, no GPU).  A step made only of decode launches is timed
by its windows (window time / launches: events between launches would cut
their programmatic overlap), with the event-bracketed launch reported beside
it as the isolated figure; the mixed step and the two-launch step use the
bracketed launches."""
import types

import bench


def _timing(prefill, launches_per_step=1):
    """The fields time_pkv returns that decode_roofline reads: bracketed
    launches of 1 GB in 0.2 ms; steps of 2 GB in 0.3 ms."""
    return dict(W=types.SimpleNamespace(prefill=prefill), dom_bytes=1e9, dom_ms=0.2, step_bytes=2e9,
                step_ms=0.3, launches_per_step=launches_per_step, dec_p10=0.19, dec_p90=0.21,
                per_launch_gbs=5000.0, ev_stride=11)


def test_all_decode_step_uses_window_time_per_launch():
    out = bench.decode_roofline(_timing(None, launches_per_step=2), 8000.0, "measured", True, 2)
    # two launches a step: 1 GB each in 0.15 ms
    assert out["algorithmic_bytes_per_launch"] == 10 ** 9 and out["avg_launch_ms"] == 0.15
    assert abs(out["achieved"] - 1e9 / 0.15e-3 / 1e9) < 0.1
    assert abs(out["frac"] - out["achieved"] / 8000.0) < 1e-4
    # the bracketed launch: 1 GB in 0.2 ms = 5000 GB/s
    assert out["isolated_launch_ms"] == 0.2 and abs(out["frac_isolated"] - 5000.0 / 8000.0) < 1e-4
    assert "window time / launches" in out["timed_by"]


def test_mixed_step_uses_the_bracketed_decode_launch():
    out = bench.decode_roofline(_timing(object()), 8000.0, "measured", True, 4)
    assert out["avg_launch_ms"] == 0.2 and abs(out["achieved"] - 5000.0) < 0.1
    assert "isolated_launch_ms" not in out and "every 11-th step" in out["timed_by"]


def test_two_launch_step_uses_the_bracketed_decode_launch():
    out = bench.decode_roofline(_timing(None), 8000.0, "measured", False, 2)
    assert out["avg_launch_ms"] == 0.2 and abs(out["achieved"] - 5000.0) < 0.1
