"""The trace tool's host side on the CPU: records as the trace build writes
them (include/gemm_f16_trace.h) are decoded into GPU time, with the global
timer wrapping modulo 2^32 between launches, and summarised."""
import numpy as np
import pytest

from tensor_core_tiled_02_gb300 import trace as tr


def put(rec, i, c, r, e, clk, code, arg=0, gt=0):
    rec[i, c, r, e, 0] = clk
    rec[i, c, r, e, 1] = (code << 56) | (arg << 32) | gt


def synthetic(L=3, C=2):
    """Launch i starts at 10 us * i (the timer wrapping past 2^32 ns between
    launches), CTA c 100 ns later per CTA; each role stamps entry, one load at
    1 us + r us, and exit at 9.5 us, at 2 cycles per ns."""
    rec = np.zeros((L, C, 6, 4, 2), np.uint64)
    for i in range(L):
        for c in range(C):
            gt0 = (2 ** 32 - 5000 + i * 10000 + c * 100) % 2 ** 32
            clk0 = 10 ** 6 * (c + 1) + i * 20000
            for r in range(6):
                put(rec, i, c, r, 0, clk0, tr.CODE["entry"], c, gt0)
                put(rec, i, c, r, 1, clk0 + 2000 * (r + 1), tr.CODE["load"], r)
                put(rec, i, c, r, 2, clk0 + 19000, tr.CODE["exit"], 0, (gt0 + 9500) % 2 ** 32)
    return rec


def test_decode_places_events_by_the_sm_clock_between_entry_and_exit():
    t, clk, code, arg = tr.decode(synthetic())
    assert np.allclose(t[0, 0, :, 1] - t[0, 0, 0, 0], [1000, 2000, 3000, 4000, 5000, 6000])
    assert t[2, 1, 0, 0] - t[0, 0, 0, 0] == 20100  # across the timer's wrap
    assert np.isnan(t[0, 0, 0, 3])                 # an empty record
    assert (code[:, :, :, 1] == tr.CODE["load"]).all() and arg[0, 0, 5, 1] == 5


def test_summary_is_relative_to_the_previous_launch_end():
    s = tr.summarise(synthetic(), skip=1)
    # launch i-1 ends with its second CTA's exit, 9.6 us after it starts; launch
    # i starts 10 us after launch i-1
    assert abs(s["first CTA enters"] - 0.4) < 1e-9
    assert abs(s["launch period (end to end)"] - 10.0) < 1e-9
    # the producers' loads 1 us after their entries: 1.4 and 1.5 us, median 1.45
    assert abs(s["first step's loads issued"] - 1.45) < 1e-9
    assert abs(s["last CTA exits"] - 10.0) < 1e-9


def test_shape_and_config_arguments():
    assert tr.parse_shape("1024,8192,8192") == (1024, 8192, 8192, 0)
    assert tr.parse_shape("2048,2048,32768,1") == (2048, 2048, 32768, 1)
    for bad in ("1024,8192", "1,2,3,4,5", "1,2,3,2", "-1,2,3"):
        with pytest.raises(ValueError):
            tr.parse_shape(bad)
    assert tr.parse_config("") == {}
    assert tr.parse_config("cta_group=2,stream_k=2") == {"cta_group": 2, "stream_k": 2}
    with pytest.raises(ValueError):
        tr.parse_config("cta_group")
