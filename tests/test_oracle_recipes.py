"""Pins for oracle.recipes: hand-worked DelayedScaling tables and CurrentScaling closed forms."""
import json
import os

import numpy as np
import pytest

from oracle import recipes as Rc
from oracle import quantize as Q

GOLD = os.path.join(os.path.dirname(__file__), "golden", "delayed_scaling_e4m3_l4.json")


@pytest.mark.parametrize("algo,key", [(Rc.ALGO_MAX, "max"), (Rc.ALGO_MOST_RECENT, "most_recent")])
def test_hand_worked_table(algo, key):
    g = json.load(open(GOLD))
    st = Rc.DelayedScalingState(g["fmt"], g["history_len"], algo, g["margin"])
    used = []
    for t, a in enumerate(g["amaxes"]):
        used.append(float(st.scale))
        st.update(a, t)
    assert used == g["scale_used_" + key]
    assert float(st.scale) == g["scale_after_last_" + key]
    np.testing.assert_array_equal(st.hist, g["history_after_last"])
    assert st.scale_inv == np.float32(1.0) / st.scale


def test_saturation_under_delayed_scale():
    # step 1 of the table: amax 8 quantized with scale 224 -> 1792 saturates to 448
    q, _, _, _ = Q.fp8_quantize(np.array([[8.0, -8.0, 2.0]], np.float32), 224.0, "e4m3")
    assert list(q[0]) == [0x7E, 0xFE, 0x7E]


def test_margin_halves_and_zero_keeps():
    st = Rc.DelayedScalingState("e4m3", 4, Rc.ALGO_MAX, margin=1)
    st.update(2.0, 0)
    assert st.scale == 112.0
    st2 = Rc.DelayedScalingState("e5m2", 4)
    st2.update(0.0, 0)
    assert st2.scale == 1.0 and st2.scale_inv == 1.0
    st2.update(np.inf, 1)
    assert st2.scale == 1.0
    for t in (2, 3, 4):               # the inf stays in the max-window for L steps
        st2.update(2.0, t)
        assert st2.scale == 1.0
    st2.update(2.0, 5)                # slot 1 overwritten: inf left the window
    assert st2.scale == 28672.0


def test_nan_amax_holds_the_scale_while_in_the_window():
    # reading: a NaN amax is not finite, like +Inf -- the maximum over a window holding it is
    # NaN and the scale is kept; most_recent keeps it for that step only
    st = Rc.DelayedScalingState("e4m3", 4, Rc.ALGO_MAX)
    st.update(2.0, 0)
    assert st.scale == 224.0
    st.update(np.nan, 1)
    assert st.scale == 224.0 and np.isnan(st.hist[1])
    for t in (2, 3, 4):
        st.update(8.0, t)
        assert st.scale == 224.0
    st.update(8.0, 5)                 # slot 1 overwritten: the NaN left the window
    assert st.scale == 56.0
    mr = Rc.DelayedScalingState("e4m3", 4, Rc.ALGO_MOST_RECENT)
    mr.update(2.0, 0)
    mr.update(np.nan, 1)
    assert mr.scale == 224.0
    mr.update(8.0, 2)
    assert mr.scale == 56.0


def test_interval_and_history_len_one():
    st = Rc.DelayedScalingState("e4m3", 8, Rc.ALGO_MAX, interval=2)
    st.update(4.0, 0)
    assert st.scale == 1.0            # recomputed only after steps 1, 3, 5, ...
    st.update(2.0, 1)
    assert st.scale == 112.0          # max(4, 2)
    a = Rc.DelayedScalingState("e4m3", 1, Rc.ALGO_MAX)
    b = Rc.DelayedScalingState("e4m3", 1, Rc.ALGO_MOST_RECENT)
    for t, v in enumerate([3.0, 0.7, 12.5, 1e-3]):
        a.update(v, t)
        b.update(v, t)
        assert a.scale == b.scale


def test_history_wraps_after_L_steps():
    L = 16
    st = Rc.DelayedScalingState("e4m3", L)
    st.update(100.0, 0)
    for t in range(1, L):
        st.update(1.0, t)
        assert st.scale == np.float32(4.48)
    st.update(1.0, L)                 # the 100 leaves the window
    assert st.scale == 448.0


def test_current_scaling_closed_forms():
    for a in [1.0, 0.5, 2.0 ** -20, 4.0, 448.0]:
        s, si = Rc.current_scale(a, "e4m3")
        assert s == np.float32(448.0) / np.float32(a)
        x = np.array([[a, -a, 0.0]], np.float32)
        q = Q.fp8_cast(x, s, "e4m3")
        assert list(q[0]) == [0x7E, 0xFE, 0x00]
    s, si = Rc.current_scale(0.0, "e5m2")
    assert s == 1.0 and si == 1.0
    s, si = Rc.current_scale(2.0 ** -3, "e5m2")
    assert s == 57344.0 * 8 and si == np.float32(1) / np.float32(57344.0 * 8)
