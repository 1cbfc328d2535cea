"""Adaptive draft length (sxl-space.tk "【大模型】- 推测解码", 自适应推测解码,
AdaptiveSpeculativeDecoder.adapt_k): the CPU restatement pinned by hand-derived
trajectories, and the device controller (spec_adapt_*) against it."""
from __future__ import annotations

import numpy as np
import pytest

from oracle.adapt import AdaptiveK, offsets, run_batch


def trajectory(counts, min_k=1, max_k=10, counts_are_fraction_of_k=None):
    c = AdaptiveK(min_k, max_k)
    ks = [c.current_k]
    for n in counts:
        if counts_are_fraction_of_k is not None:
            n = counts_are_fraction_of_k(c.current_k)
        ks.append(c.adapt(n))
    return ks


# ---------------------------------------------------------------- pins (CPU)
def test_starts_at_the_midpoint():
    assert AdaptiveK(1, 10).current_k == 5
    assert AdaptiveK(2, 6).current_k == 4
    assert AdaptiveK(3, 3).current_k == 3


def test_full_acceptance_grows_after_ten_rounds():
    # rates 1.0: no change until the history holds 10 rates, then +1 a round up to 10
    ks = trajectory([None] * 20, counts_are_fraction_of_k=lambda k: k)
    assert ks == [5] * 10 + [6, 7, 8, 9, 10, 10, 10, 10, 10, 10, 10]


def test_zero_acceptance_shrinks_after_ten_rounds():
    ks = trajectory([0] * 20)
    assert ks == [5] * 10 + [4, 3, 2, 1, 1, 1, 1, 1, 1, 1, 1]


def test_mean_exactly_at_the_thresholds_changes_nothing():
    # k = 5, 4 accepted: every rate is exactly 4/5, the mean is exactly 0.8
    assert trajectory([4] * 30) == [5] * 31
    # k = 4 (bounds 2..6), 2 accepted: the mean is exactly 1/2
    assert trajectory([2] * 30, 2, 6) == [4] * 31


def test_only_the_last_ten_rates_count():
    # ten rounds at rate 1 (k: 5 -> 6 at round 10), then rate 0; worked by hand:
    # round 11 mean 0.9 (-> 7), 12: 0.8 (tie), 13: 0.7, 14: 0.6, 15: 0.5 (tie),
    # 16: 0.4 (-> 6), 17: 0.3 (-> 5), 18: 0.2 (-> 4), 19: 0.1 (-> 3), 20: 0 (-> 2),
    # 21: (-> 1), 22: stays 1
    c = AdaptiveK(1, 10)
    ks = [c.current_k]
    for r in range(22):
        ks.append(c.adapt(c.current_k if r < 10 else 0))
    assert ks == [5] * 10 + [6, 7, 7, 7, 7, 7, 6, 5, 4, 3, 2, 1, 1]


def test_history_keeps_its_last_hundred_rates():
    c = AdaptiveK(1, 10)
    for _ in range(250):
        c.adapt(1)
    assert len(c.acceptance_history) == 100


def test_rounds_without_a_rate_leave_the_state():
    c = AdaptiveK(1, 10)
    for n in (-1, 6, 7):  # data error, more accepted than drafted
        assert c.adapt(n) == 5
    assert c.acceptance_history == []


def test_same_as_the_float_statement_away_from_ties():
    """The pages' loop in Python floats gives the same lengths, except after a
    mean that float rounding puts on the other side of 0.8 or 0.5."""
    rng = np.random.default_rng(5)
    for trial in range(200):
        c = AdaptiveK(1, 10)
        k, hist, tied = 5, [], False
        for _ in range(60):
            n = int(rng.integers(0, k + 1))
            hist.append(n / k)
            hist = hist[-100:]
            exact = c.adapt(n)
            if len(hist) >= 10:
                avg = sum(hist[-10:]) / 10
                tied |= abs(avg - 0.8) < 1e-12 or abs(avg - 0.5) < 1e-12
                if avg > 0.8:
                    k = min(k + 1, 10)
                elif avg < 0.5:
                    k = max(k - 1, 1)
            if tied:
                break
            assert k == exact


def test_offsets_and_batch_runner():
    assert offsets([3, 0, 2]).tolist() == [0, 3, 3, 5]
    out = run_batch([np.array([5, 0])] * 10, B=2)
    assert out[0].tolist() == [0, 5, 10]
    assert out[-1].tolist() == [0, 6, 10]


# ---------------------------------------------------------------- host-side API
def test_state_bytes_and_argument_checks():
    import ctypes
    import speculative_decoding_verification_61_gb300 as sv
    L = sv.lib()
    assert L.spec_adapt_state_bytes(0) == 0
    assert L.spec_adapt_state_bytes(4096) == 23 * 4 * 4096
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the checks come first
    assert L.spec_adapt_init(fake, 0, 1, 10, fake, None) == -1
    assert L.spec_adapt_init(fake, 4, 5, 4, fake, None) == -1
    assert L.spec_adapt_init(fake, 4, 1, 33, fake, None) == -1
    assert L.spec_adapt_init(None, 4, 1, 10, fake, None) == -1
    assert L.spec_adapt_update(fake, None, 4, 1, 10, fake, None) == -1
    assert L.spec_adapt_init(ctypes.c_void_p((1 << 20) + 4), 4, 1, 10, fake, None) == -2


# ---------------------------------------------------------------- device (GPU)
@pytest.mark.gpu
@pytest.mark.parametrize("B,min_k,max_k", [(1, 1, 10), (7, 2, 6), (1000, 1, 32), (4096, 1, 10), (33, 3, 3)])
def test_device_controller_matches_the_oracle(B, min_k, max_k):
    import torch
    import speculative_decoding_verification_61_gb300 as sv
    rng = np.random.default_rng(1000 + B)
    ctl = sv.AdaptiveK(B, min_k, max_k)
    ora = [AdaptiveK(min_k, max_k) for _ in range(B)]
    torch.cuda.synchronize()
    assert ctl.k_offsets.cpu().numpy().tolist() == offsets([c.current_k for c in ora]).tolist()
    # acceptance drifts from high to low and back, so lengths move both ways;
    # a few rounds carry no rate (-1, or more accepted than drafted)
    for r in range(130):
        p = 0.95 if (r // 25) % 2 == 0 else 0.3
        ks = np.array([c.current_k for c in ora])
        n = rng.binomial(ks, p)
        n[rng.random(B) < 0.03] = -1
        bad = rng.random(B) < 0.01
        n[bad] = ks[bad] + 1
        got = ctl.update(torch.from_numpy(n.astype(np.int32)).cuda())
        want = offsets([c.adapt(int(x)) for c, x in zip(ora, n)])
        assert np.array_equal(got.cpu().numpy(), want), r


@pytest.mark.gpu
def test_device_controller_ties_and_skips():
    import torch
    import speculative_decoding_verification_61_gb300 as sv
    ctl = sv.AdaptiveK(3, 1, 10)
    for _ in range(30):  # rates exactly 4/5, 1, 0: k stays / grows / shrinks
        ko = ctl.k_offsets.cpu().numpy()
        ks = np.diff(ko)
        n = np.array([4 if ks[0] == 5 else -1, ks[1], 0], dtype=np.int32)
        ctl.update(torch.from_numpy(n).cuda())
    ks = np.diff(ctl.k_offsets.cpu().numpy())
    assert ks.tolist() == [5, 10, 1]
