"""Pins of the verify-length / fallback policy oracle (flashmap_drafter.js,
``specGenerate``) against closed forms of its averages and hand-worked
sequences.  CPU only."""
from __future__ import annotations

import math

from oracle.policy import PLAIN, PLAIN_LIMIT, ROUND, VerifyPolicy


def test_adaptive_length_follows_the_acceptance_average():
    # ema_n = a + (4 - a) 0.6^n for a constant acceptance a (closed form of the recurrence)
    p = VerifyPolicy(block=16, fallback=False)
    assert p.next_action(100, 4096) == (ROUND, 7)          # ema starts at 4 < 5: an 8-token verify block
    for n in range(1, 12):
        p.after_round(16, 10.0)
        assert math.isclose(p.ema, 16 + (4 - 16) * 0.6 ** n, rel_tol=1e-12)
    # first n with 16 - 12 * 0.6^n >= 5 is n = 1 (16 - 7.2 = 8.8)
    p = VerifyPolicy(block=16, fallback=False)
    p.after_round(16, 10.0)
    assert p.next_action(100, 4096) == (ROUND, 16)
    # a run of zero acceptance: 4 * 0.6^n stays below 5
    p = VerifyPolicy(block=16, fallback=False)
    for _ in range(5):
        p.after_round(0, 10.0)
        assert p.next_action(100, 4096) == (ROUND, 7)
    # the threshold is inclusive: ema exactly 5
    p = VerifyPolicy(block=16, fallback=False, ema=5.0)
    assert p.next_action(100, 4096) == (ROUND, 16)


def test_fixed_verify_length_is_capped_by_the_block():
    assert VerifyPolicy(block=16, verify=4).next_action(0, 4096) == (ROUND, 4)
    assert VerifyPolicy(block=16, verify=40).next_action(0, 4096) == (ROUND, 16)


def test_context_limit_forces_plain_steps_and_keeps_no_statistics():
    p = VerifyPolicy(block=16, plain_left=3)
    # position + 2 * 16 + 2 > max_ctx: 1000 + 34 > 1033
    assert p.next_action(1000, 1033) == (PLAIN_LIMIT, 0)
    assert p.next_action(999, 1033) == (PLAIN, 0)
    assert p.plain_left == 3


def test_fallback_starts_after_four_losing_rounds_and_probes_again():
    p = VerifyPolicy(block=16, probe_every=16)
    # a round costs 100 ms and yields 1 token; plain steps cost 30 ms: rounds lose
    for i in range(3):
        p.after_round(0, 100.0)
        assert p.plain_left == 0                 # fewer than 4 rounds: no decision yet
    p.after_round(0, 100.0)
    # ema_tokens after 4 rounds of 1 token: 1 + 4 * 0.75^4; round_ms = 100
    et = 1 + 4 * 0.75 ** 4
    assert math.isclose(p.ema_tokens, et, rel_tol=1e-12)
    assert et * 30 < 0.85 * 100 and p.plain_left == 16
    for k in range(16):
        assert p.next_action(10, 4096) == (PLAIN, 0)
        p.after_plain(30.0, rows_handed=(k == 15))
    assert p.plain_left == 0 and p.catch_up
    assert p.next_action(10, 4096)[0] == ROUND
    # the probe round right after the stretch is left out of the round average
    p.after_round(16, 5000.0)
    assert p.round_ms == 100.0 and not p.catch_up


def test_winning_rounds_never_fall_back():
    p = VerifyPolicy(block=16)
    for _ in range(20):
        p.after_round(16, 40.0)      # 17 tokens per 40 ms round vs 30 ms plain steps
        assert p.plain_left == 0


def test_break_even_boundary_is_strict():
    # ema_tokens * step_ms == 0.85 * round_ms exactly: no fallback (strict <)
    q = VerifyPolicy(block=16, ema_tokens=2.0, step_ms=85.0, rounds=3, round_ms=100.0)
    q.after_round(1, 100.0)          # ema_tokens = 0.75 * 2 + 0.25 * 2 = 2; 2 * 85 = 170 vs 0.85 * 100 = 85
    assert q.plain_left == 0
    r = VerifyPolicy(block=16, ema_tokens=1.0, step_ms=85.0, rounds=3, round_ms=100.0)
    r.after_round(0, 100.0)          # ema_tokens = 0.75 + 0.25 = 1; 85 == 0.85 * 100 -> not below
    assert r.ema_tokens == 1.0 and r.plain_left == 0
    s = VerifyPolicy(block=16, ema_tokens=1.0, step_ms=84.9, rounds=3, round_ms=100.0)
    s.after_round(0, 100.0)
    assert s.plain_left == 16
