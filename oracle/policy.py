"""The verify-length and fallback policy of the speculative loop, plain Python
(oracle).  TEST INFRASTRUCTURE: see oracle/common.py for who may use this
package.

Source: diskformer 0.5.4 -> 0.6.6, package/engines/flashmap_drafter.js --
``specGenerate`` (its header comment and the round / plain-step bookkeeping).

What the page decides, per round or plain step of the target:
  * near the drafter's context limit (position + 2 * block + 2 > max_ctx) the
    loop only takes plain steps;
  * while a plain stretch is running (plain_left > 0) it takes a plain step;
    each updates the plain-step time average step_ms = 0.7 step_ms + 0.3 dt;
  * otherwise a round verifies K drafts: with the adaptive setting K = block
    when the acceptance average ema >= 5, else 7 (an 8-token verify block);
    with a fixed setting K = min(block, verify);
  * after a round with acc accepted drafts: ema = 0.6 ema + 0.4 acc,
    ema_tokens = 0.75 ema_tokens + 0.25 (acc + 1), rounds += 1, and the round
    time average round_ms = dt (first round) or 0.6 round_ms + 0.4 dt -- except
    the first round after a plain stretch whose context rows were just handed to
    the drafter (catch_up), whose time is left out;
  * fallback (when enabled): after at least 4 rounds, when
    ema_tokens * step_ms < 0.85 * round_ms, a plain stretch of probe_every steps
    starts.
Initial values: ema = 4, ema_tokens = 5, round_ms unset, step_ms = 30.

Readings taken where the page leaves a step open:
  * the caller reports when a plain stretch's feature rows were handed to the
    drafter (the page does it when the stretch ends, when a chunk of rows is
    full, at a stop token or at the token budget); that report sets catch_up.
"""
from __future__ import annotations

from dataclasses import dataclass


ROUND, PLAIN, PLAIN_LIMIT = 0, 1, 2   # a round; a step of a plain stretch; a plain step at the context limit


@dataclass
class VerifyPolicy:
    block: int
    verify: int = 0            # 0: adaptive, else a fixed verify length
    fallback: bool = True
    probe_every: int = 16
    ema: float = 4.0
    ema_tokens: float = 5.0
    round_ms: float | None = None
    step_ms: float = 30.0
    plain_left: int = 0
    rounds: int = 0
    catch_up: bool = False

    def next_action(self, position: int, max_ctx: int):
        """(ROUND, K), (PLAIN, 0) or (PLAIN_LIMIT, 0) for the next step of the
        loop; the context limit is checked first and keeps no statistics."""
        if position + 2 * self.block + 2 > max_ctx:
            return PLAIN_LIMIT, 0
        if self.plain_left > 0:
            return PLAIN, 0
        if self.verify == 0:
            k = self.block if self.ema >= 5 else 7
        else:
            k = min(self.block, self.verify)
        return ROUND, k

    def after_round(self, accepted: int, ms: float) -> None:
        self.ema = 0.6 * self.ema + 0.4 * accepted
        self.ema_tokens = 0.75 * self.ema_tokens + 0.25 * (accepted + 1)
        self.rounds += 1
        if not self.catch_up:
            self.round_ms = ms if self.round_ms is None else 0.6 * self.round_ms + 0.4 * ms
        self.catch_up = False
        if (self.fallback and self.rounds >= 4 and self.round_ms is not None
                and self.ema_tokens * self.step_ms < 0.85 * self.round_ms):
            self.plain_left = self.probe_every

    def after_plain(self, ms: float, rows_handed: bool) -> None:
        """A step of a plain stretch (action PLAIN) took ms; rows_handed: the
        stretch's feature rows went to the drafter after this step (the next
        round's time is then left out of the round average)."""
        self.step_ms = 0.7 * self.step_ms + 0.3 * ms
        self.plain_left -= 1
        if rows_handed:
            self.catch_up = True
