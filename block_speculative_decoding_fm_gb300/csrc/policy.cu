// policy.cu -- the verify-length and fallback policy of the speculative loop
// (flashmap_drafter.js, ``specGenerate``), as a caller-owned state record and
// four host functions.  It decides, per step of the loop, whether to run a
// draft round and how many drafts to verify, or a plain step of the target.
//   * near the drafter's context limit (position + 2 block + 2 > max_ctx): plain
//     steps only, no statistics;
//   * during a plain stretch: plain steps; each updates the plain-step time
//     average (0.7 / 0.3);
//   * a round verifies K = block when the acceptance average is >= 5, else 7
//     (adaptive), or min(block, verify) (fixed);
//   * after a round: acceptance average 0.6 / 0.4, tokens-per-round average
//     0.75 / 0.25 (accepted + 1), round-time average 0.6 / 0.4 (the first round
//     after a stretch whose rows were just handed to the drafter is left out);
//     from the fourth round on, when tokens-per-round x plain-step time falls
//     below 0.85 x round time, a plain stretch of probe_every steps starts.
#include "../../include/fm.h"

extern "C" {

fm_status fm_policy_init(fm_verify_policy *p, int32_t block, int32_t verify, int32_t fallback, int32_t probe_every) {
  if (!p || block < 1 || verify < 0 || probe_every < 1) return FM_ERR_INVALID_ARG;
  p->block = block;
  p->verify = verify;
  p->fallback = fallback ? 1 : 0;
  p->probe_every = probe_every;
  p->ema = 4.0;
  p->ema_tokens = 5.0;
  p->round_ms = -1.0;   // not measured yet
  p->step_ms = 30.0;
  p->plain_left = 0;
  p->rounds = 0;
  p->catch_up = 0;
  p->pad = 0;
  return FM_OK;
}

fm_status fm_policy_next(const fm_verify_policy *p, int32_t position, int32_t max_ctx, int32_t *action, int32_t *k) {
  if (!p || !action || !k) return FM_ERR_INVALID_ARG;
  *k = 0;
  if ((int64_t)position + 2 * (int64_t)p->block + 2 > max_ctx) {
    *action = FM_ACT_PLAIN_LIMIT;
    return FM_OK;
  }
  if (p->plain_left > 0) {
    *action = FM_ACT_PLAIN;
    return FM_OK;
  }
  *action = FM_ACT_ROUND;
  if (p->verify == 0)
    *k = p->ema >= 5.0 ? p->block : 7;
  else
    *k = p->verify < p->block ? p->verify : p->block;
  return FM_OK;
}

fm_status fm_policy_after_round(fm_verify_policy *p, int32_t accepted, double ms) {
  if (!p || accepted < 0) return FM_ERR_INVALID_ARG;
  p->ema = 0.6 * p->ema + 0.4 * accepted;
  p->ema_tokens = 0.75 * p->ema_tokens + 0.25 * (accepted + 1);
  p->rounds += 1;
  if (!p->catch_up) p->round_ms = p->round_ms < 0.0 ? ms : 0.6 * p->round_ms + 0.4 * ms;
  p->catch_up = 0;
  if (p->fallback && p->rounds >= 4 && p->round_ms >= 0.0 && p->ema_tokens * p->step_ms < 0.85 * p->round_ms)
    p->plain_left = p->probe_every;
  return FM_OK;
}

fm_status fm_policy_after_plain(fm_verify_policy *p, double ms, int32_t rows_handed) {
  if (!p || p->plain_left < 1) return FM_ERR_INVALID_ARG;
  p->step_ms = 0.7 * p->step_ms + 0.3 * ms;
  p->plain_left -= 1;
  if (rows_handed) p->catch_up = 1;
  return FM_OK;
}

}  // extern "C"
