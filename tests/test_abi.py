"""The C ABI library loads and exports every entry point include/fm.h declares;
host-only logic (argument checks that run before any device work, the pure
host acceptance rule) behaves as documented.  No GPU needed."""
from __future__ import annotations

import ctypes
import itertools
import os
import re

import numpy as np
import pytest

import block_speculative_decoding_fm_gb300 as fm
import fm_synth as S
from block_speculative_decoding_fm_gb300 import build as fmbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fmbuild.build()
    return fm.load_library()


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "fm.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(fm_[a-z_]+)\s*\(", txt)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for s in ("fm_create", "fm_context_append", "fm_draft", "fm_accept", "fm_accept_batched", "fm_debug_copy",
              "fm_destroy", "fm_status_str", "fm_last_error"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), s
    assert set(declared_symbols()) <= set(fm.EXPORTS)


def test_no_internal_symbols_exported(lib):
    out = os.popen(f"nm -D --defined-only {fm.LIB_PATH}").read()
    names = [l.split()[-1] for l in out.splitlines() if " T " in l]
    assert names and all(n.startswith("fm_") for n in names), names


def test_status_strings(lib):
    for s in range(8):
        assert lib.fm_status_str(s)
    assert lib.fm_status_str(99) == b"unknown status"


def test_accept_host_rule_brute_force(lib):
    for k in range(5):
        for d in itertools.product(range(3), repeat=4):
            for t in itertools.product(range(3), repeat=5):
                acc, bonus = fm.fm_accept(d, t, k)
                want = next((i for i in range(k) if d[i] != t[i]), k)
                assert (acc, bonus) == (want, t[want])


def test_accept_rejects_bad_arguments(lib):
    acc, bonus = ctypes.c_int32(), ctypes.c_int32()
    d = np.zeros(4, np.int32)
    assert lib.fm_accept(None, d.ctypes.data, 2, ctypes.byref(acc), ctypes.byref(bonus)) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_accept(d.ctypes.data, d.ctypes.data, -1, ctypes.byref(acc), ctypes.byref(bonus)) == \
        fm.FM_ERR_INVALID_ARG


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 96, fm.FM_ERR_UNSUPPORTED),
    ("dim", 200, fm.FM_ERR_INVALID_ARG),
    ("block", 17, fm.FM_ERR_UNSUPPORTED),
    ("n_layers", 0, fm.FM_ERR_UNSUPPORTED),
    ("lm_format", 7, fm.FM_ERR_INVALID_ARG),
    ("max_seqs", 0, fm.FM_ERR_INVALID_ARG),
    ("variant", 3, fm.FM_ERR_INVALID_ARG),
    ("target_dim", 100, fm.FM_ERR_UNSUPPORTED),
])
def test_create_rejects_bad_configs_before_device_work(lib, field, value, status):
    cfg = S.tiny_config().replace(**{field: value})
    with pytest.raises(fm.FmError) as e:
        fm.fm_create(cfg, [], None)
    assert e.value.status == status
    assert lib.fm_last_error(None)


def test_null_handle_calls_are_rejected(lib):
    assert lib.fm_context_append(None, 0, None, 0, 0, None) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_draft(None, 1, None, None, None, None, None) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_debug_copy(None, 0, 0, 0, 0, None, 0, None) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_context_append_host(None, 0, None, 0, 0, None) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_context_append_batched_host(None, 1, None, None, None, None, None) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_draft_host(None, 1, None, None, None, None, None) == fm.FM_ERR_INVALID_ARG
    lib.fm_destroy(None)
    assert lib.fm_last_error(None) is not None


def test_host_buffer_binding_checks():
    """The binding's checks of a host-buffer call's rows and tokens (before any
    library call): dtype, a host (not CUDA) buffer, C order, enough values."""
    import torch
    ok = [np.zeros(12, np.float32), torch.zeros(12), torch.zeros((3, 4))]
    for x in ok:
        assert fm._host_buffer(x, np.float32, "rows", 12) is x
    assert fm._host_buffer(torch.zeros(8, dtype=torch.int32), np.int32, "tokens", 8) is not None
    bad = [np.zeros(12, np.float64), torch.zeros(12, dtype=torch.float64), np.zeros((4, 3), np.float32).T,
           torch.zeros((4, 3)).t(), np.zeros(12, np.int32)]
    for x in bad:
        with pytest.raises(ValueError):
            fm._host_buffer(x, np.float32, "rows", 12)
    with pytest.raises(ValueError):
        fm._host_buffer(np.zeros(11, np.float32), np.float32, "rows", 12)


def test_verify_policy_matches_the_oracle_step_for_step(lib):
    """fm_policy_* (the library's host policy) against oracle.policy on seeded
    random loops: the same actions, verify lengths and state, bit for bit."""
    from oracle.policy import PLAIN, PLAIN_LIMIT, ROUND, VerifyPolicy
    rng = np.random.default_rng(21)
    for trial in range(40):
        block = int(rng.choice([5, 8, 16]))
        verify = int(rng.choice([0, 0, 3, 40]))
        fallback = bool(rng.integers(0, 2))
        probe = int(rng.integers(1, 20))
        c = fm.fm_policy_init(block, verify, fallback, probe)
        o = VerifyPolicy(block, verify, fallback, probe)
        max_ctx = 4096
        for step in range(300):
            pos = int(rng.integers(0, max_ctx)) if rng.random() < 0.1 else int(rng.integers(0, max_ctx // 2))
            act_c, k_c = fm.fm_policy_next(c, pos, max_ctx)
            act_o, k_o = o.next_action(pos, max_ctx)
            assert (act_c, k_c) == (act_o, k_o), (trial, step)
            if act_o == ROUND:
                acc = int(rng.integers(0, k_o + 1)) if rng.random() < 0.5 else int(rng.integers(0, 2))
                ms = float(rng.uniform(5, 200))
                fm.fm_policy_after_round(c, acc, ms)
                o.after_round(acc, ms)
            elif act_o == PLAIN:
                ms = float(rng.uniform(5, 60))
                handed = o.plain_left == 1 or rng.random() < 0.1
                fm.fm_policy_after_plain(c, ms, handed)
                o.after_plain(ms, handed)
            else:
                assert act_o == PLAIN_LIMIT
            assert (c.ema, c.ema_tokens, c.step_ms, c.plain_left, c.rounds, bool(c.catch_up)) == \
                (o.ema, o.ema_tokens, o.step_ms, o.plain_left, o.rounds, o.catch_up), (trial, step)
            assert (c.round_ms < 0) == (o.round_ms is None)
            if o.round_ms is not None:
                assert c.round_ms == o.round_ms


def test_verify_policy_rejects_bad_arguments(lib):
    p = fm.FmVerifyPolicy()
    assert lib.fm_policy_init(ctypes.byref(p), 0, 0, 1, 16) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_policy_init(ctypes.byref(p), 16, -1, 1, 16) == fm.FM_ERR_INVALID_ARG
    assert lib.fm_policy_init(ctypes.byref(p), 16, 0, 1, 16) == fm.FM_OK
    assert lib.fm_policy_after_plain(ctypes.byref(p), 10.0, 0) == fm.FM_ERR_INVALID_ARG   # no stretch running
    assert lib.fm_policy_after_round(ctypes.byref(p), -1, 10.0) == fm.FM_ERR_INVALID_ARG
