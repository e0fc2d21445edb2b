"""fm_lm_head_argmax_noalloc -- the lm_head + argmax for callers that may not
allocate device memory while they run (its scratch is static device memory of
the library) -- returns the same tokens as fm_draft's own fused lm_head on the
same rows, on two calls in a row: the second call finds the ticket the first
one left at zero.  The tokens also agree with the oracle's argmax of E . y, and
misaligned or mis-shaped rows are refused before any launch.  The file name makes pytest collect it last, so a run that
stops at the first failure has run every other test before it."""
from __future__ import annotations

import numpy as np
import pytest

import fm_synth as S
from gpu_common import Pair, tokens_match

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_speculative_decoding_fm_gb300 import build
    build.build()


@pytest.mark.parametrize("lm", [S.LM_BF16, S.LM_Q8_0])
def test_noalloc_lm_head_matches_draft(lm):
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    cfg = S.tiny_config(max_ctx=128).replace(lm_format=lm)
    p = Pair(cfg, 1101)
    p.append(0, S.gen_features(S.streams(1101)["features"], 40, cfg.feat_dim), 0, oracle=False)
    tok = torch.zeros((1, cfg.block), dtype=torch.int32, device="cuda")
    fm.fm_draft(p.h, [0], [77], [40], tok)
    torch.cuda.synchronize()
    want = tok.cpu().numpy()[0]
    y = torch.from_numpy(p.head_out()).cuda()      # the rows fm_draft's lm_head read
    for _ in range(2):
        out = torch.full((cfg.block,), -7, dtype=torch.int32, device="cuda")
        fm.fm_lm_head_argmax_noalloc(p.h, y, out)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), want)
    # fewer rows: the tokens of those rows
    out = torch.full((5,), -7, dtype=torch.int32, device="cuda")
    fm.fm_lm_head_argmax_noalloc(p.h, y[:5].contiguous(), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), want[:5])
    # against the oracle: the argmax of E . y in fp64 over the same table, a slot
    # excused only where its top-2 margin is below 1e-3
    logits = y.cpu().numpy().astype(np.float64) @ p.oracle.E.T
    assert tokens_match(want, np.argmax(logits, axis=-1), logits)
    # more rows than the kernel's 16 slots: rejected before any launch
    with pytest.raises(fm.FmError) as e:
        fm.fm_lm_head_argmax_noalloc(p.h, torch.zeros((17, cfg.target_dim), device="cuda"),
                                     torch.zeros(17, dtype=torch.int32, device="cuda"))
    assert e.value.status == fm.FM_ERR_INVALID_ARG
    # rows that start 4 bytes past a 16-byte boundary: rejected (the kernel reads float4)
    flat = torch.zeros(cfg.block * cfg.target_dim + 4, device="cuda")
    shifted = flat[1:1 + 2 * cfg.target_dim].view(2, cfg.target_dim)
    with pytest.raises(fm.FmError) as e:
        fm.fm_lm_head_argmax_noalloc(p.h, shifted, torch.zeros(2, dtype=torch.int32, device="cuda"))
    assert e.value.status == fm.FM_ERR_INVALID_ARG
    # the binding refuses a row width other than the drafter's
    with pytest.raises(ValueError):
        fm.fm_lm_head_argmax_noalloc(p.h, torch.zeros((2, cfg.target_dim - 4), device="cuda"),
                                     torch.zeros(2, dtype=torch.int32, device="cuda"))
    p.close()
