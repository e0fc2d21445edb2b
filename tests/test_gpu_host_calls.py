"""GPU: the host-buffer calls of the C ABI (fm_context_append_host,
fm_context_append_batched_host, fm_draft_host) against the device-pointer
calls.  Two sequences of one handle get the same rows and anchors, one
through each form: their cache rows and drafted tokens must be identical
(the same kernels on the same values; no reduction depends on timing), from
pinned and from pageable host memory, and across a call larger than the
staging buffer first held (it grows).  The draft of each is also checked
against the oracle."""
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


def caches_equal(p, a, b, hi):
    for l in range(p.cfg.n_layers):
        for which in ("k", "v"):
            ka, kb = p.cache(a, l, which)[:hi], p.cache(b, l, which)[:hi]
            assert np.array_equal(ka, kb), (l, which, np.abs(ka - kb).max())


def test_single_sequence_host_calls_match_device_calls():
    """Tiny FlashMap: a 1100-row append (the tensor-core prefill; more rows
    than the first staging buffer holds), then two cycles of a 17-row append
    (the deferred path) and a draft; sequence 0 through the device-pointer
    calls, sequence 1 through the host-buffer calls."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    cfg = S.tiny_config(max_ctx=1200).replace(max_seqs=2)
    p = Pair(cfg, 1501, keep_hidden=False)
    fr = S.streams(1501)["features"]
    ctx = S.gen_features(fr, 1100, cfg.feat_dim)
    assert ctx.size > 1 << 20
    fm.fm_context_append(p.h, 0, torch.from_numpy(ctx).cuda(), 1100, 0)
    fm.fm_context_append_host(p.h, 1, ctx, 1100, 0)          # pageable numpy rows
    p.oracle.context_append(p.state(0), ctx, 0)
    torch.cuda.synchronize()
    caches_equal(p, 0, 1, 1100)
    pos = 1100
    for cycle, anchor in enumerate((11, 2222)):
        rows = S.gen_features(fr, 17, cfg.feat_dim)
        fm.fm_context_append(p.h, 0, torch.from_numpy(rows).cuda(), 17, pos)
        pinned = torch.from_numpy(rows).pin_memory()
        fm.fm_context_append_host(p.h, 1, pinned, 17, pos)   # pinned tensor rows
        p.oracle.context_append(p.state(0), rows, pos)
        pos += 17
        tok_dev = torch.full((1, cfg.block), -1, dtype=torch.int32, device="cuda")
        fm.fm_draft(p.h, [0], [anchor], [pos], tok_dev)
        tok_host = torch.full((1, cfg.block), -1, dtype=torch.int32).pin_memory()
        fm.fm_draft_host(p.h, [1], [anchor], [pos], tok_host)
        fm.fm_synchronize(p.h)
        a, b = tok_dev.cpu().numpy(), tok_host.numpy()
        assert np.array_equal(a, b), (cycle, a, b)
        ref = p.oracle.draft(p.state(0), anchor, pos)
        assert tokens_match(a[0], ref.tokens, ref.logits), (cycle, a[0], ref.tokens)
        caches_equal(p, 0, 1, pos + 1)
    # the binding refuses a device tensor or a short buffer for the host forms
    with pytest.raises(ValueError):
        fm.fm_draft_host(p.h, [1], [5], [pos], torch.zeros((1, cfg.block), dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError):
        fm.fm_context_append_host(p.h, 1, np.zeros((2, cfg.feat_dim), np.float32), 3, pos)
    p.close()


def test_batched_host_calls_match_device_calls():
    """Eight sequences (head dim 128): 0..3 through the device-pointer batched
    append and draft, 4..7 through the host-buffer forms with the same rows
    and anchors; each group of four is one batched pass."""
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    cfg = S.DrafterConfig(S.VARIANT_FLASHMAP, dim=512, n_heads=4, head_dim=128, n_layers=2, ff_dim=1024, block=16,
                          target_dim=256, n_taps=2, vocab=4096, lm_format=S.LM_Q8_0, max_ctx=320, max_seqs=8)
    p = Pair(cfg, 1502, keep_hidden=False)
    fr = S.streams(1502)["features"]
    base = [40, 1, 130, 77]
    add = [5, 17, 0, 9]
    ctx = [S.gen_features(fr, n, cfg.feat_dim) for n in base]
    new = [S.gen_features(fr, n, cfg.feat_dim) for n in add]
    dev_ids, host_ids = [0, 1, 2, 3], [4, 5, 6, 7]
    fm.fm_context_append_batched(p.h, dev_ids, torch.from_numpy(np.concatenate(ctx)).cuda(), base, [0] * 4)
    fm.fm_context_append_batched_host(p.h, host_ids, np.concatenate(ctx), base, [0] * 4)
    fm.fm_context_append_batched(p.h, dev_ids, torch.from_numpy(np.concatenate(new)).cuda(), add, base)
    fm.fm_context_append_batched_host(p.h, host_ids, torch.from_numpy(np.concatenate(new)).pin_memory(), add, base)
    pos = [b + a for b, a in zip(base, add)]
    anchors = [3, 300, 3000, 4095]
    tok_dev = torch.full((4, cfg.block), -1, dtype=torch.int32, device="cuda")
    fm.fm_draft(p.h, dev_ids, anchors, pos, tok_dev)
    tok_host = np.full((4, cfg.block), -1, np.int32)           # pageable: the copy completes before return
    fm.fm_draft_host(p.h, host_ids, anchors, pos, tok_host)
    fm.fm_synchronize(p.h)
    a = tok_dev.cpu().numpy()
    assert np.array_equal(a, tok_host), (a, tok_host)
    for i in range(4):
        caches_equal(p, dev_ids[i], host_ids[i], pos[i] + 1)
        st = p.state(dev_ids[i])
        p.oracle.context_append(st, ctx[i], 0)
        if add[i]:
            p.oracle.context_append(st, new[i], base[i])
        ref = p.oracle.draft(st, anchors[i], pos[i])
        assert tokens_match(a[i], ref.tokens, ref.logits), (i, a[i], ref.tokens)
    p.close()
