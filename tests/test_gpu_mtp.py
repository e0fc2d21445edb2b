"""GPU parity of the MTP draft head (ternary_bonsai_2_mtp.js, ``MTPHead.forward``
and ``MTPRunner``'s draft loop) through fm_mtp_* against the oracle: the head
output h' of every row (relative L2 within 2e-3), the head's K/V cache rows
(within 1e-3), and the drafted tokens (exact unless the oracle's top-2 logit margin is below
1e-3; after an excused difference the chain follows another token and the
later drafts are not compared)."""
from __future__ import annotations

import numpy as np
import pytest

import fm_synth as S
from gpu_common import MARGIN, REL_L2, rel_l2
from oracle.common import top2_margin
from oracle.mtp import MtpHead

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_speculative_decoding_fm_gb300 import build
    build.build()


def mid_config(kv_cap=160):
    """Split-K products (eh_proj and ffn_down in two slices) at a size the oracle runs quickly."""
    return S.MtpConfig(hidden=1024, inter=2048, n_heads=8, n_kv_heads=2, head_dim=128, rot_dims=64, theta=1e6,
                       vocab=8192, kv_cap=kv_cap)


class MtpPair:
    def __init__(self, cfg, seed):
        import block_speculative_decoding_fm_gb300 as fm
        self.fm, self.cfg, self.seed = fm, cfg, seed
        self.w = S.gen_mtp_weights(cfg, seed)
        self.h = fm.fm_mtp_create(cfg, fm.weight_items(self.w))
        self.o = MtpHead(cfg, {n: t.data for n, t in self.w.items()})
        self.st = self.o.new_state()
        self.rng = S.streams(seed)["features"]

    def forward(self, tokens, pos0, kv_lo):
        import torch
        hn = S.gen_mtp_hidden(self.rng, len(tokens), self.cfg.hidden)
        t = torch.tensor(tokens, dtype=torch.int32, device="cuda")
        hout = torch.zeros((len(tokens), self.cfg.hidden), dtype=torch.float32, device="cuda")
        drafts = torch.full((len(tokens),), -1, dtype=torch.int32, device="cuda")
        self.fm.fm_mtp_forward(self.h, t, torch.from_numpy(hn).cuda(), pos0, kv_lo, hout, drafts)
        torch.cuda.synchronize()
        ref = self.o.forward(self.st, self.o.embed(tokens), hn.astype(np.float64), pos0, kv_lo)
        return hout.cpu().numpy(), drafts.cpu().numpy(), ref

    def check_cache(self, rows):
        c = self.cfg
        for which, want in ((0, self.st.k), (1, self.st.v)):
            got = self.fm.fm_mtp_cache(self.h, which, rows, np.empty((rows, c.n_kv_heads * c.head_dim), np.float32))
            # the K/V rows come out of Q8_0 products whose weights the tensor cores see rounded to f16
            # (<= 2^-11 relative per weight): the same 1e-3 bound as the drafter's f16 cache rows
            assert rel_l2(got[:rows], want[:rows]) < 1e-3, (which, rel_l2(got[:rows], want[:rows]))

    def close(self):
        self.fm.fm_mtp_destroy(self.h)


def check_tokens(got, want, logits):
    for k in range(len(want)):
        if int(got[k]) != int(want[k]):
            m = float(top2_margin(np.asarray(logits[k])[None])[0])
            assert m < MARGIN, (k, int(got[k]), int(want[k]), m)
            return k
    return len(want)


@pytest.mark.parametrize("make", [S.mtp_micro_config, mid_config])
def test_mtp_passes_match_oracle(make):
    """Three passes (3 rows, then 1, then 8 = the maximum) over a growing
    cache with a window start kv_lo > 0: h' per row, the per-row drafts and the
    cache rows against the oracle."""
    cfg = make()
    p = MtpPair(cfg, 1201)
    pos, kv_lo = 4, 2
    # rows below pos are written first (the head's own earlier passes)
    p.forward([7, 8], 2, 2)
    for tokens in ([5, 17, 63], [11], list(range(100, 108))):
        hout, drafts, ref = p.forward(tokens, pos, kv_lo)
        assert rel_l2(hout, ref.hout) < REL_L2, rel_l2(hout, ref.hout)
        lg = p.o.logits(ref.hout)
        check_tokens(drafts, np.argmax(lg, axis=-1), lg)
        pos += len(tokens)
    p.check_cache(pos)
    p.close()


@pytest.mark.parametrize("make", [S.mtp_micro_config, mid_config])
def test_mtp_draft_chain_matches_oracle(make):
    """fm_mtp_draft: one pass over two pending rows, then three chained
    single-row passes on the device's own drafts; tokens and the cache rows
    every pass wrote."""
    import torch
    cfg = make()
    p = MtpPair(cfg, 1202)
    p.forward([3, 4, 5, 6], 0, 0)                  # history rows 0..3
    hn = S.gen_mtp_hidden(p.rng, 2, cfg.hidden)
    drafts = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    p.fm.fm_mtp_draft(p.h, torch.tensor([21, 22], dtype=torch.int32, device="cuda"), torch.from_numpy(hn).cuda(),
                      4, 1, 4, drafts)
    torch.cuda.synchronize()
    got = drafts.cpu().numpy()
    want, lg, _ = p.o.draft(p.st, [21, 22], hn.astype(np.float64), 4, 1, 4)
    n = check_tokens(got, want, lg)
    if n == 4:
        p.check_cache(4 + 2 + 3)
    assert p.fm.fm_mtp_last_launch_count(p.h) > 0
    p.close()


def test_mtp_errors():
    import torch
    import block_speculative_decoding_fm_gb300 as fm
    cfg = S.mtp_micro_config()
    w = S.gen_mtp_weights(cfg, 1203)
    with pytest.raises(fm.FmError) as e:
        fm.fm_mtp_create(cfg, fm.weight_items({k: v for k, v in w.items() if k != "ffn_up"}))
    assert e.value.status == fm.FM_ERR_INVALID_ARG
    with pytest.raises(fm.FmError) as e:
        fm.fm_mtp_create(cfg.replace(hidden=200), fm.weight_items(w))
    assert e.value.status == fm.FM_ERR_UNSUPPORTED
    h = fm.fm_mtp_create(cfg, fm.weight_items(w))
    t = torch.zeros((9,), dtype=torch.int32, device="cuda")
    hn = torch.zeros((9, cfg.hidden), dtype=torch.float32, device="cuda")
    with pytest.raises(fm.FmError) as e:
        fm.fm_mtp_forward(h, t, hn, 0, 0)                 # 9 rows > max_rows
    assert e.value.status == fm.FM_ERR_INVALID_ARG
    with pytest.raises(fm.FmError) as e:
        fm.fm_mtp_forward(h, t[:2], hn[:2], 3, 4)         # kv_lo > pos0
    assert e.value.status == fm.FM_ERR_INVALID_ARG
    with pytest.raises(fm.FmError) as e:
        fm.fm_mtp_forward(h, t[:2], hn[:2], cfg.kv_cap - 1, 0)
    assert e.value.status == fm.FM_ERR_INVALID_ARG
    fm.fm_mtp_destroy(h)


def test_mtp_full_shape():
    """The page's MCFG head (H 5120, I 17408, 24 / 4 heads of 256, NEOX on 64,
    vocab 248,320; eh_proj, attn_output and ffn_down in four K slices): a pass
    over four history rows, then a depth-3 draft from two pending rows."""
    import torch
    cfg = S.mtp_config(kv_cap=64)
    p = MtpPair(cfg, 1204)
    hout, drafts, ref = p.forward([1, 2, 3, 4], 0, 0)
    assert rel_l2(hout, ref.hout) < REL_L2, rel_l2(hout, ref.hout)
    hn = S.gen_mtp_hidden(p.rng, 2, cfg.hidden)
    d = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    p.fm.fm_mtp_draft(p.h, torch.tensor([10, 20], dtype=torch.int32, device="cuda"), torch.from_numpy(hn).cuda(),
                      4, 0, 3, d)
    torch.cuda.synchronize()
    want, lg, _ = p.o.draft(p.st, [10, 20], hn.astype(np.float64), 4, 0, 3)
    check_tokens(d.cpu().numpy(), want, lg)
    p.close()
