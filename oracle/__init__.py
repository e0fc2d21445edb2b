"""CPU oracle of the block-parallel drafter forward pass (fp64, numpy).

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and
``bench.py``'s cpu_baseline leg (and ``bench.py --impl reference``) may import
this package.  It shares no code with the CUDA library in
block_speculative_decoding_fm_gb300/ and the library never calls it.

Parity pins: every function here is checked by ``tests/test_oracle_*.py``
(``-m "not gpu"``) against closed forms, invariants, library routines and
brute force on tiny inputs; nothing in the oracle is "parity unpinned".
"""
from .accept import accept
from .common import argmax_rows, top2_margin
from .dflash import DFlash, DFlashResult, DFlashState
from .flashmap import DraftResult, FlashMap, FlashMapState

__all__ = ["accept", "argmax_rows", "top2_margin", "DFlash", "DFlashResult", "DFlashState",
           "DraftResult", "FlashMap", "FlashMapState"]
