"""The oracle's bf16 rounding against torch's cast on every fp32 bit pattern.

Round to nearest, ties to even, is the cast both sides of the parity check
use for every bf16 they write.  torch's CPU conversion is the reference
(the cast the pages' frameworks apply).  All 2^32 patterns are compared in
chunks of 2^24.  Non-NaN inputs must give the same bits.  NaN inputs must stay
NaN with the quiet bit set; their payload bits are not part of parity.
"""
import numpy as np
import torch

import oracle

CHUNK = 1 << 24


def test_bf16_rounding_exhaustive_against_torch():
    prev = oracle.get_threads()
    oracle.set_threads(max(1, min(8, torch.get_num_threads())))
    try:
        for start in range(0, 1 << 32, CHUNK):
            bits = np.arange(start, start + CHUNK, dtype=np.uint64).astype(np.uint32)
            x = bits.view(np.float32)
            got = oracle.bf16_round(x)
            want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            nan = np.isnan(x)
            if not np.array_equal(got[~nan], want[~nan]):
                bad = np.nonzero((got != want) & ~nan)[0][0]
                raise AssertionError(f"bf16 of 0x{bits[bad]:08x}: oracle 0x{got[bad]:04x}, "
                                     f"torch 0x{want[bad]:04x}")
            g = got[nan].astype(np.uint32)
            assert np.all(((g >> 7) & 0xFF) == 0xFF) and np.all(g & 0x7F) and np.all(g & 0x40)
    finally:
        oracle.set_threads(prev)
