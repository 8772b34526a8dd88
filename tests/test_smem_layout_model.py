"""Shared-memory bank arithmetic behind two layout constants of the prefill GEMM,
read from its source so that a change to either is checked.

Shared memory has 32 four-byte banks. A 16-byte access covers 4 consecutive
banks, and 8 lanes' 16-byte accesses are served together. They are conflict-free
when the 8 accesses cover all 32 banks.

- Q6_K packed blocks sit in a kQ6Win-byte window per weight row. The dequant
  threads of 8 consecutive rows read the same column. The kernel chose 240
  bytes over the minimal 224, whose 56-word pitch makes every fourth row collide.
- The split-K exchange stores a peer's fp32 partial tile with rows padded to
  BN·4 + 16 bytes. The 8 lanes of a wavefront write 8 rows at the same column.
  Without the padding the pitch is a multiple of 16 words, and the 8 rows pile
  onto the same banks.
"""
import os
import re

import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "quantized_q4_matmul_gb300", "csrc",
                   "qk_gemm_tc.cu")


def source():
    with open(SRC) as f:
        return f.read()


def conflict_free(pitch_bytes, rows=8):
    assert pitch_bytes % 16 == 0  # 16-byte accesses stay 16-byte aligned
    words = pitch_bytes // 4
    banks = [(r * words + i) % 32 for r in range(rows) for i in range(4)]
    return len(set(banks)) == 32


def test_q6k_window_is_conflict_free():
    win = int(re.search(r"constexpr int kQ6Win = (\d+);", source()).group(1))
    assert win >= 224            # the 210-byte block plus up to 14 bytes of misalignment
    assert conflict_free(win)
    assert not conflict_free(224)  # the minimal window: rows 0 and 4 share banks


@pytest.mark.parametrize("BN", range(16, 257, 16))
def test_split_k_exchange_pitch_is_conflict_free(BN):
    pad = int(re.search(r"peer_pitch = \(uint32_t\)BN \* 4 \+ (\d+);", source()).group(1))
    assert conflict_free(BN * 4 + pad)
    assert not conflict_free(BN * 4)  # unpadded: a multiple of 16 words
