"""Shared-memory bank arithmetic behind two layout constants of the prefill GEMM,
read from its source so that a change to either is checked.

Shared memory has 32 four-byte banks. A 16-byte access covers 4 consecutive
banks, and 8 lanes' 16-byte accesses are served together. They are conflict-free
when the 8 accesses cover all 32 banks.

- Q6_K packed blocks sit in a kQ6Win-byte window per weight row. The dequant
  threads of 8 consecutive rows read the same column. The kernel chose 240
  bytes over the minimal 224, whose 56-word pitch makes every fourth row collide.
- The split-K exchange stores a slice of fp32 partial sums (c chunks of 16
  columns) with rows padded to 64·c + 16 bytes. The 8 lanes of a wavefront
  write 8 rows at the same column. Without the padding the pitch is a multiple
  of 16 words, and the 8 rows pile onto the same banks.
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
@pytest.mark.parametrize("ks", range(2, 9))
def test_split_k_exchange_pitch_is_conflict_free(BN, ks):
    m = re.search(r"return \(uint32_t\)\(\(BN / 16 \+ ks - 1\) / ks\) \* 64u \+ (\d+)u;", source())
    pad = int(m.group(1))
    chunks = (BN // 16 + ks - 1) // ks
    assert conflict_free(chunks * 64 + pad)
    assert not conflict_free(chunks * 64)  # unpadded: a multiple of 16 words


def _chunk(zz, n, ks):  # first token chunk of rank zz's slice: ceil(zz * n / ks)
    return (zz * n + ks - 1) // ks


@pytest.mark.parametrize("BN", range(16, 257, 16))
@pytest.mark.parametrize("ks", range(2, 9))
def test_split_k_exchange_slots(BN, ks):
    """The exchange's slot layout, restated: rank zz owns chunks
    [c(zz), c(zz + 1)); an owner keeps ks - 1 receive slots (sender s at slot
    s, or s - 1 above the owner) followed by one send slot per other owner; a
    rank without a slice sends from slot 0 on.  Every slice is owned once,
    rank 0 always owns one, no rank uses a slot twice, and every rank stays
    within max(ks - 2 + owners, owners) slots, the bound the host checks
    against the stage region.  The device evaluates c(zz) as
    ((zz * n + ks - 1) * kinv) >> 16 with kinv = ceil(65536 / ks)."""
    n = BN // 16
    owns = [_chunk(z + 1, n, ks) > _chunk(z, n, ks) for z in range(ks)]
    owners = sum(owns)
    assert owners == min(ks, n) and owns[0] and _chunk(ks, n, ks) == n
    kinv = (65536 + ks - 1) // ks
    assert all(((z * n + ks - 1) * kinv) >> 16 == _chunk(z, n, ks) for z in range(ks + 1))
    bound = max(ks - 2 + owners, owners)
    for z in range(ks):
        used = set()
        if owns[z]:
            used |= {s if s < z else s - 1 for s in range(ks) if s != z}
        for d in range(ks):
            if d == z or not owns[d]:
                continue
            below = min(d, _chunk(d, n, ks))
            assert below == sum(owns[:d])
            k = (ks - 1 if owns[z] else 0) + below - (1 if owns[z] and z < d else 0)
            assert k not in used and k < bound
            used.add(k)
