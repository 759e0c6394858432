"""Launch-plan properties (host logic, no GPU): how the units (batch row,
channel tile) are grouped into segments and cut in time.

* The segments cover every unit once, in order.
* A split happens only when the units fill at least one round (8 warps on
  each of the GPU's 152 SMs: 608 two-warp blocks, 1216 one-warp blocks) and
  leave a partial round: the first segment is then a whole number of rounds
  of one-chunk units, the second the remaining units cut in time.
* A split never takes a problem out of the no-allocation forward: its chunk
  summaries stay within that entry point's 2 MiB scratch.
* The saved-state buffer (states, then the pre-gate readout) does not depend
  on the split.
"""

import itertools

import pytest

import mamba_selective_scan_fwd_gb300 as ss
from mamba_selective_scan_fwd_gb300 import binding

SMS = 152


def tile_of(N):
    # a lane holds 4 states (all of them below 4) of a channel pair; a warp covers
    # 16 pairs for N = 8, 16, 8 pairs for N = 32, 32 pairs for N <= 4
    return {32: 16, 16: 32, 8: 32}.get(N, 64)


def round_of(N):
    return 8 * SMS // (2 if N >= 16 else 1)


SHAPES = [(b, L, d, n) for b, L, d, n in itertools.product(
    (1, 2, 4, 8), (1, 100, 256, 4096), (1, 130, 4864, 5120, 9913, 19488), (1, 4, 16, 32))]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}L{s[1]}D{s[2]}N{s[3]}" for s in SHAPES])
def test_plan_segments(shape):
    Bsz, L, Dch, N = shape
    p = ss.plan_info(Bsz, L, Dch, N, ss.SS_BF16)
    units = Bsz * -(-Dch // tile_of(N))
    segs = p["segments"]
    assert sum(u for u, _ in segs) == units
    assert p["chunks"] == max(k for _, k in segs)
    assert p["fwd_kernels"] == sum(1 + (k > 1) for _, k in segs)
    # the backward adds a carry pass after each chunked segment's reverse summaries
    assert p["bwd_saved_kernels"] == p["fwd_kernels"] + sum(k > 1 for _, k in segs) + 2
    assert p["bwd_kernels"] == p["fwd_kernels"] + p["bwd_saved_kernels"]
    if len(segs) == 2:
        (u0, k0), (u1, k1) = segs
        assert k0 == 1 and u0 % round_of(N) == 0 and u0 > 0 and 0 < u1 < round_of(N) and k1 > 1
        assert ss.fwd_workspace_bytes(Bsz, L, Dch, N, ss.SS_BF16) <= binding.FWD_NOALLOC_MAX_SCRATCH_BYTES
    slots = -(-L // 32) * 4  # one saved state every 8 steps of L rounded up to 32
    states = -(-(units * tile_of(N) * slots * N * 4) // 256) * 256
    assert ss.saved_bytes(Bsz, L, Dch, N, ss.SS_BF16) == states + Bsz * L * Dch * 4  # states, then y0


def test_split_appears_for_a_partial_round():
    # 640 units = 4 rounds of 152 + 32: the 32 are cut in time
    assert ss.plan_info(4, 4096, 5120, 16, ss.SS_BF16)["segments"] == [(608, 1), (32, 19)]
    # 1216 units = 2 whole rounds: no split
    assert ss.plan_info(4, 4096, 32 * 304, 16, ss.SS_BF16)["segments"] == [(1216, 1)]
    # 760 units = a round of 608 + 152: the 152 are cut into 4 chunks (one more round of blocks)
    assert ss.plan_info(4, 4096, 6080, 16, ss.SS_BF16)["segments"] == [(608, 1), (152, 4)]
    # 1064 = 608 + 456: cutting the 456 takes more than the partial round
    assert ss.plan_info(1, 4096, 32 * 1064, 16, ss.SS_BF16)["segments"] == [(1064, 1)]
