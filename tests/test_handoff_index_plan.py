"""The handoff kernel's copy plan, restated on the CPU (no GPU, no kernel
code): for every 64-aligned block of a request's positions, the producer
warp issues one 1-D bulk copy per prefill page the block touches and
tensor, and writes each position's decode-pool offset into the stage header.
Checked here for every page-size pair, both head dims and many start
offsets and lengths:
- the copies cover exactly the positions [first, first + count) of the block
  whose prefill page is in the pool, once each;
- every copy stays inside its prefill page and inside the stage's rows, and
  its addresses and size are multiples of 16 bytes (the bulk-copy rule);
- the byte count announced to the stage's barrier equals the bytes copied;
- the decode offsets stay inside the decode pool;
- the launch grid gives every block group of a request to exactly one CTA.
"""
import itertools

import numpy as np

BLOCK = 64         # positions per stage
BLOCKS_PER_CTA = 2


def _plan(f, n, Ps, Pd, D, H, sbt, dbt, src_pages, dst_pages):
    """Per block: (copies, tx, header) as the producer forms them.  A copy is
    (smem row, prefill page, slot, rows); header[r] is the decode element
    offset of head 0 for position blk*64 + r, or -1."""
    row_bytes = 2 * D
    out = []
    for blk in range(f // BLOCK, (f + n - 1) // BLOCK + 1):
        lo, hi = max(blk * BLOCK, f), min(blk * BLOCK + BLOCK, f + n)
        copies, header, tx = [], [-1] * BLOCK, 0
        for r in range(BLOCK):
            p = blk * BLOCK + r
            if not (lo <= p < hi):
                continue
            sp, dp = sbt[p // Ps], dbt[p // Pd]
            src_ok = 0 <= sp < src_pages
            if src_ok and 0 <= dp < dst_pages:
                header[r] = (dp * H * Pd + p % Pd) * D
            if src_ok and (p == lo or p % Ps == 0):
                run = min(hi, (p // Ps + 1) * Ps) - p
                copies.append((r, sp, p % Ps, run))
                tx += 2 * run * row_bytes
        out.append((blk, lo, hi, copies, tx, header))
    return out


def test_copy_plan_covers_each_position_once():
    rng = np.random.default_rng(3)
    for Ps, Pd, D in itertools.product((16, 32, 64), (16, 32, 64), (64, 128)):
        H = 8
        row_bytes = 2 * D
        src_MP, dst_MP = 40, 60
        src_pages, dst_pages = 100, 150
        for _ in range(30):
            f = int(rng.integers(0, 200))
            cap = min(src_MP * Ps, dst_MP * Pd)
            n = int(rng.integers(0, cap - f + 1))
            sbt = rng.permutation(src_pages)[:src_MP].astype(np.int64)
            dbt = rng.permutation(dst_pages)[:dst_MP].astype(np.int64)
            sbt[rng.integers(0, src_MP)] = -1          # a prefill page outside the pool
            dbt[rng.integers(0, dst_MP)] = dst_pages   # a decode page outside the pool
            if n == 0:
                continue
            seen = set()
            for blk, lo, hi, copies, tx, header in _plan(f, n, Ps, Pd, D, H, sbt, dbt,
                                                         src_pages, dst_pages):
                copied = 0
                for r, sp, slot, run in copies:
                    assert 0 <= r and r + run <= BLOCK          # inside the stage's rows
                    assert slot + run <= Ps                    # inside the prefill page
                    assert run > 0
                    # element offsets are multiples of D; byte addresses and sizes of 16
                    src_byte = ((sp * H + 0) * Ps + slot) * D * 2
                    assert src_byte % 16 == 0 and (r * row_bytes) % 16 == 0
                    assert (run * row_bytes) % 16 == 0
                    for k in range(run):
                        p = blk * BLOCK + r + k
                        assert p not in seen
                        seen.add(p)
                        assert sbt[p // Ps] == sp
                    copied += 2 * run * row_bytes
                assert copied == tx
                for r, off in enumerate(header):
                    if off >= 0:
                        assert off + (H - 1) * Pd * D + D <= dst_pages * H * Pd * D
            want = {p for p in range(f, f + n) if 0 <= sbt[p // Ps] < src_pages}
            assert seen == want


def test_grid_reaches_every_block():
    """The grid's x extent is min(ceil(ceil(min capacity / 64) / 2), about 16
    waves of CTAs / requests); CTA x takes block groups x, x + gx, ...: every
    block group of every request that fits both tables falls to exactly one
    CTA of the request's row."""
    sms = 152
    for Ps, Pd in itertools.product((16, 32, 64), repeat=2):
        for src_MP, dst_MP in ((1, 1), (3, 7), (40, 60), (129, 513), (2048, 8192)):
            max_tok = min(src_MP * Ps, dst_MP * Pd)
            blocks = -(-max_tok // BLOCK)
            for B in (1, 8, 64, 4096):
                gy = min(B, 65535)
                gx = min(-(-blocks // BLOCKS_PER_CTA), max(1, -(-(16 * 2 * sms) // gy)))
                for f in range(0, max_tok, max(1, max_tok // 17)):
                    n = max_tok - f
                    groups = -(-((f + n - 1) // BLOCK - f // BLOCK + 1) // BLOCKS_PER_CTA)
                    owners = [[] for _ in range(groups)]
                    for bx in range(gx):
                        for x in range(bx, groups, gx):
                            owners[x].append(bx)
                    assert all(len(o) == 1 for o in owners)
