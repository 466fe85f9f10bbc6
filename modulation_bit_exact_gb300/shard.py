"""Row sharding of the norm/modulation path across ranks.

Every operation is independent per row (the QKV epilogue per token and head),
so N processes split the rows into contiguous blocks and run the same calls on
their blocks with no collective on the data path.  The only constraint is the
modulation mapping: row r uses modulation row r // (rows // mod_rows), and a
shard must keep that mapping expressible for its own call, i.e. it must be
whole samples (their modulation rows) or lie inside one sample (its one
modulation row).  `row_shard` returns such a split.
"""
from __future__ import annotations


def row_shard(rows: int, mod_rows: int, world: int, rank: int) -> tuple[int, int, int, int]:
    """(row_lo, row_hi, mod_lo, mod_hi) of `rank`'s contiguous block of a
    [rows, D] operation whose modulation has `mod_rows` rows.

    Per-token modulation (mod_rows == rows), or whole samples when
    mod_rows % world == 0: equal contiguous blocks (the first rows % world
    ranks take one row more).  Otherwise, when world % mod_rows == 0, each
    sample is split among world // mod_rows ranks, each block inside one
    sample.  Any other combination raises ValueError."""
    if not (0 <= rank < world) or rows <= 0 or mod_rows <= 0 or rows % mod_rows:
        raise ValueError("bad shard arguments")
    seq = rows // mod_rows

    def split(n, parts, i):
        q, r = divmod(n, parts)
        lo = i * q + min(i, r)
        return lo, lo + q + (1 if i < r else 0)

    if mod_rows == rows:
        lo, hi = split(rows, world, rank)
        return lo, hi, lo, hi
    if mod_rows % world == 0:
        m_lo, m_hi = split(mod_rows, world, rank)
        return m_lo * seq, m_hi * seq, m_lo, m_hi
    if world % mod_rows == 0:
        per = world // mod_rows
        m = rank // per
        lo, hi = split(seq, per, rank % per)
        return m * seq + lo, m * seq + hi, m, m + 1
    raise ValueError(f"{mod_rows} modulation rows cannot be split evenly over {world} ranks")
