"""Bounds of the B-scale span copy (host-side arithmetic, no GPU).

A tile's B scales are copied in one bulk copy of the 16-byte aligned span of
global memory that holds the rows of its (up to 3) 128-column blocks, into a
shared-memory buffer of `sb_buf_words(kb)` 32-bit words (csrc/dg_params.h).
For every row length (fp32: K/128 words, packed UE8M0: ceil(K/512)), every
start offset within a 16-byte unit and every row count, the copy must fit the
buffer, be a multiple of 16 bytes, cover the rows, and the promotion's reads
(the tile's rows from `lead` words into the buffer) must stay inside it."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def sb_buf_words_from_header():
    src = open(os.path.join(ROOT, "moe_grouped_gemm_bf16_gb300", "csrc", "dg_params.h")).read()
    m = re.search(r"constexpr int sb_buf_words\(int kb\) \{ return (.+?); \}", src)
    assert m, "sb_buf_words not found"
    expr = m.group(1)
    assert re.fullmatch(r"[\s\dkb+*&~()]+", expr), expr
    return lambda kb: eval(expr, {}, {"kb": kb})


def test_span_copy_fits_and_covers_the_rows():
    words = sb_buf_words_from_header()
    for kb in range(1, 513):
        buf = words(kb)
        assert buf % 4 == 0 and buf >= 3 * kb
        for packed in (False, True):
            row = (kb + 3) // 4 if packed else kb
            for lead in range(4):                  # first row's word offset in its 16-byte unit
                for nrows in (1, 2, 3):
                    a = 4 * lead                   # byte address mod 16 (a 16-byte base added)
                    a0 = a & ~15
                    a1 = (a + nrows * row * 4 + 15) & ~15
                    size = a1 - a0
                    assert size % 16 == 0 and size <= 4 * buf, (kb, packed, lead, nrows)
                    assert a0 <= a and a1 >= a + nrows * row * 4
                    # the promotion reads word (lead + jb * row + idx) for rows jb < 3
                    # (rows past the copied ones hold stale words, never stored)
                    last_idx = (kb - 1) >> 2 if packed else kb - 1
                    assert lead + 2 * row + last_idx < buf, (kb, packed, lead)
