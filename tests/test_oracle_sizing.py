"""Pins of the oracle's sizing arithmetic against the values the pages print."""
import os

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


@pytest.mark.parametrize("row", list(_rows("kv_sizing.txt")), ids=lambda r: "-".join(r[:6]))
def test_kv_sizing_matches_pages(row):
    L, H, d, b, tokens = (int(x) for x in row[:5])
    quantity, expected = row[5], row[6]
    per_tok = oracle.kv_bytes_per_token(L, H, d, b)
    total = per_tok * tokens
    if quantity == "bytes_per_token":
        assert per_tok == int(expected)
    elif quantity == "gib_5":
        assert f"{total / 2**30:.5f}" == expected
    elif quantity == "gib_3":
        assert f"{total / 2**30:.3f}" == expected
    elif quantity == "gib_2f":
        assert f"{total / 1024**3:.2f}" == expected
    elif quantity == "kib_per_token_0f":
        assert f"{per_tok / 1024:.0f}" == expected
    elif quantity == "gib_0f":
        assert f"{total / 2**30:.0f}" == expected
    else:  # pragma: no cover
        raise AssertionError(quantity)


def test_gqa_factor_seven():
    # "Basics of LLM Inference ...", s.11: MHA would be 7 times larger than 4 KV heads of 28 query heads
    assert oracle.kv_bytes_per_token(28, 28, 128, 2) == 7 * oracle.kv_bytes_per_token(28, 4, 128, 2)


def test_fp8_halves_bytes():
    # s.2: an FP8 cache makes b = 1, halving the bytes again
    assert 2 * oracle.kv_bytes_per_token(28, 2, 128, 1) == oracle.kv_bytes_per_token(28, 2, 128, 2)


def test_concurrency_banner():
    # drpranayjha.com, "Watching the vLLM scheduler under load": 151,552 cache tokens -> 18.5x at 8,192
    assert f"{151552 / 8192:.1f}" == "18.5"


@pytest.mark.parametrize("row", list(_rows("block_counts.txt")), ids=lambda r: r[0])
def test_block_counts_match_pages(row):
    tokens, blocks, last = (int(x) for x in row)
    assert oracle.num_logical_blocks(tokens, 16) == blocks
    assert oracle.last_block_fill(tokens, 16) == last


def test_usable_blocks_after_null_block():
    # s.4: of 1,345 blocks one is the null block
    assert oracle.num_logical_blocks(21520) - 1 == 1344
