"""The benchmark's algorithmic bytes against the unified page format.

The roofline fractions divide these byte counts by measured times, so each
per-token figure is derived here from the page layout (K row, V share of a
value row, the two 4-byte metadata words, score and position) rather than
restated: attention reads a stored token's codes and metadata, the score
update reads and writes its fp32 score, the prompt compaction reads fp16 K
and V (512 B a token-head) and writes the whole slot."""
import pytest

import bench
from tests import pagefmt

D = pagefmt.D


def read_bytes(tier):
    """Codes and metadata of one stored token, as the attention kernel reads them."""
    kb, vb = pagefmt.BITS[tier]
    g = 8 // vb
    return D * kb // 8 + 128 // g + 4 + 4


def slot_bytes(tier):
    """Everything a token occupies in its page: codes, metadata, score, position."""
    return read_bytes(tier) + 4 + 4


@pytest.mark.parametrize("tier,name", [(pagefmt.HI, "HI_BYTES"), (pagefmt.LO, "LO_BYTES"),
                                       (pagefmt.MID, "MID_BYTES")])
def test_attention_bytes_per_token_follow_the_page_format(tier, name):
    assert getattr(bench, name) == read_bytes(tier)


def test_attention_bytes_of_a_call():
    n_req, hq = 3, 12
    per_head = hq * (D * 2 + D * 4)   # q fp16 in, out fp32 back, per query head
    assert bench.attn_bytes(5, 7, n_req, hq, False) == 5 * read_bytes(pagefmt.HI) + 7 * read_bytes(pagefmt.LO) \
        + n_req * per_head
    upd = bench.attn_bytes(5, 7, n_req, hq, True, mid_tokens=2)
    assert upd == 5 * read_bytes(pagefmt.HI) + 7 * read_bytes(pagefmt.LO) + 2 * read_bytes(pagefmt.MID) \
        + 8 * (5 + 7 + 2) + n_req * per_head


def test_prompt_bytes_of_a_call():
    hi, lo, mid, n_th, n_req, hq = 11, 13, 3, 40, 2, 8
    obs = n_req * 32 * hq * D * 2      # the observation queries, fp16
    want = 2 * D * 2 * n_th + slot_bytes(pagefmt.HI) * hi + slot_bytes(pagefmt.LO) * lo \
        + slot_bytes(pagefmt.MID) * mid + obs
    assert bench.prompt_bytes(hi, lo, n_th, n_req, hq, mid_tokens=mid) == want
    # a pruned token costs its read only
    assert bench.prompt_bytes(0, 0, 1, 0, hq) == 2 * D * 2


def test_page_prefix_read_by_attention_holds_the_counted_bytes():
    # the bytes counted per token fit in the K | V | meta prefix of a page of
    # that tier (the attention kernel copies that prefix), for the 3.5 KB pages
    for tier, t in ((pagefmt.HI, 16), (pagefmt.LO, 32), (pagefmt.MID, 16)):
        offs, end = pagefmt.segment_offsets(t, *pagefmt.BITS[tier])
        assert offs[4] >= t * read_bytes(tier)
        assert end <= 3584
