"""The forward's launch layout (``maxsim_forward_plan``, host only): the
M-tile choice, CTAs per SM, the row-group / part grid and the K-block-half
streaming choice for the shapes the benchmark and the tests use."""
import pytest

import late_interaction_retrieval_maxsim_gb300 as m

SMS = 152
COLBERT_TOKENS = 8_319_285      # 50,000 documents, Ld ~ U[32, 300]


def plan(n_q, lq, n_docs, total, dtype="fp16", argmax=True):
    return m.maxsim_forward_plan(n_q, lq, n_docs, total, dtype, with_argmax=argmax, sm_count=SMS)


@pytest.mark.parametrize("n_q,nmt,ctas,groups", [
    (1, 1, 2, 1),     # 32 rows: one M-tile, two CTAs per SM
    (4, 1, 2, 1),     # 128 rows
    (8, 2, 2, 1),     # 256 rows
    (9, 4, 1, 1),     # 288 rows: one CTA of four M-tiles (one empty)
    (12, 4, 1, 1),    # 384 rows
    (14, 2, 2, 2),    # 448 rows
    (16, 2, 2, 2),    # 512 rows: the ColBERT benchmark
    (20, 2, 2, 3),    # 640 rows: a half-empty last group of two
    (32, 2, 2, 4),
])
def test_m_tiles_ctas_and_groups(n_q, nmt, ctas, groups):
    p = plan(n_q, 32, 50_000, COLBERT_TOKENS)
    assert (p["m_tiles"], p["ctas_per_sm"], p["row_groups"]) == (nmt, ctas, groups)
    assert p["parts"] == ctas * SMS // groups            # every SM holds its CTAs


def test_k_block_halves_choice():
    # two M-tiles, short documents: only without argmax
    assert not plan(16, 32, 50_000, COLBERT_TOKENS)["k_block_halves"]
    assert plan(16, 32, 50_000, COLBERT_TOKENS, argmax=False)["k_block_halves"]
    # ColPali pages (1024 tokens on average): with argmax too
    p = plan(1, 1024, 10_000, 10_000 * 1024)
    assert (p["m_tiles"], p["row_groups"], p["parts"], p["k_block_halves"]) == (2, 4, 76, True)
    # one or four M-tiles never stream halves
    assert not plan(1, 32, 50_000, COLBERT_TOKENS, argmax=False)["k_block_halves"]
    assert not plan(12, 32, 50_000, COLBERT_TOKENS, argmax=False)["k_block_halves"]


def test_int8_layouts():
    p = plan(32, 32, 100_000, 27_200_000, "int8")
    assert (p["m_tiles"], p["ctas_per_sm"], p["row_groups"], p["parts"]) == (4, 1, 2, 76)
    assert not p["k_block_halves"]
    p = plan(1, 32, 100_000, 27_200_000, "int8")
    assert (p["m_tiles"], p["ctas_per_sm"]) == (1, 2)
    assert plan(8, 32, 100_000, 27_200_000, "int8")["ctas_per_sm"] == 1     # two M-tiles, one CTA


def test_query_padding():
    assert plan(2, 100, 10, 1000)["m_tiles"] == 2      # 100 tokens pad to 128: 256 rows
    assert plan(3, 7, 10, 1000)["m_tiles"] == 1        # 7 pads to 8


def test_no_kernel_and_errors():
    for args in ((0, 32, 10, 100), (2, 0, 10, 100), (2, 32, 0, 0), (2, 32, 10, 0)):
        assert plan(*args) == {"m_tiles": 0, "ctas_per_sm": 0, "row_groups": 0, "parts": 0,
                               "k_block_halves": False}
    with pytest.raises(Exception):
        m.maxsim_forward_plan(-1, 32, 10, 100, sm_count=SMS)
    with pytest.raises(Exception):
        m.maxsim_forward_plan(1, 32, 10, 100, sm_count=0)


def test_sizes_the_forward_rejects_are_rejected_here_too():
    """The plan applies the forward's own size limits: a token count beyond
    the kernels' 32-bit row range, or padded rows beyond int32, is an
    argument error (status 1), as maxsim_forward reports it."""
    with pytest.raises(m.MaxSimError) as e:
        m.maxsim_forward_plan(1, 32, 10, 2**31 - 1, sm_count=SMS)
    assert e.value.status == 1
    with pytest.raises(m.MaxSimError) as e:
        m.maxsim_forward_plan(2**26, 32, 10, 1000, sm_count=SMS)      # 2^31 padded rows
    assert e.value.status == 1
    assert plan(1, 32, 10, 2**31 - 1 - 256)["m_tiles"] == 1       # the largest token count accepted
