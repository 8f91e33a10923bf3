"""The byte ledger used for every GB/s figure, pinned to the pages' ledger formulas.

"case_norm_rope_quant.py" (Ch.28), Shape defaults (4096 tokens, 32 q + 8 kv heads, head_dim 128,
bf16 in, fp8 out, fp32 table): payload = elems*2 + elems*1 + rows*4, ideal lookup =
2*head_dim*2 + 2*tokens*head_dim*4. Our ledger differs only in the table term (half-width tables).
"""
from fp8_quant_memory_gb300 import ledger


def test_page_prologue_ledger_at_default_shape():
    rows = 4096 * 40
    elems = rows * 128
    payload = elems * 2 + elems * 1 + rows * 4
    lookup = 2 * 128 * 2 + 2 * 4096 * 128 * 4
    assert ledger.page_prologue_ideal_bytes(4096, 32, 8, 128) == payload + lookup
    assert payload + lookup == 67_764_736  # 67.76 MB


def test_our_prologue_ledger_halves_the_table_term():
    page = ledger.page_prologue_ideal_bytes(4096, 32, 8, 128)
    ours = ledger.qk_prologue_bytes(4096, 32, 8, 128)
    assert page - ours == 4096 * 128 * 4  # the page counts cos and sin at full head_dim width
    assert ours == 65_667_584


def test_large_prologue_ledger():
    assert ledger.qk_prologue_bytes(32768, 64, 8, 128) == (32768 * 72 * 128 * 3 + 32768 * 72 * 4
                                                           + 2 * 32768 * 64 * 4 + 2 * 128 * 2)


def test_fused_norm_rope_quant_ledger_matches_ch13_rule():
    """Ch.13 ledger, fused_norm_rope_quant: reads x, w, cos, sin; writes q and amax (one fp32 per row).
    At m = n = 4096, rope 128, bf16: 2mn + 2n + 2*(m*64*2) + mn + 4m bytes."""
    m = n = 4096
    expect = 2 * m * n + 2 * n + 2 * (m * 64 * 2) + m * n + 4 * m
    assert ledger.rope_quant_bytes(m, n, 128, "bf16", "bf16", write_y=False) == expect
    assert round(expect / 1e6, 2) == 51.4


def test_rmsnorm_ledgers():
    assert ledger.rmsnorm_fwd_bytes(8192, 4096) == 134_225_920
    assert ledger.rmsnorm_bwd_bytes(8192, 4096) == 201_342_976
    assert ledger.rope_bytes(65536, 192, 64, "fp16", "fp16") == 2 * 65536 * 192 * 2 + 192 * 2 + 2 * 65536 * 32 * 2


def test_page_norm_rope_quant_plans_at_the_page_shape():
    """Ch.13 ledger, fused_norm_rope_quant at 4096 x 4096, rope 128, bf16: 185.62 MB unfused, 51.40 MB fused."""
    from fp8_quant_memory_gb300 import ledger

    assert round(ledger.page_unfused_norm_rope_quant_bytes(4096, 4096, 128) / 1e6, 2) == 185.62
    assert round(ledger.page_fused_norm_rope_quant_bytes(4096, 4096, 128) / 1e6, 2) == 51.40
    assert ledger.page_fused_norm_rope_quant_bytes(4096, 4096, 128) == ledger.rope_quant_bytes(
        4096, 4096, 128, "bf16", "bf16", write_y=False)


def test_prologue_flops_match_the_pages_ledger():
    """10 * head_dim + 3 FLOP per row: 210.2 MFLOP for the 4096-token prologue and 3027 MFLOP for the
    32768-token one, as the Ch.28 page's ledger gives for these shapes (about 3.2 FLOP per byte)."""
    from fp8_quant_memory_gb300 import ledger

    assert ledger.qk_prologue_flops(4096, 32, 8, 128) == 4096 * 40 * 1283 == 210206720
    assert ledger.qk_prologue_flops(32768, 64, 8, 128) == 3026976768
    ai = ledger.qk_prologue_flops(4096, 32, 8, 128) / ledger.qk_prologue_bytes(4096, 32, 8, 128)
    assert 3.1 < ai < 3.3
