"""The C-ABI library builds for sm_103a, loads without a GPU, exports every symbol
include/mla.h declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

from mla_decode_attention_absorbed_gb300 import build, mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mla.load()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_symbols())
    for n in ("mla_absorb_q", "mla_decode_attn", "mla_out_proj", "mla_naive_decode", "mla_decode_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) == set(mla.EXPORTS)


def test_abi_version_and_status_strings(lib):
    assert lib.mla_abi_version() == 2
    for code in range(10):
        assert lib.mla_status_string(code).decode().startswith("MLA_")
    assert lib.mla_status_string(99).decode() == "unknown mla status"


def dsv3(B=4, s_q=1):
    return mla.Problem(B, 128, s_q, 512, 64, 128, 128, 192 ** -0.5)


def fake_cache(T=4096, paged=False):
    # addresses are never dereferenced: these calls fail or size on the host only
    kv, lens = 0x10000, 0x20000
    if paged:
        return mla.Cache(kv, 0, 0, 0x30000, T // 64, 64, 1000, lens, 0)
    return mla.Cache(kv, T * 576, T, None, 0, 64, 0, lens, 0)


def test_host_validation_without_gpu(lib):
    d = dsv3().dims()
    c = fake_cache()
    nul = ctypes.c_void_p(0)
    a = ctypes.c_void_p(0x40000)
    # NULL dims / pointers
    assert lib.mla_absorb_q(None, a, a, a, a, nul) == 1
    assert lib.mla_absorb_q(ctypes.byref(d), nul, a, a, a, nul) == 1
    # misaligned pointer
    assert lib.mla_absorb_q(ctypes.byref(d), ctypes.c_void_p(0x40008), a, a, a, nul) == 4
    # unsupported shapes
    for bad in (dict(d_c=96), dict(d_c=1024), dict(d_rope=8), dict(d_nope=24), dict(d_v=512), dict(H=65537),
                dict(H=65536), dict(B=65536), dict(B=65535, s_q=129)):
        p = dsv3()
        for k, v in bad.items():
            setattr(p, k, v)
        dd = p.dims()
        assert lib.mla_absorb_q(ctypes.byref(dd), a, a, a, a, nul) == 6, bad
    # negative sizes
    p = dsv3()
    p.B = -1
    dd = p.dims()
    assert lib.mla_out_proj(ctypes.byref(dd), a, a, a, nul) == 2
    # decode: workspace too small, bad split count, bad cache
    need = lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c), 4)
    assert need > 256
    assert lib.mla_decode_attn(ctypes.byref(d), a, ctypes.byref(c), a, a, a, need - 16, 4, nul) == 5
    assert lib.mla_decode_attn(ctypes.byref(d), a, ctypes.byref(c), a, a, a, need, 65, nul) == 2
    assert lib.mla_decode_attn(ctypes.byref(d), a, None, a, a, a, need, 4, nul) == 1
    bad_stride = mla.Cache(0x10000, 100, 4096, None, 0, 64, 0, 0x20000, 0)
    assert lib.mla_decode_attn(ctypes.byref(d), a, ctypes.byref(bad_stride), a, a, a, need, 4, nul) == 2
    odd_page = mla.Cache(0x10000, 0, 0, 0x30000, 64, 32, 100, 0x20000, 0)
    assert lib.mla_decode_attn(ctypes.byref(d), a, ctypes.byref(odd_page), a, a, a, need, 4, nul) == 6
    assert lib.mla_read_status(None, None, nul) == 1


def test_workspace_and_split_queries(lib):
    d = dsv3(B=64).dims()
    for paged in (False, True):
        c = fake_cache(4096, paged)
        s = lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(c))
        assert 1 <= s <= 152
        one = lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c), 1)
        four = lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c), 4)
        assert one >= 4 and four >= 64 * 4 * 128 * 512 * 4
    assert lib.mla_decode_workspace_size(None, None, 0) == 0
    naive = lib.mla_naive_workspace_size(ctypes.byref(d), ctypes.byref(fake_cache(4096)))
    assert naive >= 64 * 128 * 4096 * 256 * 2


def one_cta(B, s_q):
    """Dims whose attention runs one CTA per 128-row work item (d_c <= 256)."""
    return mla.Problem(B, 128, s_q, 256, 64, 128, 128, 0.1)


def test_tail_plan_fills_the_last_wave(lib):
    """One-CTA dims, more 128-row work items than a wave of 152 SMs holds: the plan
    leaves them whole except the sequences of the partly filled last wave, which it
    splits, and the workspace holds only their partials."""
    d = one_cta(B=40, s_q=4).dims()  # 160 work items = 1 wave + 8 (2 sequences)
    c = fake_cache(8192)
    # 152 // 8 = 19 pieces, capped at 16 (pieces of at least 8 of the 128 tiles)
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(c)) == 16
    tail_rows = 2 * 16 * 4 * 128  # the last 2 sequences, 16 pieces, 512 rows each
    need = lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c), 0)
    assert tail_rows * 256 * 4 <= need < 2 * tail_rows * 256 * 4
    # an explicit count splits every sequence
    assert lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c), 2) >= 40 * 2 * 512 * 256 * 4
    # whole waves, or one wave, keep the plain plan
    d = one_cta(B=38, s_q=4).dims()
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(c)) == 1
    assert lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c), 0) < 4096
    d = one_cta(B=30, s_q=4).dims()
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(c)) == 1
    # pieces stay at least 8 tiles long: a 1024-token history allows 2 pieces
    d = one_cta(B=39, s_q=4).dims()  # 156 work items: one sequence in the last wave
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(fake_cache(1024))) == 2
    # the tail's pieces must still fit the grid: 65,535 sequences leave no room for them
    d = one_cta(B=65535, s_q=1).dims()  # 65,535 items = 431 waves + 23
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(c)) == 1
    d = one_cta(B=65535 - 152, s_q=1).dims()  # 65,383 items = 430 waves + 23: 23 x 6 pieces fit
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(c)) == 6


def test_balanced_plan_for_pair_kernels(lib):
    """DeepSeek-V3 widths (CTA pairs), MLA_SPLITS_BALANCED: the batch's tiles are
    dealt out to groups of pairs, one group per 76 // (128-row blocks) pair slots,
    capped so that a range holds at least 8 tiles of what max_seq_len allows; the
    workspace holds the merge counters, the tile prefix, the (m, l) hand-over and
    two bf16 pieces per pair.  The library's choice takes it on a contiguous cache
    where it gives the busiest pair slot at least 16 tiles fewer than the split
    plans; FP8 caches, one-CTA widths and 4096 sequences or more cannot have it."""
    def rup(n):
        return (n + 255) // 256 * 256

    def balanced_bytes(B, pairs, n_rb, d_c=512):
        # status, merge counters, tile prefix, (m, l) hand-over, pieces' (m, l), pieces' rows
        return (256 + rup(B * n_rb * 2 * 4) + rup((B + 1) * 4) + rup(pairs * 2 * 2 * 128 * 3 * 4)
                + rup(pairs * 2 * 128 * 16) + pairs * 2 * 128 * d_c * 2)

    BAL = mla.SPLITS_BALANCED
    c = fake_cache(4096)
    # (3 sequences x 64 tiles allow 192 / 8 = 24 ranges, fewer than the 76 // 3 = 25 slots)
    for B, s_q, groups in ((64, 1, 76), (16, 1, 76), (64, 4, 19), (64, 2, 38), (3, 3, 24)):
        d = dsv3(B=B, s_q=s_q).dims()
        need = lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c), BAL)
        assert need == balanced_bytes(B, groups * s_q, s_q), (B, s_q)
    # few tiles: 2 sequences of at most 256 tokens (8 tiles) make one range
    d = dsv3(B=2, s_q=1).dims()
    assert lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(fake_cache(256)), BAL) == balanced_bytes(2, 1, 1)
    # the library's choice: 64 x 4096 tokens, one sequence a pair (64 tiles) against
    # 54 balanced: the unsplit plan
    d = dsv3(B=64, s_q=1).dims()
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(c)) == 1
    # 16 x 32768 tokens: 4 pieces of 128 tiles against 108 balanced: the balanced plan
    d = dsv3(B=16, s_q=1).dims()
    c32 = fake_cache(32768)
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(c32)) == 76
    assert lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c32), 0) == balanced_bytes(16, 76, 1)
    # 16 x 4096 tokens: 16 tiles a piece against 14: the split plan
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(c)) == 4
    # more than one wave of 76 pairs (256 items = 3 waves + 28): the busiest slot
    # streams 3 x 128 + 64 tiles on the tail plan, 432 balanced (19 ranges a block):
    # the balanced plan on a contiguous cache, the tail plan on a paged one
    d = dsv3(B=64, s_q=4).dims()
    c8 = fake_cache(8192)
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(c8)) == 19
    assert lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c8), 0) == balanced_bytes(64, 76, 4)
    c8p = fake_cache(8192, True)
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(c8p)) == 2  # 76 // 28
    tail_rows = 7 * 2 * 4 * 128  # the last 7 sequences, 2 pieces, 512 rows each
    need = lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c8p), 0)
    assert tail_rows * 512 * 4 <= need < 2 * tail_rows * 512 * 4
    # one wave on a paged cache keeps the split plan even where the tiles favour the
    # balanced one (16 x 32768 tokens: 4 pieces)
    d16 = dsv3(B=16, s_q=1).dims()
    assert lib.mla_decode_num_splits(ctypes.byref(d16), ctypes.byref(fake_cache(32768, True))) == 4
    # many sequences: 1000 x 4096 tokens, 843 tiles the busiest slot either way: the tail plan
    d1k = dsv3(B=1000, s_q=1).dims()
    assert lib.mla_decode_num_splits(ctypes.byref(d1k), ctypes.byref(c)) == 6
    # an explicit count keeps the split plan
    d = dsv3(B=64, s_q=1).dims()
    assert lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c), 2) >= 64 * 2 * 128 * 512 * 4
    # not available: 4096 sequences, an FP8 cache, one-CTA widths; below -1 is no count
    nul = ctypes.c_void_p(0)
    a = ctypes.c_void_p(0x1000)
    fp8 = mla.Cache(0x10000, 4096 * 576, 4096, None, 0, 64, 0, 0x20000, 0, 1, 0.5)
    for dd, cc in ((dsv3(B=4096, s_q=1).dims(), c), (dsv3(B=64, s_q=1).dims(), fp8), (one_cta(8, 1).dims(), c)):
        assert lib.mla_decode_workspace_size(ctypes.byref(dd), ctypes.byref(cc), BAL) == 0
        assert lib.mla_decode_attn(ctypes.byref(dd), a, ctypes.byref(cc), a, a, a, 1 << 30, BAL, nul) == 6
    d = dsv3(B=64, s_q=1).dims()
    assert lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c), -2) == 0
    assert lib.mla_decode_attn(ctypes.byref(d), a, ctypes.byref(c), a, a, a, 1 << 30, -2, nul) == 2
    assert lib.mla_decode_num_splits(ctypes.byref(d), ctypes.byref(fp8)) == 1  # one wave of 64 pairs


def test_expand_path_grid_limit(lib):
    """The expanded prefill runs one work item per (sequence, head): past 65535 of
    them it is unsupported, and the dispatch sizes the absorbed form instead."""
    nul = ctypes.c_void_p(0)
    a = ctypes.c_void_p(0x40000)
    c = fake_cache(4096)
    ok = dsv3(B=511, s_q=256).dims()  # 511 x 128 = 65,408 work items
    big = dsv3(B=512, s_q=256).dims()  # 65,536
    assert lib.mla_prefill_expand_workspace_size(ctypes.byref(ok), ctypes.byref(c)) > 0
    assert lib.mla_prefill_expand_workspace_size(ctypes.byref(big), ctypes.byref(c)) == 0
    assert lib.mla_prefill_expand(ctypes.byref(big), a, a, ctypes.byref(c), a, a, a, a, a, 1 << 40, nul) == 6
    assert lib.mla_prefill_workspace_size(ctypes.byref(big), ctypes.byref(c)) > 0  # the absorbed form


def test_prefill_crossover_matches_the_pages_formula(lib):
    """The library's dispatch point (host code) against the oracle's counter, which
    the page figures pin (S* = 128 at L = 512, 170 at 32K, 171 at 128K)."""
    from oracle import counts
    prob = mla.Problem(B=1, H=128, s_q=1, d_c=512, d_rope=64, d_nope=128, d_v=128, scale=1.0)
    for L in (512, 4096, 32768, 131072):
        assert abs(mla.prefill_crossover(prob, L) - counts.crossover_S(512, 128, 128, L)) < 1e-9
    assert 127.5 < mla.prefill_crossover(prob, 512) < 128.5
    assert mla.prefill_crossover(prob, 0) == 0.0


def test_naive_path_grid_limit(lib):
    """The naive path runs one grid slice per (sequence, head): past 65535 of them
    it is an argument error on the host, never a failed launch."""
    nul = ctypes.c_void_p(0)
    a = ctypes.c_void_p(0x40000)
    c = fake_cache(256)
    ok = dsv3(B=511).dims()  # 511 x 128 = 65,408
    big = dsv3(B=513).dims()  # 65,664
    assert lib.mla_naive_workspace_size(ctypes.byref(ok), ctypes.byref(c)) > 0
    assert lib.mla_naive_workspace_size(ctypes.byref(big), ctypes.byref(c)) == 0
    assert lib.mla_naive_decode(ctypes.byref(big), a, a, ctypes.byref(c), a, a, a, a, a, 1 << 40, nul) == 6
    # at DeepSeek-V3 widths the expansion holds rows [V_h | K_h | k_rope] (320 bf16)
    d = dsv3(B=64).dims()
    assert lib.mla_naive_workspace_size(ctypes.byref(d), ctypes.byref(fake_cache(4096))) >= 64 * 128 * 4096 * 320 * 2


NOALLOC_BYTES = 32 << 20  # the no-allocation entry point's array


def test_library_plan_fits_the_noalloc_array(lib):
    """mla_decode_attn_noalloc runs the library's own plan (num_splits 0) in a fixed
    32 MiB array: over the supported envelope that plan's workspace never exceeds it
    (split partials stay near one wave of 128-row work items), nor does the
    balanced plan's (two bf16 pieces per pair slot)."""
    worst = 0
    for d_c, d_rope in ((64, 16), (256, 64), (320, 16), (512, 64)):
        for H, s_q in ((16, 1), (128, 1), (128, 2), (128, 4), (64, 3), (1, 1), (512, 128)):
            for B in (1, 2, 3, 7, 20, 64, 65, 100, 151, 1000, 20000):
                for T in (64, 1000, 4096, 32768, 1 << 20):
                    if s_q > T or B * s_q > 65535 * 128:
                        continue
                    p = mla.Problem(B, H, s_q, d_c, d_rope, 128, 128, 0.1)
                    d = p.dims()
                    for paged in (False, True):
                        c = fake_cache(T, paged)
                        if not paged:
                            c = mla.Cache(0x10000, T * (d_c + d_rope), T, None, 0, 64, 0, 0x20000, 0)
                        n = lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c), 0)
                        worst = max(worst, n)
                        # the balanced plan, where the dims allow it, fits as well
                        n = lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(c), mla.SPLITS_BALANCED)
                        worst = max(worst, n)
    assert 0 < worst <= NOALLOC_BYTES, worst
