"""GPU parity of the prefill paths against the fp64 oracle's decompress-then-attend
form (orc_naive, pinned equal to the absorbed form): the expand path
(mla_prefill_expand) on full and chunked prefills, contiguous and paged, and the
dispatch (mla_prefill) on both sides of the crossover S*."""
import numpy as np
import pytest
import torch

import oracle
from helpers import sample_rows, to_dev, within_tolerance
from mla_decode_attention_absorbed_gb300 import mla
from mla_decode_attention_absorbed_gb300.workloads import MLAConfig, make_inputs

pytestmark = pytest.mark.gpu

_DSV3 = dict(H=128, d_c=512, d_rope=64, d_nope=128, d_v=128)


def _gpu(cfg, inp, dispatch=False):
    d = to_dev(inp)
    prob = mla.Problem.of(cfg)
    cache = mla.make_cache(prob, d["kv"], d["seq_lens"], d["block_table"], cfg.page_size,
                           max_seq_len=int(inp["seq_lens"].max()))
    if dispatch:
        out, lse, ws, path = mla.prefill(prob, d["q_nope"], d["q_rope"], cache, d["w_uk"], d["w_uv"])
    else:
        out, lse, ws = mla.prefill_expand(prob, d["q_nope"], d["q_rope"], cache, d["w_uk"], d["w_uv"])
        path = mla.PATH_EXPAND
    st = mla.read_status(ws)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu(), st, path


def _check(cfg, inp, rows=None, dispatch=False):
    out, lse, st, path = _gpu(cfg, inp, dispatch)
    ref, lse_ref = oracle.naive(cfg, inp["q_nope"], inp["q_rope"], inp["kv"], inp["seq_lens"], inp["w_uk"],
                                inp["w_uv"], inp["block_table"], cfg.page_size, rows=rows)
    sel = slice(None) if rows is None else torch.as_tensor(np.asarray(rows, dtype=np.int64))
    within_tolerance(out.view(-1, cfg.d_v)[sel], ref.view(-1, cfg.d_v)[sel], "prefill out")
    within_tolerance(lse.view(-1)[sel], lse_ref.view(-1)[sel], "prefill lse")
    return st, path


def _small(**kw):
    base = dict(name="prefill_small", B=2, H=4, d_c=64, d_rope=16, d_nope=64, d_v=64, seed=51)
    base.update(kw)
    return MLAConfig(**base)


@pytest.mark.parametrize("paged", [False, True])
def test_expand_full_prefill_small(paged):
    """Every token new (s_q = L): causal attention over the whole sequence."""
    cfg = _small(s_q=200, T=200, paged=paged)
    assert _check(cfg, make_inputs(cfg))[0] == 0


@pytest.mark.parametrize("paged", [False, True])
def test_expand_chunked_prefill_small(paged):
    """A chunk of 150 new tokens after a ragged history."""
    cfg = _small(B=3, s_q=150, len_lo=150, len_hi=420, paged=paged, seed=52)
    assert _check(cfg, make_inputs(cfg))[0] == 0


def test_expand_dsv3_widths_sampled():
    """DeepSeek-V3 widths, one 1024-token prompt: sampled rows against fp64."""
    cfg = MLAConfig("prefill_dsv3", B=1, s_q=1024, T=1024, seed=53, **_DSV3)
    assert _check(cfg, make_inputs(cfg), rows=sample_rows(cfg, 40))[0] == 0


def test_expand_dsv3_chunk_paged_sampled():
    cfg = MLAConfig("prefill_chunk", B=2, s_q=256, len_lo=600, len_hi=1500, paged=True, seed=54, **_DSV3)
    assert _check(cfg, make_inputs(cfg), rows=sample_rows(cfg, 40))[0] == 0


def test_dispatch_follows_the_crossover():
    """Below S* the absorbed path, at or above it the expanded one; both agree
    with the oracle."""
    prob = mla.Problem(B=1, H=128, s_q=1, d_c=512, d_rope=64, d_nope=128, d_v=128, scale=1.0)
    s_star = mla.prefill_crossover(prob, 1024)
    assert 128 < s_star < 171
    lo = MLAConfig("prefill_lo", B=2, s_q=8, T=1024, seed=55, **_DSV3)
    st, path = _check(lo, make_inputs(lo), rows=sample_rows(lo, 24), dispatch=True)
    assert st == 0 and path == mla.PATH_ABSORB
    hi = MLAConfig("prefill_hi", B=1, s_q=512, T=1024, seed=56, **_DSV3)
    st, path = _check(hi, make_inputs(hi), rows=sample_rows(hi, 24), dispatch=True)
    assert st == 0 and path == mla.PATH_EXPAND


def test_expand_matches_absorbed_on_the_gpu():
    """The two bracketings on the same chunk: GPU against GPU within the tolerance."""
    cfg = MLAConfig("prefill_both", B=2, s_q=24, T=700, seed=57, **_DSV3)
    inp = make_inputs(cfg)
    out_e, lse_e, st, _ = _gpu(cfg, inp)
    assert st == 0
    d = to_dev(inp)
    prob = mla.Problem.of(cfg)
    cache = mla.make_cache(prob, d["kv"], d["seq_lens"], None, cfg.page_size)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    o_lat, lse_a, _ = mla.decode_attn(prob, q_cat, cache)
    out_a = mla.out_proj(prob, o_lat, d["w_uv"])
    within_tolerance(out_e, out_a.cpu().double(), "expand vs absorbed out")
    within_tolerance(lse_e, lse_a.cpu().double(), "expand vs absorbed lse")


def test_expand_flags_a_bad_length():
    cfg = _small(B=3, s_q=64, len_lo=64, len_hi=200, seed=58)
    inp = make_inputs(cfg)
    lens = inp["seq_lens"].clone()
    lens[1] = 10  # shorter than s_q: invalid
    inp = dict(inp, seq_lens=lens)
    out, lse, st, _ = _gpu(cfg, inp)
    assert st == 3  # MLA_ERR_SEQLEN
    assert torch.equal(out[1], torch.zeros_like(out[1])) and bool(torch.isneginf(lse[1]).all())
