"""GPU parity of the sparse top-k decode (attention over listed cached tokens)
against the fp64 oracle, stage-isolated from the GPU's own q_cat."""
import numpy as np
import pytest
import torch

import oracle
from helpers import gpu_cache, sample_rows, to_dev, within_tolerance
from mla_decode_attention_absorbed_gb300 import mla
from mla_decode_attention_absorbed_gb300.workloads import MLAConfig, make_inputs, make_sparse_indices

pytestmark = pytest.mark.gpu

_DSV3 = dict(H=128, d_c=512, d_rope=64, d_nope=128, d_v=128)


def _run(cfg, inp, idx, num_splits=0):
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    o, lse, ws = mla.decode_attn_sparse(prob, q_cat, cache, idx.cuda(), num_splits=num_splits)
    st = mla.read_status(ws)
    torch.cuda.synchronize()
    return q_cat.cpu(), o.cpu(), lse.cpu(), st


def _check(cfg, inp, idx, num_splits=0, rows=None):
    q, o, lse, st = _run(cfg, inp, idx, num_splits)
    o_ref, lse_ref = oracle.attend_sparse(cfg, q, inp["kv"], inp["seq_lens"], idx, inp["block_table"],
                                          cfg.page_size, rows=rows)
    sel = slice(None) if rows is None else torch.as_tensor(np.asarray(rows, dtype=np.int64))
    within_tolerance(o.view(-1, cfg.d_c)[sel], o_ref.view(-1, cfg.d_c)[sel], "sparse o_lat")
    within_tolerance(lse.view(-1)[sel], lse_ref.view(-1)[sel], "sparse lse")
    return st


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("topk", [1, 100, 300])
def test_sparse_small(paged, topk):
    cfg = MLAConfig("sparse_small", B=3, H=16, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=1,
                    len_lo=20, len_hi=400, paged=paged, seed=31)
    inp = make_inputs(cfg)
    idx = make_sparse_indices(cfg, inp["seq_lens"], topk)
    assert _check(cfg, inp, idx) == 0


@pytest.mark.parametrize("paged,s_q", [(False, 1), (True, 2)])
@pytest.mark.parametrize("splits", [0, 3])
def test_sparse_dsv3_widths(paged, s_q, splits):
    cfg = MLAConfig("sparse_dsv3", B=6, s_q=s_q, len_lo=300, len_hi=5000, paged=paged, seed=32, **_DSV3)
    inp = make_inputs(cfg)
    idx = make_sparse_indices(cfg, inp["seq_lens"], 2048)
    assert _check(cfg, inp, idx, num_splits=splits) == 0


def test_sparse_full_list_matches_dense_attention():
    cfg = MLAConfig("sparse_full", B=4, T=700, s_q=1, seed=33, **_DSV3)
    inp = make_inputs(cfg)
    L = int(inp["seq_lens"][0])
    idx = torch.arange(L, dtype=torch.int32).view(1, 1, L).repeat(cfg.B, 1, 1)
    q, o_s, l_s, st = _run(cfg, inp, idx)
    assert st == 0
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d)
    o_d, l_d, _ = mla.decode_attn(prob, q.cuda(), cache)
    within_tolerance(o_s, o_d.cpu().double(), "sparse(all) vs dense o_lat")
    within_tolerance(l_s, l_d.cpu().double(), "sparse(all) vs dense lse")


def test_sparse_padding_future_entries_and_bad_page():
    cfg = MLAConfig("sparse_edge", B=3, H=16, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=1,
                    len_lo=70, len_hi=300, paged=True, seed=34)
    inp = make_inputs(cfg)
    idx = make_sparse_indices(cfg, inp["seq_lens"], 64)
    idx[0, 0, 5] = -1
    idx[1, 0, 7] = int(inp["seq_lens"][1]) + 3  # a future token (NaN canary in the cache)
    idx[2, 0, :] = -1                            # nothing visible: o = 0, lse = -inf
    assert _check(cfg, inp, idx) == 0
    _, o, lse, _ = _run(cfg, inp, idx)
    assert torch.equal(o[2], torch.zeros_like(o[2])) and bool(torch.isneginf(lse[2]).all())
    # an entry on a page outside the pool is skipped and flagged
    bt = inp["block_table"].clone()
    j = int(idx[0, 0, 10])
    bt[0, j // cfg.page_size] = 10 ** 6
    bad = dict(inp, block_table=bt)
    _, _, _, st = _run(cfg, bad, idx)
    assert st == 9  # MLA_ERR_PAGE


def test_sparse_rejects_unsupported_rows():
    cfg = MLAConfig("sparse_bad", B=2, H=16, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=2, T=128, seed=35)
    inp = make_inputs(cfg)
    idx = make_sparse_indices(cfg, inp["seq_lens"], 32)
    with pytest.raises(mla.MLAError):
        _run(cfg, inp, idx)


def test_sparse_full_size_sampled():
    """64 sequences of 32768 tokens, k = 2048: sampled rows against the oracle."""
    cfg = MLAConfig("sparse_long", B=64, T=32768, s_q=1, seed=36, **_DSV3)
    inp = make_inputs(cfg)
    idx = make_sparse_indices(cfg, inp["seq_lens"], 2048)
    assert _check(cfg, inp, idx, rows=sample_rows(cfg, 48)) == 0
