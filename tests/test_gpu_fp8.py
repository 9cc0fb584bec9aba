"""GPU parity of the FP8 (E4M3) latent cache: dense and sparse decode against
the fp64 oracle reading the same codes with the same scale, stage-isolated from
the GPU's own q_cat, plus the end-to-end step."""
import numpy as np
import pytest
import torch

import oracle
from helpers import lse_close, sample_rows, to_dev, within_tolerance
from mla_decode_attention_absorbed_gb300 import mla
from mla_decode_attention_absorbed_gb300.workloads import (KV_FP8_SCALE, MLAConfig, make_inputs,
                                                           make_sparse_indices, to_fp8_cache)

pytestmark = pytest.mark.gpu

_DSV3 = dict(H=128, d_c=512, d_rope=64, d_nope=128, d_v=128)


def _fp8_inputs(cfg, scale=KV_FP8_SCALE):
    inp = make_inputs(cfg)
    inp["kv"] = to_fp8_cache(inp["kv"], scale)
    return inp


def _run(cfg, inp, scale, idx=None, num_splits=0):
    d = to_dev(inp)
    prob = mla.Problem.of(cfg)
    cache = mla.make_cache(prob, d["kv"], d["seq_lens"], d["block_table"], cfg.page_size, kv_scale=scale)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    if idx is None:
        o, lse, ws = mla.decode_attn(prob, q_cat, cache, num_splits=num_splits)
    else:
        o, lse, ws = mla.decode_attn_sparse(prob, q_cat, cache, idx.cuda(), num_splits=num_splits)
    out = mla.out_proj(prob, o, d["w_uv"])
    st = mla.read_status(ws)
    torch.cuda.synchronize()
    return dict(q_cat=q_cat.cpu(), o_lat=o.cpu(), lse=lse.cpu(), out=out.cpu(), status=st)


def _check(cfg, inp, scale=KV_FP8_SCALE, idx=None, num_splits=0, rows=None, end_to_end=False):
    g = _run(cfg, inp, scale, idx, num_splits)
    sel = slice(None) if rows is None else torch.as_tensor(np.asarray(rows, dtype=np.int64))
    args = (cfg, g["q_cat"], inp["kv"], inp["seq_lens"])
    if idx is None:
        o_ref, lse_ref = oracle.attend(*args, inp["block_table"], cfg.page_size, rows=rows, kv_scale=scale)
    else:
        o_ref, lse_ref = oracle.attend_sparse(*args, idx, inp["block_table"], cfg.page_size, rows=rows,
                                              kv_scale=scale)
    within_tolerance(g["o_lat"].view(-1, cfg.d_c)[sel], o_ref.view(-1, cfg.d_c)[sel], "fp8 o_lat")
    lse_close(g["lse"].view(-1)[sel], lse_ref.view(-1)[sel], "fp8 lse")
    if end_to_end:
        e2e = oracle.decode(cfg, inp["q_nope"], inp["q_rope"], inp["kv"], inp["seq_lens"], inp["w_uk"],
                            inp["w_uv"], block_table=inp["block_table"], page_size=cfg.page_size, rows=rows,
                            kv_scale=scale)
        within_tolerance(g["out"].view(-1, cfg.d_v)[sel], e2e["out"].view(-1, cfg.d_v)[sel], "fp8 out (end to end)")
    return g["status"]


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("s_q", [1, 3])
def test_fp8_small(paged, s_q):
    cfg = MLAConfig("fp8_small", B=3, H=16, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=s_q,
                    len_lo=5, len_hi=300, paged=paged, seed=41)
    assert _check(cfg, _fp8_inputs(cfg), end_to_end=True) == 0


@pytest.mark.parametrize("paged,s_q", [(False, 1), (True, 2), (False, 4)])
@pytest.mark.parametrize("splits", [0, 3])
def test_fp8_dsv3_widths(paged, s_q, splits):
    cfg = MLAConfig("fp8_dsv3", B=4, s_q=s_q, len_lo=100, len_hi=1500, paged=paged, seed=42, **_DSV3)
    assert _check(cfg, _fp8_inputs(cfg), num_splits=splits, end_to_end=True) == 0


def test_fp8_scale_not_a_power_of_two():
    """The scale enters the scores and the values: a scale with a full mantissa."""
    s = 0.0371
    cfg = MLAConfig("fp8_scale", B=3, s_q=2, len_lo=64, len_hi=700, seed=43, **_DSV3)
    assert _check(cfg, _fp8_inputs(cfg, s), scale=s) == 0


def test_fp8_equals_bf16_cache_of_its_values():
    """With a power-of-two scale the FP8 cache holds bf16 numbers: the GPU result must
    match the bf16 path over those values within the tolerance (different kernels:
    fp16 vs bf16 operands)."""
    cfg = MLAConfig("fp8_vs_bf16", B=3, s_q=1, len_lo=200, len_hi=900, seed=44, **_DSV3)
    inp = _fp8_inputs(cfg)
    g8 = _run(cfg, inp, KV_FP8_SCALE)
    deq = (inp["kv"].view(torch.float8_e4m3fn).to(torch.float32) * KV_FP8_SCALE).to(torch.bfloat16)
    d = to_dev(dict(inp, kv=deq))
    prob = mla.Problem.of(cfg)
    cache = mla.make_cache(prob, d["kv"], d["seq_lens"], None, cfg.page_size)
    o, lse, _ = mla.decode_attn(prob, g8["q_cat"].cuda(), cache)
    within_tolerance(g8["o_lat"], o.cpu().double(), "fp8 vs bf16 o_lat")
    within_tolerance(g8["lse"], lse.cpu().double(), "fp8 vs bf16 lse")


@pytest.mark.parametrize("paged", [False, True])
def test_fp8_sparse(paged):
    cfg = MLAConfig("fp8_sparse", B=4, s_q=1, len_lo=300, len_hi=5000, paged=paged, seed=45, **_DSV3)
    inp = _fp8_inputs(cfg)
    idx = make_sparse_indices(cfg, inp["seq_lens"], 2048)
    assert _check(cfg, inp, idx=idx) == 0


def test_fp8_sparse_small_with_padding():
    cfg = MLAConfig("fp8_sparse_small", B=3, H=16, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=1,
                    len_lo=20, len_hi=400, paged=True, seed=46)
    inp = _fp8_inputs(cfg)
    idx = make_sparse_indices(cfg, inp["seq_lens"], 100)
    idx[0, 0, 3] = -1
    idx[1, 0, 5] = int(inp["seq_lens"][1]) + 2  # future token: a NaN code sits there
    assert _check(cfg, inp, idx=idx) == 0


def test_fp8_full_size_sampled():
    """The dsv3 decode workload (64 x 4096 tokens) with an FP8 cache, sampled rows."""
    cfg = MLAConfig("fp8_dsv3_full", B=64, T=4096, s_q=1, seed=47, **_DSV3)
    assert _check(cfg, _fp8_inputs(cfg), rows=sample_rows(cfg, 48)) == 0


@pytest.mark.parametrize("paged", [False, True])
def test_fp8_last_wave_tail(paged):
    """80 work items on 76 cluster slots with an FP8 cache: the last sequence runs in
    pieces merged by the tail combine (no longest-first order for FP8); its rows and
    a sample of the others against the oracle."""
    cfg = MLAConfig("fp8_tail", B=20, s_q=4, T=1024, paged=paged, seed=63, **_DSV3)
    inp = _fp8_inputs(cfg)
    d = to_dev(inp)
    prob = mla.Problem.of(cfg)
    cache = mla.make_cache(prob, d["kv"], d["seq_lens"], d["block_table"], cfg.page_size, kv_scale=KV_FP8_SCALE)
    assert mla.decode_num_splits(prob, cache) == 2
    rows = cfg.s_q * cfg.H
    tail = list(range((cfg.B - 1) * rows, cfg.B * rows, 29))
    assert _check(cfg, inp, rows=sorted(set(sample_rows(cfg, 16) + tail)), end_to_end=True) == 0


def test_fp8_rejected_where_unsupported():
    cfg = MLAConfig("fp8_bad", B=2, H=16, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=1, T=128, seed=48)
    inp = to_dev(_fp8_inputs(cfg))
    prob = mla.Problem.of(cfg)
    cache = mla.make_cache(prob, inp["kv"], inp["seq_lens"], None, cfg.page_size, kv_scale=KV_FP8_SCALE)
    with pytest.raises(mla.MLAError):  # the comparison path takes bf16 caches only
        mla.naive_decode(prob, inp["q_nope"], inp["q_rope"], cache, inp["w_uk"], inp["w_uv"])
    bad = mla.make_cache(prob, inp["kv"], inp["seq_lens"], None, cfg.page_size, kv_scale=KV_FP8_SCALE)
    bad.kv_scale = 0.0
    q_cat = mla.absorb_q(prob, inp["q_nope"], inp["q_rope"], inp["w_uk"])
    with pytest.raises((mla.MLAError, ValueError)):  # the size query already refuses it
        mla.decode_attn(prob, q_cat, bad)
