"""Device-side error reporting: bad lengths and bad page ids are recorded in the
workspace status word, the affected outputs are zero (lse -inf), the other
sequences stay correct, and nothing faults."""
import pytest
import torch

from mla_decode_attention_absorbed_gb300 import mla
from mla_decode_attention_absorbed_gb300.workloads import MLAConfig, make_inputs

from helpers import check_against_oracle, gpu_cache, run_gpu, to_dev

pytestmark = pytest.mark.gpu

DSV3_DIMS = dict(H=128, d_c=512, d_rope=64, d_nope=128, d_v=128)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_decode_attention_absorbed_gb300 import build
    build.build()
    mla.load()


@pytest.mark.parametrize("splits", [mla.SPLITS_BALANCED, 0, 1, 3])  # balanced: its merge writes them
def test_bad_lengths_flagged(splits):
    cfg = MLAConfig("bl", B=4, s_q=2, T=200, **DSV3_DIMS)
    inp = make_inputs(cfg, seq_lens=[150, 1, 200, 0])  # 1 < s_q and 0 are invalid
    d = to_dev(inp)
    d["seq_lens"] = torch.tensor([150, 1, 200, 0], dtype=torch.int32, device="cuda")
    prob, cache = gpu_cache(cfg, d)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    o_lat, lse, ws = mla.decode_attn(prob, q_cat, cache, num_splits=splits)
    assert mla.read_status(ws) == 3  # MLA_ERR_SEQLEN
    o = o_lat.cpu()
    assert torch.equal(o[1], torch.zeros_like(o[1])) and torch.equal(o[3], torch.zeros_like(o[3]))
    assert torch.isinf(lse[1]).all() and torch.isinf(lse[3]).all()
    # the valid sequences are unaffected
    good = MLAConfig("g", B=2, s_q=2, T=200, **DSV3_DIMS)
    ginp = {k: (v[[0, 2]] if k in ("q_nope", "q_rope", "kv", "seq_lens") else v) for k, v in inp.items()}
    ginp["seq_lens"] = torch.tensor([150, 200], dtype=torch.int32)
    g = dict(q_cat=q_cat.cpu()[[0, 2]], o_lat=o[[0, 2]], lse=lse.cpu()[[0, 2]],
             out=mla.out_proj(prob, o_lat, d["w_uv"]).cpu()[[0, 2]])
    check_against_oracle(good, ginp, g)


def test_length_beyond_capacity_flagged():
    cfg = MLAConfig("cap", B=2, s_q=1, T=128, **DSV3_DIMS)
    inp = make_inputs(cfg, seq_lens=[128, 64])
    d = to_dev(inp)
    d["seq_lens"] = torch.tensor([129, 64], dtype=torch.int32, device="cuda")
    prob, cache = gpu_cache(cfg, d)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    o_lat, lse, ws = mla.decode_attn(prob, q_cat, cache)
    assert mla.read_status(ws) == 3
    assert torch.isinf(lse[0].cpu()).all() and torch.isfinite(lse[1].cpu()).all()


def test_bad_page_flagged():
    cfg = MLAConfig("bp", B=2, s_q=1, len_lo=100, len_hi=300, paged=True, **DSV3_DIMS)
    inp = make_inputs(cfg)
    d = to_dev(inp)
    bt = inp["block_table"].clone()
    bt[0, 1] = 10_000  # outside the pool
    d["block_table"] = bt.cuda()
    prob, cache = gpu_cache(cfg, d)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    o_lat, lse, ws = mla.decode_attn(prob, q_cat, cache)
    assert mla.read_status(ws) == 9  # MLA_ERR_PAGE
    assert torch.isfinite(lse.cpu()).all()


def test_status_resets_between_calls():
    cfg = MLAConfig("r", B=1, s_q=1, T=64, **DSV3_DIMS)
    inp = make_inputs(cfg)
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    ws = mla.alloc_workspace(mla.decode_workspace_size(prob, cache), "cuda")
    ws.fill_(7)
    mla.decode_attn(prob, q_cat, cache, workspace=ws)
    assert mla.read_status(ws) == 0


def test_host_errors_raise():
    cfg = MLAConfig("h", B=1, s_q=1, T=64, **DSV3_DIMS)
    inp = make_inputs(cfg)
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.decode_attn(prob, q_cat, cache, workspace=small, num_splits=4)
    assert e.value.code == 5
    mis = torch.empty(q_cat.numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + q_cat.numel()]
    with pytest.raises(mla.MLAError) as e:
        mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"], q_cat=mis)
    assert e.value.code == 4


def test_wait_timeout_reported_and_recovered():
    """A bounded wait that runs out: with the attention kernels' wait bound set to
    1 ns (the tiny workload, one CTA per work item), some wait for work gives up,
    the kernel records MLA_ERR_TIMEOUT, drains its copies and MMAs in flight (those
    waits keep the 2 s bound) and returns; the next call, with the default bound
    restored, runs clean and matches the oracle."""
    from mla_decode_attention_absorbed_gb300.workloads import CONFIGS
    cfg = CONFIGS["tiny"]
    inp = make_inputs(cfg)
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    try:
        mla.set_wait_limit_ns(1)
        _, _, ws = mla.decode_attn(prob, q_cat, cache)
        torch.cuda.synchronize()
        assert mla.read_status(ws) == 8  # MLA_ERR_TIMEOUT
    finally:
        mla.set_wait_limit_ns(0)
    g = run_gpu(cfg, inp)
    assert g["status"] == 0
    check_against_oracle(cfg, inp, g)


def test_wait_timeout_balanced_plan():
    """The same on the balanced plan's persistent pair kernel (DeepSeek-V3 widths,
    three sequences cut between tile ranges): waits give up in every role, the
    epilogue warps agree before leaving their item loop (none is left at a barrier
    the others passed), the pair meets at its closing cluster barrier, and the next
    call, with the default bound, runs clean and matches the oracle."""
    cfg = MLAConfig("to_bal", B=3, s_q=1, T=1500, seed=31, **DSV3_DIMS)
    inp = make_inputs(cfg)
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    try:
        mla.set_wait_limit_ns(1)
        _, _, ws = mla.decode_attn(prob, q_cat, cache, num_splits=mla.SPLITS_BALANCED)
        torch.cuda.synchronize()
        assert mla.read_status(ws) == 8  # MLA_ERR_TIMEOUT
    finally:
        mla.set_wait_limit_ns(0)
    g = run_gpu(cfg, inp, num_splits=mla.SPLITS_BALANCED)
    assert g["status"] == 0
    check_against_oracle(cfg, inp, g)
