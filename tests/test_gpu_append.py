"""GPU parity of the cache append (latent down-projection of the new tokens)
against the fp64 oracle: the new rows within the tolerance, every other cache
row bitwise unchanged, bad lengths / pages flagged and left unwritten."""
import pytest
import torch

import oracle
from helpers import within_tolerance
from mla_decode_attention_absorbed_gb300 import mla
from mla_decode_attention_absorbed_gb300.workloads import MLAConfig, make_append_inputs, make_inputs

pytestmark = pytest.mark.gpu

_DSV3 = dict(H=128, d_c=512, d_rope=64, d_nope=128, d_v=128)


def _run(cfg, inp, app, seq_lens=None, block_table=None):
    dev = "cuda"
    kv = inp["kv"].to(dev).clone()
    lens = (seq_lens if seq_lens is not None else inp["seq_lens"]).to(dev)
    bt = block_table if block_table is not None else inp["block_table"]
    bt = bt.to(dev) if bt is not None else None
    prob = mla.Problem.of(cfg)
    cache = mla.make_cache(prob, kv, lens, bt, cfg.page_size)
    ws = mla.cache_append(prob, app["x"].to(dev), app["w_dkv"].to(dev), app["k_rope"].to(dev), cache)
    status = mla.read_status(ws)
    torch.cuda.synchronize()
    return kv.cpu(), status


def _check(cfg, inp, app, seq_lens=None, block_table=None):
    lens = seq_lens if seq_lens is not None else inp["seq_lens"]
    bt = block_table if block_table is not None else inp["block_table"]
    got, status = _run(cfg, inp, app, seq_lens, block_table)
    ref, written = oracle.cache_append(cfg, app["x"], app["w_dkv"], app["k_rope"], inp["kv"], lens, bt,
                                       cfg.page_size)
    old = inp["kv"]
    # untouched rows: bitwise (NaN canaries included)
    assert torch.equal(got[~written].view(torch.int16), old[~written].view(torch.int16))
    if written.any():
        new = got[written]
        within_tolerance(new[:, :cfg.d_c], ref[written][:, :cfg.d_c], "appended c_kv")
        assert torch.equal(new[:, cfg.d_c:].view(torch.int16),
                           ref[written][:, cfg.d_c:].to(torch.bfloat16).view(torch.int16)), "k_rope copied"
    return status, written


@pytest.mark.parametrize("paged,s_q", [(False, 1), (True, 2)])
def test_append_small(paged, s_q):
    cfg = MLAConfig("append_small", B=3, H=16, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=s_q,
                    len_lo=s_q, len_hi=300, paged=paged, seed=5)
    inp = make_inputs(cfg)
    app = make_append_inputs(cfg, d_model=200)
    status, written = _check(cfg, inp, app)
    assert status == 0
    assert int(written.sum()) == cfg.B * s_q


@pytest.mark.parametrize("paged,s_q", [(False, 1), (True, 2)])
def test_append_dsv3_widths(paged, s_q):
    """DeepSeek-V3 widths: d_model = 7168 (split along d_model over the GPU), d_c = 512."""
    cfg = MLAConfig("append_dsv3", B=64, s_q=s_q, len_lo=s_q, len_hi=700, paged=paged, seed=9, **_DSV3)
    inp = make_inputs(cfg)
    app = make_append_inputs(cfg, d_model=7168)
    status, written = _check(cfg, inp, app)
    assert status == 0
    assert int(written.sum()) == cfg.B * s_q


def test_append_flags_bad_length_and_page():
    cfg = MLAConfig("append_bad", B=4, H=16, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=1,
                    len_lo=70, len_hi=200, paged=True, seed=6)
    inp = make_inputs(cfg)
    app = make_append_inputs(cfg, d_model=64)
    lens = inp["seq_lens"].clone()
    bt = inp["block_table"].clone()
    lens[0] = 0
    bt[2, (int(lens[2]) - 1) // cfg.page_size] = 10 ** 6
    status, written = _check(cfg, inp, app, seq_lens=lens, block_table=bt)
    assert status in (3, 9)  # MLA_ERR_SEQLEN or MLA_ERR_PAGE (the first one recorded)
    assert int(written.sum()) == cfg.B - 2


def test_append_host_errors():
    cfg = MLAConfig("append_err", B=2, H=16, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=1, T=64, seed=1)
    inp = make_inputs(cfg)
    app = make_append_inputs(cfg, d_model=60)  # not a multiple of 8
    with pytest.raises(mla.MLAError):
        _run(cfg, inp, app)


# ------------------------------------------------------------------ FP8 (E4M3) cache
def _fp8_codes_ok(got, exact):
    """got: E4M3 codes from the GPU; exact: the float64 values they quantise.  The
    code must be the nearest one (ties to even, saturating), or -- where the exact
    value lies within fp32 summation error of the midpoint between two codes --
    its other neighbour."""
    ref = oracle.e4m3_encode(exact)
    same = got == ref
    if bool(same.all()):
        return
    g = got[~same].view(torch.float8_e4m3fn).to(torch.float64)
    r = ref[~same].view(torch.float8_e4m3fn).to(torch.float64)
    v = exact[~same]
    mid = (g + r) / 2
    # neighbouring codes, and v within 1e-4 relative of their midpoint
    assert bool(((mid - v).abs() <= 1e-4 * v.abs().clamp(min=1e-3)).all()), (g[:5], r[:5], v[:5])
    assert bool(((g - r).abs() <= (v.abs() * 2.0 ** -2).clamp(min=2.0 ** -9)).all())


@pytest.mark.parametrize("paged,s_q,scale", [(False, 1, 1.0 / 16), (True, 2, 1.0 / 16), (False, 2, 0.0371)])
def test_append_fp8(paged, s_q, scale):
    """Appending into an FP8 cache: every element of the new rows is the E4M3 code
    of value / kv_scale; every other code is unchanged."""
    from mla_decode_attention_absorbed_gb300.workloads import to_fp8_cache
    cfg = MLAConfig("append_fp8", B=16, s_q=s_q, len_lo=s_q, len_hi=500, paged=paged, seed=12, **_DSV3)
    inp = make_inputs(cfg)
    app = make_append_inputs(cfg, d_model=7168)
    codes = to_fp8_cache(inp["kv"], scale)
    dev = "cuda"
    kv = codes.to(dev).clone()
    lens = inp["seq_lens"].to(dev)  # the descriptor holds raw pointers: keep the tensors alive
    bt = inp["block_table"].to(dev) if inp["block_table"] is not None else None
    prob = mla.Problem.of(cfg)
    cache = mla.make_cache(prob, kv, lens, bt, cfg.page_size, kv_scale=scale)
    ws = mla.cache_append(prob, app["x"].to(dev), app["w_dkv"].to(dev), app["k_rope"].to(dev), cache)
    assert mla.read_status(ws) == 0
    got = kv.cpu()
    exact, written = oracle.cache_append(cfg, app["x"], app["w_dkv"], app["k_rope"], codes, inp["seq_lens"],
                                         inp["block_table"], cfg.page_size, kv_scale=scale)
    assert int(written.sum()) == cfg.B * s_q
    assert torch.equal(got[~written], codes[~written])
    _fp8_codes_ok(got[written], exact[written])
