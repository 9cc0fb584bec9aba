"""mla_decode_attn_noalloc: the decode attention for callers that cannot
allocate scratch memory (a plain C / FFI host holding only its inputs and
outputs, or a serving loop whose device memory belongs to a framework pool).
Its scratch is a fixed array inside the library, shared by every call.

Checked through the C ABI against mla_decode_attn (same tolerance as the other
parity tests), on two calls in a row, so the second call runs on an array that
still holds the first call's contents.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

from mla_decode_attention_absorbed_gb300 import mla
from mla_decode_attention_absorbed_gb300.workloads import CONFIGS, MLAConfig, make_inputs

from helpers import gpu_cache, to_dev, within_tolerance

pytestmark = pytest.mark.gpu

DSV3_DIMS = dict(H=128, d_c=512, d_rope=64, d_nope=128, d_v=128)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_decode_attention_absorbed_gb300 import build
    build.build()
    mla.load()


def _prepare(cfg, seq_lens=None):
    inp = make_inputs(cfg, seq_lens=seq_lens)
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    return d, prob, cache, q_cat


def _noalloc(prob, q_cat, cache, splits):
    o = torch.full((prob.B, prob.s_q, prob.H, prob.d_c), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((prob.B, prob.s_q, prob.H), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    mla.decode_attn_noalloc(prob, q_cat, cache, o, lse, num_splits=splits, device_status=status)
    torch.cuda.synchronize()
    return o, lse, int(status.item())


@pytest.mark.parametrize("name,cfg,splits", [
    ("ragged_split3", MLAConfig("na", B=3, s_q=2, len_lo=70, len_hi=900, seed=21, **DSV3_DIMS), 3),
    ("dsv3_auto", CONFIGS["dsv3"], 0),
])
def test_matches_workspace_entry_point_twice(name, cfg, splits):
    d, prob, cache, q_cat = _prepare(cfg)
    ref_o, ref_lse, ws = mla.decode_attn(prob, q_cat, cache, num_splits=splits)
    assert mla.read_status(ws) == 0
    for call in range(2):
        o, lse, st = _noalloc(prob, q_cat, cache, splits)
        assert st == 0, f"call {call}: device status {st}"
        within_tolerance(o, ref_o.double(), f"o_lat, call {call}")
        within_tolerance(lse, ref_lse.double(), f"lse, call {call}")


def test_status_word_is_cleared_between_calls():
    cfg = MLAConfig("nb", B=2, s_q=1, T=200, seed=22, **DSV3_DIMS)
    d, prob, cache, q_cat = _prepare(cfg, seq_lens=[150, 200])
    good_o, good_lse, _ = _noalloc(prob, q_cat, cache, 2)
    d["seq_lens"][1] = 0  # invalid: recorded on the device, not a fault
    o, lse, st = _noalloc(prob, q_cat, cache, 2)
    assert st == 3
    d["seq_lens"][1] = 200
    o, lse, st = _noalloc(prob, q_cat, cache, 2)
    assert st == 0
    assert torch.equal(o, good_o) and torch.equal(lse, good_lse)


def test_rejects_partials_beyond_the_array():
    cfg = CONFIGS["dsv3"]
    d, prob, cache, q_cat = _prepare(cfg)
    o = torch.empty(prob.B, prob.s_q, prob.H, prob.d_c, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(prob.B, prob.s_q, prob.H, dtype=torch.float32, device="cuda")
    with pytest.raises(mla.MLAError) as e:
        mla.decode_attn_noalloc(prob, q_cat, cache, o, lse, num_splits=16)
    assert e.value.code == 5  # MLA_ERR_WORKSPACE: more than the built-in 32 MiB
