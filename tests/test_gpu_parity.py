"""Parity of the CUDA path with the fp64 oracle, per output tensor, within
max|gpu - ref| <= 2e-2 * max|ref| + 1e-3 (bf16 inputs, fp32 accumulation).

Small cases are compared element by element on every row; the full-size
workloads run in the launch configuration the benchmark times (automatic split
count) and are compared on sampled rows the oracle computes one by one."""
import pytest
import torch

import oracle
from mla_decode_attention_absorbed_gb300 import mla
from mla_decode_attention_absorbed_gb300.workloads import CONFIGS, MLAConfig, make_inputs

from helpers import check_against_oracle, gpu_cache, run_gpu, sample_rows, to_dev, within_tolerance

pytestmark = pytest.mark.gpu

DSV3_DIMS = dict(H=128, d_c=512, d_rope=64, d_nope=128, d_v=128)
# widths whose attention runs one CTA per 128-row work item (the tail and
# longest-first plans are theirs; the pair kernels take the balanced plan)
ONE_CTA_DIMS = dict(H=128, d_c=256, d_rope=64, d_nope=128, d_v=128)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from mla_decode_attention_absorbed_gb300 import build
    build.build()
    mla.load()


def test_tiny_config_all_rows():
    cfg = CONFIGS["tiny"]
    inp = make_inputs(cfg)
    g = run_gpu(cfg, inp)
    assert g["status"] == 0
    check_against_oracle(cfg, inp, g)


# several 64-token tiles, ragged tails, s_q 1/2/4, paged and contiguous, split counts
CASES = [
    ("contig_sq1", MLAConfig("c1", B=3, s_q=1, len_lo=65, len_hi=700, **DSV3_DIMS), 0),
    ("contig_sq1_split1", MLAConfig("c1", B=3, s_q=1, len_lo=65, len_hi=700, **DSV3_DIMS), 1),
    ("contig_sq1_split7", MLAConfig("c1", B=3, s_q=1, len_lo=65, len_hi=700, **DSV3_DIMS), 7),
    ("contig_sq2", MLAConfig("c2", B=2, s_q=2, len_lo=100, len_hi=400, seed=3, **DSV3_DIMS), 2),
    ("contig_sq4", MLAConfig("c4", B=2, s_q=4, len_lo=4, len_hi=300, seed=4, **DSV3_DIMS), 3),
    ("paged_sq2", MLAConfig("p2", B=3, s_q=2, len_lo=2, len_hi=500, paged=True, seed=5, **DSV3_DIMS), 0),
    ("paged_sq1_split5", MLAConfig("p1", B=2, s_q=1, len_lo=1, len_hi=900, paged=True, seed=6, **DSV3_DIMS), 5),
    ("small_dims", MLAConfig("sd", B=3, H=16, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=3, len_lo=3,
                             len_hi=300, seed=7), 2),
    ("mid_dims", MLAConfig("md", B=2, H=40, d_c=192, d_rope=32, d_nope=64, d_v=48, s_q=2, len_lo=70,
                           len_hi=260, seed=8), 0),
    # pair kernel shapes other than DeepSeek-V3's: a partial RoPE box (d_rope 48), two query
    # tokens per 128-row block (H 64), a CTA whose second score chain is empty (d_c 320, d_rope 16)
    ("pair_dc384_rope48", MLAConfig("q1", B=2, H=64, d_c=384, d_rope=48, d_nope=64, d_v=64, s_q=2, len_lo=70,
                                    len_hi=400, seed=21), 0),
    ("pair_dc320_rope16", MLAConfig("q2", B=3, H=128, d_c=320, d_rope=16, d_nope=64, d_v=64, s_q=1, len_lo=1,
                                    len_hi=300, paged=True, seed=22), 2),
    ("pair_dc448_rope32", MLAConfig("q3", B=2, H=128, d_c=448, d_rope=32, d_nope=128, d_v=128, s_q=3, len_lo=3,
                                    len_hi=260, seed=23), 0),
    # the balanced plan on the same shapes: its pieces are stored per CTA (the second CTA's
    # block d_c - 256 columns wide), two query tokens share a row block, three row blocks
    ("contig_sq4_balanced", MLAConfig("c4", B=2, s_q=4, len_lo=4, len_hi=300, seed=4, **DSV3_DIMS),
     mla.SPLITS_BALANCED),
    ("pair_dc384_rope48_balanced", MLAConfig("q1", B=2, H=64, d_c=384, d_rope=48, d_nope=64, d_v=64, s_q=2,
                                             len_lo=70, len_hi=400, seed=21), mla.SPLITS_BALANCED),
    ("pair_dc320_rope16_balanced", MLAConfig("q2", B=3, H=128, d_c=320, d_rope=16, d_nope=64, d_v=64, s_q=1,
                                             len_lo=1, len_hi=300, paged=True, seed=22), mla.SPLITS_BALANCED),
    ("pair_dc448_rope32_balanced", MLAConfig("q3", B=2, H=128, d_c=448, d_rope=32, d_nope=128, d_v=128, s_q=3,
                                             len_lo=3, len_hi=260, seed=23), mla.SPLITS_BALANCED),
]


@pytest.mark.parametrize("name,cfg,splits", CASES, ids=[c[0] for c in CASES])
def test_parity_small(name, cfg, splits):
    inp = make_inputs(cfg)
    g = run_gpu(cfg, inp, num_splits=splits)
    assert g["status"] == 0
    check_against_oracle(cfg, inp, g)


def test_edge_lengths():
    """L = s_q (every token new), L = 1, L on a tile boundary, L = capacity."""
    cfg = MLAConfig("e", B=5, s_q=1, T=256, **DSV3_DIMS)
    inp = make_inputs(cfg, seq_lens=[1, 64, 65, 255, 256])
    check_against_oracle(cfg, inp, run_gpu(cfg, inp))
    cfg4 = MLAConfig("e4", B=3, s_q=4, T=130, **DSV3_DIMS)
    inp4 = make_inputs(cfg4, seq_lens=[4, 68, 130])
    check_against_oracle(cfg4, inp4, run_gpu(cfg4, inp4, num_splits=2))


def test_more_splits_than_tiles():
    cfg = MLAConfig("e", B=2, s_q=2, T=100, **DSV3_DIMS)
    inp = make_inputs(cfg, seq_lens=[70, 100])
    check_against_oracle(cfg, inp, run_gpu(cfg, inp, num_splits=9))


def test_split_counts_agree():
    cfg = MLAConfig("s", B=2, s_q=1, T=2000, **DSV3_DIMS)
    inp = make_inputs(cfg, seq_lens=[1999, 1333])
    base = run_gpu(cfg, inp, num_splits=1)
    for s in (2, 7, 64):
        g = run_gpu(cfg, inp, num_splits=s)
        within_tolerance(g["o_lat"], base["o_lat"].double(), f"o_lat splits={s}", rel=1e-2, abs_=1e-3)
        within_tolerance(g["lse"], base["lse"].double(), f"lse splits={s}", rel=1e-4, abs_=1e-4)


def test_paged_equals_contiguous_and_strided():
    cfg = MLAConfig("pc", B=3, s_q=2, T=300, **DSV3_DIMS)
    inp = make_inputs(cfg, seq_lens=[300, 131, 64])
    ref = run_gpu(cfg, inp, num_splits=2)
    # same tokens in shuffled 64-token pages
    pages, table = [], []
    for b, L in enumerate(inp["seq_lens"].tolist()):
        ids = []
        for p0 in range(0, L, 64):
            blk = torch.full((64, cfg.W), float("nan"), dtype=torch.bfloat16)
            take = inp["kv"][b, p0:min(L, p0 + 64)]
            blk[:take.shape[0]] = take
            ids.append(len(pages))
            pages.append(blk)
        table.append(ids)
    perm = torch.randperm(len(pages), generator=torch.Generator().manual_seed(11))
    pool = torch.stack(pages)[torch.argsort(perm)]
    bt = torch.full((cfg.B, 6), -1, dtype=torch.int32)
    for b, ids in enumerate(table):
        bt[b, :len(ids)] = perm[torch.tensor(ids)].to(torch.int32)
    pinp = dict(inp, kv=pool, block_table=bt)
    pcfg = cfg.with_(paged=True)
    g = run_gpu(pcfg, pinp, num_splits=2)
    assert torch.equal(g["o_lat"], ref["o_lat"]) and torch.equal(g["lse"], ref["lse"])
    # a contiguous cache whose sequences sit further apart than T_max rows
    big = torch.full((cfg.B, 400, cfg.W), float("nan"), dtype=torch.bfloat16)
    big[:, :300] = inp["kv"]
    sinp = dict(inp, kv=big[:, :300])
    g2 = run_gpu(cfg, sinp, num_splits=2)
    assert torch.equal(g2["o_lat"], ref["o_lat"]) and torch.equal(g2["out"], ref["out"])


def test_deterministic():
    cfg = MLAConfig("d", B=2, s_q=2, T=500, **DSV3_DIMS)
    inp = make_inputs(cfg)
    a, b = run_gpu(cfg, inp, num_splits=3), run_gpu(cfg, inp, num_splits=3)
    for k in ("q_cat", "o_lat", "lse", "out"):
        assert torch.equal(a[k], b[k]), k


def test_empty_batch():
    cfg = MLAConfig("z", B=0, s_q=1, T=64, **DSV3_DIMS)
    prob = mla.Problem.of(cfg)
    kv = torch.zeros(1, 64, cfg.W, dtype=torch.bfloat16, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = mla.make_cache(prob, kv, lens)
    q = torch.zeros(1, 1, 128, 576, dtype=torch.bfloat16, device="cuda")
    o, lse, ws = mla.decode_attn(prob, q, cache)
    assert mla.read_status(ws) == 0


# ---------------------------------------------------------------- full-size workloads, sampled rows
@pytest.mark.parametrize("name", ["dsv3", "long", "spec", "ragged_paged"])
def test_full_size_sampled(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg)
    g = run_gpu(cfg, inp)
    assert g["status"] == 0
    rows = sample_rows(cfg, 48)
    check_against_oracle(cfg, inp, g, rows=rows)
    for k in ("o_lat", "lse", "out"):
        assert torch.isfinite(g[k].float()).all(), k


def test_tail_plan_matches_unsplit_and_oracle():
    """156 work items on 152 SM slots (one CTA per item): the last sequence runs in
    two pieces (the grid's last work items, merged), the others unsplit; the result
    agrees with the unsplit launch and the oracle, and the fused step with the same
    plan is bit-identical."""
    from helpers import sample_rows
    cfg = MLAConfig("tail", B=39, s_q=4, T=1024, seed=61, **ONE_CTA_DIMS)
    inp = make_inputs(cfg)
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d)
    assert mla.decode_num_splits(prob, cache) == 2
    auto = run_gpu(cfg, inp)
    one = run_gpu(cfg, inp, num_splits=1)
    assert auto["status"] == 0 and one["status"] == 0
    within_tolerance(auto["o_lat"].double(), one["o_lat"].double(), "tail plan vs unsplit o_lat")
    within_tolerance(auto["lse"].double(), one["lse"].double(), "tail plan vs unsplit lse")
    # the head sequences run exactly as in the unsplit launch
    head = (cfg.B - 1) * cfg.s_q * cfg.H
    assert torch.equal(auto["o_lat"].view(-1, cfg.d_c)[:head], one["o_lat"].view(-1, cfg.d_c)[:head])
    tail_rows = list(range(head, head + cfg.s_q * cfg.H, 37)) + [cfg.B * cfg.s_q * cfg.H - 1]
    check_against_oracle(cfg, inp, auto, rows=sorted(set(sample_rows(cfg, 16) + tail_rows)))
    dec = mla.Decoder(prob, d["kv"], d["seq_lens"], d["w_uk"], d["w_uv"], d["block_table"], cfg.page_size)
    out_f = dec.step(d["q_nope"], d["q_rope"]).clone()
    lse_f = dec.lse.clone()
    out_s = dec(d["q_nope"], d["q_rope"]).clone()
    torch.cuda.synchronize()
    assert mla.read_status(dec.workspace) == 0
    assert torch.equal(out_f, out_s) and torch.equal(lse_f, dec.lse)
    assert torch.equal(lse_f.cpu(), auto["lse"])


def test_longest_first_order_ragged():
    """200 ragged sequences on 152 SM slots (one CTA per item): the work order is
    longest first (ranked on the device) and the 48 shortest sequences, the last
    wave, run in 3 pieces each; whole sequences match the explicit unsplit launch
    bit for bit, everything matches the oracle, and the fused step is
    bit-identical."""
    from helpers import sample_rows
    cfg = MLAConfig("lpt", B=200, s_q=1, len_lo=64, len_hi=2048, paged=True, seed=62, **ONE_CTA_DIMS)
    inp = make_inputs(cfg)
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d)
    assert mla.decode_num_splits(prob, cache) == 3
    auto = run_gpu(cfg, inp)
    one = run_gpu(cfg, inp, num_splits=1)
    assert auto["status"] == 0 and one["status"] == 0
    within_tolerance(auto["o_lat"].double(), one["o_lat"].double(), "longest first + tail vs unsplit o_lat")
    lens = inp["seq_lens"].tolist()
    order = sorted(range(cfg.B), key=lambda b: (-lens[b], b))
    rows = cfg.s_q * cfg.H
    for b in order[:152]:  # whole sequences
        assert torch.equal(auto["o_lat"].view(cfg.B, -1)[b], one["o_lat"].view(cfg.B, -1)[b]), b
    split_rows = [b * rows + r for b in order[152:] for r in (0, rows - 1)]
    check_against_oracle(cfg, inp, auto, rows=sorted(set(sample_rows(cfg, 16) + split_rows)))
    dec = mla.Decoder(prob, d["kv"], d["seq_lens"], d["w_uk"], d["w_uv"], d["block_table"], cfg.page_size)
    out_f = dec.step(d["q_nope"], d["q_rope"]).clone()
    lse_f = dec.lse.clone()
    out_s = dec(d["q_nope"], d["q_rope"]).clone()
    torch.cuda.synchronize()
    assert mla.read_status(dec.workspace) == 0
    assert torch.equal(out_f, out_s) and torch.equal(lse_f, dec.lse)
    assert torch.equal(lse_f.cpu(), auto["lse"])


# ---------------------------------------------------------------- balanced plan (pair kernels)
def _balanced_case(cfg, inp, rows=None):
    """The balanced plan (MLA_SPLITS_BALANCED) against the explicit unsplit launch
    and the oracle; the fused step with the same plan is bit-identical to separate
    calls."""
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d)
    auto = run_gpu(cfg, inp, num_splits=mla.SPLITS_BALANCED)
    one = run_gpu(cfg, inp, num_splits=1)
    assert auto["status"] == 0 and one["status"] == 0
    within_tolerance(auto["o_lat"].double(), one["o_lat"].double(), "balanced vs unsplit o_lat")
    within_tolerance(auto["lse"].double(), one["lse"].double(), "balanced vs unsplit lse", rel=1e-3, abs_=1e-3)
    check_against_oracle(cfg, inp, auto, rows=rows)
    dec = mla.Decoder(prob, d["kv"], d["seq_lens"], d["w_uk"], d["w_uv"], d["block_table"], cfg.page_size,
                      num_splits=mla.SPLITS_BALANCED)
    out_f = dec.step(d["q_nope"], d["q_rope"]).clone()
    lse_f = dec.lse.clone()
    out_s = dec(d["q_nope"], d["q_rope"]).clone()
    torch.cuda.synchronize()
    assert mla.read_status(dec.workspace) == 0
    assert torch.equal(out_f, out_s) and torch.equal(lse_f, dec.lse)
    assert torch.equal(lse_f.cpu(), auto["lse"])
    return prob, cache


def test_balanced_plan_ragged_paged():
    """Ragged paged sequences, two query tokens (two row blocks, 38 groups): ranges
    start and end inside sequences, so pieces of most sequences merge."""
    cfg = MLAConfig("bal", B=9, s_q=2, len_lo=1, len_hi=3000, paged=True, seed=71, **DSV3_DIMS)
    inp = make_inputs(cfg)
    _balanced_case(cfg, inp, rows=sample_rows(cfg, 64))


def test_balanced_plan_one_long_sequence():
    """One 8,257-token sequence (130 tiles) dealt out to 16 ranges of about 8 tiles."""
    cfg = MLAConfig("bal1", B=1, s_q=1, T=8257, seed=72, **DSV3_DIMS)
    inp = make_inputs(cfg)
    _balanced_case(cfg, inp)


def test_balanced_plan_many_short_sequences():
    """300 short sequences: each range holds many whole sequences (written out
    directly) between the pieces at its two ends."""
    cfg = MLAConfig("bal2", B=300, s_q=1, len_lo=1, len_hi=300, seed=73, **DSV3_DIMS)
    inp = make_inputs(cfg)
    _balanced_case(cfg, inp, rows=sample_rows(cfg, 64) + [128 * b for b in range(0, 300, 7)])


def test_balanced_plan_empty_causal_piece():
    """Two ranges of 20 tiles; the second starts at the first sequence's last tile,
    which holds tokens 640 and 641 only: with four query tokens the first two row
    blocks (queries 0 and 1, limits 638 and 639) see nothing of it, so their piece
    is empty and must merge as nothing."""
    cfg = MLAConfig("bal3", B=2, s_q=4, T=642, seed=74, **DSV3_DIMS)
    inp = make_inputs(cfg, seq_lens=[642, 576])
    _balanced_case(cfg, inp)


# ---------------------------------------------------------------- naive comparison path
def _run_naive(cfg, inp):
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d)
    out, lse, ws = mla.naive_decode(prob, d["q_nope"], d["q_rope"], cache, d["w_uk"], d["w_uv"])
    st = mla.read_status(ws)
    return out.cpu(), lse.cpu(), st


@pytest.mark.parametrize("cfg", [CONFIGS["tiny"],
                                 MLAConfig("n", B=2, s_q=2, len_lo=60, len_hi=300, seed=2, **DSV3_DIMS),
                                 MLAConfig("np", B=2, s_q=1, len_lo=60, len_hi=300, paged=True, seed=9,
                                           **DSV3_DIMS)], ids=["tiny", "dsv3dims", "paged"])
def test_naive_path_matches_oracle(cfg):
    inp = make_inputs(cfg)
    out, lse, st = _run_naive(cfg, inp)
    assert st == 0
    ref_out, ref_lse = oracle.naive(cfg, inp["q_nope"], inp["q_rope"], inp["kv"], inp["seq_lens"],
                                    inp["w_uk"], inp["w_uv"], inp["block_table"], cfg.page_size)
    within_tolerance(out, ref_out, "naive out")
    within_tolerance(lse, ref_lse, "naive lse")
    # and the absorbed GPU path agrees with it
    g = run_gpu(cfg, inp)
    within_tolerance(g["out"], ref_out, "absorbed vs naive reference")


@pytest.mark.parametrize("name,splits", [("dsv3", 0), ("long", 0), ("spec", 0)])
def test_fused_step_matches_separate_calls(name, splits):
    """mla_decode_step (programmatically overlapped launches) gives bit for bit the
    results of the three separate calls, and matches the oracle on sampled rows."""
    from helpers import sample_rows
    cfg = CONFIGS[name].with_(B=min(CONFIGS[name].B, 16))
    inp = make_inputs(cfg)
    d = to_dev(inp)
    prob = mla.Problem.of(cfg)
    dec = mla.Decoder(prob, d["kv"], d["seq_lens"], d["w_uk"], d["w_uv"], d["block_table"], cfg.page_size,
                      num_splits=splits)
    for _ in range(2):
        out_f = dec.step(d["q_nope"], d["q_rope"]).clone()
    lse_f = dec.lse.clone()
    assert mla.read_status(dec.workspace) == 0
    out_s = dec(d["q_nope"], d["q_rope"]).clone()
    torch.cuda.synchronize()
    assert torch.equal(out_f, out_s) and torch.equal(lse_f, dec.lse)
    rows = sample_rows(cfg, 24)
    g = dict(q_cat=dec.q_cat.cpu(), o_lat=dec.o_lat.cpu(), lse=lse_f.cpu(), out=out_f.cpu())
    check_against_oracle(cfg, inp, g, rows=rows)
