"""Pins for the fp64 CPU oracle: it is checked against things other than itself.

- counters: the figures the pages print (tests/golden/page_figures.json);
- library routines: torch.einsum and torch's scaled_dot_product_attention in
  float64 (the naive and the absorbed form both reduce to them);
- closed forms and special cases: T = 1, uniform weights, a dominant score,
  s_q = L, a constant RoPE key, selection-matrix weights, huge scores;
- invariants: naive == absorbed (two bracketings, two independent code paths),
  token permutation, paged == contiguous, split-and-merge == whole.

Each is chosen so that a plausible slip in the oracle (dropped RoPE term, wrong
scale, off-by-one causal limit, transposed or mis-indexed weight, a softmax
without max subtraction, a mis-indexed page) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import counts
from mla_decode_attention_absorbed_gb300.workloads import MLAConfig, make_append_inputs, make_inputs, make_sparse_indices

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")


def small(**kw):
    base = dict(name="t", B=2, H=4, d_c=16, d_rope=8, d_nope=8, d_v=12, s_q=1, T=24)
    base.update(kw)
    return MLAConfig(**base)


def f64(t):
    return t.to(torch.float64)


# ------------------------------------------------------------------ counters vs the pages
@pytest.mark.parametrize("entry", json.load(open(GOLDEN))["entries"], ids=lambda e: e["id"])
def test_counter_matches_page_figure(entry):
    fn = getattr(counts, entry["fn"])
    got = float(fn(**entry["args"]))
    if entry.get("unit") == "GiB":
        got /= 2 ** 30
    want = float(entry["value"])
    if entry["rel"] == 0:
        assert got == want, entry["cite"]
    else:
        assert abs(got - want) <= entry["rel"] * abs(want), (got, want, entry["cite"])


def test_visible_pairs_closed_form():
    # causal prefill of T tokens sees T(T+1)/2 pairs ("MLA, dim by dim", MHA Prefill)
    for T in (1, 2, 7, 64):
        assert counts.visible_pairs(T, T) == T * (T + 1) // 2
    # brute-force enumeration of the reading "query i sees j <= L - s_q + i"
    for L, s_q in ((5, 1), (9, 4), (4, 4), (130, 2)):
        n = sum(1 for i in range(s_q) for j in range(L) if j <= L - s_q + i)
        assert counts.visible_pairs(L, s_q) == n


# ------------------------------------------------------------------ library routines
def _naive_sdpa(cfg, inp):
    """Naive form via torch.einsum + scaled_dot_product_attention, float64."""
    B, H, s_q = cfg.B, cfg.H, cfg.s_q
    outs, lses = [], []
    for b in range(B):
        L = int(inp["seq_lens"][b])
        C = f64(inp["kv"][b, :L, :cfg.d_c])
        KR = f64(inp["kv"][b, :L, cfg.d_c:])
        K = torch.einsum("tc,hcn->htn", C, f64(inp["w_uk"]))
        V = torch.einsum("tc,hcv->htv", C, f64(inp["w_uv"]))
        K = torch.cat([K, KR.unsqueeze(0).expand(H, L, cfg.d_rope)], dim=-1)
        q = torch.cat([f64(inp["q_nope"][b]), f64(inp["q_rope"][b])], dim=-1).transpose(0, 1)  # H, s_q, dk
        mask = torch.tensor([[j <= L - s_q + i for j in range(L)] for i in range(s_q)])
        o = F.scaled_dot_product_attention(q, K, V, attn_mask=mask, scale=cfg.scale)
        s = torch.einsum("hid,htd->hit", q, K) * cfg.scale
        s = s.masked_fill(~mask, float("-inf"))
        outs.append(o.transpose(0, 1))
        lses.append(torch.logsumexp(s, dim=-1).transpose(0, 1))
    return torch.stack(outs), torch.stack(lses)


@pytest.mark.parametrize("kw", [dict(), dict(s_q=3, T=20), dict(B=3, len_lo=5, len_hi=30, s_q=2)])
def test_naive_matches_library_sdpa(kw):
    cfg = small(**kw)
    inp = make_inputs(cfg)
    out, lse = oracle.naive(cfg, inp["q_nope"], inp["q_rope"], inp["kv"], inp["seq_lens"],
                            inp["w_uk"], inp["w_uv"])
    ref_out, ref_lse = _naive_sdpa(cfg, inp)
    torch.testing.assert_close(out, ref_out, rtol=1e-11, atol=1e-12)
    torch.testing.assert_close(lse, ref_lse, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("kw", [dict(), dict(s_q=4, T=19), dict(B=3, len_lo=4, len_hi=40, s_q=2)])
def test_absorbed_stages_match_library(kw):
    cfg = small(**kw)
    inp = make_inputs(cfg)
    r = oracle.decode(cfg, inp["q_nope"], inp["q_rope"], inp["kv"], inp["seq_lens"], inp["w_uk"], inp["w_uv"])
    # absorb_q == einsum with W_UK, then concat of the RoPE query
    q_abs = torch.einsum("bihn,hcn->bihc", f64(inp["q_nope"]), f64(inp["w_uk"]))
    torch.testing.assert_close(r["q_cat"], torch.cat([q_abs, f64(inp["q_rope"])], -1), rtol=1e-13, atol=1e-13)
    # attention over the latent rows == SDPA as one shared K (all 576 columns) and V = c_kv
    for b in range(cfg.B):
        L = int(inp["seq_lens"][b])
        rows = f64(inp["kv"][b, :L])
        q = r["q_cat"][b].transpose(0, 1)  # H, s_q, W
        mask = torch.tensor([[j <= L - cfg.s_q + i for j in range(L)] for i in range(cfg.s_q)])
        o = F.scaled_dot_product_attention(q, rows.expand(cfg.H, L, cfg.W), rows[:, :cfg.d_c].expand(cfg.H, L, cfg.d_c),
                                           attn_mask=mask, scale=cfg.scale)
        torch.testing.assert_close(r["o_lat"][b], o.transpose(0, 1), rtol=1e-11, atol=1e-12)
    # out_proj == einsum with W_UV
    out = torch.einsum("bihc,hcv->bihv", r["o_lat"], f64(inp["w_uv"]))
    torch.testing.assert_close(r["out"], out, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ two bracketings agree
@pytest.mark.parametrize("kw", [dict(), dict(s_q=4, T=33), dict(B=3, len_lo=6, len_hi=50, s_q=3),
                                dict(B=2, len_lo=3, len_hi=70, s_q=2, paged=True, page_size=8)])
def test_naive_equals_absorbed(kw):
    """'The scores are identical' ("Why MLA and MTP Fight Each Other", 3.1) and W^V
    before or after the sum is the same (5.1): the two forms agree in fp64."""
    cfg = small(**kw)
    inp = make_inputs(cfg)
    args = (inp["q_nope"], inp["q_rope"], inp["kv"], inp["seq_lens"], inp["w_uk"], inp["w_uv"])
    a = oracle.decode(cfg, *args, block_table=inp["block_table"], page_size=cfg.page_size)
    n_out, n_lse = oracle.naive(cfg, *args, block_table=inp["block_table"], page_size=cfg.page_size)
    scale = a["out"].abs().max()
    assert (a["out"] - n_out).abs().max() <= 1e-10 * scale
    assert (a["lse"] - n_lse).abs().max() <= 1e-10 * a["lse"].abs().max()


def test_dsv3_shape_naive_equals_absorbed_sampled():
    """DeepSeek-V3 widths (H=128, d_c=512, d_rope=64, d_nope=d_v=128) on a short
    history, sampled rows."""
    cfg = MLAConfig("d", B=2, H=128, d_c=512, d_rope=64, d_nope=128, d_v=128, s_q=2, T=40)
    inp = make_inputs(cfg)
    rows = [0, 5, 127, 128 + 64, 3 * 128 + 1]
    args = (inp["q_nope"], inp["q_rope"], inp["kv"], inp["seq_lens"], inp["w_uk"], inp["w_uv"])
    a = oracle.decode(cfg, *args, rows=rows)
    n_out, _ = oracle.naive(cfg, *args, rows=rows)
    ao, no = a["out"].view(-1, cfg.d_v)[rows], n_out.view(-1, cfg.d_v)[rows]
    assert (ao - no).abs().max() <= 1e-10 * ao.abs().max()


# ------------------------------------------------------------------ special cases
def _q_cat_from(cfg, q):
    return q.reshape(cfg.B, cfg.s_q, cfg.H, cfg.W).to(torch.float64)


def test_single_token_returns_that_latent():
    cfg = small(T=1)
    inp = make_inputs(cfg)
    q_cat = oracle.absorb_q(cfg, inp["q_nope"], inp["q_rope"], inp["w_uk"])
    o, lse = oracle.attend(cfg, q_cat, inp["kv"], inp["seq_lens"])
    c0 = f64(inp["kv"][:, 0, :cfg.d_c])  # [B, d_c]
    assert torch.equal(o[:, 0], c0.unsqueeze(1).expand_as(o[:, 0]))
    s0 = cfg.scale * torch.einsum("bhw,bw->bh", q_cat[:, 0], f64(inp["kv"][:, 0]))
    torch.testing.assert_close(lse[:, 0], s0, rtol=1e-14, atol=1e-14)


def test_zero_query_gives_uniform_weights():
    cfg = small(s_q=2, B=3, len_lo=3, len_hi=40)
    inp = make_inputs(cfg)
    q_cat = torch.zeros(cfg.B, cfg.s_q, cfg.H, cfg.W, dtype=torch.float64)
    o, lse = oracle.attend(cfg, q_cat, inp["kv"], inp["seq_lens"])
    for b in range(cfg.B):
        L = int(inp["seq_lens"][b])
        for i in range(cfg.s_q):
            n = L - cfg.s_q + i + 1
            mean = f64(inp["kv"][b, :n, :cfg.d_c]).mean(0)
            torch.testing.assert_close(o[b, i], mean.expand(cfg.H, cfg.d_c), rtol=1e-13, atol=1e-14)
            assert torch.allclose(lse[b, i], torch.full((cfg.H,), math.log(n), dtype=torch.float64), atol=1e-14)


def test_dominant_score_selects_its_row():
    """One-hot latents; the query aims one token 60 units above the rest."""
    cfg = small(B=1, H=2, d_c=8, d_rope=4, T=8)
    inp = make_inputs(cfg)
    kv = torch.zeros(1, 8, cfg.W, dtype=torch.bfloat16)
    for j in range(8):
        kv[0, j, j] = 1.0
    q_cat = torch.zeros(1, 1, cfg.H, cfg.W, dtype=torch.float64)
    q_cat[0, 0, 0, 3] = 60.0 / cfg.scale   # head 0 -> token 3
    q_cat[0, 0, 1, 6] = 60.0 / cfg.scale   # head 1 -> token 6
    o, lse = oracle.attend(cfg, q_cat, kv, inp["seq_lens"])
    for h, j in ((0, 3), (1, 6)):
        expect = torch.zeros(cfg.d_c, dtype=torch.float64)
        w = math.exp(60.0)
        expect[:] = 1.0 / (w + 7)
        expect[j] = w / (w + 7)
        torch.testing.assert_close(o[0, 0, h], expect, rtol=1e-14, atol=1e-30)
        assert abs(lse[0, 0, h].item() - (60.0 + math.log1p(7 * math.exp(-60.0)))) < 1e-13


def test_huge_scores_need_max_subtraction():
    """Scores around 1e4: exp() without the running maximum would overflow."""
    cfg = small(B=1, H=1, d_c=8, d_rope=0, T=4)
    kv = torch.zeros(1, 4, 8, dtype=torch.bfloat16)
    for j in range(4):
        kv[0, j, j] = 1.0
    q_cat = torch.zeros(1, 1, 1, 8, dtype=torch.float64)
    base = 1.0e4 / cfg.scale
    q_cat[0, 0, 0, :4] = torch.tensor([base, base + 1 / cfg.scale, base, base - 2 / cfg.scale], dtype=torch.float64)
    o, lse = oracle.attend(cfg, q_cat, kv, torch.tensor([4], dtype=torch.int32))
    s = [1.0e4, 1.0e4 + 1, 1.0e4, 1.0e4 - 2]
    ref = counts.log_sum_exp(s)
    assert abs(lse.item() - ref) < 1e-9
    p = [math.exp(x - ref) for x in s]
    torch.testing.assert_close(o[0, 0, 0, :4], torch.tensor(p, dtype=torch.float64), rtol=1e-12, atol=1e-15)


def test_causal_limit_when_all_tokens_are_new():
    """s_q == L: query 0 sees token 0 only, the last query sees all L."""
    cfg = small(s_q=5, T=5)
    inp = make_inputs(cfg)
    q_cat = oracle.absorb_q(cfg, inp["q_nope"], inp["q_rope"], inp["w_uk"])
    o, lse = oracle.attend(cfg, q_cat, inp["kv"], inp["seq_lens"])
    c0 = f64(inp["kv"][:, 0, :cfg.d_c])
    assert torch.equal(o[:, 0], c0.unsqueeze(1).expand_as(o[:, 0]))
    # the last query equals an s_q = 1 decode over the same L tokens
    cfg1 = cfg.with_(s_q=1)
    o1, lse1 = oracle.attend(cfg1, q_cat[:, -1:], inp["kv"], inp["seq_lens"])
    torch.testing.assert_close(o[:, -1:], o1, rtol=0, atol=0)
    torch.testing.assert_close(lse[:, -1:], lse1, rtol=0, atol=0)


def test_constant_rope_key_shifts_lse_only():
    """A RoPE key shared by every token adds one constant to every score: weights and
    o_lat stay, lse moves by scale * q_rope . k_rope (pins the RoPE term and its scale)."""
    cfg = small(s_q=2, T=30)
    inp = make_inputs(cfg)
    kv = inp["kv"].clone()
    kv[:, :, cfg.d_c:] = kv[:, :1, cfg.d_c:]
    q_cat = oracle.absorb_q(cfg, inp["q_nope"], inp["q_rope"], inp["w_uk"])
    o, lse = oracle.attend(cfg, q_cat, kv, inp["seq_lens"])
    q0 = q_cat.clone()
    q0[..., cfg.d_c:] = 0
    o0, lse0 = oracle.attend(cfg, q0, kv, inp["seq_lens"])
    shift = cfg.scale * torch.einsum("bihr,br->bih", q_cat[..., cfg.d_c:], f64(kv[:, 0, cfg.d_c:]))
    torch.testing.assert_close(o, o0, rtol=1e-12, atol=1e-13)
    torch.testing.assert_close(lse, lse0 + shift, rtol=1e-12, atol=1e-12)


def test_token_permutation_invariance():
    cfg = small(T=40)
    inp = make_inputs(cfg)
    q_cat = oracle.absorb_q(cfg, inp["q_nope"], inp["q_rope"], inp["w_uk"])
    o, lse = oracle.attend(cfg, q_cat, inp["kv"], inp["seq_lens"])
    perm = torch.randperm(40, generator=torch.Generator().manual_seed(7))
    o2, lse2 = oracle.attend(cfg, q_cat, inp["kv"][:, perm], inp["seq_lens"])
    torch.testing.assert_close(o, o2, rtol=1e-13, atol=1e-14)
    torch.testing.assert_close(lse, lse2, rtol=1e-14, atol=1e-14)


def test_absorb_q_selection_weights():
    """W_UK[h, c, n] = (h+1) if c == 2n + h else 0: q_abs[c] = (h+1) q_nope[(c-h)/2]."""
    cfg = small(H=3, d_c=20, d_nope=8)
    inp = make_inputs(cfg)
    w = torch.zeros(cfg.H, cfg.d_c, cfg.d_nope, dtype=torch.bfloat16)
    for h in range(cfg.H):
        for n in range(cfg.d_nope):
            w[h, 2 * n + h, n] = h + 1
    q_cat = oracle.absorb_q(cfg, inp["q_nope"], inp["q_rope"], w)
    qn = f64(inp["q_nope"])
    for h in range(cfg.H):
        for c in range(cfg.d_c):
            if (c - h) % 2 == 0 and 0 <= (c - h) // 2 < cfg.d_nope:
                expect = (h + 1) * qn[:, :, h, (c - h) // 2]
            else:
                expect = torch.zeros_like(qn[:, :, h, 0])
            assert torch.equal(q_cat[:, :, h, c], expect)
    assert torch.equal(q_cat[..., cfg.d_c:], f64(inp["q_rope"]))


def test_out_proj_selection_weights():
    """W_UV[h, c, v] = 1 if c == v + h: out[v] = o_lat[v + h]."""
    cfg = small(H=3, d_c=16, d_v=10)
    w = torch.zeros(cfg.H, cfg.d_c, cfg.d_v, dtype=torch.bfloat16)
    for h in range(cfg.H):
        for v in range(cfg.d_v):
            w[h, v + h, v] = 1
    o_lat = torch.randn(cfg.B, cfg.s_q, cfg.H, cfg.d_c, dtype=torch.float64)
    out = oracle.out_proj(cfg, o_lat, w)
    for h in range(cfg.H):
        assert torch.equal(out[:, :, h], o_lat[:, :, h, h:h + cfg.d_v])


# ------------------------------------------------------------------ layout invariants
def test_paged_equals_contiguous():
    cfg = small(B=3, len_lo=5, len_hi=60, s_q=2)
    inp = make_inputs(cfg)
    q_cat = oracle.absorb_q(cfg, inp["q_nope"], inp["q_rope"], inp["w_uk"])
    o, lse = oracle.attend(cfg, q_cat, inp["kv"], inp["seq_lens"])
    ps = 8
    pages = []
    table = []
    for b in range(cfg.B):
        L = int(inp["seq_lens"][b])
        n = -(-L // ps)
        ids = []
        for p in range(n):
            blk = torch.full((ps, cfg.W), float("nan"), dtype=torch.bfloat16)
            take = inp["kv"][b, p * ps:min(L, (p + 1) * ps)]
            blk[:take.shape[0]] = take
            ids.append(len(pages))
            pages.append(blk)
        table.append(ids)
    perm = torch.randperm(len(pages), generator=torch.Generator().manual_seed(3))
    pool = torch.stack(pages)[torch.argsort(perm)]  # page k of the table sits at slot perm[k]
    max_pages = max(len(t) for t in table)
    bt = torch.full((cfg.B, max_pages + 2), -1, dtype=torch.int32)
    for b, ids in enumerate(table):
        bt[b, :len(ids)] = perm[torch.tensor(ids)].to(torch.int32)
    o2, lse2 = oracle.attend(cfg, q_cat, pool, inp["seq_lens"], block_table=bt, page_size=ps)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_row_subset_matches_full():
    cfg = small(s_q=2, T=33)
    inp = make_inputs(cfg)
    q_cat = oracle.absorb_q(cfg, inp["q_nope"], inp["q_rope"], inp["w_uk"])
    o, lse = oracle.attend(cfg, q_cat, inp["kv"], inp["seq_lens"])
    rows = [1, 6, 13]
    o2, lse2 = oracle.attend(cfg, q_cat, inp["kv"], inp["seq_lens"], rows=rows)
    assert torch.equal(o.view(-1, cfg.d_c)[rows], o2.view(-1, cfg.d_c)[rows])
    assert torch.isnan(o2.view(-1, cfg.d_c)[0]).all()


# ------------------------------------------------------------------ split-T merge
def test_split_and_merge_equals_whole():
    cfg = small(s_q=3, T=50, B=1)
    inp = make_inputs(cfg)
    q_cat = oracle.absorb_q(cfg, inp["q_nope"], inp["q_rope"], inp["w_uk"])
    o, lse = oracle.attend(cfg, q_cat, inp["kv"], inp["seq_lens"])
    g = np.random.default_rng(0)
    for row in range(cfg.s_q * cfg.H):
        cuts = sorted(set(g.integers(1, 50, size=4).tolist()))
        bounds = [0] + cuts + [50, 60]  # the last chunk lies wholly past every query's limit
        parts = [oracle.attend_partial(cfg, q_cat, inp["kv"], inp["seq_lens"], row, a, b)
                 for a, b in zip(bounds[:-1], bounds[1:])]
        m = [p[0] for p in parts]
        assert m[-1] == float("-inf")
        ob, lb = oracle.combine(m, [p[1] for p in parts], torch.stack([p[2] for p in parts]))
        torch.testing.assert_close(ob, o.view(-1, cfg.d_c)[row], rtol=1e-12, atol=1e-13)
        assert abs(lb - lse.view(-1)[row].item()) < 1e-12


def test_merge_of_nothing():
    o, lse = oracle.combine([float("-inf")] * 2, [0.0, 0.0], torch.zeros(2, 4, dtype=torch.float64))
    assert lse == float("-inf") and torch.equal(o, torch.zeros(4, dtype=torch.float64))


# ----------------------------------------------------------------------------- cache append
# "MLA, dim by dim", "MLA Decode": the new token's hidden state is compressed,
# x . W_DKV -> c^KV (2 d d_c FLOPs), and appended to the latent cache.

def test_down_proj_selection_matrix():
    """A one-hot W_DKV picks columns of x: c[m, k] = x[m, perm[k]] exactly."""
    g = torch.Generator().manual_seed(3)
    d_model, d_c = 40, 16
    x = torch.randn(3, 2, d_model, generator=g).bfloat16()
    perm = torch.randperm(d_model, generator=g)[:d_c]
    w = torch.zeros(d_model, d_c)
    w[perm, torch.arange(d_c)] = 1.0
    c = oracle.down_proj(x, w.bfloat16())
    assert torch.equal(c, x.double()[..., perm])


def test_down_proj_linearity():
    """c is linear in x: c(2 x1 - x2) = 2 c(x1) - c(x2) to rounding of the fp64 sums."""
    g = torch.Generator().manual_seed(4)
    x1 = torch.randint(-8, 8, (4, 24), generator=g).float().bfloat16()
    x2 = torch.randint(-8, 8, (4, 24), generator=g).float().bfloat16()
    w = (torch.randint(-8, 8, (24, 8), generator=g).float() / 8).bfloat16()
    lhs = oracle.down_proj((2 * x1.float() - x2.float()).bfloat16(), w)
    rhs = 2 * oracle.down_proj(x1, w) - oracle.down_proj(x2, w)
    assert torch.equal(lhs, rhs)  # small integers and eighths: every sum is exact


def _append_case(paged: bool, s_q: int = 2):
    cfg = MLAConfig("append_pin", B=3, H=4, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=s_q,
                    len_lo=5, len_hi=150, paged=paged, page_size=64, seed=11, canary=False)
    inp = make_inputs(cfg)
    app = make_append_inputs(cfg, d_model=48)
    new, written = oracle.cache_append(cfg, app["x"], app["w_dkv"], app["k_rope"], inp["kv"], inp["seq_lens"],
                                       inp["block_table"], cfg.page_size)
    return cfg, inp, app, new, written


def _logical_rows(cfg, inp, cache64):
    """[b][j] -> fp64 row of token j of sequence b (contiguous or through the block table)."""
    out = {}
    for b in range(cfg.B):
        L = int(inp["seq_lens"][b])
        for j in range(L):
            if inp["block_table"] is None:
                out[(b, j)] = cache64[b, j]
            else:
                page = int(inp["block_table"][b, j // cfg.page_size])
                out[(b, j)] = cache64[page, j % cfg.page_size]
    return out


def test_append_writes_the_new_positions_only():
    for paged in (False, True):
        cfg, inp, app, new, written = _append_case(paged)
        old = inp["kv"].double()
        c = oracle.down_proj(app["x"], app["w_dkv"])
        rows = _logical_rows(cfg, inp, new)
        n_new = 0
        for b in range(cfg.B):
            L = int(inp["seq_lens"][b])
            for i in range(cfg.s_q):
                r = rows[(b, L - cfg.s_q + i)]
                assert torch.equal(r[:cfg.d_c], c[b, i])
                assert torch.equal(r[cfg.d_c:], app["k_rope"][b, i].double())
                n_new += 1
        assert int(written.sum()) == n_new
        assert torch.equal(new[~written], old[~written])


def test_append_paged_equals_contiguous():
    cfg_c, inp_c, _, new_c, _ = _append_case(False)
    cfg_p, inp_p, _, new_p, _ = _append_case(True)
    # same lengths (same seed, same draw order for the lengths)
    assert torch.equal(inp_c["seq_lens"], inp_p["seq_lens"])
    rc, rp = _logical_rows(cfg_c, inp_c, new_c), _logical_rows(cfg_p, inp_p, new_p)
    for b in range(cfg_c.B):
        L = int(inp_c["seq_lens"][b])
        for i in range(cfg_c.s_q):
            assert torch.equal(rc[(b, L - cfg_c.s_q + i)], rp[(b, L - cfg_c.s_q + i)])


def test_append_skips_invalid_lengths_and_pages():
    cfg, inp, app, _, _ = _append_case(True, s_q=1)
    lens = inp["seq_lens"].clone()
    lens[0] = 0                      # shorter than s_q
    bt = inp["block_table"].clone()
    L1 = int(lens[1])
    bt[1, (L1 - 1) // cfg.page_size] = 10 ** 6  # page outside the pool
    new, written = oracle.cache_append(cfg, app["x"], app["w_dkv"], app["k_rope"], inp["kv"], lens, bt,
                                       cfg.page_size)
    assert int(written.sum()) == cfg.B - 2


# ----------------------------------------------------------------------------- sparse top-k decode
# "Why MLA and MTP Fight Each Other", 6: the selected tokens are gathered by
# index and the scoring and the weighted sum run over those only.

def _sparse_case(s_q=2, paged=False):
    cfg = MLAConfig("sparse_pin", B=3, H=4, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=s_q,
                    len_lo=40, len_hi=130, paged=paged, seed=21, canary=True)
    inp = make_inputs(cfg)
    q_cat = oracle.absorb_q(cfg, inp["q_nope"], inp["q_rope"], inp["w_uk"]).to(torch.bfloat16)
    return cfg, inp, q_cat


def _full_lists(cfg, lens, extra=0):
    """Every visible token of every (b, i), in order, padded with -1 (plus `extra` pads)."""
    topk = int(lens.max()) + extra
    idx = torch.full((cfg.B, cfg.s_q, topk), -1, dtype=torch.int32)
    for b in range(cfg.B):
        for i in range(cfg.s_q):
            n = int(lens[b]) - cfg.s_q + i + 1
            idx[b, i, :n] = torch.arange(n, dtype=torch.int32)
    return idx


@pytest.mark.parametrize("paged", [False, True])
def test_sparse_with_every_token_is_dense(paged):
    cfg, inp, q = _sparse_case(paged=paged)
    idx = _full_lists(cfg, inp["seq_lens"], extra=5)
    o_s, l_s = oracle.attend_sparse(cfg, q, inp["kv"], inp["seq_lens"], idx, inp["block_table"], cfg.page_size)
    o_d, l_d = oracle.attend(cfg, q, inp["kv"], inp["seq_lens"], inp["block_table"], cfg.page_size)
    assert torch.allclose(o_s, o_d, rtol=0, atol=1e-12) and torch.allclose(l_s, l_d, rtol=0, atol=1e-12)


def test_sparse_order_padding_and_future_entries_do_not_matter():
    cfg, inp, q = _sparse_case()
    lens = inp["seq_lens"]
    idx = make_sparse_indices(cfg, lens, topk=24)
    o0, l0 = oracle.attend_sparse(cfg, q, inp["kv"], lens, idx)
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(idx.shape[-1], generator=g)
    o1, l1 = oracle.attend_sparse(cfg, q, inp["kv"], lens, idx[..., perm])
    assert torch.allclose(o0, o1, atol=1e-12) and torch.allclose(l0, l1, atol=1e-12)
    # -1 padding and entries past the causal limit (future tokens, NaN canaries) take no part
    fut = torch.empty(cfg.B, cfg.s_q, 3, dtype=torch.int32)
    for b in range(cfg.B):
        for i in range(cfg.s_q):
            fut[b, i] = torch.tensor([-1, int(lens[b]) - cfg.s_q + i + 1, int(lens[b]) + 7])
    o2, l2 = oracle.attend_sparse(cfg, q, inp["kv"], lens, torch.cat([idx, fut], dim=-1))
    assert torch.allclose(o0, o2, atol=1e-12) and torch.allclose(l0, l2, atol=1e-12)


def test_sparse_single_token_is_that_latent():
    cfg, inp, q = _sparse_case(s_q=1)
    lens = inp["seq_lens"]
    idx = torch.full((cfg.B, 1, 4), -1, dtype=torch.int32)
    idx[:, 0, 2] = 3
    o, lse = oracle.attend_sparse(cfg, q, inp["kv"], lens, idx)
    for b in range(cfg.B):
        row = inp["kv"][b, 3].double()
        assert torch.equal(o[b, 0], row[:cfg.d_c].expand(cfg.H, -1))
        s = cfg.scale * (q[b, 0].double() @ row)
        assert torch.allclose(lse[b, 0], s, atol=1e-12)


def test_sparse_no_visible_entry_gives_zero_and_minus_inf():
    cfg, inp, q = _sparse_case(s_q=1)
    idx = torch.full((cfg.B, 1, 8), -1, dtype=torch.int32)
    o, lse = oracle.attend_sparse(cfg, q, inp["kv"], inp["seq_lens"], idx)
    assert torch.equal(o, torch.zeros_like(o)) and bool(torch.isneginf(lse).all())


# ------------------------------------------------------------------ FP8 (E4M3) latent cache
def test_e4m3_decode_matches_library_for_every_code():
    """The oracle's E4M3 decoder against torch's float8_e4m3fn for all 256 codes,
    plus the format's landmarks (1, max 448, smallest subnormal 2^-9, NaN)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64)
    mine = torch.tensor([oracle.e4m3_to_f64(c) for c in range(256)], dtype=torch.float64)
    nan = torch.isnan(lib)
    assert torch.equal(nan, torch.isnan(mine)) and int(nan.sum()) == 2  # 0x7F and 0xFF
    assert torch.equal(lib[~nan], mine[~nan])
    assert oracle.e4m3_to_f64(0x38) == 1.0 and oracle.e4m3_to_f64(0x7E) == 448.0
    assert oracle.e4m3_to_f64(0x01) == 2.0 ** -9 and oracle.e4m3_to_f64(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_f64(0xB8) == -1.0


def _fp8_case(paged=False, s_q=2, kv_scale=1.0 / 16.0):
    from mla_decode_attention_absorbed_gb300.workloads import to_fp8_cache
    cfg = MLAConfig("fp8_pin", B=3, H=4, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=s_q,
                    len_lo=20, len_hi=90, paged=paged, seed=31, canary=True)
    inp = make_inputs(cfg)
    codes = to_fp8_cache(inp["kv"], kv_scale)
    q_cat = oracle.absorb_q(cfg, inp["q_nope"], inp["q_rope"], inp["w_uk"]).to(torch.bfloat16)
    return cfg, inp, codes, q_cat


@pytest.mark.parametrize("paged", [False, True])
def test_fp8_cache_equals_bf16_cache_of_its_values(paged):
    """With a power-of-two scale every kv_scale * code is a bf16 number: attention
    over the FP8 cache must equal, bit for bit, attention over that bf16 cache."""
    cfg, inp, codes, q = _fp8_case(paged)
    deq = (codes.view(torch.float8_e4m3fn).to(torch.float32) / 16.0).to(torch.bfloat16)
    o8, l8 = oracle.attend(cfg, q, codes, inp["seq_lens"], inp["block_table"], cfg.page_size, kv_scale=1.0 / 16.0)
    ob, lb = oracle.attend(cfg, q, deq, inp["seq_lens"], inp["block_table"], cfg.page_size)
    assert torch.equal(o8, ob) and torch.equal(l8, lb)


def test_fp8_cache_scale_enters_scores_and_values():
    """A non-power-of-two scale against SDPA on the library-decoded values: the
    scale multiplies both the keys (scores) and the values (latent sum)."""
    s = 0.0371
    cfg, inp, codes, q = _fp8_case(kv_scale=s)
    o8, l8 = oracle.attend(cfg, q, codes, inp["seq_lens"], kv_scale=s)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64) * s
    for b in range(cfg.B):
        L = int(inp["seq_lens"][b])
        rows = vals[b, :L]
        qq = f64(q[b]).transpose(0, 1)
        mask = torch.tensor([[j <= L - cfg.s_q + i for j in range(L)] for i in range(cfg.s_q)])
        o = F.scaled_dot_product_attention(qq, rows.expand(cfg.H, L, cfg.W), rows[:, :cfg.d_c].expand(cfg.H, L, cfg.d_c),
                                           attn_mask=mask, scale=cfg.scale)
        torch.testing.assert_close(o8[b], o.transpose(0, 1), rtol=1e-11, atol=1e-12)


def test_fp8_sparse_full_list_is_dense():
    cfg, inp, codes, q = _fp8_case(paged=True)
    idx = _full_lists(cfg, inp["seq_lens"], extra=3)
    o_s, l_s = oracle.attend_sparse(cfg, q, codes, inp["seq_lens"], idx, inp["block_table"], cfg.page_size,
                                    kv_scale=1.0 / 16.0)
    o_d, l_d = oracle.attend(cfg, q, codes, inp["seq_lens"], inp["block_table"], cfg.page_size, kv_scale=1.0 / 16.0)
    assert torch.allclose(o_s, o_d, rtol=0, atol=1e-12) and torch.allclose(l_s, l_d, rtol=0, atol=1e-12)


def test_fp8_canaries_stay_unread():
    """NaN codes sit in every row past a sequence's length; no output may be NaN."""
    cfg, inp, codes, q = _fp8_case()
    assert bool((codes == 0x7F).any())
    o8, l8 = oracle.attend(cfg, q, codes, inp["seq_lens"], kv_scale=1.0 / 16.0)
    assert not torch.isnan(o8).any() and not torch.isnan(l8).any()


def test_e4m3_encode_roundtrip_ties_and_saturation():
    """Encoding every finite code's value gives the code back; midpoints round to
    the even code; values past 448 saturate; the library cast agrees in range."""
    vals = torch.tensor([oracle.e4m3_to_f64(c) for c in range(256)], dtype=torch.float64)
    codes = oracle.e4m3_encode(vals)
    fin = ~torch.isnan(vals)
    idx = torch.arange(256)[fin]
    back = codes[fin].to(torch.int64)
    # +0 and -0 both encode to themselves
    assert torch.equal(back, idx)
    # midpoints between consecutive positive codes go to the even one
    for c in range(0, 0x7E):
        mid = (oracle.e4m3_to_f64(c) + oracle.e4m3_to_f64(c + 1)) / 2
        assert int(oracle.e4m3_encode([mid])[0]) == (c if c % 2 == 0 else c + 1)
    assert int(oracle.e4m3_encode([1e6])[0]) == 0x7E and int(oracle.e4m3_encode([-500.0])[0]) == 0xFE
    x = torch.randn(4000, generator=torch.Generator().manual_seed(5), dtype=torch.float64) * 40
    assert torch.equal(oracle.e4m3_encode(x), x.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8))


def test_fp8_append_rows_are_the_quantised_down_projection():
    from mla_decode_attention_absorbed_gb300.workloads import to_fp8_cache
    cfg, inp, a, _, _ = _append_case(paged=False)
    codes = to_fp8_cache(inp["kv"])
    out8, w8 = oracle.cache_append(cfg, a["x"], a["w_dkv"], a["k_rope"], codes, inp["seq_lens"], kv_scale=1.0 / 16.0)
    outb, wb = oracle.cache_append(cfg, a["x"], a["w_dkv"], a["k_rope"], inp["kv"], inp["seq_lens"])
    assert torch.equal(w8, wb)
    # written rows: the exact values divided by the scale; others: the old codes' values
    assert torch.allclose(out8[w8], outb[wb] * 16.0, rtol=0, atol=0)
    old = codes.view(torch.float8_e4m3fn).to(torch.float64)
    assert torch.equal(out8[~w8].nan_to_num(1e9), old[~w8].nan_to_num(1e9))
