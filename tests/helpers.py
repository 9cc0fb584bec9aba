"""Shared helpers of the test suite: run the CUDA path, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mla_decode_attention_absorbed_gb300 import mla
from mla_decode_attention_absorbed_gb300.workloads import MLAConfig, make_inputs

# Spec tolerance per output tensor: max|gpu - ref| <= 2e-2 * max|ref| + 1e-3
REL_TOL = 2e-2
ABS_TOL = 1e-3


def within_tolerance(gpu: torch.Tensor, ref: torch.Tensor, what: str = "", rel=REL_TOL, abs_=ABS_TOL):
    g = gpu.detach().to("cpu", torch.float64)
    r = ref.detach().to("cpu", torch.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    fin = torch.isfinite(r)
    assert torch.equal(torch.isfinite(g), fin), f"{what}: non-finite values differ"
    if fin.sum() == 0:
        return 0.0
    err = (g[fin] - r[fin]).abs().max().item()
    bound = rel * r[fin].abs().max().item() + abs_
    assert err <= bound, f"{what}: max|gpu-ref| = {err:.3e} > {bound:.3e}"
    return err / max(bound, 1e-30)


# lse is an fp32 output of the normaliser: besides the per-tensor bound above it must
# agree with the oracle to 1e-2 nats everywhere (the relative bound alone would allow
# about 0.2 nats at lse ~ 9)
LSE_ABS_TOL = 1e-2


def lse_close(gpu: torch.Tensor, ref: torch.Tensor, what: str = "lse"):
    within_tolerance(gpu, ref, what)
    g = gpu.detach().to("cpu", torch.float64)
    r = ref.detach().to("cpu", torch.float64)
    fin = torch.isfinite(r)
    if fin.any():
        err = (g[fin] - r[fin]).abs().max().item()
        assert err <= LSE_ABS_TOL, f"{what}: max|gpu-ref| = {err:.3e} nats > {LSE_ABS_TOL}"


def to_dev(inp: dict, device="cuda") -> dict:
    out = {}
    for k, v in inp.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


def gpu_cache(cfg: MLAConfig, d: dict, max_seq_len=0):
    prob = mla.Problem.of(cfg)
    cache = mla.make_cache(prob, d["kv"], d["seq_lens"], d["block_table"], cfg.page_size, max_seq_len)
    return prob, cache


def run_gpu(cfg: MLAConfig, inp: dict, num_splits: int = 0, max_seq_len: int = 0):
    """absorb_q -> decode_attn -> out_proj on the GPU; returns CPU tensors and the status word."""
    d = to_dev(inp)
    prob, cache = gpu_cache(cfg, d, max_seq_len)
    q_cat = mla.absorb_q(prob, d["q_nope"], d["q_rope"], d["w_uk"])
    o_lat, lse, ws = mla.decode_attn(prob, q_cat, cache, num_splits=num_splits)
    out = mla.out_proj(prob, o_lat, d["w_uv"])
    status = mla.read_status(ws)
    torch.cuda.synchronize()
    return dict(q_cat=q_cat.cpu(), o_lat=o_lat.cpu(), lse=lse.cpu(), out=out.cpu(), status=status)


def oracle_args(cfg, inp):
    return (inp["q_nope"], inp["q_rope"], inp["kv"], inp["seq_lens"], inp["w_uk"], inp["w_uv"])


def check_against_oracle(cfg: MLAConfig, inp: dict, g: dict, rows=None):
    """Stage-isolated and end-to-end comparison (all rows, or the listed flat rows)."""
    ref_q = oracle.absorb_q(cfg, inp["q_nope"], inp["q_rope"], inp["w_uk"])
    within_tolerance(g["q_cat"], ref_q, "q_cat")
    # attention from the GPU's own q_cat (stage-isolated)
    o_ref, lse_ref = oracle.attend(cfg, g["q_cat"], inp["kv"], inp["seq_lens"], inp["block_table"],
                                   cfg.page_size, rows=rows)
    sel = slice(None) if rows is None else torch.as_tensor(np.asarray(rows, dtype=np.int64))
    within_tolerance(g["o_lat"].view(-1, cfg.d_c)[sel], o_ref.view(-1, cfg.d_c)[sel], "o_lat")
    lse_close(g["lse"].view(-1)[sel], lse_ref.view(-1)[sel], "lse")
    # projection from the GPU's own o_lat (stage-isolated)
    out_ref = oracle.out_proj(cfg, g["o_lat"], inp["w_uv"])
    within_tolerance(g["out"].view(-1, cfg.d_v)[sel], out_ref.view(-1, cfg.d_v)[sel], "out (stage)")
    # end to end from the inputs in fp64
    e2e = oracle.decode(cfg, *oracle_args(cfg, inp), block_table=inp["block_table"], page_size=cfg.page_size,
                        rows=rows)
    within_tolerance(g["out"].view(-1, cfg.d_v)[sel], e2e["out"].view(-1, cfg.d_v)[sel], "out (end to end)")
    lse_close(g["lse"].view(-1)[sel], e2e["lse"].view(-1)[sel], "lse (end to end)")


def sample_rows(cfg: MLAConfig, n: int, seed: int = 1):
    """n flat rows spread over sequences, query positions and heads, always
    including the first and the last row."""
    total = cfg.B * cfg.s_q * cfg.H
    g = np.random.default_rng(seed)
    rows = set(g.choice(total, size=min(n, total), replace=False).tolist())
    rows |= {0, total - 1}
    return sorted(rows)
