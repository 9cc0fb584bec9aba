"""Closed-form FLOP and byte counters for MLA decode -- TEST INFRASTRUCTURE.

These are the counting rules the pages state, written as functions so the
test suite can pin them against the numbers the pages print.  One multiply-add
is 2 FLOPs ("MLA, dim by dim", "Tensor View": FLOPs = 2 * output dims * contracted
dim).  Softmax, masking and rotation are not counted ("MLA, dim by dim",
"Notation and Preliminaries"; "Why MLA and MTP Fight Each Other", section 1).

Symbols: H heads, d_c latent width, d_rope (d_s) decoupled RoPE key width,
d_k / d_v per-head key / value widths, L cached tokens, S query tokens, b bytes
per cached element.
"""
from __future__ import annotations

import math


# ------------------------------------------------------------------ per cached token, decode
def latent_bytes_per_token(d_c: int, d_rope: int, b: int = 2) -> int:
    """Bytes of one cached token of one layer: the latent plus the RoPE key
    ("Decode attention intensity...", "A strong answer")."""
    return (d_c + d_rope) * b


def absorbed_flops_per_token(H: int, d_c: int, d_rope: int) -> int:
    """FLOPs one query token spends on one cached token with absorption: every
    head scores against the full d_c + d_rope row and aggregates over the d_c
    latent ("Decode attention intensity...", "A strong answer"; "Why MLA and MTP
    Fight Each Other", Appendix A)."""
    return H * (2 * (d_c + d_rope) + 2 * d_c)


def absorbed_intensity(H: int, d_c: int, d_rope: int, b: int = 2, s_q: int = 1) -> float:
    """FLOP/B of the attention core for s_q query tokens against one cache read
    (causal triangle ignored, as in "Decode attention intensity...", reversal paragraph)."""
    return s_q * absorbed_flops_per_token(H, d_c, d_rope) / latent_bytes_per_token(d_c, d_rope, b)


def decompress_flops_per_token(H: int, d_c: int, d_k: int, d_v: int) -> int:
    """FLOPs to re-expand one cached latent into every head's K and V
    ("Decode attention intensity...", paragraph on absorption; "Why MLA and MTP
    Fight Each Other", 3.3): 2 * d_c * H * (d_k + d_v)."""
    return 2 * d_c * H * (d_k + d_v)


def gqa_intensity(g: int, b: int = 2) -> float:
    """2g/b: decode attention intensity with g query heads per KV head
    ("Decode attention intensity...", first equation)."""
    return 2 * g / b


# ------------------------------------------------------------------ per pair (MACs), one head
def pair_macs(d_c: int, d_k: int, d_v: int, d_rope: int = 0, absorbed: bool = True) -> int:
    """Multiply-accumulates per query-token x cached-token pair and head
    ("Why MLA and MTP Fight Each Other", 5.1 and A.3): absorbed = score over
    d_c + d_rope plus a d_c-wide aggregate; expanded = score over d_k + d_rope plus a
    d_v-wide aggregate."""
    if absorbed:
        return (d_c + d_rope) + d_c
    return (d_k + d_rope) + d_v


def projection_macs(d_c: int, d_k: int, d_v: int) -> int:
    """Per-head projection MACs of either bracketing for one token: d_c (d_k + d_v)
    ("Why MLA and MTP Fight Each Other", 5.2)."""
    return d_c * (d_k + d_v)


# ------------------------------------------------------------------ whole-layer decode / prefill
def mla_algorithm_flops(H: int, d_c: int, d_k: int, d_v: int, S: int, L: int,
                        causal: bool = False) -> int:
    """Absorb bracketing: projections billed per query token, 2 d_c MACs per pair
    ("Why MLA and MTP Fight Each Other", 5.3).  ``causal`` counts the S(S+1)/2
    visible pairs of a prefill where S == L (5.5)."""
    pairs = S * (S + 1) // 2 if causal else S * L
    return 2 * H * (S * projection_macs(d_c, d_k, d_v) + pairs * 2 * d_c)


def mha_algorithm_flops(H: int, d_c: int, d_k: int, d_v: int, S: int, L: int,
                        causal: bool = False) -> int:
    """Expand bracketing: projections billed per cached token, d_k + d_v MACs per pair."""
    pairs = S * (S + 1) // 2 if causal else S * L
    return 2 * H * (L * projection_macs(d_c, d_k, d_v) + pairs * (d_k + d_v))


def mla_algorithm_bytes(d_c: int, L: int, b: int = 2) -> int:
    """Decode bytes of the absorb bracketing: the latent history, read once."""
    return L * d_c * b


def mha_algorithm_bytes(H: int, d_c: int, d_k: int, d_v: int, L: int, b: int = 2) -> int:
    """Decode bytes of the expand bracketing: the latent history plus the
    materialised per-head K and V."""
    return L * (d_c + H * (d_k + d_v)) * b


def crossover_S(d_c: int, d_k: int, d_v: int, L: float) -> float:
    """Query count S* at which both bracketings cost the same FLOPs
    ("Why MLA and MTP Fight Each Other", 5.6): setting the two 5.3 totals equal,
    S* = L d_c (d_k + d_v) / (d_c (d_k + d_v) + L (2 d_c - d_k - d_v)).  H cancels."""
    p = projection_macs(d_c, d_k, d_v)
    return L * p / (p + L * (2 * d_c - d_k - d_v))


def crossover_L_decode(d_c: int, d_k: int, d_v: int) -> float:
    """History length at which the two bracketings tie for S = 1 (5.4)."""
    p = projection_macs(d_c, d_k, d_v)
    return p / (p + (d_k + d_v) - 2 * d_c)


def fixed_decode_flops(d_model: int, H: int, d_c: int, d_k: int, d_v: int) -> int:
    """History-independent decode FLOPs of one token ("Why MLA and MTP Fight Each
    Other", 4.1): latent compression, query projection, K-side absorption and the
    per-head latent-to-value projection."""
    return 2 * d_model * d_c + 2 * d_model * H * d_k + 2 * H * d_k * d_c + 2 * H * d_c * d_v


def per_token_history_flops(H: int, d_c: int) -> int:
    """History-dependent decode FLOPs per cached token without RoPE: 4 H d_c (4.1)."""
    return 4 * H * d_c


def sparse_mla_flops(H: int, d_c: int, d_k: int, d_v: int, k: int) -> int:
    """Absorbed decode over k gathered tokens ("Why MLA and MTP Fight Each Other", 6)."""
    return mla_algorithm_flops(H, d_c, d_k, d_v, 1, k)


def cache_bytes(numbers_per_token: int, ctx: int, layers: int, b: int = 2) -> int:
    """Cache size for a context of ``ctx`` tokens ("Why MLA and MTP Fight Each Other", 3)."""
    return numbers_per_token * ctx * layers * b


def input_projection_flops_per_token(d: int, h: int, d_k: int, d_v: int, d_c: int,
                                     d_qc: int | None, kind: str) -> int:
    """Prefill input-projection FLOPs per token ("MLA, dim by dim", Prefill Comparison table)."""
    if kind == "mha":
        return 2 * d * h * (2 * d_k + d_v)
    if kind == "mla_noq":
        return 2 * d * d_c + 2 * h * d * d_k + 2 * h * d_c * (d_k + d_v)
    if kind == "mla_qcomp":
        return 2 * d * d_c + 2 * d * d_qc + 2 * h * d_qc * d_k + 2 * h * d_c * (d_k + d_v)
    raise ValueError(kind)


def ridge(peak_flops: float, bandwidth_bytes: float) -> float:
    """Roofline balance point, FLOP/B ("Why MLA and MTP Fight Each Other", 1)."""
    return peak_flops / bandwidth_bytes


# ------------------------------------------------------------------ the workloads this library runs
def visible_pairs(L: int, s_q: int) -> int:
    """(query, cached-token) pairs under the causal rule among the s_q new tokens:
    query i sees L - s_q + i + 1 tokens, so sum = s_q L - s_q (s_q - 1) / 2."""
    return s_q * L - s_q * (s_q - 1) // 2


def attention_flops(H: int, d_c: int, d_rope: int, seq_lens, s_q: int) -> int:
    """Algorithmic FLOPs of the attention core over a batch."""
    per_pair = 2 * (d_c + d_rope) + 2 * d_c
    return sum(visible_pairs(int(L), s_q) for L in seq_lens) * H * per_pair


def attention_bytes(H: int, d_c: int, d_rope: int, seq_lens, s_q: int, b: int = 2) -> int:
    """Algorithmic HBM bytes of the attention core: each cached token read once,
    q_cat read once, o_lat (bf16) and lse (fp32) written once."""
    B = len(seq_lens)
    cache = sum(int(L) for L in seq_lens) * (d_c + d_rope) * b
    q = B * s_q * H * (d_c + d_rope) * b
    o = B * s_q * H * d_c * b
    lse = B * s_q * H * 4
    return cache + q + o + lse


def absorb_flops(B: int, s_q: int, H: int, d_nope: int, d_c: int) -> int:
    return 2 * B * s_q * H * d_nope * d_c


def absorb_bytes(B: int, s_q: int, H: int, d_nope: int, d_c: int, d_rope: int, b: int = 2) -> int:
    """q_nope + q_rope read, W_UK read once, q_cat written."""
    return b * (B * s_q * H * (d_nope + d_rope) + H * d_c * d_nope + B * s_q * H * (d_c + d_rope))


def out_proj_flops(B: int, s_q: int, H: int, d_c: int, d_v: int) -> int:
    return 2 * B * s_q * H * d_c * d_v


def out_proj_bytes(B: int, s_q: int, H: int, d_c: int, d_v: int, b: int = 2) -> int:
    """o_lat read, W_UV read once, out written."""
    return b * (B * s_q * H * d_c + H * d_c * d_v + B * s_q * H * d_v)


def naive_flops(H: int, d_c: int, d_rope: int, d_nope: int, d_v: int, seq_lens, s_q: int) -> int:
    """Decompress every cached token per head, then attend with per-head K (d_nope + d_rope) and V (d_v)."""
    tokens = sum(int(L) for L in seq_lens)
    pairs = sum(visible_pairs(int(L), s_q) for L in seq_lens)
    return tokens * decompress_flops_per_token(H, d_c, d_nope, d_v) + pairs * H * 2 * (d_nope + d_rope + d_v)


def log_sum_exp(xs) -> float:
    m = max(xs)
    return m + math.log(sum(math.exp(x - m) for x in xs))
