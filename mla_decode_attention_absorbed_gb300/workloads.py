"""Seeded synthetic workloads for MLA decode.

This module only draws random inputs and describes shapes; it holds none of
the method's arithmetic.  The tests, the benchmark and the smoke check all take
their inputs from here, so the CUDA path and the CPU oracle see the very same
bf16 buffers.

Recipe (one CPU ``torch.Generator`` seeded with ``cfg.seed``; draws in this order):
  1. ragged configs only: sequence lengths, uniform integers in [len_lo, len_hi];
  2. q_nope [B, s_q, H, d_nope]   ~ N(0, 1)
  3. q_rope [B, s_q, H, d_rope]   ~ N(0, 1)
  4. latent cache rows [c_kv | k_rope] ~ N(0, 1): contiguous [B, T_max, d_c + d_rope],
     or a pool [P, page, d_c + d_rope] with P = sum_b ceil(L_b / page);
  5. W_UK [H, d_c, d_nope]        ~ N(0, 1 / d_c)
  6. W_UV [H, d_c, d_v]           ~ N(0, 1 / d_c)
  7. paged configs only: a permutation of the pool's pages, dealt to the
     sequences in order to build the block table.
Every draw is fp32 ``randn`` rounded to bf16 (round-to-nearest-even).  Cache rows
no sequence may read (tokens at or beyond a sequence's length) are set to NaN so
that any read of them shows up in the outputs; unused block-table entries are -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class MLAConfig:
    name: str
    B: int
    H: int
    d_c: int
    d_rope: int
    d_nope: int
    d_v: int
    s_q: int
    T: int = 0                 # fixed length of every sequence (when len_lo == 0)
    len_lo: int = 0            # ragged lengths: uniform in [len_lo, len_hi]
    len_hi: int = 0
    paged: bool = False
    page_size: int = 64
    seed: int = 0
    canary: bool = True        # NaN in cache rows nobody may read

    @property
    def scale(self) -> float:
        """1 / sqrt(d_nope + d_rope): the query-key width before absorption."""
        return 1.0 / math.sqrt(self.d_nope + self.d_rope)

    @property
    def W(self) -> int:
        return self.d_c + self.d_rope

    def with_(self, **kw) -> "MLAConfig":
        return replace(self, **kw)


_DSV3 = dict(H=128, d_c=512, d_rope=64, d_nope=128, d_v=128)

CONFIGS = {
    # correctness case the oracle finishes in well under a second
    "tiny": MLAConfig("tiny", B=2, H=16, d_c=64, d_rope=16, d_nope=32, d_v=32, s_q=1, T=128),
    # DeepSeek-V3-shaped layer, the headline decode case
    "dsv3": MLAConfig("dsv3", B=64, s_q=1, T=4096, **_DSV3),
    # long context
    "long": MLAConfig("long", B=16, s_q=1, T=32768, **_DSV3),
    # speculative verify: 3 drafts + bonus, causal among the 4
    "spec": MLAConfig("spec", B=64, s_q=4, T=8192, **_DSV3),
    # sparse top-k decode: long histories, k = 2048 listed tokens per query token
    "sparse": MLAConfig("sparse", B=64, s_q=1, T=32768, **_DSV3),
    # prefill: one 4096-token prompt (every token new), and a 512-token chunk after
    # 3584 cached tokens (above the crossover S* ~ 142 at L = 4096)
    "prefill": MLAConfig("prefill", B=1, s_q=4096, T=4096, **_DSV3),
    "chunk": MLAConfig("chunk", B=1, s_q=512, T=4096, **_DSV3),
    # ragged lengths over a shuffled paged pool
    "ragged_paged": MLAConfig("ragged_paged", B=128, s_q=2, len_lo=512, len_hi=16384, paged=True,
                              page_size=64, **_DSV3),
}


def _randn_bf16(g: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def draw_lengths(cfg: MLAConfig, g: torch.Generator) -> torch.Tensor:
    if cfg.len_lo:
        return torch.randint(cfg.len_lo, cfg.len_hi + 1, (cfg.B,), generator=g, dtype=torch.int64).to(torch.int32)
    return torch.full((cfg.B,), cfg.T, dtype=torch.int32)


def make_inputs(cfg: MLAConfig, seq_lens=None) -> dict:
    """CPU tensors for one decode step of ``cfg``.

    ``seq_lens`` (optional) overrides the drawn lengths (tests of edge cases).
    Returns q_nope, q_rope, kv, w_uk, w_uv, seq_lens (int32), block_table (int32 or
    None), page_size, T_max (contiguous capacity per sequence)."""
    g = torch.Generator().manual_seed(cfg.seed)
    drawn = draw_lengths(cfg, g)
    lens = drawn if seq_lens is None else torch.as_tensor(seq_lens, dtype=torch.int32).clone()
    B, s_q, H = cfg.B, cfg.s_q, cfg.H
    q_nope = _randn_bf16(g, (B, s_q, H, cfg.d_nope))
    q_rope = _randn_bf16(g, (B, s_q, H, cfg.d_rope))
    if cfg.paged:
        ps = cfg.page_size
        pages_per_seq = [max(1, -(-int(L) // ps)) for L in lens.tolist()]
        n_pages = sum(pages_per_seq)
        kv = _randn_bf16(g, (n_pages, ps, cfg.W))
    else:
        t_max = max(int(cfg.T), int(lens.max().item()) if B else 0, 1)
        kv = _randn_bf16(g, (B, t_max, cfg.W))
    w_uk = _randn_bf16(g, (H, cfg.d_c, cfg.d_nope), std=1.0 / math.sqrt(cfg.d_c))
    w_uv = _randn_bf16(g, (H, cfg.d_c, cfg.d_v), std=1.0 / math.sqrt(cfg.d_c))
    block_table = None
    if cfg.paged:
        perm = torch.randperm(n_pages, generator=g).to(torch.int32)
        max_pages = max(pages_per_seq) if B else 1
        block_table = torch.full((B, max_pages), -1, dtype=torch.int32)
        off = 0
        for b, n in enumerate(pages_per_seq):
            block_table[b, :n] = perm[off:off + n]
            off += n
    if cfg.canary:
        nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
        if cfg.paged:
            ps = cfg.page_size
            for b, L in enumerate(lens.tolist()):
                n = max(1, -(-L // ps))
                tail = L - (n - 1) * ps
                if tail < ps:
                    kv[int(block_table[b, n - 1]), max(tail, 0):] = nan
        else:
            for b, L in enumerate(lens.tolist()):
                kv[b, max(L, 0):] = nan
    return dict(q_nope=q_nope, q_rope=q_rope, kv=kv, w_uk=w_uk, w_uv=w_uv, seq_lens=lens,
                block_table=block_table, page_size=cfg.page_size,
                T_max=(kv.shape[1] if not cfg.paged else block_table.shape[1] * cfg.page_size))


# Scale of the FP8 latent-cache workloads: codes hold value / 2^-4, so the
# N(0, 1) values of the drawn cache use E4M3's range (max 448) without clipping.
KV_FP8_SCALE = 1.0 / 16.0


def to_fp8_cache(kv: torch.Tensor, kv_scale: float = KV_FP8_SCALE) -> torch.Tensor:
    """E4M3 codes (uint8, same shape) of a drawn bf16 cache, for the FP8-cache
    workloads: each value divided by ``kv_scale`` and cast by torch's
    float8_e4m3fn conversion (round to nearest even); NaN canaries stay NaN."""
    return (kv.to(torch.float32) / kv_scale).to(torch.float8_e4m3fn).view(torch.uint8)


def make_append_inputs(cfg: MLAConfig, d_model: int, seed: int = 7) -> dict:
    """Inputs of the cache-append step (latent down-projection of the new tokens).

    One CPU generator seeded with ``seed``; draws in this order, each fp32
    ``randn`` rounded to bf16:
      1. x [B, s_q, d_model]      ~ N(0, 1)        (the new tokens' hidden states)
      2. W_DKV [d_model, d_c]     ~ N(0, 1 / d_model)
      3. k_rope [B, s_q, d_rope]  ~ N(0, 1)        (their RoPE keys, already rotated)"""
    g = torch.Generator().manual_seed(seed)
    x = _randn_bf16(g, (cfg.B, cfg.s_q, d_model))
    w_dkv = _randn_bf16(g, (d_model, cfg.d_c), std=1.0 / math.sqrt(d_model))
    k_rope = _randn_bf16(g, (cfg.B, cfg.s_q, cfg.d_rope))
    return dict(x=x, w_dkv=w_dkv, k_rope=k_rope, d_model=d_model)


def make_sparse_indices(cfg: MLAConfig, seq_lens: torch.Tensor, topk: int, seed: int = 13) -> torch.Tensor:
    """Top-k token lists of the sparse decode, int32 [B, s_q, topk].

    Stands in for a learned selector (which needs trained weights): for every
    sequence b and query token i, ``topk`` distinct positions drawn uniformly
    from the tokens it may see (0 .. L_b - s_q + i), listed in increasing order;
    when fewer are visible, all of them, padded with -1.  One CPU generator
    seeded with ``seed``; one ``randperm`` per (b, i) in that order."""
    g = torch.Generator().manual_seed(seed)
    out = torch.full((cfg.B, cfg.s_q, topk), -1, dtype=torch.int32)
    for b in range(cfg.B):
        L = int(seq_lens[b])
        for i in range(cfg.s_q):
            n_vis = max(0, L - cfg.s_q + i + 1)
            if n_vis == 0:
                continue
            pick = torch.randperm(n_vis, generator=g)[:topk]
            pick, _ = torch.sort(pick)
            out[b, i, : pick.numel()] = pick.to(torch.int32)
    return out

