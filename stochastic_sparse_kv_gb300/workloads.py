"""Seeded synthetic decode-attention inputs (shared by the tests, the benchmark and the
oracle checks).  This module only draws random tensors of the right shapes; it holds
none of the method's arithmetic.

The workloads stand in for the pages' measurement setting (Llama-3.1-8B-Instruct at
32k-token contexts, "Stochastic Sparse Attention for Memory-Bound Inference",
abstract): no weights or datasets are used, only the model's attention shape
(32 query heads, 8 KV heads, head dim 128, bf16 KV cache).

Recipe (all from ``torch.Generator('cpu').manual_seed(seed)``):
  * K, V ~ N(0, 1) in fp32, rounded to bf16, layout [B, H_kv, n_max, d].
  * q: per query head, g ~ N(0, I_d) and q = score_std * sqrt(d) * g / |g|, so that
    s = q.k / sqrt(d) has standard deviation exactly score_std for k ~ N(0, I);
    rounded to bf16, layout [B, H_q, d].  With score_std=None q ~ N(0, 1) directly.
  * heavy hitters (optional): a seeded fraction of the keys of each (b, h_kv) gets
    k += c * qbar_hat, with qbar_hat the unit mean of the G query vectors of that KV
    head and c chosen so that the group-mean score of those keys rises by
    heavy_sigmas * score_std; then re-rounded to bf16.
  * seq_lens: fixed n, or per-sequence uniform integers in [lo, hi] (ragged batch).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H_q: int
    H_kv: int
    d: int
    n_max: int
    S: int
    modes: tuple
    seq_lo: int | None = None      # ragged: seq_lens ~ U{seq_lo..seq_hi}
    seq_hi: int | None = None
    score_std: float | None = 3.0  # None: q ~ N(0,1)
    heavy_frac: float = 0.0
    heavy_sigmas: float = 3.0
    seed: int = 0

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv


# The five workloads: a tiny parity case, the Llama-shaped single sequence, the batched
# decode step the headline metric is quoted on, a ragged batch with heavy hitters, and
# a long-context sweep (one entry per context length).
TINY = Workload("tiny", 1, 1, 1, 64, 256, 16, ("systematic",), score_std=None)
LLAMA_B1 = Workload("llama8b_b1_32k", 1, 32, 8, 128, 32768, 256,
                    ("systematic", "stratified", "dense"))
BATCHED = Workload("llama8b_b16_32k", 16, 32, 8, 128, 32768, 256,
                   ("systematic", "stratified", "dense"))
RAGGED = Workload("llama8b_ragged_b32", 32, 32, 8, 128, 65536, 256, ("systematic",),
                  seq_lo=4096, seq_hi=65536, heavy_frac=0.01)
LONG = tuple(Workload(f"llama8b_b4_{n // 1024}k", 4, 32, 8, 128, n, 256,
                      ("systematic", "stratified", "dense")) for n in (8192, 32768, 131072))
BATCHED_S_SWEEP = (64, 128, 256, 512)
# A value-stage CTA keeps a head's chunk arrays in shared memory up to 4096 chunks of 32
# keys (131072 keys), or 10240 chunks (327680 keys) when the batch has at most one head
# per SM (its wide team of 1024 threads); beyond that they stay in global memory.  One
# Llama-shaped sequence of 400000 keys takes that path.
LONG_GLOBAL = Workload("llama8b_b1_400k", 1, 32, 8, 128, 400000, 256, ("systematic", "stratified", "dense"))


def seq_lens_for(w: Workload) -> torch.Tensor:
    if w.seq_lo is None:
        return torch.full((w.B,), w.n_max, dtype=torch.int32)
    g = torch.Generator("cpu").manual_seed(w.seed + 7919)
    return torch.randint(w.seq_lo, w.seq_hi + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)


def make_q(B: int, H_q: int, d: int, score_std: float | None, gen: torch.Generator) -> torch.Tensor:
    g = torch.randn(B, H_q, d, generator=gen, dtype=torch.float32)
    if score_std is not None:
        g = g.double()
        g = score_std * math.sqrt(d) * g / g.norm(dim=-1, keepdim=True)
        g = g.float()
    return g.to(torch.bfloat16)


def make_inputs(w: Workload, seed: int | None = None, device: str | torch.device = "cpu"):
    """Return (q, k_cache, v_cache, seq_lens) for a workload, all on ``device``
    (seq_lens int32).  Tensors are drawn on the CPU one batch row at a time, so that
    the same seed gives the same values on any device."""
    seed = w.seed if seed is None else seed
    gen = torch.Generator("cpu").manual_seed(seed)
    q = make_q(w.B, w.H_q, w.d, w.score_std, gen)
    shape = (w.H_kv, w.n_max, w.d)
    k = torch.empty((w.B,) + shape, dtype=torch.bfloat16, device=device)
    v = torch.empty((w.B,) + shape, dtype=torch.bfloat16, device=device)
    for b in range(w.B):
        kb = torch.randn(shape, generator=gen, dtype=torch.float32)
        if w.heavy_frac > 0:
            kb = _boost(kb, q[b].float(), w, gen)
        k[b].copy_(kb.to(torch.bfloat16))
        del kb
        v[b].copy_(torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16))
    return q.to(device), k, v, seq_lens_for(w).to(device)


def _boost(kb: torch.Tensor, qb: torch.Tensor, w: Workload, gen: torch.Generator) -> torch.Tensor:
    """Heavy-hitter keys: raise the group-mean score of a seeded 1% of the keys of each
    KV head by heavy_sigmas * score_std."""
    G, d = w.G, w.d
    std = w.score_std if w.score_std is not None else 1.0
    n_heavy = max(1, int(round(w.heavy_frac * w.n_max)))
    for g in range(w.H_kv):
        qbar = qb[g * G:(g + 1) * G].double().mean(0)
        qhat = qbar / qbar.norm()
        # scale * qbar . (c * qhat) = c * |qbar| / sqrt(d) = heavy_sigmas * std
        c = w.heavy_sigmas * std * math.sqrt(d) / float(qbar.norm())
        pick = torch.randperm(w.n_max, generator=gen)[:n_heavy]
        kb[g, pick] += (c * qhat).float()
    return kb


def make_inputs_device(w: Workload, device, seed: int | None = None):
    """The same recipe as make_inputs, drawn on `device` with a device generator: the
    same shapes and distributions (and the same seq_lens), but other random values.  For
    timing runs over large caches, where drawing on the host would take minutes."""
    seed = w.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    g = torch.randn(w.B, w.H_q, w.d, generator=gen, device=device, dtype=torch.float32)
    if w.score_std is not None:
        g = (w.score_std * math.sqrt(w.d) * g.double() / g.double().norm(dim=-1, keepdim=True)).float()
    q = g.to(torch.bfloat16)
    shape = (w.B, w.H_kv, w.n_max, w.d)
    k = torch.empty(shape, dtype=torch.bfloat16, device=device)
    v = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for b in range(w.B):
        kb = torch.randn(shape[1:], generator=gen, device=device, dtype=torch.float32)
        if w.heavy_frac > 0:
            qb = q[b].float()
            G, d = w.G, w.d
            std = w.score_std if w.score_std is not None else 1.0
            n_heavy = max(1, int(round(w.heavy_frac * w.n_max)))
            for hk in range(w.H_kv):
                qbar = qb[hk * G:(hk + 1) * G].double().mean(0)
                c = w.heavy_sigmas * std * math.sqrt(d) / float(qbar.norm())
                pick = torch.randperm(w.n_max, generator=gen, device=device)[:n_heavy]
                kb[hk, pick] += (c * qbar / qbar.norm()).float()
        k[b].copy_(kb.to(torch.bfloat16))
        v[b].copy_(torch.randn(shape[1:], generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16))
        del kb
    return q, k, v, seq_lens_for(w).to(device)


def small(name: str, B: int, H_q: int, H_kv: int, d: int, n_max: int, S: int, *,
          seq_lens=None, score_std: float | None = 3.0, heavy_frac: float = 0.0, seed: int = 0):
    """An ad-hoc small workload (parity tests): optional explicit seq_lens list."""
    w = Workload(name, B, H_q, H_kv, d, n_max, S, ("systematic", "stratified", "dense"),
                 score_std=score_std, heavy_frac=heavy_frac, seed=seed)
    q, k, v, sl = make_inputs(w)
    if seq_lens is not None:
        sl = torch.tensor(seq_lens, dtype=torch.int32)
    return w, q, k, v, sl
