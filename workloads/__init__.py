"""Seeded synthetic inputs for long-context decode attention.

Shared by the tests, the smoke check and the benchmark; used by both the CUDA
path and the CPU oracle.  It holds none of the method's arithmetic: only random
draws, the bf16 rounding of those draws (round to nearest even, by torch), the
structured score peaks that the workload recipes ask for, and page-table
layout.

Workload recipes (decode of one new token per sequence):
  tiny        B=1, Hq=Hkv=1, d=64, L=1024, scale 1/8, 4 splits, fp32 output
  mha32k      B=1, Hq=Hkv=32, d=128, L=32768, scale 1/sqrt(128), auto splits
  gqa_paged   B=8, Hq=64, Hkv=8, d=128, L_b ~ U{16384..131072}, 64-token pages
              placed by a seeded random permutation
  million     B=1, Hq=32, Hkv=8, d=128, L=1048576; keys of tokens 0-3 get
              +3*q_hat (attention sinks)
  ffd         B=4, Hq=32, Hkv=8, d=128, L=131072; keys of tokens 0-3 and of
              the last 64 tokens get +2.5*q_hat; round(1% of L) distinct
              tokens in [4, L-64) get +c*q_hat with c ~ N(2, 0.5) each
  ladder      any B and L at Hq=32, Hkv=8, d=128, unstructured (the
              context-length ladder of the split-count sweep)
q, K, V ~ N(0, 1) in fp32, structure added in fp32, then rounded to bf16.
q_hat for KV head h is u/|u| with u the sum of the group's query vectors
(after their bf16 rounding), so one direction serves all heads of the group.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

PAGE_SIZE = 64


@dataclass
class Problem:
    """One decode call's inputs (device tensors) and its configuration."""
    name: str
    q: torch.Tensor                      # [B, Hq, d] bf16
    k: Optional[torch.Tensor]            # [B, Hkv, L_max, d] bf16 (contiguous cache)
    v: Optional[torch.Tensor]
    seq_lens: torch.Tensor               # [B] int32
    scale: float
    L_max: int
    num_splits: int = 0                  # 0 = planner's choice
    out_dtype: str = "bf16"              # "bf16" or "f32"
    k_pages: Optional[torch.Tensor] = None   # [P, Hkv, page_size, d] bf16
    v_pages: Optional[torch.Tensor] = None
    page_table: Optional[torch.Tensor] = None  # [B, max_pages] int32 (-1 = unused)
    num_pages: int = 0
    page_size: int = PAGE_SIZE
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def d(self):
        return self.q.shape[2]

    @property
    def Hkv(self):
        t = self.k if self.k is not None else self.k_pages
        return t.shape[1]

    @property
    def paged(self):
        return self.k_pages is not None

    def kv_tokens(self) -> int:
        """Sum over sequences of the cached tokens."""
        return int(self.seq_lens.to(torch.int64).sum().item())


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def group_direction(q_bf16: torch.Tensor, Hkv: int) -> torch.Tensor:
    """q_hat [B, Hkv, d] (fp32): normalised sum of each group's query vectors."""
    B, Hq, d = q_bf16.shape
    G = Hq // Hkv
    u = q_bf16.float().reshape(B, Hkv, G, d).sum(dim=2)
    return u / u.norm(dim=-1, keepdim=True)


def random_problem(B, Hq, Hkv, L_max, d, seed=0, device="cpu", seq_lens=None, scale=None,
                   num_splits=0, out_dtype="bf16", name="random", std=1.0):
    """Unstructured q, K, V ~ N(0, std^2) rounded to bf16."""
    g = _gen(seed, device)
    q = (_randn((B, Hq, d), g, device) * std).to(torch.bfloat16)
    k = (_randn((B, Hkv, L_max, d), g, device) * std).to(torch.bfloat16)
    v = _randn((B, Hkv, L_max, d), g, device).to(torch.bfloat16)
    if seq_lens is None:
        sl = torch.full((B,), L_max, dtype=torch.int32, device=device)
    else:
        sl = torch.as_tensor(seq_lens, dtype=torch.int32).to(device)
    return Problem(name, q, k, v, sl, scale if scale is not None else 1.0 / math.sqrt(d), L_max,
                   num_splits=num_splits, out_dtype=out_dtype)


def _structured_keys(q, B, Hkv, L, d, g, device, boosts):
    """K ~ N(0,1) with `boosts(b, h) -> (positions LongTensor, coefficients fp32 Tensor)`
    added along q_hat[b, h] before the bf16 rounding.  Built one (b, h) slab at a time."""
    qh = group_direction(q, Hkv)
    k = torch.empty((B, Hkv, L, d), dtype=torch.bfloat16, device=device)
    for b in range(B):
        for h in range(Hkv):
            slab = _randn((L, d), g, device)
            pos, coef = boosts(b, h)
            if pos is not None and pos.numel():
                slab[pos] += coef[:, None] * qh[b, h][None, :]
            k[b, h] = slab.to(torch.bfloat16)
    return k


def _values(B, Hkv, L, d, g, device):
    v = torch.empty((B, Hkv, L, d), dtype=torch.bfloat16, device=device)
    for b in range(B):
        for h in range(Hkv):
            v[b, h] = _randn((L, d), g, device).to(torch.bfloat16)
    return v


def tiny(seed=0, device="cpu") -> Problem:
    p = random_problem(1, 1, 1, 1024, 64, seed=seed, device=device, scale=1.0 / 8.0,
                       num_splits=4, out_dtype="f32", name="tiny")
    return p


def mha32k(seed=0, device="cpu", L=32768) -> Problem:
    return random_problem(1, 32, 32, L, 128, seed=seed, device=device,
                          scale=1.0 / math.sqrt(128), name="mha32k")


def million(seed=0, device="cpu", L=1 << 20) -> Problem:
    B, Hq, Hkv, d = 1, 32, 8, 128
    g = _gen(seed, device)
    q = _randn((B, Hq, d), g, device).to(torch.bfloat16)
    sinks = torch.arange(0, min(4, L), device=device)
    three = torch.full((sinks.numel(),), 3.0, device=device)
    k = _structured_keys(q, B, Hkv, L, d, g, device, lambda b, h: (sinks, three))
    v = _values(B, Hkv, L, d, g, device)
    sl = torch.full((B,), L, dtype=torch.int32, device=device)
    return Problem("million", q, k, v, sl, 1.0 / math.sqrt(d), L)


def ffd(seed=0, device="cpu", B=4, L=131072, Hq=32, Hkv=8, d=128, anchor_boost=2.5, plant_mean=2.0,
        plant_std=0.5, plant_frac=0.01) -> Problem:
    """The FFD recipe; the keyword arguments after d change it into a sparser
    cache (e.g. anchor_boost=20, plant_mean=20, plant_frac=0.001: the anchors
    and the planted tokens score ~13 units above the rest at G=4, so at
    delta 5 the candidates are those tokens alone, and the 64-token tiles
    holding one are ~1 - (1 - plant_frac)^64 of the cache)."""
    g = _gen(seed, device)
    q = _randn((B, Hq, d), g, device).to(torch.bfloat16)
    n_planted = int(round(plant_frac * L))
    anchors = torch.cat([torch.arange(0, min(4, L), device=device),
                         torch.arange(max(0, L - 64), L, device=device)]).unique()
    anchor_coef = torch.full((anchors.numel(),), float(anchor_boost), device=device)
    lo, hi = 4, L - 64

    def boosts(b, h):
        if hi > lo and n_planted > 0:
            pl = torch.randperm(hi - lo, generator=g, device=device)[:n_planted] + lo
            c = plant_mean + plant_std * _randn((pl.numel(),), g, device)
            return torch.cat([anchors, pl]), torch.cat([anchor_coef, c])
        return anchors, anchor_coef

    k = _structured_keys(q, B, Hkv, L, d, g, device, boosts)
    v = _values(B, Hkv, L, d, g, device)
    sl = torch.full((B,), L, dtype=torch.int32, device=device)
    return Problem("ffd", q, k, v, sl, 1.0 / math.sqrt(d), L,
                   meta=dict(n_sink=4, window=64, deltas=(5.0, 7.0), n_planted=n_planted))


def ladder(B=1, L=32768, seed=0, device="cpu", Hq=32, Hkv=8, d=128) -> Problem:
    """Context-length ladder shape (GQA group of 4, d=128) at any batch and
    length: unstructured q, K, V ~ N(0,1) rounded to bf16, drawn one
    (sequence, head) slab at a time so that large caches need no fp32 copy."""
    g = _gen(seed, device)
    q = _randn((B, Hq, d), g, device).to(torch.bfloat16)
    k = _structured_keys(q, B, Hkv, L, d, g, device, lambda b, h: (None, None))
    v = _values(B, Hkv, L, d, g, device)
    sl = torch.full((B,), L, dtype=torch.int32, device=device)
    return Problem("ladder", q, k, v, sl, 1.0 / math.sqrt(d), L)


def page_layout(seq_lens, page_size, g, device, max_pages=None):
    """Physical page ids for every (sequence, logical page): a seeded random
    permutation of the P = sum ceil(L_b / page_size) pages, assigned in
    (sequence, page) order.  Unused table entries are -1."""
    sl = [int(x) for x in seq_lens]
    npg = [(x + page_size - 1) // page_size for x in sl]
    P = sum(npg)
    if max_pages is None:
        max_pages = max(npg) if npg else 0
    perm = torch.randperm(P, generator=g, device=device).to(torch.int32) if P else \
        torch.empty(0, dtype=torch.int32, device=device)
    table = torch.full((len(sl), max(max_pages, 1)), -1, dtype=torch.int32, device=device)
    off = 0
    for b, n in enumerate(npg):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, P


def gqa_paged(seed=0, device="cpu", B=8, Hq=64, Hkv=8, d=128, L_min=16384, L_max=131072,
              lengths=None, page_size=PAGE_SIZE) -> Problem:
    g = _gen(seed, device)
    if lengths is None:
        lens = torch.randint(L_min, L_max + 1, (B,), generator=g, device=device)
        lengths = [int(x) for x in lens.tolist()]
    max_pages = (L_max + page_size - 1) // page_size
    table, P = page_layout(lengths, page_size, g, device, max_pages=max_pages)
    q = _randn((B, Hq, d), g, device).to(torch.bfloat16)
    kp = torch.empty((P, Hkv, page_size, d), dtype=torch.bfloat16, device=device)
    vp = torch.empty_like(kp)
    step = 1024
    for p0 in range(0, P, step):
        p1 = min(P, p0 + step)
        kp[p0:p1] = _randn((p1 - p0, Hkv, page_size, d), g, device).to(torch.bfloat16)
        vp[p0:p1] = _randn((p1 - p0, Hkv, page_size, d), g, device).to(torch.bfloat16)
    sl = torch.tensor(lengths, dtype=torch.int32, device=device)
    return Problem("gqa_paged", q, None, None, sl, 1.0 / math.sqrt(d), max_pages * page_size,
                   k_pages=kp, v_pages=vp, page_table=table, num_pages=P, page_size=page_size)


def to_paged(p: Problem, seed=1, page_size=PAGE_SIZE, identity=False, poison_tail=True) -> Problem:
    """Re-lay a contiguous problem's cache into pages (same values, same tokens).
    With poison_tail, rows past each sequence's end inside its last page are NaN,
    so any read of them shows up in the output."""
    g = _gen(seed, p.q.device)
    B, Hkv, L_max, d = p.k.shape
    lens = [int(x) for x in p.seq_lens.tolist()]
    max_pages = max(1, (L_max + page_size - 1) // page_size)
    if identity:
        npg = [(x + page_size - 1) // page_size for x in lens]
        P = sum(npg)
        table = torch.full((B, max_pages), -1, dtype=torch.int32, device=p.q.device)
        off = 0
        for b, n in enumerate(npg):
            table[b, :n] = torch.arange(off, off + n, dtype=torch.int32, device=p.q.device)
            off += n
    else:
        table, P = page_layout(lens, page_size, g, p.q.device, max_pages=max_pages)
    kp = torch.zeros((max(P, 1), Hkv, page_size, d), dtype=torch.bfloat16, device=p.q.device)
    vp = torch.zeros_like(kp)
    if poison_tail:
        kp.fill_(float("nan"))
        vp.fill_(float("nan"))
    for b, L in enumerate(lens):
        for lp in range((L + page_size - 1) // page_size):
            t0, t1 = lp * page_size, min(L, (lp + 1) * page_size)
            pid = int(table[b, lp])
            kp[pid, :, : t1 - t0] = p.k[b, :, t0:t1]
            vp[pid, :, : t1 - t0] = p.v[b, :, t0:t1]
    return Problem(p.name + "_paged", p.q, None, None, p.seq_lens, p.scale, max_pages * page_size,
                   num_splits=p.num_splits, out_dtype=p.out_dtype, k_pages=kp, v_pages=vp,
                   page_table=table, num_pages=P, page_size=page_size)


CONFIGS = {
    "tiny": tiny,
    "mha32k": mha32k,
    "gqa_paged": gqa_paged,
    "million": million,
    "ffd": ffd,
}
