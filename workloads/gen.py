"""Workload recipes and seeded tensors.

Shapes follow the Llama-70B attention geometry of the visual appendix
("KV-Cache Offloading for LLM Inference -- Visual Reference", section 1:
80 layers, 64 query heads, 8 KV heads, head dim 128) and its 16-token
blocks; the tiny case is a 2-layer, 4:1 GQA cut used for CPU-sized checks.

Recency skew (input shaping only).  The appendix (section 6) assumes about
80 % of attention mass lands on the most recent 10 % of tokens.  To give the
synthetic inputs that shape, each (layer, KV head) gets a fixed random unit
direction u; queries are z + sqrt(d)*u with z ~ N(0, I), and keys of the
recent 10 % of the prefill, of every decode-appended token and of block 0
get +c*u.  For such a key the scaled score sigma*q.k gains c on average, so
with c = ln 36 the boosted tenth of tokens takes 0.1*36 / (0.1*36 + 0.9) =
80 % of the weight.  Nothing in the oracle or the kernels depends on this.

Every tensor is a pure function of (workload seed, content id, position or
step), generated in fixed 256-token chunks so any token range can be
regenerated on its own.  Tensors are generated on the device asked for; the
CPU and CUDA generators give different streams, so a comparison must use
tensors from one device (GPU tests copy them to the host for the oracle).
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np
import torch

CHUNK = 256          # tokens per generator chunk
BOOST_C = math.log(36.0)
_MASK64 = (1 << 64) - 1


def _mix(*vals: int) -> int:
    """splitmix64-style hash of a tuple of integers (seed derivation only)."""
    h = 0x9E3779B97F4A7C15
    for v in vals:
        h = (h ^ (v & _MASK64)) & _MASK64
        h = (h + 0x9E3779B97F4A7C15) & _MASK64
        z = h
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        h = z ^ (z >> 31)
    return h & ((1 << 63) - 1)


@dataclass(frozen=True)
class Workload:
    name: str
    L: int
    Hq: int
    Hkv: int
    d: int
    prefill_lens: tuple
    steps: int
    alphas: tuple
    skew: bool
    seed: int
    block_tokens: int = 16
    shared_prefix_tokens: int = 0
    pool_pages: int = 0
    demote_every: int = 0
    demote_frac: float = 0.0
    recency_window: int = 64
    weights: tuple = (0.25, 0.55, 0.20)
    cuts: tuple = (0.3, 0.6)
    meta: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def nseq(self) -> int:
        return len(self.prefill_lens)

    @property
    def token_bytes(self) -> int:
        """K and V bytes of one token over all layers and KV heads (bf16)."""
        return 2 * self.L * self.Hkv * self.d * 2

    @property
    def page_bytes(self) -> int:
        return self.token_bytes * self.block_tokens

    def max_blocks_per_seq(self) -> int:
        B = self.block_tokens
        return max((n + self.steps + B - 1) // B for n in self.prefill_lens) + 1

    def unique_blocks_needed(self) -> int:
        """Physical pages the run needs if nothing is evicted."""
        B = self.block_tokens
        total = sum((n + self.steps + B - 1) // B for n in self.prefill_lens)
        shared = self.shared_prefix_tokens // B
        return total - shared * (self.nseq - 1)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _lens_uniform(seed: int, n: int, lo: int, hi: int, multiple: int) -> tuple:
    rng = np.random.Generator(np.random.PCG64(seed))
    raw = rng.integers(lo, hi + 1, size=n)
    if multiple > 1:
        raw = (raw // multiple) * multiple
    return tuple(int(x) for x in raw)


def _build() -> dict:
    base = 0x6B76
    w = {}
    w["tiny"] = Workload(
        name="tiny", L=2, Hq=8, Hkv=2, d=64, prefill_lens=(256,), steps=4,
        alphas=(0.15,), skew=False, seed=base + 0, pool_pages=17)
    w["l70b_8k"] = Workload(
        name="l70b_8k", L=80, Hq=64, Hkv=8, d=128, prefill_lens=(8192,),
        steps=32, alphas=(0.15,), skew=True, seed=base + 1, pool_pages=514)
    lens3 = _lens_uniform(base + 2, 16, 1024, 8192, 16)
    wl3 = Workload(
        name="l70b_batch16", L=80, Hq=64, Hkv=8, d=128, prefill_lens=lens3,
        steps=16, alphas=(0.01, 0.15), skew=True, seed=base + 2,
        shared_prefix_tokens=1024)
    w["l70b_batch16"] = wl3.with_(pool_pages=wl3.unique_blocks_needed() + 16)
    w["l70b_128k"] = Workload(
        name="l70b_128k", L=80, Hq=64, Hkv=8, d=128, prefill_lens=(131072,),
        steps=64, alphas=(0.01, 0.05, 0.15), skew=True, seed=base + 3,
        pool_pages=8192 + 8)
    lens5 = _lens_uniform(base + 4, 32, 4096, 16384, 1)
    B = 16
    need5 = sum((n + 32 + B - 1) // B for n in lens5)
    w["l70b_mixed32"] = Workload(
        name="l70b_mixed32", L=80, Hq=64, Hkv=8, d=128, prefill_lens=lens5,
        steps=32, alphas=(0.05,), skew=True, seed=base + 4,
        pool_pages=int(math.ceil(1.10 * need5)), demote_every=8,
        demote_frac=0.10)
    return w


WORKLOADS = _build()


def workload(name: str, **overrides) -> Workload:
    wl = WORKLOADS[name]
    return wl.with_(**overrides) if overrides else wl


def unit_dirs(wl: Workload) -> np.ndarray:
    """Fixed unit direction per (layer, KV head): float32 [L][Hkv][d]."""
    rng = np.random.Generator(np.random.PCG64(_mix(wl.seed, 0x75)))
    u = rng.standard_normal((wl.L, wl.Hkv, wl.d))
    u /= np.linalg.norm(u, axis=-1, keepdims=True)
    return u.astype(np.float32)


def _content_id(wl: Workload, seq: int, pos: int) -> int:
    return 0 if pos < wl.shared_prefix_tokens else seq


def _boosted(wl: Workload, seq: int, pos: torch.Tensor) -> torch.Tensor:
    n = wl.prefill_lens[seq]
    recent_from = max((9 * n) // 10, wl.shared_prefix_tokens)
    return (pos < wl.block_tokens) | (pos >= recent_from)


def _chunk(wl: Workload, cid: int, chunk: int, device) -> tuple:
    shape = (CHUNK, wl.L, wl.Hkv, wl.d)
    gk = torch.Generator(device=device)
    gk.manual_seed(_mix(wl.seed, cid, chunk, 1))
    k = torch.randn(shape, generator=gk, device=device, dtype=torch.float32)
    gv = torch.Generator(device=device)
    gv.manual_seed(_mix(wl.seed, cid, chunk, 2))
    v = torch.randn(shape, generator=gv, device=device, dtype=torch.float32)
    return k, v


def kv_tokens(wl: Workload, seq: int, p0: int, p1: int, device="cpu") -> tuple:
    """K, V of sequence `seq` for token positions [p0, p1).

    Returns two bf16 tensors [p1-p0][L][Hkv][d] (token-major, the order in
    which tokens are appended).
    """
    assert 0 <= p0 <= p1
    n = p1 - p0
    K = torch.empty((n, wl.L, wl.Hkv, wl.d), dtype=torch.bfloat16, device=device)
    V = torch.empty_like(K)
    if n == 0:
        return K, V
    u = torch.from_numpy(unit_dirs(wl)).to(device) if wl.skew else None
    c0, c1 = p0 // CHUNK, (p1 - 1) // CHUNK
    for c in range(c0, c1 + 1):
        a, b = max(p0, c * CHUNK), min(p1, (c + 1) * CHUNK)
        pos = torch.arange(a, b, device=device)
        lo, hi = a - c * CHUNK, b - c * CHUNK
        cid_a, cid_b = _content_id(wl, seq, a), _content_id(wl, seq, b - 1)
        kk, vv = _chunk(wl, cid_a, c, device)
        kk, vv = kk[lo:hi], vv[lo:hi]
        if cid_b != cid_a:  # chunk straddles the end of a shared prefix
            k1, v1 = _chunk(wl, cid_b, c, device)
            sel = (pos < wl.shared_prefix_tokens).view(-1, 1, 1, 1)
            kk = torch.where(sel, kk, k1[lo:hi])
            vv = torch.where(sel, vv, v1[lo:hi])
        if wl.skew:
            m = _boosted(wl, seq, pos).to(torch.float32).view(-1, 1, 1, 1)
            kk = kk + m * (BOOST_C * u).unsqueeze(0)
        K[a - p0:b - p0] = kk.to(torch.bfloat16)
        V[a - p0:b - p0] = vv.to(torch.bfloat16)
    return K, V


def kv_stream(wl: Workload, seq: int, l: int, g: int, p0: int, p1: int,
              device="cpu") -> tuple:
    """K, V of one (layer, KV head) stream: bf16 [p1-p0][d] each."""
    K, V = kv_tokens(wl, seq, p0, p1, device)
    return K[:, l, g, :].contiguous(), V[:, l, g, :].contiguous()


def queries(wl: Workload, seq: int, step: int, device="cpu") -> torch.Tensor:
    """Query of sequence `seq` at decode step `step` (1-based): bf16 [L][Hq][d]."""
    g = torch.Generator(device=device)
    g.manual_seed(_mix(wl.seed, seq, step, 3))
    q = torch.randn((wl.L, wl.Hq, wl.d), generator=g, device=device,
                    dtype=torch.float32)
    if wl.skew:
        u = torch.from_numpy(unit_dirs(wl)).to(device)
        q = q + math.sqrt(wl.d) * u.repeat_interleave(wl.G, dim=1)
    return q.to(torch.bfloat16)


def synthetic_masses(seed: int, nb: int) -> np.ndarray:
    """Seeded positive fp32 per-block masses for driving the scoring step
    directly (tests that bypass attention).  About a third of the blocks
    sit on the uniform share 1/nb exactly, the rest are spread around it."""
    rng = np.random.Generator(np.random.PCG64(_mix(seed, nb, 9)))
    x = rng.exponential(1.0, size=nb) / nb
    exact = rng.random(nb) < 0.33
    x = np.where(exact, 1.0 / nb, x)
    return x.astype(np.float32)
