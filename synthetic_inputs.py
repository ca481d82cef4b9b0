"""Seeded synthetic inputs for the InfLLM v2 sparse-attention path.

This module is shared by the fp64 oracle (``oracle/``) and by the CUDA path's
tests and benchmark.  It only *draws* data: it holds none of the method's
arithmetic (no kernel means, no scores, no selection, no attention).

Workloads restate the five synthetic configurations that the benchmark and the
parity tests use (MiniCPM4 technical report, "InfLLM v2" section: KV blocks of
m tokens, semantic kernels of size p and stride s, GQA groups of 16 heads).
All tensors are produced as bf16 bit patterns (``uint16``) so that both sides
consume bit-identical inputs: the oracle widens them exactly to float64, the
GPU path views them as ``torch.bfloat16``.

Recipe (per workload, one ``numpy.random.Generator(PCG64(seed))``):
  1. Q, K, V drawn as float32 ``standard_normal`` with shapes
     Q [B, n_q, Hq, d], K/V [B, Hkv, L, d], in that order.
  2. Q is rounded to bf16 (round to nearest, ties to even).
  3. Planted blocks: per (b, h_kv), ``n_planted`` blocks are chosen uniformly
     without replacement among the blocks that are never forced for any of the
     queries (block index in [n_init, c_first - n_local + 1), c_first being
     the block of the first query), unless the workload fixes them.  Every key
     of a planted block gets + ``plant_gain`` * u, u the unit vector along the
     mean of that group's bf16 queries (over its 16 heads and n_q tokens).
  4. Optional AR(1) drift (x_t = rho x_{t-1} + sigma e_t, x_{-1} = 0), drawn
     as float32 normals of shape [2, B, Hkv, L, d] and added to K (index 0)
     and V (index 1), computed in float32 with separate multiply and add.
  5. K and V are summed in float64 (base + plant + drift) and rounded once to
     bf16.
"""

from __future__ import annotations

import dataclasses
import hashlib

import numpy as np

HEAD_DIM = 128
GROUP = 16
BLOCK = 64
KERNEL = 32
STRIDE = 16


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, selection settings and data recipe."""

    name: str
    batch: int
    n_kv_heads: int
    kv_len: int          # L, including the n_q query tokens themselves
    n_q: int             # query tokens per sequence (positions L-n_q .. L-1)
    topk: int
    topk_includes_forced: bool
    seed: int
    n_planted: int = 0
    planted_blocks: tuple | None = None   # fixed planted blocks (same for all b, h)
    plant_gain: float = 3.0
    drift_rho: float = 0.0
    drift_sigma: float = 0.0
    n_init: int = 1
    n_local: int = 2
    group: int = GROUP
    head_dim: int = HEAD_DIM
    block: int = BLOCK
    kernel: int = KERNEL
    stride: int = STRIDE

    @property
    def n_heads(self) -> int:
        return self.n_kv_heads * self.group

    @property
    def k_max(self) -> int:
        """Width of the block-index output rows."""
        if self.topk_includes_forced:
            return self.topk
        return self.topk + self.n_init + self.n_local

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads (decode 4K, decode 32K, decode 128K, prefill 32K,
# speculative verify at 128K).  Sizes follow the configurations the
# benchmark and parity suite are quoted on.
WORKLOADS = {
    "decode_4k": Workload("decode_4k", batch=1, n_kv_heads=1, kv_len=4096, n_q=1,
                          topk=16, topk_includes_forced=True, seed=0, n_planted=8),
    "decode_32k": Workload("decode_32k", batch=8, n_kv_heads=2, kv_len=32768, n_q=1,
                           topk=64, topk_includes_forced=True, seed=1, n_planted=32),
    "decode_128k": Workload("decode_128k", batch=4, n_kv_heads=2, kv_len=131072, n_q=1,
                            topk=64, topk_includes_forced=True, seed=2, n_planted=64,
                            drift_rho=0.99, drift_sigma=0.1),
    "prefill_32k": Workload("prefill_32k", batch=1, n_kv_heads=2, kv_len=32768, n_q=32768,
                            topk=64, topk_includes_forced=False, seed=3,
                            planted_blocks=tuple(32 * n for n in range(16))),
    "verify_128k": Workload("verify_128k", batch=4, n_kv_heads=2, kv_len=131080, n_q=8,
                            topk=64, topk_includes_forced=True, seed=4, n_planted=64,
                            drift_rho=0.99, drift_sigma=0.1),
}


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns exactly to float64."""
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


@dataclasses.dataclass
class Inputs:
    """bf16 bit patterns (uint16) of one workload's tensors plus metadata."""

    wl: Workload
    q: np.ndarray        # [B, n_q, Hq, d] uint16
    k: np.ndarray        # [B, Hkv, L, d] uint16
    v: np.ndarray        # [B, Hkv, L, d] uint16
    kv_lens: np.ndarray  # [B] int32
    planted: np.ndarray  # [B, Hkv, n_planted] int64 (block indices)

    def sha256(self) -> dict:
        return {name: hashlib.sha256(getattr(self, name).tobytes()).hexdigest()[:16]
                for name in ("q", "k", "v")}


def _ar1(eps: np.ndarray, rho: float, sigma: float) -> np.ndarray:
    """AR(1) along axis -2 (the sequence axis) of float32 normals."""
    out = np.empty_like(eps)
    rho32 = np.float32(rho)
    sig32 = np.float32(sigma)
    prev = np.zeros(eps.shape[:-2] + eps.shape[-1:], dtype=np.float32)
    for t in range(eps.shape[-2]):
        cur = np.multiply(prev, rho32)
        cur = np.add(cur, np.multiply(eps[..., t, :], sig32))
        out[..., t, :] = cur
        prev = cur
    return out


def make_inputs(wl: Workload) -> Inputs:
    """Draw one workload's inputs following the recipe in the module docstring."""
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    B, Hkv, L, d, nq, G = wl.batch, wl.n_kv_heads, wl.kv_len, wl.head_dim, wl.n_q, wl.group
    q32 = rng.standard_normal((B, nq, Hkv * G, d), dtype=np.float32)
    k32 = rng.standard_normal((B, Hkv, L, d), dtype=np.float32)
    v32 = rng.standard_normal((B, Hkv, L, d), dtype=np.float32)
    q = bf16_bits_from_f32(q32)
    del q32
    qf = bf16_bits_to_f64(q)

    m = wl.block
    n_blocks = -(-L // m)
    if wl.planted_blocks is not None:
        planted = np.broadcast_to(np.asarray(wl.planted_blocks, dtype=np.int64),
                                  (B, Hkv, len(wl.planted_blocks))).copy()
        planted = planted[..., planted[0, 0] < n_blocks] if planted.size else planted
    else:
        c_first = (L - nq) // m
        lo, hi = wl.n_init, c_first - wl.n_local + 1
        pool = np.arange(lo, max(lo, hi), dtype=np.int64)
        n_pl = min(wl.n_planted, pool.size)
        planted = np.zeros((B, Hkv, n_pl), dtype=np.int64)
        for b in range(B):
            for h in range(Hkv):
                planted[b, h] = np.sort(rng.choice(pool, size=n_pl, replace=False))

    drift = None
    if wl.drift_sigma > 0.0:
        eps = rng.standard_normal((2, B, Hkv, L, d), dtype=np.float32)
        drift = _ar1(eps, wl.drift_rho, wl.drift_sigma)
        del eps

    k = np.empty((B, Hkv, L, d), dtype=np.uint16)
    v = np.empty((B, Hkv, L, d), dtype=np.uint16)
    for b in range(B):
        for h in range(Hkv):
            kb = k32[b, h].astype(np.float64)
            vb = v32[b, h].astype(np.float64)
            if planted.shape[-1] > 0 and wl.plant_gain != 0.0:
                mean_q = qf[b, :, h * G:(h + 1) * G, :].reshape(-1, d).mean(axis=0)
                u = mean_q / np.linalg.norm(mean_q)
                for j in planted[b, h]:
                    kb[j * m:min((j + 1) * m, L)] += wl.plant_gain * u
            if drift is not None:
                kb += drift[0, b, h]
                vb += drift[1, b, h]
            k[b, h] = bf16_bits_from_f32(kb.astype(np.float32))
            v[b, h] = bf16_bits_from_f32(vb.astype(np.float32))
    kv_lens = np.full((B,), L, dtype=np.int32)
    return Inputs(wl=wl, q=q, k=k, v=v, kv_lens=kv_lens, planted=planted)


def make_random(batch: int, n_kv_heads: int, kv_len: int, n_q: int, topk: int,
                includes_forced: bool = True, seed: int = 0, kv_lens=None,
                max_kv_len: int | None = None, n_init: int = 1, n_local: int = 2,
                scale_k: float = 1.0) -> Inputs:
    """Small iid-normal inputs for parity tests (ragged lengths allowed).

    ``kv_lens`` (per batch entry) may be shorter than ``kv_len``, which is then
    the cache capacity; entries past a sequence's length are filled with
    large finite garbage so that a kernel reading them would be caught.
    """
    wl = Workload(f"random_{seed}", batch=batch, n_kv_heads=n_kv_heads,
                  kv_len=max_kv_len or kv_len, n_q=n_q, topk=topk,
                  topk_includes_forced=includes_forced, seed=seed,
                  n_init=n_init, n_local=n_local)
    rng = np.random.Generator(np.random.PCG64(seed))
    cap = wl.kv_len
    d, G = wl.head_dim, wl.group
    q = bf16_bits_from_f32(rng.standard_normal((batch, n_q, n_kv_heads * G, d), dtype=np.float32))
    k32 = rng.standard_normal((batch, n_kv_heads, cap, d), dtype=np.float32) * np.float32(scale_k)
    v32 = rng.standard_normal((batch, n_kv_heads, cap, d), dtype=np.float32)
    lens = np.full((batch,), kv_len, dtype=np.int32) if kv_lens is None else np.asarray(kv_lens, dtype=np.int32)
    for b in range(batch):
        k32[b, :, lens[b]:, :] = 1.0e4
        v32[b, :, lens[b]:, :] = -1.0e4
    return Inputs(wl=wl, q=q, k=bf16_bits_from_f32(k32), v=bf16_bits_from_f32(v32),
                  kv_lens=lens, planted=np.zeros((batch, n_kv_heads, 0), dtype=np.int64))


def make_grad_out(wl: Workload, seed: int) -> np.ndarray:
    """Upstream gradient for the backward pass: bf16 bits of float32
    ``standard_normal`` [B, n_q, Hq, d] from its own PCG64(seed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return bf16_bits_from_f32(rng.standard_normal((wl.batch, wl.n_q, wl.n_heads, wl.head_dim), dtype=np.float32))


def make_block_sets(wl: Workload, kv_lens: np.ndarray, seed: int):
    """A fixed, valid block selection for backward tests at sizes where the
    selection itself is not recomputed: per (b, h_kv, t) with query position
    i = L - n_q + t and c = i // block, min(k_max, c + 1) distinct blocks in
    [0, c] that always include 0 and c, the rest drawn uniformly without
    replacement from [1, c - 1] by PCG64(seed), ascending.
    Returns (block_idx int32 [B, Hkv, n_q, k_max] padded with -1,
    n_selected int32 [B, Hkv, n_q])."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B, H, nq, km = wl.batch, wl.n_kv_heads, wl.n_q, wl.k_max
    idx = np.full((B, H, nq, km), -1, dtype=np.int32)
    nsel = np.zeros((B, H, nq), dtype=np.int32)
    for b in range(B):
        L = int(kv_lens[b])
        for h in range(H):
            for t in range(nq):
                c = (L - nq + t) // wl.block
                n = min(km, c + 1)
                if n == c + 1:
                    chosen = np.arange(c + 1)
                else:
                    rest = rng.choice(np.arange(1, c), size=n - 2, replace=False)
                    chosen = np.sort(np.concatenate(([0, c], rest)))
                idx[b, h, t, :n] = chosen
                nsel[b, h, t] = n
    return idx, nsel
