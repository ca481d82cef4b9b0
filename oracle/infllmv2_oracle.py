"""Plain fp64 CPU oracle of the InfLLM v2 sparse-attention path.

TEST INFRASTRUCTURE ONLY.  This module exists to check the CUDA library.  Only
the tests, the package's smoke check and the benchmark's CPU-baseline leg may
import it; the product path never calls it and has no CPU fallback.  It shares
no code with the CUDA path: the only thing both sides use is the seeded input
generator in ``synthetic_inputs`` (which holds none of the method's arithmetic).

Source of every formula: the MiniCPM4 technical report as digested on the page
"MiniCPM4: Ultra-Efficient LLMs on End Devices" (paper-graph-ui digest), section
"InfLLM v2: Trainable Sparse Attention for Both Prefilling and Decoding",
abbreviated below as [InfLLM v2 › <paragraph>, <equation>].

Every step is written the slow, obvious way, in float64, in the order the
section gives it: kernel means -> per-head kernel softmax -> group mean ->
block max -> forced blocks -> top-k -> exact softmax attention over the chosen
blocks.  Readings of points the pages leave open:

* R1  the kernel softmax is taken over ``score_scale * q . Mean(K)``; the
      section prints no scale, so the scale is a parameter (default 1/sqrt(d),
      the same as the attention scale).
* R2  only complete kernels exist: kernel j covers keys [j s, j s + p) and the
      count is floor((L - p)/s) + 1; kernel j is visible to the query at
      position i only if all its keys are <= i.
* R3  heads are averaged at kernel level (r_group), then the block takes the
      max over the kernels that intersect it.
* R4  the forced set is the first ``n_init`` blocks plus the ``n_local`` blocks
      ending at the query's own block (block-aligned, causal).
* R5  ``includes_forced`` decides whether forced blocks count toward k; forced
      blocks that coincide free their slots for scored blocks.
* R6  equal scores are ordered by the lower block index.
* R7  the query at position i attends key i itself (inclusive causal mask);
      query t of n_q sits at position L - n_q + t.
* R10 (approximation, off by default) the coarse kernels of the LSE
      approximation are the means of non-overlapping windows of s_c keys;
      one is visible to query i once all its keys are <= i; their LSE
      replaces the fine one as each head's normaliser (a count correction
      would shift every head by the same constant and change no selection);
      before the first coarse kernel is complete the exact LSE is kept.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Settings:
    """Method settings.  Defaults are the recommended InfLLM v2 shape."""

    block: int = 64          # m   [InfLLM v2 › Block-level key-value partitioning]
    kernel: int = 32         # p   [InfLLM v2 › Semantic kernels]
    stride: int = 16         # s   [InfLLM v2 › Semantic kernels]
    topk: int = 64
    n_init: int = 1          # [InfLLM v2 › Initial and local tokens always selected]
    n_local: int = 2
    includes_forced: bool = True
    score_scale: float | None = None   # None -> 1/sqrt(d)
    attn_scale: float | None = None    # None -> 1/sqrt(d)
    coarse: int = 0          # s_c: 0 = exact LSE; else the LSE over coarse kernels of
                             # s_c keys [InfLLM v2 › Efficient LSE approximation]

    def sscale(self, d: int) -> float:
        return 1.0 / math.sqrt(d) if self.score_scale is None else float(self.score_scale)

    def ascale(self, d: int) -> float:
        return 1.0 / math.sqrt(d) if self.attn_scale is None else float(self.attn_scale)


# --------------------------------------------------------------------------
# Stage 1a: semantic kernels and their mean-pooled keys
# [InfLLM v2 › Semantic kernels for block relevance scoring, eq. S_j]
# --------------------------------------------------------------------------

def n_complete_kernels(L: int, p: int, s: int) -> int:
    """Number of kernels K[j s : j s + p] that lie wholly inside L keys (R2)."""
    if L < p:
        return 0
    return (L - p) // s + 1


def visible_kernel_count(i: int, p: int, s: int) -> int:
    """Kernels whose keys are all at positions <= i (R2, R7)."""
    return n_complete_kernels(i + 1, p, s)


def compress_keys(K: np.ndarray, p: int, s: int) -> np.ndarray:
    """Mean(K[j s : j s + p]) for every complete kernel j.  K: [L, d] float64."""
    n_c = n_complete_kernels(K.shape[0], p, s)
    out = np.zeros((n_c, K.shape[1]), dtype=np.float64)
    for j in range(n_c):
        out[j] = K[j * s: j * s + p].mean(axis=0)
    return out


# --------------------------------------------------------------------------
# Stage 1b: relevance scores
# --------------------------------------------------------------------------

def window_means(K: np.ndarray, size: int, stride: int) -> np.ndarray:
    """Mean of K[j stride : j stride + size] for every complete window j.

    With (size, stride) = (p, s) these are the semantic kernels; with
    size = stride = s_c the coarse kernels of the LSE approximation.
    """
    L, d = K.shape
    n = n_complete_kernels(L, size, stride)
    out = np.zeros((n, d), dtype=np.float64)
    for j in range(n):
        out[j] = K[j * stride: j * stride + size].astype(np.float64).mean(axis=0)
    return out


def kernel_logits(q: np.ndarray, Kc: np.ndarray, scale: float) -> np.ndarray:
    """scale * q_h . Mean(K_j) for every head h and kernel j.  q: [G, d]."""
    return scale * (q @ Kc.T)


def kernel_softmax(z: np.ndarray) -> np.ndarray:
    """r_kernel: softmax over the kernels, one distribution per head.

    [InfLLM v2 › Semantic kernels, eq. r_kernel]; the normaliser is the
    log-sum-exp of pass 1 in [InfLLM v2 › Top-K implementation and the LSE
    bottleneck].
    """
    zmax = z.max(axis=1, keepdims=True)
    lse = zmax + np.log(np.exp(z - zmax).sum(axis=1, keepdims=True))
    return np.exp(z - lse)


def group_relevance(z: np.ndarray) -> np.ndarray:
    """r_group: mean over the heads of a GQA group of each head's r_kernel.

    [InfLLM v2 › Query group sharing for memory efficiency, eq. r_group]
    """
    return kernel_softmax(z).mean(axis=0)


def log_sum_exp(z: np.ndarray) -> np.ndarray:
    """Per-row log-sum-exp (pass 1 of [InfLLM v2 › Top-K implementation and
    the LSE bottleneck]).  z: [G, n], n >= 1."""
    zmax = z.max(axis=1, keepdims=True)
    return (zmax + np.log(np.exp(z - zmax).sum(axis=1, keepdims=True)))[:, 0]


def group_relevance_given_lse(z: np.ndarray, lse: np.ndarray) -> np.ndarray:
    """r_group with a given per-head normaliser: mean_h exp(z_h - lse_h)."""
    return np.exp(z - lse[:, None]).mean(axis=0)


def block_relevance(g: np.ndarray, i: int, m: int, p: int, s: int) -> np.ndarray:
    """r_block for blocks 0 .. floor(i/m): max of r over intersecting kernels.

    [InfLLM v2 › Semantic kernels, eq. r_block].  ``g`` holds one score per
    visible kernel.  A block that no visible kernel touches scores -inf.
    """
    c = i // m
    r = np.full(c + 1, -np.inf)
    for j in range(g.shape[0]):
        first = (j * s) // m
        last = (j * s + p - 1) // m
        for blk in range(first, min(last, c) + 1):
            if g[j] > r[blk]:
                r[blk] = g[j]
    return r


def forced_blocks(i: int, m: int, n_init: int, n_local: int) -> list[int]:
    """Blocks that are always selected: the initial ones and the local window.

    [InfLLM v2 › Initial and local tokens always selected]; reading R4.
    """
    c = i // m
    out = set(range(0, min(n_init, c + 1)))
    out.update(range(max(0, c - n_local + 1), c + 1))
    return sorted(out)


def top_k_blocks(r: np.ndarray, forced: list[int], topk: int, includes_forced: bool) -> np.ndarray:
    """Forced blocks plus the highest-scoring other blocks, ascending.

    Scored candidates are blocks with a finite score that are not forced,
    ordered by (score descending, index ascending) (R5, R6).  With fewer
    candidates than slots every candidate is taken, so a short context is
    exactly dense [InfLLM v2 › Initial and local tokens always selected].
    """
    n_take = topk - len(forced) if includes_forced else topk
    n_take = max(n_take, 0)
    fset = set(forced)
    cand = np.array([j for j in range(r.shape[0]) if j not in fset and np.isfinite(r[j])],
                    dtype=np.int64)
    if cand.size:
        order = np.lexsort((cand, -r[cand]))
        taken = cand[order[:n_take]]
    else:
        taken = cand
    return np.array(sorted(fset.union(int(x) for x in taken)), dtype=np.int64)


def boundary_score(r: np.ndarray, blocks: np.ndarray, forced: list[int]) -> float:
    """Score of the lowest-ranked scored block taken: the smallest r over the
    selected blocks that are not forced, nan when no scored block is taken.

    This is the k-th best score among the candidates of top_k_blocks, the one
    the acceptance rule's 1e-4 relative tie band is measured from.
    """
    fset = set(forced)
    scored = [int(j) for j in blocks if int(j) not in fset]
    return float(min(r[j] for j in scored)) if scored else float("nan")


@dataclasses.dataclass
class Selection:
    blocks: np.ndarray   # selected block indices, ascending
    r: np.ndarray        # r_block for blocks 0 .. floor(i/m)
    g: np.ndarray        # r_group for the visible kernels
    boundary: float      # score of the lowest-ranked scored block taken (nan if none)


def select_for_query(q: np.ndarray, Kc: np.ndarray, i: int, st: Settings,
                     Kcc: np.ndarray | None = None) -> Selection:
    """Stage 1 for one query token of one GQA group.  q: [G, d]; Kc: [n_c, d].

    With st.coarse, the normaliser of every head's kernel softmax is the LSE
    over the visible coarse kernels Kcc (means of s_c keys, stride s_c)
    instead of over the fine kernels [InfLLM v2 › Efficient LSE
    approximation]; before the first coarse kernel is complete the exact LSE
    is kept.
    """
    d = q.shape[1]
    n_vis = min(visible_kernel_count(i, st.kernel, st.stride), Kc.shape[0])
    if n_vis > 0:
        z = kernel_logits(q, Kc[:n_vis], st.sscale(d))
        n_vis_c = 0
        if st.coarse:
            n_vis_c = min(visible_kernel_count(i, st.coarse, st.coarse), Kcc.shape[0])
        if n_vis_c > 0:
            lse = log_sum_exp(kernel_logits(q, Kcc[:n_vis_c], st.sscale(d)))
            g = group_relevance_given_lse(z, lse)
        else:
            g = group_relevance(z)
    else:
        g = np.zeros(0)
    r = block_relevance(g, i, st.block, st.kernel, st.stride)
    forced = forced_blocks(i, st.block, st.n_init, st.n_local)
    blocks = top_k_blocks(r, forced, st.topk, st.includes_forced)
    return Selection(blocks=blocks, r=r, g=g, boundary=boundary_score(r, blocks, forced))


# --------------------------------------------------------------------------
# Stage 2: exact attention over the selected blocks
# [InfLLM v2 › Block-level key-value partitioning, eq. B_j] and the standard
# scaled dot-product softmax attention of the section's first paragraph.
# --------------------------------------------------------------------------

def sparse_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, blocks: np.ndarray,
                     i: int, m: int, scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Softmax attention of q [G, d] over keys of the selected blocks with x <= i.

    Returns (O [G, d], lse [G]) with lse the natural log-sum-exp of the scaled
    scores of the attended keys.
    """
    mask = np.zeros(K.shape[0], dtype=bool)
    for j in blocks:
        mask[j * m:(j + 1) * m] = True
    mask[i + 1:] = False
    Ks, Vs = K[mask], V[mask]
    sc = scale * (q @ Ks.T)                       # [G, n_keys]
    smax = sc.max(axis=1, keepdims=True)
    e = np.exp(sc - smax)
    denom = e.sum(axis=1, keepdims=True)
    out = (e @ Vs) / denom
    lse = (smax + np.log(denom))[:, 0]
    return out, lse


def attended_keys(n_keys: int, blocks: np.ndarray, i: int, m: int) -> np.ndarray:
    """Indices (ascending) of the keys a query at position i attends: those of
    its selected blocks with x <= i."""
    mask = np.zeros(n_keys, dtype=bool)
    for j in blocks:
        mask[j * m:(j + 1) * m] = True
    mask[i + 1:] = False
    return np.nonzero(mask)[0]


def sparse_attention_grad_selected(q: np.ndarray, K: np.ndarray, V: np.ndarray, blocks: np.ndarray, i: int,
                                   m: int, scale: float, dO: np.ndarray):
    """Gradients of sparse_attention's O with respect to q, K and V for an
    upstream gradient dO [G, d], with the selection held fixed (there is no
    gradient through the top-k; [InfLLM v2 › Training-time considerations]:
    the keys receive the stage-2 gradient).  Softmax backward written out:
        P = softmax(scale q K_sel^T),  dP = dO V_sel^T,
        D = rowsum(dO * O),  dS = P * (dP - D),
        dq = scale dS K_sel,  dK_sel = scale dS^T q,  dV_sel = P^T dO.
    Returns (dq [G, d], keys [n], dK_sel [n, d], dV_sel [n, d]) for the n
    attended keys.
    """
    keys = attended_keys(K.shape[0], blocks, i, m)
    Ks, Vs = K[keys], V[keys]
    sc = scale * (q @ Ks.T)
    P = np.exp(sc - sc.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    O = P @ Vs
    dP = dO @ Vs.T
    D = (dO * O).sum(axis=1, keepdims=True)
    dS = P * (dP - D)
    return scale * (dS @ Ks), keys, scale * (dS.T @ q), P.T @ dO


def sparse_attention_grad(q: np.ndarray, K: np.ndarray, V: np.ndarray, blocks: np.ndarray, i: int, m: int,
                          scale: float, dO: np.ndarray):
    """sparse_attention_grad_selected scattered to full size: returns
    (dq [G, d], dK [L, d], dV [L, d]) with zeros for keys not attended."""
    dq, keys, dKs, dVs = sparse_attention_grad_selected(q, K, V, blocks, i, m, scale, dO)
    dK = np.zeros(K.shape, dtype=np.float64)
    dV = np.zeros(V.shape, dtype=np.float64)
    dK[keys] = dKs
    dV[keys] = dVs
    return dq, dK, dV


def block_grad_kv(Q: np.ndarray, dO: np.ndarray, lse: np.ndarray, D: np.ndarray, pos: np.ndarray,
                  Kj: np.ndarray, Vj: np.ndarray, key0: int, scale: float, extra: np.ndarray | None = None):
    """Gradients of one key block with respect to its keys and values, from
    every query that selected the block (the selection held fixed,
    [InfLLM v2 › Training-time considerations]): the sum over those queries of
    sparse_attention_grad_selected's dK_sel and dV_sel rows for this block's
    keys, with each query's softmax normalised by its own log-sum-exp over all
    the keys it attends.

    Q, dO [T, G, d]: the T queries' rows and upstream gradients; lse, D [T, G]:
    each query's natural log-sum-exp of its scaled scores and rowsum(dO * O);
    pos [T]: the query positions (keys after a query's position are not
    attended); Kj, Vj [m, d]: the block's keys key0 .. key0 + m - 1.
        P = exp(scale q K_j^T - lse) on attended keys,  dP = dO V_j^T,
        dS = P * (dP - D),  dK_j = scale sum dS^T q,  dV_j = sum P^T dO.
    extra [T, G, d] (optional): also returns sum P^T extra.
    Returns (dK_j [m, d], dV_j [m, d], sum P^T extra or None).
    """
    T, G, d = Q.shape
    m = Kj.shape[0]
    keys = key0 + np.arange(m)
    S = scale * (Q.reshape(T * G, d) @ Kj.T).reshape(T, G, m)
    valid = (keys[None, :] <= pos[:, None])[:, None, :]
    P = np.where(valid, np.exp(np.where(valid, S, 0.0) - lse[:, :, None]), 0.0)
    dP = (dO.reshape(T * G, d) @ Vj.T).reshape(T, G, m)
    dS = P * (dP - D[:, :, None])
    dK = scale * (dS.reshape(T * G, m).T @ Q.reshape(T * G, d))
    dV = P.reshape(T * G, m).T @ dO.reshape(T * G, d)
    ex = None if extra is None else P.reshape(T * G, m).T @ extra.reshape(T * G, d)
    return dK, dV, ex


# --------------------------------------------------------------------------
# Drivers over the [B, Hkv, n_q] units of one input set
# --------------------------------------------------------------------------

def _f64(bits: np.ndarray) -> np.ndarray:
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def kc_for(inputs, b: int, h: int, st: Settings) -> np.ndarray:
    L = int(inputs.kv_lens[b])
    K = _f64(inputs.k[b, h, :L])
    return compress_keys(K, st.kernel, st.stride)


def query_position(L: int, n_q: int, t: int) -> int:
    return L - n_q + t


def run_selection(inputs, st: Settings, units=None, kc_cache=None):
    """Selections for the (b, h_kv, t) units given (all by default).

    Returns {(b, h, t): Selection}.
    """
    kcc_cache = {}
    wl = inputs.wl
    G = wl.group
    if units is None:
        units = [(b, h, t) for b in range(wl.batch) for h in range(wl.n_kv_heads)
                 for t in range(wl.n_q)]
    kc_cache = {} if kc_cache is None else kc_cache
    out = {}
    for (b, h, t) in units:
        if (b, h) not in kc_cache:
            kc_cache[(b, h)] = kc_for(inputs, b, h, st)
        L = int(inputs.kv_lens[b])
        i = query_position(L, wl.n_q, t)
        q = _f64(inputs.q[b, t, h * G:(h + 1) * G])
        Kcc = None
        if st.coarse:
            if (b, h) not in kcc_cache:
                kcc_cache[(b, h)] = window_means(_f64(inputs.k[b, h, :L]), st.coarse, st.coarse)
            Kcc = kcc_cache[(b, h)]
        out[(b, h, t)] = select_for_query(q, kc_cache[(b, h)], i, st, Kcc)
    return out


def run_attention(inputs, st: Settings, blocks_of, units=None):
    """Attention outputs for the units given, on the block sets ``blocks_of``.

    ``blocks_of`` maps (b, h, t) -> selected blocks.  Returns
    {(b, h, t): (O [G, d], lse [G])}.
    """
    wl = inputs.wl
    G, d = wl.group, wl.head_dim
    if units is None:
        units = sorted(blocks_of.keys())
    out = {}
    kv = {}
    for (b, h, t) in units:
        if (b, h) not in kv:
            L = int(inputs.kv_lens[b])
            kv = {(b, h): (_f64(inputs.k[b, h, :L]), _f64(inputs.v[b, h, :L]))}
        K, V = kv[(b, h)]
        L = int(inputs.kv_lens[b])
        i = query_position(L, wl.n_q, t)
        q = _f64(inputs.q[b, t, h * G:(h + 1) * G])
        out[(b, h, t)] = sparse_attention(q, K, V, np.asarray(blocks_of[(b, h, t)]), i,
                                          st.block, st.ascale(d))
    return out


def unit_attention_grad(inputs, st: Settings, blocks_of, dO_all: np.ndarray, unit, K=None, V=None):
    """Gradient contributions of one (b, h, t) unit: (dq [G, d], keys, dK_sel,
    dV_sel) as from sparse_attention_grad_selected."""
    wl = inputs.wl
    G, d = wl.group, wl.head_dim
    b, h, t = unit
    L = int(inputs.kv_lens[b])
    if K is None:
        K, V = _f64(inputs.k[b, h, :L]), _f64(inputs.v[b, h, :L])
    i = query_position(L, wl.n_q, t)
    q = _f64(inputs.q[b, t, h * G:(h + 1) * G])
    return sparse_attention_grad_selected(q, K, V, np.asarray(blocks_of[unit]), i, st.block, st.ascale(d),
                                          np.asarray(dO_all[b, t, h * G:(h + 1) * G], dtype=np.float64))
