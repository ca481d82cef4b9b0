"""The fp64 oracle over every unit of a large workload, in a process pool.

Test infrastructure.  The parity tests of the full-size prefill workload
compare every (b, h_kv, t) unit, which takes minutes of oracle time on one
core.  This module spreads the oracle's per-unit functions over worker
processes started with the `spawn` method (the parent has already created a
CUDA context, which a forked child must not inherit).  The inputs and the
device results reach the workers as memory-mapped .npy files in a temporary
directory; nothing here computes any part of the method itself.
"""

from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np

_W = {}


def _init(folder, names, wl, st):
    import synthetic_inputs as S
    for n in names:
        _W[n] = np.load(os.path.join(folder, n + ".npy"), mmap_mode="r")
    _W["inp"] = S.Inputs(wl=wl, q=_W["q"], k=_W["k"], v=_W["v"], kv_lens=np.asarray(_W["kv_lens"]),
                         planted=np.zeros((wl.batch, wl.n_kv_heads, 0), dtype=np.int64))
    _W["st"] = st
    _W["kc"] = {}


def _select_task(task):
    """Oracle selection of units (b, h, t0..t1-1) checked against the device's."""
    import oracle as O
    from helpers import selection_mismatch
    b, h, t0, t1 = task
    inp, st = _W["inp"], _W["st"]
    units = [(b, h, t) for t in range(t0, t1)]
    sels = O.run_selection(inp, st, units=units, kc_cache=_W["kc"])
    idx, nsel = _W["idx"], _W["nsel"]
    kmax = idx.shape[-1]
    oidx = np.full((t1 - t0, kmax), -1, dtype=np.int32)
    onsel = np.zeros(t1 - t0, dtype=np.int32)
    bad, ties = [], 0
    for (b_, h_, t), s in sels.items():
        n = int(nsel[b_, h_, t])
        row = np.asarray(idx[b_, h_, t])
        oidx[t - t0, :len(s.blocks)] = s.blocks
        onsel[t - t0] = len(s.blocks)
        if not (0 <= n <= kmax) or np.any(row[max(n, 0):] != -1) or np.any(np.diff(row[:n]) <= 0):
            bad.append(((b_, h_, t), "malformed row"))
            continue
        msg = selection_mismatch(row[:n], s)
        if msg:
            bad.append(((b_, h_, t), msg))
        elif set(row[:n].tolist()) != set(s.blocks.tolist()):
            ties += 1
    return b, h, t0, t1, bad, ties, oidx, onsel


def _attend_task(task):
    """Oracle attention of units (b, h, t0..t1-1) on the oracle selection,
    compared with the device output: per-element rule and error sums."""
    import oracle as O
    from helpers import ATT_MAX, attended_key_count_of, bf16_half_ulp
    b, h, t0, t1 = task
    inp, st = _W["inp"], _W["st"]
    oidx, onsel, out, lse = _W["oidx"], _W["onsel"], _W["out"], _W["lse"]
    units = [(b, h, t) for t in range(t0, t1)]
    blocks_of = {u: np.asarray(oidx[u][:onsel[u]]) for u in units}
    refs = O.run_attention(inp, st, blocks_of, units=units)
    wl = inp.wl
    res = {"max": 0.0, "sum": 0.0, "allow": 0.0, "count": 0, "lse": 0.0, "over": [],
           "s_max": 0.0, "s_sum": 0.0, "s_count": 0}
    for (b_, h_, t), (o_ref, l_ref) in refs.items():
        o = np.asarray(out[b_, t, h_ * 16:(h_ + 1) * 16], dtype=np.float64)
        e = np.abs(o - o_ref)
        allow = bf16_half_ulp(np.abs(o_ref) + ATT_MAX)
        if np.any(e > ATT_MAX + allow):
            res["over"].append(((b_, h_, t), float(e.max())))
        res["max"] = max(res["max"], float(e.max()))
        res["sum"] += float(e.sum())
        res["allow"] += float(allow.sum())
        res["count"] += e.size
        res["lse"] = max(res["lse"], float(np.abs(np.asarray(lse[b_, t, h_ * 16:(h_ + 1) * 16]) - l_ref).max()))
        L = int(inp.kv_lens[b_])
        if attended_key_count_of(L - wl.n_q + t, blocks_of[(b_, h_, t)], wl.block) >= _W["strict_keys"]:
            res["s_max"] = max(res["s_max"], float(e.max()))
            res["s_sum"] += float(e.sum())
            res["s_count"] += e.size
    return res


def _init_attend(folder, names, wl, st, strict_keys):
    _init(folder, names, wl, st)
    _W["strict_keys"] = strict_keys


def _kv_f64(b, h):
    """This worker's fp64 copy of one (b, h) cache, kept across its tasks."""
    import synthetic_inputs as S
    key = ("kv", b, h)
    if key not in _W:
        L = int(_W["inp"].kv_lens[b])
        for k in [k for k in _W if isinstance(k, tuple) and k[0] == "kv"]:
            del _W[k]
        _W[key] = (S.bf16_bits_to_f64(_W["inp"].k[b, h, :L]), S.bf16_bits_to_f64(_W["inp"].v[b, h, :L]))
    return _W[key]


def _grad_q_task(task):
    """Per unit of (b, h, t0..t1-1), on the given selection: the oracle's
    forward (lse, and D = rowsum(dO * O) from its own O), its dq against the
    device's, and the allowance for the bf16 forward output the device's D
    is built from (dD = |rowsum(dO * (out - O))|).  Returns the error
    statistics and each unit's lse, D and dD."""
    import oracle as O
    import synthetic_inputs as S
    b, h, t0, t1 = task
    inp, st = _W["inp"], _W["st"]
    wl = inp.wl
    G, d, m = wl.group, wl.head_dim, wl.block
    scale = st.ascale(d)
    K, V = _kv_f64(b, h)
    L = int(inp.kv_lens[b])
    idx, nsel, dO_all, out, dq = _W["idx"], _W["nsel"], _W["dout"], _W["out"], _W["dq"]
    res = {"ref": 0.0, "over": 0.0, "err": 0.0, "allow": 0.0, "count": 0}
    stats = np.zeros((t1 - t0, 3, G))
    for t in range(t0, t1):
        i = O.query_position(L, wl.n_q, t)
        blocks = np.asarray(idx[b, h, t][:nsel[b, h, t]])
        q = S.bf16_bits_to_f64(inp.q[b, t, h * G:(h + 1) * G])
        dOu = S.bf16_bits_to_f64(dO_all[b, t, h * G:(h + 1) * G])
        o_ref, lse = O.sparse_attention(q, K, V, blocks, i, m, scale)
        gq = O.sparse_attention_grad_selected(q, K, V, blocks, i, m, scale, dOu)[0]
        o_dev = S.bf16_bits_to_f64(out[b, t, h * G:(h + 1) * G])
        dD = np.abs((dOu * (o_dev - o_ref)).sum(axis=1))
        pk = O.sparse_attention(q, K, np.abs(K), blocks, i, m, scale)[0]
        allow = scale * dD[:, None] * pk
        err = np.abs(np.asarray(dq[b, t, h * G:(h + 1) * G], dtype=np.float64) - gq)
        res["ref"] = max(res["ref"], float(np.abs(gq).max()))
        res["over"] = max(res["over"], float((err - 1.001 * allow).max()))
        res["err"] += float(err.sum())
        res["allow"] += float(allow.sum())
        res["count"] += err.size
        stats[t - t0] = (lse, (dOu * o_ref).sum(axis=1), dD)
    return b, h, t0, t1, res, stats


def _grad_kv_task(task):
    """dK, dV of the key blocks j0..j1-1 of (b, h) from every query that
    selected them (oracle.block_grad_kv with the queries' own lse and D),
    the allowance for the bf16 forward output, and the keys some query
    attends."""
    import oracle as O
    import synthetic_inputs as S
    b, h, j0, j1 = task
    inp, st = _W["inp"], _W["st"]
    wl = inp.wl
    G, d, m = wl.group, wl.head_dim, wl.block
    scale = st.ascale(d)
    K, V = _kv_f64(b, h)
    L = int(inp.kv_lens[b])
    idx, nsel, dO_all, stats = _W["idx"], _W["nsel"], _W["dout"], _W["stats"]
    sel = np.asarray(idx[b, h])                       # [n_q, k_max]
    n = np.asarray(nsel[b, h])
    live = np.arange(sel.shape[1])[None, :] < n[:, None]
    lo, hi = j0 * m, min(j1 * m, L)
    rk, rv, ra = (np.zeros((max(0, hi - lo), d)) for _ in range(3))
    used = np.zeros(max(0, hi - lo), dtype=bool)
    for j in range(j0, j1):
        if j * m >= L:
            break
        toks = np.nonzero(((sel == j) & live).any(axis=1))[0]
        if toks.size == 0:
            continue
        pos = np.array([O.query_position(L, wl.n_q, int(t)) for t in toks])
        Q = S.bf16_bits_to_f64(inp.q[b, toks][:, h * G:(h + 1) * G])
        dOt = S.bf16_bits_to_f64(dO_all[b, toks][:, h * G:(h + 1) * G])
        st3 = np.asarray(stats[b, h, toks])           # [T, 3, G]: lse, D, dD
        rows = slice(j * m, min((j + 1) * m, L))
        dk, dv, ex = O.block_grad_kv(Q, dOt, st3[:, 0], st3[:, 1], pos, K[rows], V[rows], j * m, scale,
                                     st3[:, 2][:, :, None] * np.abs(Q))
        r = slice(j * m - lo, min((j + 1) * m, L) - lo)
        rk[r], rv[r], ra[r] = dk, dv, scale * ex
        used[r] = np.arange(j * m, min((j + 1) * m, L)) <= pos.max()
    return b, h, j0, j1, rk, rv, ra, used


def all_backward(inp, st, idx, nsel, dout, out, dq, chunk=256, blocks_per_task=16):
    """Oracle gradients of every unit of a workload with the selection
    (idx, nsel) held fixed.  dout, out: bf16 bits [B, n_q, Hq, d] (the
    upstream gradient and the device's forward output); dq: the device's
    dq.  Returns (dq statistics, dK ref, dV ref, dK allowance, keys used),
    the key arrays shaped like the caches."""
    wl = inp.wl
    with tempfile.TemporaryDirectory() as folder:
        arrays = {"q": inp.q, "k": inp.k, "v": inp.v, "kv_lens": inp.kv_lens, "idx": idx, "nsel": nsel,
                  "dout": dout, "out": out, "dq": dq}
        _save(folder, arrays)
        ctx = mp.get_context("spawn")
        G = wl.group
        stats = np.zeros((wl.batch, wl.n_kv_heads, wl.n_q, 3, G))
        tot = {"ref": 0.0, "over": 0.0, "err": 0.0, "allow": 0.0, "count": 0}
        with _OneBlasThread(), ctx.Pool(_workers(), initializer=_init,
                                        initargs=(folder, list(arrays), wl, st)) as pool:
            for b, h, t0, t1, r, sts in pool.imap_unordered(_grad_q_task, _tasks(inp, chunk)):
                tot["ref"] = max(tot["ref"], r["ref"])
                tot["over"] = max(tot["over"], r["over"])
                for k in ("err", "allow", "count"):
                    tot[k] += r[k]
                stats[b, h, t0:t1] = sts
        _save(folder, {"stats": stats})
        shape = (wl.batch, wl.n_kv_heads, wl.kv_len, wl.head_dim)
        rk, rv, ra = np.zeros(shape), np.zeros(shape), np.zeros(shape)
        used = np.zeros(shape[:3], dtype=bool)
        nb = (wl.kv_len + wl.block - 1) // wl.block
        tasks = [(b, h, j0, min(nb, j0 + blocks_per_task)) for b in range(wl.batch) for h in range(wl.n_kv_heads)
                 for j0 in range(0, nb, blocks_per_task)]
        with _OneBlasThread(), ctx.Pool(_workers(), initializer=_init,
                                        initargs=(folder, list(arrays) + ["stats"], wl, st)) as pool:
            for b, h, j0, j1, k_, v_, a_, u_ in pool.imap_unordered(_grad_kv_task, tasks):
                lo = j0 * wl.block
                rk[b, h, lo:lo + k_.shape[0]] = k_
                rv[b, h, lo:lo + v_.shape[0]] = v_
                ra[b, h, lo:lo + a_.shape[0]] = a_
                used[b, h, lo:lo + u_.shape[0]] = u_
    return tot, rk, rv, ra, used


def _tasks(inp, chunk):
    wl = inp.wl
    return [(b, h, t0, min(wl.n_q, t0 + chunk)) for b in range(wl.batch) for h in range(wl.n_kv_heads)
            for t0 in range(0, wl.n_q, chunk)]


def _workers():
    return max(1, min(32, (os.cpu_count() or 2)))


class _OneBlasThread:
    """Spawned workers inherit the environment: one BLAS thread each."""

    KEYS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in self.KEYS}
        for k in self.KEYS:
            os.environ[k] = "1"

    def __exit__(self, *exc):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _save(folder, arrays):
    for n, a in arrays.items():
        np.save(os.path.join(folder, n + ".npy"), np.ascontiguousarray(a))


def all_selections(inp, st, idx, nsel, chunk=256):
    """Check the device selection (idx, nsel: numpy) of every unit against the
    oracle.  Returns (bad [(unit, msg)], tie-band differences, oracle idx,
    oracle nsel) with the oracle's selection laid out like idx / nsel."""
    wl = inp.wl
    with tempfile.TemporaryDirectory() as folder:
        arrays = {"q": inp.q, "k": inp.k, "v": inp.v, "kv_lens": inp.kv_lens, "idx": idx, "nsel": nsel}
        _save(folder, arrays)
        ctx = mp.get_context("spawn")
        oidx = np.full(idx.shape, -1, dtype=np.int32)
        onsel = np.zeros(nsel.shape, dtype=np.int32)
        bad, ties = [], 0
        with _OneBlasThread(), ctx.Pool(_workers(), initializer=_init,
                                        initargs=(folder, list(arrays), wl, st)) as pool:
            for b, h, t0, t1, bd, ti, oi, on in pool.imap_unordered(_select_task, _tasks(inp, chunk)):
                bad += bd
                ties += ti
                oidx[b, h, t0:t1] = oi
                onsel[b, h, t0:t1] = on
    return bad, ties, oidx, onsel


def all_attention(inp, st, oidx, onsel, out, lse, strict_keys, chunk=256):
    """Oracle attention of every unit on the oracle selection (oidx, onsel)
    against the device output (out: float32 numpy [B, n_q, Hq, d], lse).
    Returns the merged error statistics of _attend_task."""
    wl = inp.wl
    with tempfile.TemporaryDirectory() as folder:
        arrays = {"q": inp.q, "k": inp.k, "v": inp.v, "kv_lens": inp.kv_lens, "oidx": oidx, "onsel": onsel,
                  "out": out, "lse": lse}
        _save(folder, arrays)
        ctx = mp.get_context("spawn")
        tot = {"max": 0.0, "sum": 0.0, "allow": 0.0, "count": 0, "lse": 0.0, "over": [],
               "s_max": 0.0, "s_sum": 0.0, "s_count": 0}
        with _OneBlasThread(), ctx.Pool(_workers(), initializer=_init_attend,
                                        initargs=(folder, list(arrays), wl, st, strict_keys)) as pool:
            for r in pool.imap_unordered(_attend_task, _tasks(inp, chunk)):
                for k in ("max", "lse", "s_max"):
                    tot[k] = max(tot[k], r[k])
                for k in ("sum", "allow", "count", "s_sum", "s_count"):
                    tot[k] += r[k]
                tot["over"] += r["over"]
    return tot
