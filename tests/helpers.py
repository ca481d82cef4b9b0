"""Shared helpers of the parity tests: device upload, running the CUDA path
through the binding, and the comparison rules.

Tolerances (fixed by the acceptance rule of the benchmark configurations):
  * selection: block sets equal, except blocks whose oracle score lies within
    1e-4 relative of the oracle's boundary score (the last scored block taken);
  * attention: max |O_gpu - O_ref| <= 2e-3 and mean |O_gpu - O_ref| <= 2e-4
    over all outputs, O_ref computed by the fp64 oracle on the same selection.
    The output is bf16, so an element can be no closer to O_ref than the
    rounding of the stored value allows: each element may in addition be off
    by half a bf16 ulp of its magnitude (bf16_half_ulp), and the mean by the
    mean of those half-ulps.  That allowance only matters where |O| is near 1
    (a query averaging a handful of values); units attending at least
    STRICT_MIN_KEYS keys are also held to the bare 2e-3 / 2e-4;
  * block scores r: relative error <= 1e-4 where the oracle's r is finite
    (the kernel means carry 16 significant bits, the dot products fp32);
  * lse: absolute error <= 1e-3 (fp32 accumulation of a natural log);
  * gradients dq, dk, dv (backward with the selection fixed): the attention
    rule relative to each tensor's scale, max |g_gpu - g_ref| <= 2e-3 max|g_ref|
    and mean |g_gpu - g_ref| <= 2e-4 max|g_ref| over the rows that receive a
    gradient; rows of keys no query attends are exactly 0.  The kernels carry
    P and dS at 16 significant bits (error near 4e-4 of the scale).  D =
    rowsum(dO * O) is formed from the forward output the call is given, which
    is bf16: its error dD_r = sum_d dO_rd (O_gpu - O_ref)_rd moves dq_r by
    -scale dD_r sum_j P_rj k_j and dk_j by -scale sum_r P_rj dD_r q_r.  Both
    rules widen by those terms' magnitudes, bounded with the oracle's own
    probabilities: scale |dD_r| sum_j P_rj |k_j| for dq and
    scale sum_r P_rj |dD_r| |q_r| for dk (dv does not involve D).  The term
    only matters for queries that attend a handful of keys, where |O| ~ |V|.
"""

from __future__ import annotations

import numpy as np

SEL_REL = 1e-4
ATT_MAX = 2e-3
ATT_MEAN = 2e-4
R_REL = 1e-4
LSE_ABS = 1e-3
STRICT_MIN_KEYS = 256
GRAD_MAX = 2e-3
GRAD_MEAN = 2e-4


def dev_bf16(bits: np.ndarray, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def kc_to_f64(kc) -> np.ndarray:
    """bf16 [B, Hkv, 2, n_c, d] hi/lo planes -> fp64 [B, Hkv, n_c, d] (hi + lo)."""
    import torch
    a = kc.view(torch.int16).cpu().numpy().view(np.uint16)
    f = (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return f[:, :, 0] + f[:, :, 1]


class DeviceRun:
    """Uploads one input set and runs the three stages on the device."""

    def __init__(self, inp, dev, score_scale=None, attn_scale=None):
        import torch
        import trainable_block_sparse_infllm_gb300 as T
        self.T = T
        self.inp = inp
        wl = inp.wl
        self.dev = dev
        self.p = T.make_params(wl.batch, wl.n_kv_heads, wl.kv_len, wl.topk, wl.topk_includes_forced,
                               n_init=wl.n_init, n_local=wl.n_local, score_scale=score_scale,
                               attn_scale=attn_scale)
        self.q = dev_bf16(inp.q, dev)
        self.k = dev_bf16(inp.k, dev)
        self.v = dev_bf16(inp.v, dev)
        self.lens = torch.from_numpy(inp.kv_lens.astype(np.int32)).to(dev)
        self.kmax = T.max_selected(self.p)
        self.nq = wl.n_q
        B, H = wl.batch, wl.n_kv_heads
        self.kc = T.alloc_kc(self.p, dev)
        self.idx = torch.full((B, H, self.nq, self.kmax), -7, dtype=torch.int32, device=dev)
        self.nsel = torch.full((B, H, self.nq), -7, dtype=torch.int32, device=dev)
        self.nbmax = -(-wl.kv_len // wl.block)
        self.scores = torch.empty((B, H, self.nq, self.nbmax), dtype=torch.float32, device=dev)
        self.out = torch.full_like(self.q, float("nan"))
        self.lse = torch.full((B, self.nq, wl.n_heads), float("nan"), dtype=torch.float32, device=dev)

    def compress(self, begin=0, end=-1):
        self.T.compress_keys(self.p, self.k, self.lens, self.kc, begin, end)

    def select(self, with_scores=True):
        ws = self.T.alloc_workspace(self.p, self.nq, self.T.OP_SELECT, self.dev)
        self.T.select_blocks(self.p, self.q, self.kc, self.lens, self.idx, self.nsel,
                             self.scores if with_scores else None, ws)

    def attend(self, idx=None, nsel=None, prefill=None):
        idx = self.idx if idx is None else idx
        nsel = self.nsel if nsel is None else nsel
        if prefill is None:
            prefill = self.nq > self.T.DECODE_MAX_NQ
        op = self.T.OP_PREFILL if prefill else self.T.OP_DECODE
        ws = self.T.alloc_workspace(self.p, self.nq, op, self.dev)
        fn = self.T.sparse_attn_prefill if prefill else self.T.sparse_attn_decode
        fn(self.p, self.q, self.k, self.v, self.lens, idx, nsel, self.out, self.lse, ws)

    def step(self):
        """The fused decode step (newest kernel + selection + attention)."""
        ws = self.T.alloc_workspace(self.p, self.nq, self.T.OP_DECODE_STEP, self.dev)
        self.T.decode_step(self.p, self.q, self.k, self.v, self.lens, self.kc, self.idx, self.nsel,
                           self.out, self.lse, ws)

    def blank_step_kernels(self):
        """Compress everything, then NaN the kernel means a decode step must
        recompute (those ending inside the last n_q tokens).  Returns the full
        kernel-mean buffer for comparison."""
        import torch
        from oracle import n_complete_kernels
        self.compress()
        full = self.kc.clone()
        for b, L in enumerate(self.inp.kv_lens):
            lo = n_complete_kernels(max(int(L) - self.nq, 0), 32, 16)
            hi = n_complete_kernels(int(L), 32, 16)
            if hi > lo:
                self.kc[b, :, :, lo:hi].view(torch.int16).fill_(0x7FC0)
        return full

    def backward(self, idx, nsel, dout_bits):
        """Gradients of the attention last run by ``attend`` (out, lse) for
        upstream ``dout_bits``: returns fp32 (dq, dk, dv) device tensors."""
        import torch
        wl = self.inp.wl
        dout = dev_bf16(dout_bits, self.dev)
        dq = torch.full((wl.batch, self.nq, wl.n_heads, wl.head_dim), float("nan"), dtype=torch.float32,
                        device=self.dev)
        dk = torch.full((wl.batch, wl.n_kv_heads, wl.kv_len, wl.head_dim), float("nan"), dtype=torch.float32,
                        device=self.dev)
        dv = torch.full_like(dk, float("nan"))
        ws = self.T.alloc_workspace(self.p, self.nq, self.T.OP_BACKWARD, self.dev)
        self.T.sparse_attn_backward(self.p, self.q, self.k, self.v, self.lens, idx, nsel, self.out, self.lse, dout,
                                    dq, dk, dv, ws)
        return dq, dk, dv

    def gpu_blocks(self, units):
        idx, nsel = self.idx.cpu().numpy(), self.nsel.cpu().numpy()
        return {(b, h, t): idx[b, h, t, :nsel[b, h, t]].copy() for (b, h, t) in units}

    def upload_selection(self, sels):
        """Oracle selections {(b,h,t): Selection} -> device idx/nsel tensors."""
        import torch
        B, H = self.inp.wl.batch, self.inp.wl.n_kv_heads
        idx = np.full((B, H, self.nq, self.kmax), -1, dtype=np.int32)
        nsel = np.zeros((B, H, self.nq), dtype=np.int32)
        for (b, h, t), s in sels.items():
            idx[b, h, t, :len(s.blocks)] = s.blocks
            nsel[b, h, t] = len(s.blocks)
        return torch.from_numpy(idx).to(self.dev), torch.from_numpy(nsel).to(self.dev)


def selection_mismatch(gpu_blocks, sel, rel=SEL_REL):
    """None if the GPU set is acceptable for oracle selection `sel`, else a message."""
    g = set(int(x) for x in gpu_blocks)
    o = set(int(x) for x in sel.blocks)
    if len(g) != len(gpu_blocks):
        return f"duplicate blocks {sorted(gpu_blocks)}"
    if g == o:
        return None
    if len(g) != len(o):
        return f"size {len(g)} != {len(o)}"
    rK = sel.boundary
    for j in g ^ o:
        if j < 0 or j >= sel.r.shape[0] or not np.isfinite(sel.r[j]) or not np.isfinite(rK):
            return f"block {j} outside the candidates"
        if abs(sel.r[j] - rK) > rel * abs(rK):
            return f"block {j} score {sel.r[j]:.8g} vs boundary {rK:.8g}"
    return None


def check_selections(run, sels, check_scores=True):
    idx = run.idx.cpu().numpy()
    nsel = run.nsel.cpu().numpy()
    scores = run.scores.cpu().numpy() if check_scores else None
    bad, ties = [], 0
    for (b, h, t), s in sels.items():
        n = int(nsel[b, h, t])
        row = idx[b, h, t]
        assert 0 <= n <= run.kmax, ((b, h, t), n)
        assert np.all(row[n:] == -1), ((b, h, t), row)
        blocks = row[:n]
        assert np.all(np.diff(blocks) > 0), ((b, h, t), blocks)
        msg = selection_mismatch(blocks, s)
        if msg:
            bad.append(((b, h, t), msg))
        elif set(blocks.tolist()) != set(s.blocks.tolist()):
            ties += 1
        if scores is not None:
            r_gpu = scores[b, h, t, :s.r.shape[0]]
            fin = np.isfinite(s.r)
            assert np.array_equal(np.isfinite(r_gpu), fin), ((b, h, t), "finite pattern")
            if fin.any():
                err = np.abs(r_gpu[fin] - s.r[fin]) / np.abs(s.r[fin])
                assert err.max() <= R_REL, ((b, h, t), float(err.max()))
            assert np.all(np.isneginf(scores[b, h, t, s.r.shape[0]:])), ((b, h, t), "tail")
    assert not bad, bad[:5]
    return ties


def bf16_half_ulp(x):
    """Half the spacing of bf16 values at |x| (8 significant bits): for
    2^e <= |x| < 2^(e+1) the spacing is 2^(e-7), so rounding to bf16 moves a
    value by at most 2^(e-8)."""
    _, e = np.frexp(np.abs(np.asarray(x, dtype=np.float64)))   # |x| = f 2^e, 1/2 <= f < 1
    return np.ldexp(1.0, e - 9)


def attended_key_count_of(i, blocks, m):
    """Keys a query at position i attends: those of its selected blocks
    (size m) at positions <= i."""
    return int(sum(max(0, min(m, i - int(j) * m + 1)) for j in blocks))


def strict_units(inp, blocks_of, min_keys=STRICT_MIN_KEYS):
    """The units of blocks_of {(b,h,t): blocks} that attend >= min_keys keys."""
    wl = inp.wl
    return {u for u, blk in blocks_of.items()
            if attended_key_count_of(int(inp.kv_lens[u[0]]) - wl.n_q + u[2], blk, wl.block) >= min_keys}


def check_attention(run, refs, strict=False, strict_units=None):
    """refs: {(b,h,t): (O [16, d], lse [16])}.  Returns (max, mean) abs error.

    Every element: |O_gpu - O_ref| <= 2e-3 + half a bf16 ulp at |O_ref| + 2e-3
    (the stored output is bf16; a value within 2e-3 of O_ref rounds to one
    within that of it), and the mean error <= 2e-4 + the mean of those
    half-ulps.  strict: the workload rule with no allowance, max <= 2e-3 and
    mean <= 2e-4, over the units in strict_units (all units when None).
    """
    out = run.out.float().cpu().numpy()
    lse = run.lse.cpu().numpy()
    errs, total, total_allow, count, lse_err = [], 0.0, 0.0, 0, 0.0
    s_max, s_total, s_count = 0.0, 0.0, 0
    for (b, h, t), (o_ref, l_ref) in refs.items():
        o = out[b, t, h * 16:(h + 1) * 16]
        e = np.abs(o - o_ref)
        allow = bf16_half_ulp(np.abs(o_ref) + ATT_MAX)
        assert np.all(e <= ATT_MAX + allow), ((b, h, t), float(e.max()), float((e - allow).max()))
        errs.append(e.max())
        total += e.sum()
        total_allow += allow.sum()
        count += e.size
        if strict and (strict_units is None or (b, h, t) in strict_units):
            s_max = max(s_max, float(e.max()))
            s_total += e.sum()
            s_count += e.size
        lse_err = max(lse_err, float(np.abs(lse[b, t, h * 16:(h + 1) * 16] - l_ref).max()))
    mx, mean = float(max(errs)), total / count
    assert mean <= ATT_MEAN + total_allow / count, (mean, total_allow / count)
    if strict and s_count:
        assert s_max <= ATT_MAX and s_total / s_count <= ATT_MEAN, (s_max, s_total / s_count)
    assert lse_err <= LSE_ABS, lse_err
    return mx, mean


def check_grad(name, got, ref, rows_used=None, allow=None):
    """got, ref: arrays of the same shape [..., d].  rows_used (bool over the
    leading dims, optional): rows that receive a gradient; the others must be
    exactly 0 in ``got``.  allow (same shape as ref, optional): a per-element
    bound on the error the kernel's inputs carry by themselves (the bf16
    forward output inside D); it widens both rules.  Returns
    (max err / scale, mean err / scale)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    allow = np.zeros_like(ref) if allow is None else np.asarray(allow, dtype=np.float64)
    assert np.all(np.isfinite(got)), (name, "non-finite")
    scale = float(np.abs(ref).max())
    assert scale > 0, (name, "zero reference")
    err = np.abs(got - ref)
    if rows_used is not None:
        assert np.all(got[~rows_used] == 0), (name, "gradient on a key no query attends")
        err, allow = err[rows_used], allow[rows_used]
    over = err - 1.001 * allow
    assert over.max() <= GRAD_MAX * scale, (name, float(over.max()) / scale, float(err.max()) / scale)
    assert err.mean() <= GRAD_MEAN * scale + allow.mean(), (name, float(err.mean()) / scale)
    return float(err.max()) / scale, float(err.mean()) / scale
