"""Benchmark of the InfLLM v2 hot path on GB300.

Headline: decode tokens/s at 128K context (batch 4, 32 query / 2 KV heads,
top-64 blocks).  One step = the whole decode path for one new token per
sequence through infllmv2_decode_step: the newest complete kernel mean, block
selection (scores, LSE, group mean, block max, top-k) and sparse attention
with its merge, in one cluster launch.  Eight steps over eight input replicas
form one CUDA graph.  The three separate stages (compress_keys,
select_blocks, sparse_attn_decode) are timed alone as a breakdown.  A prefill
line (32K causal prefill, 32 query / 2 KV heads) is reported alongside.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs under torch.distributed (one process per GPU); every rank decodes
its own batch (weak scaling) and the time is the max over ranks.
`--impl reference` times the fp64 CPU oracle on the same workload.
"""

from __future__ import annotations

import os

# The CPU legs (input generation, the oracle) run single-threaded so that the
# reported core count is exact.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import re
import json
import math
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic_inputs as S  # noqa: E402

DECODE = "decode_128k"
PREFILL = "prefill_32k"
METRIC = "decode tokens/s and prefill tokens/s at 128K ctx; % of HBM / bf16 TC roofline"
REPLICAS = 8          # rotating input copies: 8 x 0.57 GB >> L2 (129 MB)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# Source file of each kernel whose DRAM traffic is recorded; its hash, with
# every header it includes from the same folder (transitively), dates the
# recorded counters.
_KERNEL_SRC = {"decode_step_kernel": "decode_step.cu", "attn_tc_kernel": "attn_tc.cu", "sel_tc_kernel": "select_tc.cu",
               "bwd_dq_kernel": "attn_bwd.cu", "bwd_dkdv_kernel": "attn_bwd.cu"}


def _src_hash(kernel: str):
    csrc = os.path.join(ROOT, "trainable_block_sparse_infllm_gb300", "csrc")
    order = []

    def visit(fn):
        if fn in order:
            return
        order.append(fn)
        for line in open(os.path.join(csrc, fn)):
            m = re.match(r'\s*#include "([^"]+)"', line)
            if m and os.path.exists(os.path.join(csrc, m.group(1))):
                visit(m.group(1))

    visit(_KERNEL_SRC[kernel])
    h = hashlib.sha256()
    for fn in order:
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


def _traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(path))
        e = d[f"{kernel}@{workload}"]
        if e.get("src_hash") == _src_hash(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------- decode ---

class DecodeBench:
    """One decode-path workload (n_q <= 16 tokens per sequence) on `replicas`
    rotating device copies of its inputs; a step is one infllmv2_decode_step
    call (one fused launch for n_q = 1, compress + select + attend otherwise)."""

    def __init__(self, dev, seed_offset=0, name=DECODE, replicas=REPLICAS):
        import torch
        import trainable_block_sparse_infllm_gb300 as T
        self.T, self.torch, self.dev = T, torch, dev
        self.name, self.replicas = name, replicas
        wl = S.WORKLOADS[name]
        if seed_offset:
            wl = wl.scaled(seed=wl.seed + 1000 * seed_offset)
        self.wl = wl
        inp = S.make_inputs(wl)
        self.inp = inp
        self.sha256 = inp.sha256()
        self.p = T.make_params(wl.batch, wl.n_kv_heads, wl.kv_len, wl.topk, wl.topk_includes_forced)
        B, H, L, nq = wl.batch, wl.n_kv_heads, wl.kv_len, wl.n_q

        def up(bits):
            return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

        q0, k0, v0 = up(inp.q), up(inp.k), up(inp.v)
        self.lens = torch.from_numpy(inp.kv_lens).to(dev)
        self.kmax = T.max_selected(self.p)
        self.reps = []
        d = wl.head_dim
        nq_el, kv_el = q0.numel(), B * H * nq * d
        for r in range(replicas):
            # One device buffer per replica holds a step's inputs back to back
            # (q, then the new tokens' keys and values), so that the end-to-end
            # leg moves them with one host-to-device copy.
            packed = torch.empty(nq_el + 2 * kv_el, dtype=torch.bfloat16, device=dev)
            packed[:nq_el].copy_(q0.reshape(-1))
            k_new = packed[nq_el:nq_el + kv_el].view(B, H, nq, d)
            v_new = packed[nq_el + kv_el:].view(B, H, nq, d)
            k_new.copy_(k0[:, :, L - nq:L])
            v_new.copy_(v0[:, :, L - nq:L])
            rep = {"q": packed[:nq_el].view(q0.shape), "packed": packed, "k_new": k_new, "v_new": v_new,
                   "k": k0.clone(), "v": v0.clone(), "kc": T.alloc_kc(self.p, dev),
                   "idx": torch.empty((B, H, nq, self.kmax), dtype=torch.int32, device=dev),
                   "nsel": torch.empty((B, H, nq), dtype=torch.int32, device=dev),
                   "out": torch.empty_like(q0),
                   "lse": torch.empty((B, nq, wl.n_heads), dtype=torch.float32, device=dev),
                   "ws_sel": T.alloc_workspace(self.p, nq, T.OP_SELECT, dev),
                   "ws_att": T.alloc_workspace(self.p, nq, T.OP_DECODE, dev),
                   "ws_step": T.alloc_workspace(self.p, nq, T.OP_DECODE_STEP, dev)}
            T.compress_keys(self.p, rep["k"], self.lens, rep["kc"])      # full cache, once
            self.reps.append(rep)
        del q0, k0, v0
        torch.cuda.synchronize()

    # the three stages of one decode step on replica r
    def compress_newest(self, r):
        rep = self.reps[r]
        self.T.compress_keys(self.p, rep["k"], self.lens, rep["kc"], -1, -1)

    def select(self, r):
        rep = self.reps[r]
        self.T.select_blocks(self.p, rep["q"], rep["kc"], self.lens, rep["idx"], rep["nsel"], None,
                             rep["ws_sel"])

    def attend(self, r):
        rep = self.reps[r]
        self.T.sparse_attn_decode(self.p, rep["q"], rep["k"], rep["v"], self.lens, rep["idx"], rep["nsel"],
                                  rep["out"], rep["lse"], rep["ws_att"])

    def step(self, r):
        """One decode step on replica r: a single fused launch."""
        rep = self.reps[r]
        self.T.decode_step(self.p, rep["q"], rep["k"], rep["v"], self.lens, rep["kc"], rep["idx"], rep["nsel"],
                           rep["out"], rep["lse"], rep["ws_step"])

    def capture(self, per_graph=REPLICAS):
        """CUDA graphs: one step per replica, and `per_graph` steps back to
        back over the rotating replicas."""
        torch = self.torch
        R = self.replicas
        for r in range(R):
            self.step(r)                        # warm: module load, attributes, symbols
        torch.cuda.synchronize()
        self.graphs = []                        # one step each (end-to-end leg, remainders)
        for r in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.step(r)
            self.graphs.append(g)
        self.per_graph = per_graph
        self.round = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.round):
            for x in range(per_graph):
                self.step(x % R)
        torch.cuda.synchronize()

    def run_steps(self, n):
        """n steps: whole graphs of per_graph steps, then single steps."""
        for _ in range(n // self.per_graph):
            self.round.replay()
        for x in range(n % self.per_graph):
            self.graphs[x % self.replicas].replay()

    def timed_steps(self, n, warmup):
        """Seconds per step over n steps (CUDA events on the launching stream)."""
        torch = self.torch
        self.run_steps(max(warmup, self.per_graph))
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        self.run_steps(n)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e-3 / n

    def time_fn(self, fn, n, warm=3):
        torch = self.torch
        for i in range(warm):
            fn(i % self.replicas)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(n):
            fn(i % self.replicas)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n * 1e-3     # seconds per call

    def working_set_bytes(self):
        rep = self.reps[0]
        return sum(rep[k].numel() * rep[k].element_size() for k in ("k", "v", "kc", "q"))

    def algorithmic_bytes(self):
        """Bytes a decode step must move: queries, both kernel-mean planes, the
        K and V tiles of the union of the step's selected blocks per (b, h_kv)
        (each block once, however many of the n_q tokens chose it), outputs,
        indices and the newest kernels."""
        wl = self.wl
        B, H, nq, d = wl.batch, wl.n_kv_heads, wl.n_q, wl.head_dim
        n_c = S_n_c(wl.kv_len)
        idx = self.reps[0]["idx"].cpu().numpy()
        nsel = self.reps[0]["nsel"].cpu().numpy()
        union = 0
        for b in range(B):
            for h in range(H):
                blocks = set()
                for t in range(nq):
                    blocks.update(idx[b, h, t, :nsel[b, h, t]].tolist())
                union += len(blocks)
        self.union_blocks = union
        self.selected_blocks = int(nsel.sum())
        q_b = B * nq * wl.n_heads * d * 2
        kc_b = B * H * n_c * d * 4                      # hi + lo planes
        kv_b = union * wl.block * d * 2 * 2             # selected K and V tiles, each block once
        out_b = q_b
        idx_b = B * H * nq * (self.kmax + 1) * 4
        n_new = S_n_c(wl.kv_len) - S_n_c(wl.kv_len - nq)  # kernels ending inside the step's tokens
        comp_b = B * H * n_new * (wl.kernel * d * 2 + d * 4)   # 32 keys in, 512 B out each
        return {"compress": comp_b, "select": kc_b + q_b + idx_b,
                "attend": kv_b + q_b + out_b + idx_b + B * nq * wl.n_heads * 4,
                "step": comp_b + kc_b + q_b * 2 + kv_b + idx_b}


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def S_n_c(L, p=32, s=16):
    return (L - p) // s + 1 if L >= p else 0


# ------------------------------------------------- every decode workload ---

WORKLOAD_TEXT = {
    "decode_4k": "decode_4k: batch 1, 16 q / 1 kv head, 4096-token cache, top-16 incl. forced, 1 query/seq",
    "decode_32k": "decode_32k: batch 8, 32 q / 2 kv heads, 32768-token cache, top-64 incl. forced, 1 query/seq",
    "decode_128k": "decode_128k: batch 4, 32 q / 2 kv heads, 131072-token cache, top-64 incl. forced, 1 query/seq",
    "verify_128k": "verify_128k: batch 4, 32 q / 2 kv heads, 131072-token cache + 8 draft tokens attending "
                   "causally, top-64 per token incl. forced",
    "prefill_32k": "prefill_32k: batch 1, 32 q / 2 kv heads, causal 32768 x 32768, top-64 + init + local",
}


def _l2_bytes(dev):
    import torch
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except Exception:
        return 129 * 2 ** 20


def decode_workload_line(name, dev, steps, warmup, peaks, warm_l2=False, bench=None):
    """tokens/s and the HBM roofline of one decode-path workload.  Inputs
    rotate over enough replicas that every step reads cold HBM (three times
    L2 at least), except where one copy of the working set is already small
    enough that the step is latency-bound, which the line then says; with
    warm_l2 one more figure replays a single replica (labelled)."""
    import torch
    if bench is None:
        wl = S.WORKLOADS[name]
        probe = wl.batch * wl.n_kv_heads * wl.kv_len * wl.head_dim * 2 * 2
        l2 = _l2_bytes(dev)
        reps = 1 if probe * 16 < l2 else min(REPLICAS, max(2, -(-3 * l2 // probe)))
        bench = DecodeBench(dev, name=name, replicas=reps)
        bench.capture(per_graph=max(8, reps))
    wl = bench.wl
    t = bench.timed_steps(steps, warmup)
    ab = bench.algorithmic_bytes()
    ws = bench.working_set_bytes()
    achieved = ab["step"] / t / 1e9
    # The single-launch form of the step is the one that needs no workspace.
    launches = 1 if wl.n_q == 1 and bench.T.workspace_size(bench.p, wl.n_q, bench.T.OP_DECODE_STEP) == 0 else 3
    line = {
        "workload": WORKLOAD_TEXT[name],
        "tokens_per_s": wl.batch * wl.n_q / t,
        "us_per_step": t * 1e6,
        "launches_per_step": launches,
        "l2": (f"{bench.replicas} rotating input replicas ({bench.replicas * ws / 1e9:.2f} GB, "
               f"{bench.replicas * ws / _l2_bytes(dev):.1f}x L2)" if bench.replicas > 1 else
               f"one input copy ({ws / 1e6:.1f} MB, inside L2): latency-bound, cached bytes"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks[0], "unit": "GB/s",
                     "frac": achieved / peaks[0], "peak_kind": peaks[3],
                     "algorithmic_bytes_per_step": ab["step"],
                     "kv_blocks": {"selected": bench.selected_blocks, "union_fetched": bench.union_blocks}},
        "sha256": bench.sha256,
    }
    if warm_l2:
        one = DecodeBench(dev, name=name, replicas=1)
        one.capture(per_graph=8)
        tw = one.timed_steps(steps, warmup)
        line["warm_l2"] = {"tokens_per_s": wl.batch * wl.n_q / tw, "us_per_step": tw * 1e6,
                           "note": "one input copy replayed: the step's 50 MB of kernel means and selected "
                                   "blocks stay in L2 between steps (not a roofline figure)"}
        del one
    return line


# The oracle as it stands, timed on the host: one thread, and every core
# (independent units spread over a spawn process pool, one thread each).

_POOL = {}


def _pool_init(folder, names, wl, st):
    for n in names:
        _POOL[n] = np.load(os.path.join(folder, n + ".npy"), mmap_mode="r")
    _POOL["inp"] = S.Inputs(wl=wl, q=_POOL["q"], k=_POOL["k"], v=_POOL["v"], kv_lens=np.asarray(_POOL["kv_lens"]),
                            planted=np.zeros((wl.batch, wl.n_kv_heads, 0), dtype=np.int64))
    _POOL["st"] = st


def _oracle_units(inp, st, units):
    import oracle as O
    sels = O.run_selection(inp, st, units=units)
    O.run_attention(inp, st, {u: x.blocks for u, x in sels.items()}, units=units)
    return len(units)


def _pool_task(units):
    return _oracle_units(_POOL["inp"], _POOL["st"], units)


def oracle_baseline(name, budget_s=4.0, inp=None):
    """Oracle tokens/s on a bounded sample of the workload: one thread, then
    all host cores.  A token of a sequence is its units over every KV head."""
    import multiprocessing as mp
    import tempfile
    import oracle as O
    wl = S.WORKLOADS[name]
    inp = S.make_inputs(wl) if inp is None else inp
    st = O.Settings(topk=wl.topk, n_init=wl.n_init, n_local=wl.n_local, includes_forced=wl.topk_includes_forced)
    units = [(b, h, t) for b in range(wl.batch) for t in range(wl.n_q) for h in range(wl.n_kv_heads)]
    rng = np.random.default_rng(0)
    order = rng.permutation(len(units))
    # one thread (this process keeps BLAS at one thread)
    t0 = time.perf_counter()
    done = 0
    while done == 0 or (time.perf_counter() - t0 < budget_s and done < len(units)):
        done += _oracle_units(inp, st, [units[order[done % len(units)]]])
    one = done / wl.n_kv_heads / (time.perf_counter() - t0)
    # all cores: as many units per worker as one thread managed in the budget
    cores = os.cpu_count() or 1
    per_worker = max(1, done)
    sample = [units[order[x % len(units)]] for x in range(cores * per_worker)]
    tasks = [sample[w * per_worker:(w + 1) * per_worker] for w in range(cores)]
    with tempfile.TemporaryDirectory() as folder:
        arrays = {"q": inp.q, "k": inp.k, "v": inp.v, "kv_lens": inp.kv_lens}
        for n, a in arrays.items():
            np.save(os.path.join(folder, n + ".npy"), np.ascontiguousarray(a))
        with mp.get_context("spawn").Pool(cores, initializer=_pool_init,
                                          initargs=(folder, list(arrays), wl, st)) as pool:
            pool.map(_pool_task, [[u] for u in sample[:cores]], chunksize=1)   # workers up, inputs mapped
            t1 = time.perf_counter()
            n_all = sum(pool.map(_pool_task, tasks, chunksize=1))
            dt = time.perf_counter() - t1
    allc = n_all / wl.n_kv_heads / dt
    return {"value": allc, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "one_thread": {"value": one, "cores": 1},
            "sample": f"{name}: {done} (one thread) and {n_all} (all cores) of its {len(units)} (b, h_kv, t) units, "
                      f"kernel means + selection + attention in numpy fp64; a token counts its {wl.n_kv_heads} "
                      f"KV-head units"}


# ---------------------------------------------------------------- prefill ---

def prefill_line(dev, steps, warmup, peaks):
    import torch
    import trainable_block_sparse_infllm_gb300 as T
    wl = S.WORKLOADS[PREFILL]
    inp = S.make_inputs(wl)
    p = T.make_params(wl.batch, wl.n_kv_heads, wl.kv_len, wl.topk, wl.topk_includes_forced)

    def up(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = up(inp.q), up(inp.k), up(inp.v)
    lens = torch.from_numpy(inp.kv_lens).to(dev)
    kmax = T.max_selected(p)
    B, H, nq = wl.batch, wl.n_kv_heads, wl.n_q
    kc = T.alloc_kc(p, dev)
    idx = torch.empty((B, H, nq, kmax), dtype=torch.int32, device=dev)
    nsel = torch.empty((B, H, nq), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, nq, wl.n_heads), dtype=torch.float32, device=dev)
    ws_sel = T.alloc_workspace(p, nq, T.OP_SELECT, dev)
    ws_att = T.alloc_workspace(p, nq, T.OP_PREFILL, dev)

    stages = {
        "compress": lambda: T.compress_keys(p, k, lens, kc),
        "select": lambda: T.select_blocks(p, q, kc, lens, idx, nsel, None, ws_sel),
        "attend": lambda: T.sparse_attn_prefill(p, q, k, v, lens, idx, nsel, out, lse, ws_att),
    }

    def timed(fn, n):
        for _ in range(max(warmup, 1)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n * 1e-3

    def full():
        for f in stages.values():
            f()

    t_step = timed(full, steps)
    t_stage = {name: timed(f, steps) for name, f in stages.items()}
    # Algorithmic attention FLOPs from the selection actually made:
    # 4 d per (query head, attended key) pair.
    idx_h, nsel_h = idx.cpu().numpy(), nsel.cpu().numpy()
    pairs = 0
    m = wl.block
    for b in range(B):
        L = int(inp.kv_lens[b])
        pos = L - nq + np.arange(nq)
        for h in range(H):
            rows = idx_h[b, h]
            valid = rows >= 0
            keys = np.where(valid, np.minimum(m, pos[:, None] - rows * m + 1), 0)
            pairs += int(keys.clip(min=0).sum())
    flops = 4.0 * wl.head_dim * pairs * wl.group
    achieved = flops / t_stage["attend"] / 1e12
    issued, split_tiles, n_tiles, union_sum, sel_sum = _prefill_issued_flops(wl, inp.kv_lens, idx_h, nsel_h)

    # The coarse-kernel LSE approximation of the selection (windows of 64
    # keys): its time against the exact selection's, and how many of the
    # exact selection's blocks it keeps.
    sc = 64
    kcc = T.alloc_kcc(p, sc, dev)
    idx_c = torch.empty_like(idx)
    nsel_c = torch.empty_like(nsel)
    t_cmeans = timed(lambda: T.coarse_means(p, k, lens, sc, kcc), steps)
    t_csel = timed(lambda: T.select_blocks_coarse_lse(p, q, kc, sc, kcc, lens, idx_c, nsel_c), steps)
    idx_ch, nsel_ch = idx_c.cpu().numpy(), nsel_c.cpu().numpy()
    kept = total = 0
    for b in range(B):
        for h in range(H):
            for t_ in range(nq):
                e = set(idx_h[b, h, t_, :nsel_h[b, h, t_]].tolist())
                c = set(idx_ch[b, h, t_, :nsel_ch[b, h, t_]].tolist())
                kept += len(e & c)
                total += len(e)
    coarse = {"window": sc, "select_ms": t_csel * 1e3, "coarse_means_ms": t_cmeans * 1e3,
              "select_speedup": t_stage["select"] / t_csel, "selection_overlap": kept / max(total, 1)}

    # Backward of the attention with this selection held fixed (dq, dk, dv in
    # fp32 for a seeded upstream gradient).  Algorithmic FLOPs: five products
    # of 2 d per (query head, attended key) pair (q K^T, dO V^T, dS K, dS^T q,
    # P^T dO); the kernels recompute q K^T and dO V^T once more each.
    dout = up(S.make_grad_out(wl, seed=wl.seed + 2000))
    dq = torch.empty((B, nq, wl.n_heads, wl.head_dim), dtype=torch.float32, device=dev)
    dk = torch.empty((B, H, wl.kv_len, wl.head_dim), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    ws_bwd = T.alloc_workspace(p, nq, T.OP_BACKWARD, dev)
    t_bwd = timed(lambda: T.sparse_attn_backward(p, q, k, v, lens, idx, nsel, out, lse, dout, dq, dk, dv, ws_bwd),
                  steps)
    bflops = 10.0 * wl.head_dim * pairs * wl.group
    b_achieved = bflops / t_bwd / 1e12
    backward = {"ms": t_bwd * 1e3, "tokens_per_s": B * nq / t_bwd,
                "kernels": "index (count, scan, fill), bwd_dq_kernel (mma.sync), bwd_dkdv_kernel (tcgen05)",
                "roofline": {"bound": "tensor", "achieved": b_achieved, "peak": peaks[1], "unit": "TFLOP/s",
                             "frac": b_achieved / peaks[1], "peak_kind": peaks[3] + " burst bf16",
                             "algorithmic_flop_per_call": bflops}}
    return {
        "workload": f"{PREFILL}: batch 1, 32 q / 2 kv heads, causal 32768 x 32768, top-64 + init + local",
        "tokens_per_s": B * nq / t_step,
        "ms_per_step": t_step * 1e3,
        "stage_ms": {k_: v_ * 1e3 for k_, v_ in t_stage.items()},
        "roofline": {"kernel": "attn_tc_kernel (sparse_attn_prefill)", "bound": "tensor",
                     "achieved": achieved, "peak": peaks[1], "unit": "TFLOP/s",
                     "frac": achieved / peaks[1], "peak_kind": peaks[3] + " burst bf16",
                     "algorithmic_flop_per_launch": flops, "traffic": _traffic("attn_tc_kernel", PREFILL),
                     "issued": {"flop_per_launch": issued, "tflops": issued / t_stage["attend"] / 1e12,
                                "frac": issued / t_stage["attend"] / 1e12 / peaks[1],
                                "issued_over_useful": issued / flops,
                                "union_over_selected_blocks": union_sum / max(sel_sum, 1),
                                "tiles_with_hi_lo_probabilities": f"{split_tiles} of {n_tiles}",
                                "note": "tcgen05 products the kernel issues: S and O += P V over the union of each "
                                        "8-token tile's blocks, two blocks per item (a lone last block is issued "
                                        "as a pair), a second P V product in tiles fed hi + lo probabilities"}},
        "coarse_lse": coarse,
        "backward": backward,
    }


def _prefill_issued_flops(wl, kv_lens, idx_h, nsel_h, tile=8, split_keys=2048):
    """MMA FLOPs the prefill kernel issues for this selection: per tile of
    `tile` tokens x 16 heads (128 rows), ceil(|union| / 2) items of 128 keys,
    each an S product and a P V product of 2 * 128 * 128 * 128 FLOPs, plus a
    second P V product in tiles where some token attends < split_keys keys."""
    B, H, nq, m = wl.batch, wl.n_kv_heads, wl.n_q, wl.block
    item = 2.0 * 128 * 128 * 128
    issued, split_tiles, n_tiles, union_sum, sel_sum = 0.0, 0, 0, 0, 0
    nbmax = -(-wl.kv_len // m)
    for b in range(B):
        L = int(kv_lens[b])
        pos = L - nq + np.arange(nq)
        for h in range(H):
            rows = idx_h[b, h]
            valid = (np.arange(rows.shape[1])[None, :] < nsel_h[b, h][:, None]) & (rows >= 0)
            keys = np.where(valid, np.minimum(m, pos[:, None] - rows * m + 1), 0).clip(min=0).sum(axis=1)
            nt = -(-nq // tile)
            mask = np.zeros((nt, nbmax), dtype=bool)
            tok = np.broadcast_to(np.arange(nq)[:, None], rows.shape)
            mask[(tok[valid] // tile), rows[valid]] = True
            union = mask.sum(axis=1)
            tile_min_keys = np.full(nt, np.iinfo(np.int64).max)
            np.minimum.at(tile_min_keys, np.arange(nq) // tile, keys)
            split = tile_min_keys < split_keys
            items = -(-union // 2)
            issued += float(items.sum()) * item * 2 + float(items[split].sum()) * item
            split_tiles += int(split.sum())
            n_tiles += nt
            union_sum += int(union.sum())
            sel_sum += int(valid.sum())
    return issued, split_tiles, n_tiles, union_sum * tile, sel_sum


# ----------------------------------------------------------- CPU baseline ---

def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle as O
    wl = S.WORKLOADS[DECODE]
    inp = S.make_inputs(wl)
    st = O.Settings(topk=wl.topk, includes_forced=wl.topk_includes_forced)

    def one_step(i):
        b = i % wl.batch
        units = [(b, h, t) for h in range(wl.n_kv_heads) for t in range(wl.n_q)]
        sels = O.run_selection(inp, st, units=units)
        O.run_attention(inp, st, {u: s.blocks for u, s in sels.items()}, units=units)

    for i in range(args.warmup):
        one_step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one_step(i)
    dt = time.perf_counter() - t0
    value = args.steps * wl.n_q / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": f"{DECODE} (one sequence per step)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": "one sequence (both KV heads) of decode_128k per step, "
                                       "single-threaded numpy fp64"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- profile ---

def profile_passes(path, n):
    """n passes of one path on a single input copy, nothing timed: the decode
    path is one decode_step launch per pass (decode_128k, 0.57 GB of inputs),
    the verify path one three-stage decode step of verify_128k (0.57 GB);
    the prefill path is compress + select + attention (prefill_32k); the
    backward path is one forward, then n backward calls (prefill_32k).  The
    *8k variants run the prefill workload cut to 8192 tokens."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import trainable_block_sparse_infllm_gb300 as T
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    wl = S.WORKLOADS[{"decode": DECODE, "verify": "verify_128k"}.get(path, PREFILL)]
    if path.endswith("8k"):
        # The prefill workload cut to an 8192-token causal prefill (inputs of
        # ~150 MB, above L2): a case small enough for full ncu captures.
        wl = wl.scaled(kv_len=8192, n_q=8192)
        path = path[:-2]
    inp = S.make_inputs(wl)
    p = T.make_params(wl.batch, wl.n_kv_heads, wl.kv_len, wl.topk, wl.topk_includes_forced)

    def up(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = up(inp.q), up(inp.k), up(inp.v)
    lens = torch.from_numpy(inp.kv_lens).to(dev)
    B, H, nq = wl.batch, wl.n_kv_heads, wl.n_q
    kmax = T.max_selected(p)
    kc = T.alloc_kc(p, dev)
    idx = torch.empty((B, H, nq, kmax), dtype=torch.int32, device=dev)
    nsel = torch.empty((B, H, nq), dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, nq, wl.n_heads), dtype=torch.float32, device=dev)
    T.compress_keys(p, k, lens, kc)
    if path in ("decode", "verify"):
        ws = T.alloc_workspace(p, nq, T.OP_DECODE_STEP, dev)
        for _ in range(n):
            T.decode_step(p, q, k, v, lens, kc, idx, nsel, out, lse, ws)
    elif path == "backward":
        ws_sel = T.alloc_workspace(p, nq, T.OP_SELECT, dev)
        ws_att = T.alloc_workspace(p, nq, T.OP_PREFILL, dev)
        T.select_blocks(p, q, kc, lens, idx, nsel, None, ws_sel)
        T.sparse_attn_prefill(p, q, k, v, lens, idx, nsel, out, lse, ws_att)
        dout = up(S.make_grad_out(wl, seed=wl.seed + 2000))
        dq = torch.empty((B, nq, wl.n_heads, wl.head_dim), dtype=torch.float32, device=dev)
        dk = torch.empty((B, H, wl.kv_len, wl.head_dim), dtype=torch.float32, device=dev)
        dv = torch.empty_like(dk)
        ws_bwd = T.alloc_workspace(p, nq, T.OP_BACKWARD, dev)
        for _ in range(n):
            T.sparse_attn_backward(p, q, k, v, lens, idx, nsel, out, lse, dout, dq, dk, dv, ws_bwd)
    else:
        ws_sel = T.alloc_workspace(p, nq, T.OP_SELECT, dev)
        ws_att = T.alloc_workspace(p, nq, T.OP_PREFILL, dev)
        for _ in range(n):
            T.compress_keys(p, k, lens, kc)
            T.select_blocks(p, q, kc, lens, idx, nsel, None, ws_sel)
            T.sparse_attn_prefill(p, q, k, v, lens, idx, nsel, out, lse, ws_att)
    torch.cuda.synchronize()
    assert T.get_device_status(clear=True) == 0
    print(f"profile passes done: {path} x {n}")
    return 0


# ------------------------------------------------------------------- main ---

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="headline workload and prefill only")
    ap.add_argument("--profile", choices=["decode", "verify", "prefill", "backward", "prefill8k", "backward8k"],
                    help="run warmup + steps untimed passes of one path on one input copy and exit "
                         "(a small, fixed launch sequence for ncu)")
    args = ap.parse_args()
    if args.profile:
        return profile_passes(args.profile, args.warmup + args.steps)
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import __graft_entry__
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if rank == 0 or world == 1:
        __graft_entry__.build()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        if rank != 0:
            __graft_entry__.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    import trainable_block_sparse_infllm_gb300 as T
    peaks = _peaks()

    bench = DecodeBench(dev, seed_offset=rank)
    bench.capture()
    wl = bench.wl
    tokens_per_step = wl.batch * wl.n_q

    # Per-stage durations (each stage alone, rotating replicas).
    stage_t = {"compress": bench.time_fn(bench.compress_newest, args.steps),
               "select": bench.time_fn(bench.select, args.steps),
               "attend": bench.time_fn(bench.attend, args.steps)}

    # Timed region: exactly K steps (graph replays).
    bench.run_steps(max(args.warmup, REPLICAS))
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = Clocks(local)
    clocks.start()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record()
    bench.run_steps(args.steps)
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - w0
    if dist:
        dist.barrier()
    clk = clocks.stop()
    t = max_over_ranks(e0.elapsed_time(e1) * 1e-3, dist, dev)
    assert T.get_device_status(clear=True) == 0, "device status flagged during the bench"

    # End to end through the public API with host buffers: per step the new
    # token's q, k, v come from pinned host memory (k, v appended to the
    # cache) and the attention output goes back to pinned host memory.  Each
    # step is one launch of infllmv2_append_decode_step, which reads q, k and v
    # from pinned host memory, writes k and v into the caches and stores its
    # output into pinned host memory.  Steps are batched into CUDA graphs
    # exactly as in the device-timed leg: one graph of REPLICAS steps over the
    # rotating replicas (single-step graphs for a remainder).  A graph per step
    # would add its own launch (about 4.6 us on this path) to every step.
    B, H, nq, d = wl.batch, wl.n_kv_heads, wl.n_q, wl.head_dim
    in_h = torch.empty((REPLICAS, bench.reps[0]["packed"].numel()), dtype=torch.bfloat16).pin_memory()
    out_h = torch.empty((REPLICAS,) + tuple(bench.reps[0]["out"].shape), dtype=torch.bfloat16).pin_memory()
    for r in range(REPLICAS):
        in_h[r].copy_(bench.reps[r]["packed"])
    torch.cuda.synchronize()
    nq_el, kv_el = bench.reps[0]["q"].numel(), bench.reps[0]["k_new"].numel()

    def e2e_one(r):
        rep = bench.reps[r]
        q_h = in_h[r][:nq_el].view(rep["q"].shape)
        k_h = in_h[r][nq_el:nq_el + kv_el].view(rep["k_new"].shape)
        v_h = in_h[r][nq_el + kv_el:].view(rep["v_new"].shape)
        T.append_decode_step(bench.p, q_h, k_h, v_h, rep["k"], rep["v"], bench.lens, rep["kc"], rep["idx"],
                             rep["nsel"], out_h[r], None)

    graphs_e2e = []
    for r in range(REPLICAS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e2e_one(r)
        graphs_e2e.append(g)
    round_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(round_e2e):
        for r in range(REPLICAS):
            e2e_one(r)
    torch.cuda.synchronize()

    def e2e_steps(n):
        for _ in range(n // REPLICAS):
            round_e2e.replay()
        for x in range(n % REPLICAS):
            graphs_e2e[x].replay()

    e2e_steps(max(args.warmup, REPLICAS))
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record()
    e2e_steps(args.steps)
    f1.record()
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(f0.elapsed_time(f1) * 1e-3, dist, dev)

    prefill = None
    if not args.no_prefill and rank == 0:
        prefill = prefill_line(dev, max(3, min(10, args.steps // 20)), 3, peaks)

    # Every other workload on its own, and decode_128k's warm-L2 figure.
    workloads = {}
    if rank == 0 and not args.no_workloads:
        n_w = max(20, min(200, args.steps))
        workloads[DECODE] = decode_workload_line(DECODE, dev, n_w, args.warmup, peaks, warm_l2=True, bench=bench)
        for name in ("decode_4k", "decode_32k", "verify_128k"):
            workloads[name] = decode_workload_line(name, dev, n_w, args.warmup, peaks)
            torch.cuda.empty_cache()
        assert T.get_device_status(clear=True) == 0, "device status flagged during the workload lines"

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    ab = bench.algorithmic_bytes()
    # The step is one launch of decode_step_kernel: its average duration is
    # the timed region over K.
    t_launch = t / args.steps
    achieved = ab["step"] / t_launch / 1e9
    value = world * tokens_per_step * args.steps / t
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{DECODE}: batch 4, 32 q / 2 kv heads, head_dim 128, 131072-token bf16 "
                               f"KV cache, block 64, kernel 32/16, top-64 incl. block 0 + 2 local, 1 query/seq",
                   "global_batch": world * wl.batch, "seq_len": wl.kv_len, "parallelism": f"dp{world}",
                   "l2": f"{REPLICAS} rotating input replicas ({REPLICAS * 0.57:.1f} GB) > L2",
                   "graph": f"decode_step (newest kernel + select + attention, one launch per step), "
                            f"{REPLICAS} steps per CUDA graph"},
        "clocks": clk,
        "gpu_launches": args.steps,
        "unfused_stage_ms": {k_: v_ * 1e3 for k_, v_ in stage_t.items()},
        "roofline": {"kernel": "decode_step_kernel", "bound": "hbm", "achieved": achieved, "peak": peaks[0],
                     "unit": "GB/s", "frac": achieved / peaks[0], "peak_kind": peaks[3],
                     "algorithmic_bytes_per_launch": ab["step"],
                     "traffic": _traffic("decode_step_kernel", DECODE)},
        "e2e": {"value": world * tokens_per_step * args.steps / t_e2e, "unit": "tokens/s",
                "h2d_bytes_per_step": int(in_h[0].numel() * 2),
                "d2h_bytes_per_step": int(out_h[0].numel() * 2), "wall_s": wall,
                "transfers": "one launch per step (infllmv2_append_decode_step): it reads q, k, v from pinned host "
                             "memory, appends k, v to the caches and stores its output there",
                "graph": f"{REPLICAS} steps per CUDA graph as in the device-timed leg"},
        "prefill": prefill,
    }
    line["workloads"] = workloads
    if world == 1 and not args.no_cpu_baseline:
        for name in list(workloads) + ([PREFILL] if prefill else []):
            cb = oracle_baseline(name)
            (prefill if name == PREFILL else workloads[name])["cpu_baseline"] = cb
            if name == DECODE:
                line["cpu_baseline"] = cb
        if DECODE not in workloads:
            line["cpu_baseline"] = oracle_baseline(DECODE)
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
