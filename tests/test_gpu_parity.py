"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Every test here needs an sm_103a GPU and the built library.  Small cases span
several tiles of every kernel and ragged tails; the workload tests run the
benchmark's own launch configuration at full size and compare every decode
unit (prefill: a stratified sample of query tokens).
"""

import math

import numpy as np
import pytest

import oracle as O
import synthetic_inputs as S
from helpers import (ATT_MAX, ATT_MEAN, LSE_ABS, STRICT_MIN_KEYS, DeviceRun, bf16_half_ulp, check_attention,
                     check_selections, kc_to_f64, strict_units)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__
    __graft_entry__.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    import trainable_block_sparse_infllm_gb300 as T
    T.get_device_status(clear=True)
    yield d
    torch.cuda.synchronize()
    assert T.get_device_status(clear=True) == 0


def _settings(wl, score_scale=None, attn_scale=None):
    return O.Settings(topk=wl.topk, n_init=wl.n_init, n_local=wl.n_local,
                      includes_forced=wl.topk_includes_forced, score_scale=score_scale,
                      attn_scale=attn_scale)


# ------------------------------------------------------------- stage 1 ----

def test_compress_keys_ragged(dev):
    import torch
    inp = S.make_random(batch=3, n_kv_heads=2, kv_len=5000, n_q=1, topk=8, seed=21,
                        kv_lens=[5000, 4093, 31])
    run = DeviceRun(inp, dev)
    run.kc.view(torch.int16).fill_(0x7FC0)       # NaN sentinel: untouched rows stay NaN
    run.compress()
    torch.cuda.synchronize()
    got = kc_to_f64(run.kc)
    st = O.Settings()
    for b in range(3):
        for h in range(2):
            ref = O.kc_for(inp, b, h, st)
            n = ref.shape[0]
            err = np.abs(got[b, h, :n] - ref)
            assert np.all(err <= 2.0 ** -16 * np.abs(ref) + 1e-9), (b, h, float(err.max()))
            assert np.all(np.isnan(got[b, h, n:])), (b, h)


def test_compress_keys_incremental_ranges(dev):
    import torch
    inp = S.make_random(batch=2, n_kv_heads=1, kv_len=3000, n_q=1, topk=8, seed=22, kv_lens=[3000, 2222])
    run = DeviceRun(inp, dev)
    run.compress()
    full = run.kc.clone()
    run.kc.view(torch.int16).fill_(0x7FC0)
    run.compress(0, 50)
    run.compress(50, 100)
    run.compress(100, -1)
    assert torch.equal(run.kc.view(torch.int16)[:, :, :, :137], full.view(torch.int16)[:, :, :, :137])
    # -1: only the newest complete kernel of each sequence
    run.kc.view(torch.int16).fill_(0x7FC0)
    run.compress(-1, -1)
    for b, L in enumerate(inp.kv_lens):
        n = O.n_complete_kernels(int(L), 32, 16)
        assert torch.equal(run.kc[b, :, :, n - 1], full[b, :, :, n - 1])
        assert torch.isnan(run.kc[b, :, :, : n - 1].float()).all()


# ------------------------------------------------------------- stage 2 ----

SELECT_CASES = [
    # batch, hkv, cap, lens, n_q, topk, includes_forced, score_scale
    (2, 2, 5000, [5000, 3333], 1, 16, True, None),
    (1, 2, 9000, [9000], 1, 64, True, None),
    (2, 1, 4100, [4100, 2000], 3, 12, True, 1.0),
    (1, 2, 6000, [6000], 8, 24, True, None),
    (2, 1, 3000, [3000, 1500], 16, 10, False, None),
    (1, 2, 2600, [2600], 17, 16, True, None),          # smallest prefill-path n_q
    (2, 1, 2000, [2000, 1234], 130, 8, False, None),
    (1, 1, 700, [700], 700, 4, True, None),             # whole sequence from position 0
    (3, 1, 300, [300, 40, 20], 20, 4, True, 1.0),       # tiny contexts, no visible kernel
    (2, 1, 200, [64, 33], 1, 3, True, None),
    # Few tiles on long caches: each tile's chunks split over a cluster of up
    # to 16 CTAs; the short sequence leaves most of its cluster without chunks.
    (2, 2, 40000, [40000, 9000], 5, 32, True, None),
    (1, 2, 30000, [30000], 12, 64, False, None),        # a partial second tile
    (1, 1, 20000, [20000], 40, 16, False, None),        # prefill-path n_q
    # Short caches cap the cluster: 3 CTAs (each owning 3 tokens' score
    # rows) and 2 CTAs (4 rows each).
    (4, 2, 6000, [6000, 5000, 4100, 3000], 24, 16, True, None),
    (2, 2, 4500, [4500, 2600], 20, 12, False, None),
    # 80 tiles (no cluster) with 1563 blocks of scores per token: too many for
    # two CTAs per SM, so one CTA per SM with a three-chunk ring.
    (1, 2, 100000, [100000], 320, 32, False, None),
]


@pytest.mark.parametrize("case", SELECT_CASES, ids=[f"sel{i}" for i in range(len(SELECT_CASES))])
def test_select_blocks_parity(dev, case):
    import torch
    B, H, cap, lens, nq, topk, inc, sscale = case
    inp = S.make_random(batch=B, n_kv_heads=H, kv_len=cap, n_q=nq, topk=topk, includes_forced=inc,
                        seed=100 + sum(lens) + nq, kv_lens=lens)
    run = DeviceRun(inp, dev, score_scale=sscale)
    run.compress()
    run.select()
    torch.cuda.synchronize()
    sels = O.run_selection(inp, _settings(inp.wl, score_scale=sscale))
    check_selections(run, sels)


def test_prefill_selection_past_on_chip_capacity(dev):
    # 340,000 tokens of capacity (5313 blocks): past the 5115 blocks whose 8
    # tokens' block scores fit in shared memory, the prefill-path selection
    # keeps them in one workspace slot per SM.  Ragged lengths; the selection
    # (with its scores) and the attention on it against the oracle.
    import torch
    inp = S.make_random(batch=2, n_kv_heads=2, kv_len=340000, n_q=24, topk=48, includes_forced=False, seed=91,
                        kv_lens=[340000, 151000])
    run = DeviceRun(inp, dev)
    assert run.T.workspace_size(run.p, 24, run.T.OP_SELECT) > 0
    run.compress()
    run.select()
    torch.cuda.synchronize()
    st = _settings(inp.wl)
    sels = O.run_selection(inp, st)
    check_selections(run, sels)
    idx, nsel = run.upload_selection(sels)
    run.attend(idx, nsel)
    torch.cuda.synchronize()
    blocks_of = {u: s.blocks for u, s in sels.items()}
    refs = O.run_attention(inp, st, blocks_of)
    check_attention(run, refs, strict=True, strict_units=strict_units(inp, blocks_of))


def test_select_blocks_dense_when_context_short(dev):
    import torch
    inp = S.make_random(batch=1, n_kv_heads=2, kv_len=1024, n_q=4, topk=16, seed=5)
    run = DeviceRun(inp, dev)
    run.compress()
    run.select()
    torch.cuda.synchronize()
    nsel = run.nsel.cpu().numpy()
    idx = run.idx.cpu().numpy()
    for t in range(4):
        assert np.all(nsel[0, :, t] == 16)
        assert np.array_equal(idx[0, 0, t], np.arange(16))


# ------------------------------------------------------------- stage 3 ----

ATTN_CASES = [
    # batch, hkv, cap, lens, n_q, topk, includes_forced, prefill
    (2, 2, 5000, [5000, 3333], 1, 16, True, False),
    (1, 2, 9000, [9000], 1, 64, True, False),
    (2, 1, 4100, [4100, 2100], 5, 12, True, False),
    (1, 2, 6000, [6000], 16, 24, True, False),
    (2, 1, 3000, [3000, 1500], 16, 10, False, True),
    (2, 1, 2000, [2000, 1234], 130, 8, False, True),
    (1, 1, 700, [700], 700, 4, True, True),
    (3, 1, 300, [300, 40, 20], 20, 4, True, True),
    # Few tiles on long caches: each tile's union split over a cluster of up
    # to 16 CTAs (a partial last tile, ragged lengths).
    (1, 2, 9000, [9000], 8, 64, True, True),
    (2, 2, 20000, [20000, 7000], 13, 48, False, True),
]


@pytest.mark.parametrize("case", ATTN_CASES, ids=[f"att{i}" for i in range(len(ATTN_CASES))])
def test_sparse_attention_parity(dev, case):
    import torch
    B, H, cap, lens, nq, topk, inc, prefill = case
    inp = S.make_random(batch=B, n_kv_heads=H, kv_len=cap, n_q=nq, topk=topk, includes_forced=inc,
                        seed=200 + sum(lens) + nq, kv_lens=lens)
    st = _settings(inp.wl)
    sels = O.run_selection(inp, st)
    run = DeviceRun(inp, dev)
    idx, nsel = run.upload_selection(sels)
    run.attend(idx, nsel, prefill=prefill)
    torch.cuda.synchronize()
    blocks_of = {u: s.blocks for u, s in sels.items()}
    refs = O.run_attention(inp, st, blocks_of)
    check_attention(run, refs, strict=True, strict_units=strict_units(inp, blocks_of))


def test_attention_dense_degeneracy_matches_sdpa(dev):
    # topk covering every block: the output is plain causal attention.
    import torch
    inp = S.make_random(batch=1, n_kv_heads=1, kv_len=900, n_q=900, topk=15, seed=7)
    run = DeviceRun(inp, dev)
    run.compress()
    run.select()
    run.attend()
    torch.cuda.synchronize()
    q = torch.from_numpy(S.bf16_bits_to_f32(inp.q[0])).double().permute(1, 0, 2)[None]
    k = torch.from_numpy(S.bf16_bits_to_f32(inp.k[0, 0])).double()[None, None].expand(1, 16, 900, 128)
    v = torch.from_numpy(S.bf16_bits_to_f32(inp.v[0, 0])).double()[None, None].expand(1, 16, 900, 128)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)[0].permute(1, 0, 2)
    err = (run.out[0].double().cpu() - ref).abs().numpy()
    # The rule of helpers.check_attention: 2e-3 / 2e-4 plus what the bf16
    # output format forces (half an ulp of each stored value), and the bare
    # rule for the queries that attend at least 256 keys.
    allow = bf16_half_ulp(np.abs(ref.numpy()) + ATT_MAX)
    assert np.all(err <= ATT_MAX + allow), float((err - allow).max())
    assert err.mean() <= ATT_MEAN + allow.mean()
    late = err[STRICT_MIN_KEYS - 1:]
    assert late.max() <= ATT_MAX and late.mean() <= ATT_MEAN, (float(late.max()), float(late.mean()))


def test_split_count_does_not_change_decode_result(dev):
    # Same unit through the decode (split + merge) and prefill (single CTA)
    # entry points: the merge identity makes them agree to rounding.
    import torch
    inp = S.make_random(batch=2, n_kv_heads=2, kv_len=8000, n_q=4, topk=48, seed=9)
    st = _settings(inp.wl)
    sels = O.run_selection(inp, st)
    run = DeviceRun(inp, dev)
    idx, nsel = run.upload_selection(sels)
    run.attend(idx, nsel, prefill=False)
    a = run.out.float().clone()
    run.attend(idx, nsel, prefill=True)
    torch.cuda.synchronize()
    assert (a - run.out.float()).abs().max().item() <= 2e-3


def test_bad_kv_len_sets_device_status(dev):
    import torch
    import trainable_block_sparse_infllm_gb300 as T
    inp = S.make_random(batch=2, n_kv_heads=1, kv_len=1000, n_q=2, topk=4, seed=3, kv_lens=[1000, 1])
    run = DeviceRun(inp, dev)
    run.compress()
    run.select()
    run.attend()
    torch.cuda.synchronize()
    assert T.get_device_status(clear=True) & T.DEVICE_BAD_KV_LEN
    assert run.nsel[1].eq(0).all().item()
    assert run.out[1].float().eq(0).all().item()


# ------------------------------------------------------ fused decode step ----

STEP_CASES = [
    # batch, hkv, cap, lens, n_q, topk, includes_forced
    (2, 2, 5000, [5000, 3333], 1, 16, True),
    (1, 2, 9000, [9000], 1, 64, True),
    (3, 1, 4200, [4192, 4177, 4100], 1, 16, True),    # 4192 completes a kernel
    (2, 2, 20000, [20000, 17], 1, 32, False),          # second sequence has no kernel
    (3, 1, 300, [300, 40, 33], 1, 4, True),
    (2, 1, 200, [64, 1], 1, 3, True),                  # a one-token sequence
    (1, 2, 6000, [6000], 8, 24, True),                 # n_q > 1: the three stages in order
]


@pytest.mark.parametrize("case", STEP_CASES, ids=[f"step{i}" for i in range(len(STEP_CASES))])
def test_decode_step_parity(dev, case):
    import torch
    B, H, cap, lens, nq, topk, inc = case
    inp = S.make_random(batch=B, n_kv_heads=H, kv_len=cap, n_q=nq, topk=topk, includes_forced=inc,
                        seed=300 + sum(lens) + nq, kv_lens=lens)
    st = _settings(inp.wl)
    run = DeviceRun(inp, dev)
    full = run.blank_step_kernels()
    run.step()
    torch.cuda.synchronize()
    # The recomputed kernel means are bit-identical to the compression kernel's.
    assert torch.equal(run.kc.view(torch.int16), full.view(torch.int16))
    sels = O.run_selection(inp, st)
    check_selections(run, sels, check_scores=False)
    got = run.gpu_blocks(sels.keys())
    refs = O.run_attention(inp, st, got)
    check_attention(run, refs, strict=True, strict_units=strict_units(inp, got))


def test_decode_step_matches_separate_stages(dev):
    # Same inputs through the single launch and through the three entry
    # points: identical selections (no tie-band case here) and outputs equal
    # to rounding.
    import torch
    inp = S.make_random(batch=2, n_kv_heads=2, kv_len=30000, n_q=1, topk=48, seed=41, kv_lens=[30000, 12345])
    run = DeviceRun(inp, dev)
    run.compress()
    run.select(with_scores=False)
    run.attend()
    idx_a, out_a, lse_a = run.idx.clone(), run.out.float().clone(), run.lse.clone()
    run.idx.fill_(-7)
    run.out.fill_(float("nan"))
    run.step()
    torch.cuda.synchronize()
    assert torch.equal(idx_a, run.idx)
    assert (out_a - run.out.float()).abs().max().item() <= 2e-3
    assert (lse_a - run.lse).abs().max().item() <= 1e-3


def test_decode_step_bad_kv_len(dev):
    import torch
    import trainable_block_sparse_infllm_gb300 as T
    inp = S.make_random(batch=2, n_kv_heads=1, kv_len=1000, n_q=1, topk=4, seed=3, kv_lens=[1000, 900])
    run = DeviceRun(inp, dev)
    run.compress()
    run.lens[1] = 1001                      # beyond max_kv_len
    run.step()
    torch.cuda.synchronize()
    assert T.get_device_status(clear=True) & T.DEVICE_BAD_KV_LEN
    assert run.nsel[1].eq(0).all().item()
    assert run.idx[1].eq(-1).all().item()
    assert run.out[1].float().eq(0).all().item()
    assert run.nsel[0].eq(4).all().item()


def test_append_decode_step_one_launch_long_cache(dev):
    # The same check on a 131,072-token cache, where the step runs as
    # clusters of up to 16 CTAs: the appended key and value are stored by
    # CTA 0 and read by whichever CTA attends the local block.  Pinned host
    # inputs; the newest kernel ends on the appended key for the first
    # sequence (131072) and not for the second (99999).
    import torch
    import trainable_block_sparse_infllm_gb300 as T
    inp = S.make_random(batch=2, n_kv_heads=2, kv_len=131072, n_q=1, topk=64, seed=58,
                        kv_lens=[131072, 99999])
    run = DeviceRun(inp, dev)
    full_k, full_v = run.k.clone(), run.v.clone()
    kc_full = run.blank_step_kernels()
    run.step()
    torch.cuda.synchronize()
    out_ref, idx_ref = run.out.clone(), run.idx.clone()
    k_new = torch.stack([full_k[b, :, int(L) - 1:int(L)] for b, L in enumerate(inp.kv_lens)]).cpu().pin_memory()
    v_new = torch.stack([full_v[b, :, int(L) - 1:int(L)] for b, L in enumerate(inp.kv_lens)]).cpu().pin_memory()
    q = run.q.cpu().pin_memory()
    out = torch.empty(run.out.shape, dtype=torch.bfloat16).pin_memory()
    run.blank_step_kernels()
    for b, L in enumerate(inp.kv_lens):
        run.k[b, :, int(L) - 1].view(torch.int16).fill_(0x7FC0)
        run.v[b, :, int(L) - 1].view(torch.int16).fill_(0x7FC0)
    run.idx.fill_(-7)
    T.append_decode_step(run.p, q, k_new, v_new, run.k, run.v, run.lens, run.kc, run.idx, run.nsel, out)
    torch.cuda.synchronize()
    assert T.get_device_status(clear=True) == 0
    assert torch.equal(run.k.view(torch.int16), full_k.view(torch.int16))
    assert torch.equal(run.v.view(torch.int16), full_v.view(torch.int16))
    assert torch.equal(run.kc.view(torch.int16), kc_full.view(torch.int16))
    assert torch.equal(run.idx, idx_ref)
    assert torch.equal(out.to(dev).view(torch.int16), out_ref.view(torch.int16))


def test_append_decode_step_bad_kv_len(dev):
    # A sequence whose kv_len lies past max_kv_len: status flagged, its caches
    # untouched, an empty selection and a zero output; the other sequence's
    # row is appended.
    import torch
    import trainable_block_sparse_infllm_gb300 as T
    inp = S.make_random(batch=2, n_kv_heads=1, kv_len=1000, n_q=1, topk=4, seed=4, kv_lens=[1000, 900])
    run = DeviceRun(inp, dev)
    run.compress()
    k0, v0 = run.k.clone(), run.v.clone()
    k_new = torch.randn((2, 1, 1, 128), device=dev).to(torch.bfloat16)
    v_new = torch.randn((2, 1, 1, 128), device=dev).to(torch.bfloat16)
    run.lens[1] = 1001
    out = torch.full_like(run.out, float("nan"))
    T.append_decode_step(run.p, run.q, k_new, v_new, run.k, run.v, run.lens, run.kc, run.idx, run.nsel, out)
    torch.cuda.synchronize()
    assert T.get_device_status(clear=True) & T.DEVICE_BAD_KV_LEN
    assert torch.equal(run.k[1].view(torch.int16), k0[1].view(torch.int16))
    assert torch.equal(run.v[1].view(torch.int16), v0[1].view(torch.int16))
    assert run.nsel[1].eq(0).all().item() and run.idx[1].eq(-1).all().item()
    assert out[1].float().eq(0).all().item()
    assert torch.equal(run.k[0, :, 999].view(torch.int16), k_new[0, :, 0].view(torch.int16))
    assert torch.equal(run.v[0, :, 999].view(torch.int16), v_new[0, :, 0].view(torch.int16))
    assert torch.isfinite(out[0].float()).all().item()


# --------------------------------------------------------- full workloads ----

@pytest.mark.parametrize("name", ["decode_4k", "decode_32k", "decode_128k", "verify_128k"])
def test_workload_parity(dev, name):
    # Every unit of the workload, in the benchmark's launch configuration.
    import torch
    wl = S.WORKLOADS[name]
    inp = S.make_inputs(wl)
    st = _settings(wl)
    run = DeviceRun(inp, dev)
    run.compress()
    run.select()
    run.attend()
    torch.cuda.synchronize()
    units = [(b, h, t) for b in range(wl.batch) for h in range(wl.n_kv_heads) for t in range(wl.n_q)]
    kc_cache = {}
    sels = O.run_selection(inp, st, units=units, kc_cache=kc_cache)
    ties = check_selections(run, sels, check_scores=False)
    if name in ("decode_4k", "decode_32k"):
        # Free slots >= planted blocks: every planted block is selected.
        idx = run.idx.cpu().numpy()
        for (b, h, t) in units:
            assert set(inp.planted[b, h].tolist()) <= set(idx[b, h, t].tolist())
    # Attention on the oracle's selection.
    idx, nsel = run.upload_selection(sels)
    run.out.fill_(float("nan"))
    run.attend(idx, nsel)
    torch.cuda.synchronize()
    blocks_of = {u: s.blocks for u, s in sels.items()}
    refs = O.run_attention(inp, st, blocks_of, units=units)
    mx, mean = check_attention(run, refs, strict=True, strict_units=strict_units(inp, blocks_of))
    print(f"{name}: units={len(units)} tie-band differences={ties} max|dO|={mx:.2e} mean={mean:.2e}")
    if wl.n_q == 1:
        # The fused decode step on the same inputs, in the benchmark's launch
        # configuration: kernel means, selection and attention in one launch.
        full = run.blank_step_kernels()
        run.idx.fill_(-7)
        run.out.fill_(float("nan"))
        run.step()
        torch.cuda.synchronize()
        assert torch.equal(run.kc.view(torch.int16), full.view(torch.int16))
        ties = check_selections(run, sels, check_scores=False)
        got = run.gpu_blocks(units)
        same = {u for u in units if np.array_equal(got[u], sels[u].blocks)}
        refs = {u: refs[u] for u in same}
        refs.update(O.run_attention(inp, st, got, units=[u for u in units if u not in same]))
        mx, mean = check_attention(run, refs, strict=True, strict_units=strict_units(inp, got))
        print(f"{name} fused step: tie-band differences={ties} max|dO|={mx:.2e} mean={mean:.2e}")


def test_workload_parity_prefill_32k(dev):
    # Every one of the 32768 x 2 query tokens: the selection against the
    # oracle's, then the attention on the oracle's selection against the
    # oracle's output (the oracle runs in a pool of worker processes).
    import torch
    import oracle_pool
    wl = S.WORKLOADS["prefill_32k"]
    inp = S.make_inputs(wl)
    st = _settings(wl)
    run = DeviceRun(inp, dev)
    run.compress()
    run.select(with_scores=False)
    torch.cuda.synchronize()
    bad, ties, oidx, onsel = oracle_pool.all_selections(inp, st, run.idx.cpu().numpy(), run.nsel.cpu().numpy())
    assert not bad, (len(bad), bad[:5])
    run.out.fill_(float("nan"))
    run.attend(torch.from_numpy(oidx).to(dev), torch.from_numpy(onsel).to(dev))
    torch.cuda.synchronize()
    r = oracle_pool.all_attention(inp, st, oidx, onsel, run.out.float().cpu().numpy(), run.lse.cpu().numpy(),
                                  STRICT_MIN_KEYS)
    assert r["count"] == wl.n_q * wl.n_heads * wl.head_dim
    assert not r["over"], (len(r["over"]), r["over"][:5])
    assert r["sum"] / r["count"] <= ATT_MEAN + r["allow"] / r["count"], r["sum"] / r["count"]
    assert r["s_max"] <= ATT_MAX and r["s_sum"] / r["s_count"] <= ATT_MEAN, (r["s_max"], r["s_sum"] / r["s_count"])
    assert r["lse"] <= LSE_ABS, r["lse"]
    print(f"prefill_32k: {wl.n_q * wl.n_kv_heads} units, tie-band differences={ties}, max|dO|={r['max']:.2e} "
          f"mean={r['sum'] / r['count']:.2e}; on {r['s_count'] // (16 * 128)} units attending >= "
          f"{STRICT_MIN_KEYS} keys: max={r['s_max']:.2e} mean={r['s_sum'] / r['s_count']:.2e}")


def test_chunked_prefill_on_a_cache(dev):
    # A 2048-token chunk appended to caches of different lengths (the query
    # position rule i = L - n_q + t): selection over each token's visible
    # kernels and the tcgen05 attention, on a stratified sample of tokens.
    import torch
    nq = 2048
    inp = S.make_random(batch=2, n_kv_heads=2, kv_len=20000, n_q=nq, topk=32, includes_forced=False,
                        seed=77, kv_lens=[20000, 9000])
    st = _settings(inp.wl)
    run = DeviceRun(inp, dev)
    run.compress()
    run.select(with_scores=False)
    run.attend()
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    toks = sorted(set(range(0, 64)) | set(range(nq - 64, nq)) | set(rng.choice(nq, 128, replace=False).tolist()))
    units = [(b, h, t) for b in range(2) for h in range(2) for t in toks]
    sels = O.run_selection(inp, st, units=units)
    check_selections(run, sels, check_scores=False)
    idx, nsel = run.upload_selection(sels)
    run.out.fill_(float("nan"))
    run.attend(idx, nsel)
    torch.cuda.synchronize()
    blocks_of = {u: s.blocks for u, s in sels.items()}
    refs = O.run_attention(inp, st, blocks_of, units=units)
    mx, mean = check_attention(run, refs, strict=True, strict_units=strict_units(inp, blocks_of))
    print(f"chunked prefill: units={len(units)} max|dO|={mx:.2e} mean={mean:.2e}")


# ------------------------------------------- coarse-LSE approximation ----

@pytest.mark.parametrize("sc", [64, 128])
def test_coarse_means_match_oracle(dev, sc):
    import torch
    inp = S.make_random(batch=2, n_kv_heads=2, kv_len=5000, n_q=1, topk=8, seed=61, kv_lens=[5000, 1111])
    run = DeviceRun(inp, dev)
    kcc = run.T.alloc_kcc(run.p, sc, dev)
    kcc.view(torch.int16).fill_(0x7FC0)
    run.T.coarse_means(run.p, run.k, run.lens, sc, kcc)
    torch.cuda.synchronize()
    got = kc_to_f64(kcc)
    for b in range(2):
        for h in range(2):
            L = int(inp.kv_lens[b])
            ref = O.window_means(S.bf16_bits_to_f32(inp.k[b, h, :L]).astype(np.float64), sc, sc)
            n = ref.shape[0]
            err = np.abs(got[b, h, :n] - ref)
            assert np.all(err <= 2.0 ** -16 * np.abs(ref) + 1e-7), (b, h, float(err.max()))
            assert np.all(np.isnan(got[b, h, n:])), (b, h)


COARSE_CASES = [
    # batch, hkv, cap, lens, n_q, topk, includes_forced, sc
    (2, 2, 5000, [5000, 3333], 100, 16, True, 64),
    (1, 2, 4000, [4000], 300, 24, False, 128),
    (1, 1, 700, [700], 700, 4, True, 64),        # from position 0: the first tokens keep the exact LSE
    (2, 1, 2000, [2000, 90], 90, 6, True, 64),   # a sequence barely past its first window
]


@pytest.mark.parametrize("case", COARSE_CASES, ids=[f"coarse{i}" for i in range(len(COARSE_CASES))])
def test_select_coarse_lse_parity(dev, case):
    import torch
    B, H, cap, lens, nq, topk, inc, sc = case
    inp = S.make_random(batch=B, n_kv_heads=H, kv_len=cap, n_q=nq, topk=topk, includes_forced=inc,
                        seed=400 + sum(lens) + nq, kv_lens=lens)
    run = DeviceRun(inp, dev)
    run.compress()
    kcc = run.T.alloc_kcc(run.p, sc, dev)
    run.T.coarse_means(run.p, run.k, run.lens, sc, kcc)
    run.T.select_blocks_coarse_lse(run.p, run.q, run.kc, sc, kcc, run.lens, run.idx, run.nsel, run.scores)
    torch.cuda.synchronize()
    st = O.Settings(topk=topk, includes_forced=inc, coarse=sc)
    sels = O.run_selection(inp, st)
    check_selections(run, sels)


def test_select_exact_ties_break_to_lower_block(dev):
    # The key sequence repeats after `half` keys, so block j and block
    # j + half/64 see bit-identical kernel means and score exactly alike; both
    # sides must keep the lower block of every tied pair (ties go to the lower
    # index).  A second case makes every block identical, which exercises the
    # many-way tie path of the top-k.
    import torch
    for period_blocks, L in ((40, 80 * 64), (1, 20000)):
        inp = S.make_random(batch=1, n_kv_heads=2, kv_len=L, n_q=2, topk=12, seed=31)
        half = period_blocks * 64
        k = inp.k.copy()
        for start in range(half, L, half):
            n = min(half, L - start)
            k[:, :, start:start + n] = inp.k[:, :, :n]
        inp.k[...] = k
        run = DeviceRun(inp, dev)
        run.compress()
        run.select()
        torch.cuda.synchronize()
        sels = O.run_selection(inp, _settings(inp.wl))
        idx, nsel = run.idx.cpu().numpy(), run.nsel.cpu().numpy()
        for (b, h, t), s in sels.items():
            assert idx[b, h, t, :nsel[b, h, t]].tolist() == s.blocks.tolist(), ((b, h, t), period_blocks)


@pytest.mark.parametrize("nq", [1, 3])
def test_append_kv_then_decode_step(dev, nq):
    # The append writes the newest rows bit-exactly, leaves every other row
    # alone, and append + decode step gives the step on a cache that already
    # held those rows.
    import torch
    import trainable_block_sparse_infllm_gb300 as T
    inp = S.make_random(batch=2, n_kv_heads=2, kv_len=3000, n_q=nq, topk=16, seed=31 + nq, kv_lens=[3000, 2100])
    run = DeviceRun(inp, dev)
    run.compress()
    full_k, full_v = run.k.clone(), run.v.clone()
    run.blank_step_kernels()
    run.step()
    out_ref, idx_ref = run.out.clone(), run.idx.clone()
    k_new = torch.stack([full_k[b, :, int(L) - nq:int(L)] for b, L in enumerate(inp.kv_lens)]).contiguous()
    v_new = torch.stack([full_v[b, :, int(L) - nq:int(L)] for b, L in enumerate(inp.kv_lens)]).contiguous()
    for b, L in enumerate(inp.kv_lens):
        run.k[b, :, int(L) - nq:int(L)].view(torch.int16).fill_(0x7FC0)
        run.v[b, :, int(L) - nq:int(L)].view(torch.int16).fill_(0x7FC0)
    T.append_kv(run.p, k_new, v_new, run.lens, run.k, run.v)
    run.blank_step_kernels()
    run.idx.fill_(-7)
    run.out.fill_(float("nan"))
    run.step()
    torch.cuda.synchronize()
    assert torch.equal(run.k.view(torch.int16), full_k.view(torch.int16))
    assert torch.equal(run.v.view(torch.int16), full_v.view(torch.int16))
    assert torch.equal(run.idx, idx_ref)
    assert torch.equal(run.out.view(torch.int16), out_ref.view(torch.int16))


@pytest.mark.parametrize("where", ["device", "host"])
def test_append_decode_step_one_launch(dev, where):
    # The cache append fused into the decode step gives the caches, kernel
    # means, selection, output and lse of the step on a cache that already
    # held the token.  The appended rows start out as NaN in the caches; with
    # lengths 4096 and 2080 the newest kernel ends on the appended key, with
    # 3000 it does not.  "host": q, k_new, v_new, out and lse in pinned host
    # memory.
    import torch
    import trainable_block_sparse_infllm_gb300 as T
    inp = S.make_random(batch=3, n_kv_heads=2, kv_len=4096, n_q=1, topk=16, seed=57, kv_lens=[4096, 3000, 2080])
    run = DeviceRun(inp, dev)
    full_k, full_v = run.k.clone(), run.v.clone()
    kc_full = run.blank_step_kernels()
    run.step()
    torch.cuda.synchronize()
    assert torch.equal(run.kc.view(torch.int16), kc_full.view(torch.int16))
    out_ref, lse_ref = run.out.clone(), run.lse.clone()
    idx_ref, nsel_ref = run.idx.clone(), run.nsel.clone()
    k_new = torch.stack([full_k[b, :, int(L) - 1:int(L)] for b, L in enumerate(inp.kv_lens)]).contiguous()
    v_new = torch.stack([full_v[b, :, int(L) - 1:int(L)] for b, L in enumerate(inp.kv_lens)]).contiguous()
    q = run.q.clone()
    out = torch.full_like(run.out, float("nan"))
    lse = torch.full_like(run.lse, float("nan"))
    if where == "host":
        k_new, v_new, q = k_new.cpu().pin_memory(), v_new.cpu().pin_memory(), q.cpu().pin_memory()
        out, lse = out.cpu().pin_memory(), lse.cpu().pin_memory()
    run.blank_step_kernels()
    for b, L in enumerate(inp.kv_lens):
        run.k[b, :, int(L) - 1].view(torch.int16).fill_(0x7FC0)
        run.v[b, :, int(L) - 1].view(torch.int16).fill_(0x7FC0)
    run.idx.fill_(-7)
    run.nsel.fill_(-7)
    T.append_decode_step(run.p, q, k_new, v_new, run.k, run.v, run.lens, run.kc, run.idx, run.nsel, out, lse)
    torch.cuda.synchronize()
    assert T.get_device_status(clear=True) == 0
    assert torch.equal(run.k.view(torch.int16), full_k.view(torch.int16))
    assert torch.equal(run.v.view(torch.int16), full_v.view(torch.int16))
    assert torch.equal(run.kc.view(torch.int16), kc_full.view(torch.int16))
    assert torch.equal(run.idx, idx_ref) and torch.equal(run.nsel, nsel_ref)
    assert torch.equal(out.to(dev).view(torch.int16), out_ref.view(torch.int16))
    assert torch.equal(lse.to(dev), lse_ref)


def test_append_kv_bad_kv_len(dev):
    import torch
    import trainable_block_sparse_infllm_gb300 as T
    inp = S.make_random(batch=2, n_kv_heads=1, kv_len=500, n_q=2, topk=4, seed=6, kv_lens=[500, 1])
    run = DeviceRun(inp, dev)
    before_k, before_v = run.k.clone(), run.v.clone()
    k_new = torch.zeros((2, 1, 2, 128), dtype=torch.bfloat16, device=dev)
    T.append_kv(run.p, k_new, k_new, run.lens, run.k, run.v)
    torch.cuda.synchronize()
    assert T.get_device_status(clear=True) & T.DEVICE_BAD_KV_LEN
    assert torch.equal(run.k[1].view(torch.int16), before_k[1].view(torch.int16))
    assert bool((run.k[0, 0, 498:500] == 0).all()) and bool((run.v[0, 0, 498:500] == 0).all())
    assert torch.equal(run.k[0, 0, :498].view(torch.int16), before_k[0, 0, :498].view(torch.int16))


@pytest.mark.parametrize("sc", [0, 64])
def test_select_long_capacity(dev, sc):
    # A cache capacity of 250K tokens (3907 blocks): the prefill selection
    # keeps 8 tokens' block scores on chip with a 2-stage ring and its top-k
    # scratch laid over the ring; the result rule is the same.
    import torch
    inp = S.make_random(batch=1, n_kv_heads=2, kv_len=3000, n_q=40, topk=16, seed=77, max_kv_len=250_000)
    run = DeviceRun(inp, dev)
    run.compress()
    if sc:
        kcc = run.T.alloc_kcc(run.p, sc, dev)
        run.T.coarse_means(run.p, run.k, run.lens, sc, kcc)
        run.T.select_blocks_coarse_lse(run.p, run.q, run.kc, sc, kcc, run.lens, run.idx, run.nsel, run.scores)
    else:
        run.select()
    torch.cuda.synchronize()
    st = O.Settings(topk=16, coarse=sc)
    check_selections(run, O.run_selection(inp, st))


@pytest.mark.parametrize("nq", [1, 3])
def test_decode_step_output_to_pinned_host_memory(dev, nq):
    # The step stores its output with ordinary stores, so a pinned host buffer
    # receives the same bytes as device memory: the single launch (n_q = 1)
    # and the three stages in order (n_q = 3).
    import torch
    inp = S.make_random(batch=2, n_kv_heads=2, kv_len=3000, n_q=nq, topk=16, seed=44, kv_lens=[3000, 2500])
    run = DeviceRun(inp, dev)
    run.blank_step_kernels()
    run.step()
    ref_out, ref_lse = run.out.clone(), run.lse.clone()
    run.blank_step_kernels()
    out_h = torch.full(tuple(run.out.shape), float("nan"), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.full(tuple(run.lse.shape), float("nan"), dtype=torch.float32).pin_memory()
    ws = run.T.alloc_workspace(run.p, run.nq, run.T.OP_DECODE_STEP, dev)
    run.T.decode_step(run.p, run.q, run.k, run.v, run.lens, run.kc, run.idx, run.nsel, out_h, lse_h, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16), ref_out.cpu().view(torch.int16))
    assert torch.equal(lse_h, ref_lse.cpu())


def test_append_kv_from_pinned_host_memory_with_queries(dev):
    # k_new, v_new and the step's queries read straight from pinned host
    # memory; the cache rows and the query buffer receive the same bytes.
    import torch
    import trainable_block_sparse_infllm_gb300 as T
    inp = S.make_random(batch=2, n_kv_heads=2, kv_len=1500, n_q=2, topk=8, seed=45, kv_lens=[1500, 700])
    run = DeviceRun(inp, dev)
    full_k, full_v, q_ref = run.k.clone(), run.v.clone(), run.q.clone()
    k_h = torch.stack([full_k[b, :, int(L) - 2:int(L)] for b, L in enumerate(inp.kv_lens)]).cpu().pin_memory()
    v_h = torch.stack([full_v[b, :, int(L) - 2:int(L)] for b, L in enumerate(inp.kv_lens)]).cpu().pin_memory()
    q_h = q_ref.cpu().pin_memory()
    for b, L in enumerate(inp.kv_lens):
        run.k[b, :, int(L) - 2:int(L)].view(torch.int16).fill_(0x7FC0)
        run.v[b, :, int(L) - 2:int(L)].view(torch.int16).fill_(0x7FC0)
    run.q.view(torch.int16).fill_(0x7FC0)
    T.append_kv(run.p, k_h, v_h, run.lens, run.k, run.v, q_src=q_h, q_dst=run.q)
    torch.cuda.synchronize()
    assert torch.equal(run.k.view(torch.int16), full_k.view(torch.int16))
    assert torch.equal(run.v.view(torch.int16), full_v.view(torch.int16))
    assert torch.equal(run.q.view(torch.int16), q_ref.view(torch.int16))


def test_decode_step_256k_capacity(dev):
    # A 262,144-token cache (4096 blocks) with two KV heads, one of them
    # filled to 261,500 tokens: the fused step stays one launch (16-CTA
    # clusters, 16 kernel-mean chunks per CTA) and matches the oracle, and
    # the three separate stages agree with it.
    import torch
    cap = 262_144
    inp = S.make_random(batch=2, n_kv_heads=1, kv_len=cap, n_q=1, topk=64, seed=91, kv_lens=[cap, 261_500])
    st = _settings(inp.wl)
    run = DeviceRun(inp, dev)
    assert run.T.workspace_size(run.p, 1, run.T.OP_DECODE_STEP) == 0   # the single-launch form
    full = run.blank_step_kernels()
    run.step()
    torch.cuda.synchronize()
    assert torch.equal(run.kc.view(torch.int16), full.view(torch.int16))
    sels = O.run_selection(inp, st)
    check_selections(run, sels, check_scores=False)
    got = run.gpu_blocks(sels.keys())
    refs = O.run_attention(inp, st, got)
    mx, mean = check_attention(run, refs, strict=True, strict_units=strict_units(inp, got))
    out_step = run.out.float().clone()
    run.select(with_scores=False)
    run.attend()
    torch.cuda.synchronize()
    check_selections(run, sels, check_scores=False)
    assert (run.out.float() - out_step).abs().max().item() <= 2e-3
    print(f"256K capacity: fused step max|dO|={mx:.2e} mean={mean:.2e}")
