"""GPU parity of the backward of stage 3 (dq, dk, dv with the block selection
held fixed) against the fp64 oracle, through the C ABI.

The forward runs first on the GPU to give out and lse (the backward's inputs,
as in training); the expected gradients come from the oracle alone, from q, K,
V, the upstream gradient and the selection.
"""

import numpy as np
import pytest

import oracle as O
import synthetic_inputs as S
from helpers import DeviceRun, check_grad

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


def _settings(wl):
    return O.Settings(topk=wl.topk, n_init=wl.n_init, n_local=wl.n_local, includes_forced=wl.topk_includes_forced)


def _used_rows(wl, kv_lens, blocks_of):
    """[B, Hkv, L_max] bool: keys attended by at least one query."""
    used = np.zeros((wl.batch, wl.n_kv_heads, wl.kv_len), dtype=bool)
    for (b, h, t), blocks in blocks_of.items():
        i = O.query_position(int(kv_lens[b]), wl.n_q, t)
        used[b, h, O.attended_keys(wl.kv_len, np.asarray(blocks), i, wl.block)] = True
    return used


def _unit_refs(inp, st, blocks, dO, out_gpu, unit, K, V):
    """Oracle gradients of one unit and the allowances for the bf16 forward
    output inside D: (dq, keys, dK_sel, dV_sel, allow_dq, allow_dK_sel)."""
    wl = inp.wl
    b, h, t = unit
    G, d = wl.group, wl.head_dim
    scale = st.ascale(d)
    i = O.query_position(int(inp.kv_lens[b]), wl.n_q, t)
    blocks = np.asarray(blocks)
    gq, keys, gk, gv = O.unit_attention_grad(inp, st, {unit: blocks}, dO, unit, K, V)
    q = S.bf16_bits_to_f64(inp.q[b, t, h * G:(h + 1) * G])
    o_ref, _ = O.sparse_attention(q, K, V, blocks, i, wl.block, scale)
    dOu = dO[b, t, h * G:(h + 1) * G]
    dD = np.abs((dOu * (out_gpu[b, t, h * G:(h + 1) * G] - o_ref)).sum(axis=1))[:, None]
    pk, _ = O.sparse_attention(q, K, np.abs(K), blocks, i, wl.block, scale)        # sum_j P_j |k_j|
    _, _, _, pq = O.sparse_attention_grad_selected(q, K, V, blocks, i, wl.block, scale, dD * np.abs(q))
    return gq, keys, gk, gv, scale * dD * pk, scale * pq


def _refs_all(inp, st, blocks_of, dO, out_gpu):
    wl = inp.wl
    G = wl.group
    shape_kv = (wl.batch, wl.n_kv_heads, wl.kv_len, wl.head_dim)
    rq = np.zeros((wl.batch, wl.n_q, wl.n_heads, wl.head_dim))
    aq = np.zeros_like(rq)
    rk, rv, ak = np.zeros(shape_kv), np.zeros(shape_kv), np.zeros(shape_kv)
    for b in range(wl.batch):
        L = int(inp.kv_lens[b])
        for h in range(wl.n_kv_heads):
            K, V = S.bf16_bits_to_f64(inp.k[b, h, :L]), S.bf16_bits_to_f64(inp.v[b, h, :L])
            for t in range(wl.n_q):
                gq, keys, gk, gv, alq, alk = _unit_refs(inp, st, blocks_of[(b, h, t)], dO, out_gpu, (b, h, t), K, V)
                rq[b, t, h * G:(h + 1) * G] = gq
                aq[b, t, h * G:(h + 1) * G] = alq
                rk[b, h, keys] += gk
                rv[b, h, keys] += gv
                ak[b, h, keys] += alk
    return rq, rk, rv, aq, ak


BWD_CASES = [
    # batch, hkv, cap, lens, n_q, topk, includes_forced
    (2, 1, 4100, [4100, 2100], 5, 12, True),     # few queries (decode-path forward)
    (1, 2, 9000, [9000], 1, 64, True),           # one query token
    (2, 2, 2000, [2000, 1234], 130, 8, False),   # ragged lengths, partial query tiles
    (1, 1, 700, [700], 700, 4, True),            # from position 0: block 0 has three work items
    (3, 1, 300, [300, 40, 20], 20, 4, True),     # tiny contexts, rows with one key
    (1, 1, 1000, [1000], 1000, 16, True),        # capacity not a multiple of the block
]


@pytest.mark.parametrize("case", BWD_CASES, ids=[f"bwd{i}" for i in range(len(BWD_CASES))])
def test_backward_parity(dev, case):
    import torch
    B, H, cap, lens, nq, topk, inc = case
    inp = S.make_random(batch=B, n_kv_heads=H, kv_len=cap, n_q=nq, topk=topk, includes_forced=inc,
                        seed=300 + sum(lens) + nq, kv_lens=lens)
    wl = inp.wl
    st = _settings(wl)
    sels = O.run_selection(inp, st)
    blocks = {u: s.blocks for u, s in sels.items()}
    run = DeviceRun(inp, dev)
    idx, nsel = run.upload_selection(sels)
    run.attend(idx, nsel)
    dout = S.make_grad_out(wl, seed=900 + nq)
    dq, dk, dv = run.backward(idx, nsel, dout)
    torch.cuda.synchronize()
    rq, rk, rv, aq, ak = _refs_all(inp, st, blocks, S.bf16_bits_to_f64(dout), run.out.double().cpu().numpy())
    used = _used_rows(wl, inp.kv_lens, blocks)
    stats = [check_grad("dq", dq.cpu().numpy(), rq, allow=aq),
             check_grad("dk", dk.cpu().numpy(), rk, used, allow=ak),
             check_grad("dv", dv.cpu().numpy(), rv, used)]
    print(" ".join(f"{n}: max {a:.2e} mean {m:.2e}" for n, (a, m) in zip(("dq", "dk", "dv"), stats)))


def test_backward_dense_degeneracy_matches_autograd(dev):
    # topk covering every block: the gradients are those of plain causal
    # attention, here from torch autograd in float64 on the CPU.
    import torch
    inp = S.make_random(batch=1, n_kv_heads=1, kv_len=600, n_q=600, topk=10, seed=8)
    run = DeviceRun(inp, dev)
    run.compress()
    run.select()
    run.attend()
    dout = S.make_grad_out(inp.wl, seed=81)
    dq, dk, dv = run.backward(run.idx, run.nsel, dout)
    torch.cuda.synchronize()
    assert np.all(run.nsel.cpu().numpy() == np.arange(600)[None, None] // 64 + 1)
    q = torch.from_numpy(S.bf16_bits_to_f64(inp.q[0])).permute(1, 0, 2).requires_grad_()
    k = torch.from_numpy(S.bf16_bits_to_f64(inp.k[0, 0])).requires_grad_()
    v = torch.from_numpy(S.bf16_bits_to_f64(inp.v[0, 0])).requires_grad_()
    o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None, None].expand(1, 16, 600, 128),
                                                         v[None, None].expand(1, 16, 600, 128), is_causal=True)
    o.backward(torch.from_numpy(S.bf16_bits_to_f64(dout[0])).permute(1, 0, 2)[None])
    # Allowances for the bf16 forward output inside D, from the oracle.
    blocks_of = {(0, 0, t): np.arange(t // 64 + 1) for t in range(600)}
    _, _, _, aq, ak = _refs_all(inp, O.Settings(topk=10), blocks_of, S.bf16_bits_to_f64(dout),
                                run.out.double().cpu().numpy())
    check_grad("dq", dq[0].cpu().numpy(), q.grad.permute(1, 0, 2).numpy(), allow=aq[0])
    check_grad("dk", dk[0, 0].cpu().numpy(), k.grad.numpy(), allow=ak[0, 0])
    check_grad("dv", dv[0, 0].cpu().numpy(), v.grad.numpy())


def test_backward_bad_kv_len(dev):
    import torch
    import trainable_block_sparse_infllm_gb300 as T
    inp = S.make_random(batch=2, n_kv_heads=1, kv_len=1000, n_q=2, topk=4, seed=4, kv_lens=[1000, 1])
    run = DeviceRun(inp, dev)
    idx = torch.zeros((2, 1, 2, run.kmax), dtype=torch.int32, device=dev)
    nsel = torch.ones((2, 1, 2), dtype=torch.int32, device=dev)
    run.attend(idx, nsel)
    dq, dk, dv = run.backward(idx, nsel, S.make_grad_out(inp.wl, seed=5))
    torch.cuda.synchronize()
    assert T.get_device_status(clear=True) & T.DEVICE_BAD_KV_LEN
    assert bool((dq[1] == 0).all()) and bool((dk[1] == 0).all()) and bool((dv[1] == 0).all())
    assert bool(torch.isfinite(dq[0]).all()) and bool((dk[0, 0, 64:] == 0).all())


def test_backward_prefill_32k_workload(dev):
    # Full-size prefill workload with a seeded block selection: dq of every
    # one of the 65,536 (head group, token) units, and dK, dV of every key,
    # against the oracle in a spawn process pool (dq per query; dK and dV per
    # key block from all the queries that selected it).
    import torch
    import oracle_pool
    from helpers import GRAD_MAX, GRAD_MEAN
    wl = S.WORKLOADS["prefill_32k"]
    inp = S.make_inputs(wl)
    st = _settings(wl)
    idx_np, nsel_np = S.make_block_sets(wl, inp.kv_lens, seed=wl.seed + 1000)
    run = DeviceRun(inp, dev)
    idx = torch.from_numpy(idx_np).to(dev)
    nsel = torch.from_numpy(nsel_np).to(dev)
    run.attend(idx, nsel)
    dout = S.make_grad_out(wl, seed=wl.seed + 2000)
    dq, dk, dv = run.backward(idx, nsel, dout)
    torch.cuda.synchronize()
    dq, dk, dv = dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy()
    assert np.all(np.isfinite(dk)) and np.all(np.isfinite(dv)) and np.all(np.isfinite(dq))
    out_bits = run.out.cpu().view(torch.int16).numpy()
    tot, rk, rv, ra, used = oracle_pool.all_backward(inp, st, idx_np, nsel_np, dout, out_bits, dq)
    # dq: check_grad's rule over all units, from the pooled statistics.
    assert tot["over"] <= GRAD_MAX * tot["ref"], ("dq", tot["over"] / tot["ref"])
    mean = tot["err"] / tot["count"]
    assert mean <= GRAD_MEAN * tot["ref"] + tot["allow"] / tot["count"], ("dq mean", mean / tot["ref"])
    print(f"dq: {tot['count'] // (16 * 128)} units, max over allowance {tot['over'] / tot['ref']:.2e}, "
          f"mean {mean / tot['ref']:.2e} (relative to max |dq|)")
    for h in range(wl.n_kv_heads):
        mk = check_grad(f"dk h{h}", dk[0, h], rk[0, h], rows_used=used[0, h], allow=ra[0, h])
        mv = check_grad(f"dv h{h}", dv[0, h], rv[0, h], rows_used=used[0, h])
        print(f"h{h}: {int(used[0, h].sum())} keys, dk max {mk[0]:.2e} mean {mk[1]:.2e}, "
              f"dv max {mv[0]:.2e} mean {mv[1]:.2e}")
