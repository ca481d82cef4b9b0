"""The process pool that runs the oracle over every unit of a large workload
(tests/oracle_pool.py): on a small case, fed the oracle's own selection and
its own bf16-rounded output, it reports no mismatch, no tie, and every unit."""

import numpy as np

import oracle as O
import oracle_pool
import synthetic_inputs as S
from helpers import STRICT_MIN_KEYS


def test_pool_accepts_the_oracles_own_results():
    inp = S.make_random(batch=2, n_kv_heads=1, kv_len=700, n_q=300, topk=4, includes_forced=False, seed=5,
                        kv_lens=[700, 450])
    wl = inp.wl
    st = O.Settings(topk=4, includes_forced=False)
    sels = O.run_selection(inp, st)
    idx = np.full((2, 1, wl.n_q, wl.k_max), -1, dtype=np.int32)
    nsel = np.zeros((2, 1, wl.n_q), dtype=np.int32)
    for (b, h, t), s in sels.items():
        idx[b, h, t, :len(s.blocks)] = s.blocks
        nsel[b, h, t] = len(s.blocks)
    bad, ties, oidx, onsel = oracle_pool.all_selections(inp, st, idx, nsel, chunk=64)
    assert bad == [] and ties == 0
    assert np.array_equal(oidx, idx) and np.array_equal(onsel, nsel)
    # A scored block swapped for the one block left out (query 299 of the
    # second sequence sits at 449 in block 7 and takes 4 of blocks 1..5) is
    # reported, for that unit only.
    row = sels[(1, 0, 299)].blocks.tolist()
    assert len(row) == 7
    missing = (set(range(8)) - set(row)).pop()
    sw = sorted(set(row) - {1 if missing != 1 else 2} | {missing})
    idx2 = idx.copy()
    idx2[1, 0, 299, :7] = sw
    bad2, _, _, _ = oracle_pool.all_selections(inp, st, idx2, nsel, chunk=64)
    assert [u for u, _ in bad2] == [(1, 0, 299)]
    refs = O.run_attention(inp, st, {u: s.blocks for u, s in sels.items()})
    out = np.zeros((2, wl.n_q, wl.n_heads, wl.head_dim), dtype=np.float32)
    lse = np.zeros((2, wl.n_q, wl.n_heads), dtype=np.float32)
    for (b, h, t), (o, l) in refs.items():
        out[b, t, h * 16:(h + 1) * 16] = S.bf16_bits_to_f32(S.bf16_bits_from_f32(o.astype(np.float32)))
        lse[b, t, h * 16:(h + 1) * 16] = l
    r = oracle_pool.all_attention(inp, st, oidx, onsel, out, lse, STRICT_MIN_KEYS, chunk=64)
    assert r["count"] == 2 * wl.n_q * wl.n_heads * wl.head_dim
    assert r["over"] == [] and r["sum"] <= r["allow"] and r["lse"] < 1e-6
    assert r["s_count"] > 0
