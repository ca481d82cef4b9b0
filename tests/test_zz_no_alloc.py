"""The allocation-free selection entry point against the workspace one (GPU).

infllmv2_select_blocks_static serves callers that cannot hand the library
device scratch at the call site (start-up-planned device memory, C hosts
without a device allocator); it uses an 8 MiB array built into the library.
It must return what infllmv2_select_blocks returns, on consecutive calls that
reuse that array.  This file is collected last so that a failure here does
not hide the rest of the GPU suite.
"""

import numpy as np
import pytest

import synthetic_inputs as S

pytestmark = pytest.mark.gpu


def _run_both(dev, batch, n_kv_heads, kv_len, n_q, topk, kv_lens, seed):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import trainable_block_sparse_infllm_gb300 as T
    from helpers import R_REL, dev_bf16

    inp = S.make_random(batch=batch, n_kv_heads=n_kv_heads, kv_len=kv_len, n_q=n_q, topk=topk, seed=seed,
                        kv_lens=kv_lens)
    wl = inp.wl
    p = T.make_params(batch, n_kv_heads, wl.kv_len, topk, True)
    q, k = dev_bf16(inp.q, dev), dev_bf16(inp.k, dev)
    lens = torch.from_numpy(inp.kv_lens.astype(np.int32)).to(dev)
    kc = T.alloc_kc(p, dev)
    T.compress_keys(p, k, lens, kc)
    kmax = T.max_selected(p)
    nbmax = -(-wl.kv_len // 64)

    def outputs():
        return (torch.full((batch, n_kv_heads, n_q, kmax), -7, dtype=torch.int32, device=dev),
                torch.full((batch, n_kv_heads, n_q), -7, dtype=torch.int32, device=dev),
                torch.full((batch, n_kv_heads, n_q, nbmax), float("nan"), dtype=torch.float32, device=dev))

    ref_idx, ref_n, ref_r = outputs()
    ws = T.alloc_workspace(p, n_q, T.OP_SELECT, dev)
    T.select_blocks(p, q, kc, lens, ref_idx, ref_n, ref_r, ws)
    results = []
    for _ in range(2):                       # two calls in a row share the built-in scratch
        idx, n, r = outputs()
        T.select_blocks_static(p, q, kc, lens, idx, n, r)
        results.append((idx, n, r))
    torch.cuda.synchronize()
    assert T.get_device_status(clear=True) == 0
    for idx, n, r in results:
        assert torch.equal(idx, ref_idx)
        assert torch.equal(n, ref_n)
        a, b = r.cpu().numpy(), ref_r.cpu().numpy()
        fin = np.isfinite(b)
        assert np.array_equal(np.isfinite(a), fin)
        assert np.all(np.abs(a[fin] - b[fin]) <= R_REL * np.abs(b[fin]))


@pytest.fixture(scope="module")
def dev():
    import torch
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def test_static_scratch_matches_workspace_decode(dev):
    _run_both(dev, batch=2, n_kv_heads=2, kv_len=9000, n_q=1, topk=32, kv_lens=[9000, 5555], seed=41)


def test_static_scratch_matches_workspace_verify(dev):
    _run_both(dev, batch=2, n_kv_heads=2, kv_len=6000, n_q=6, topk=16, kv_lens=[6000, 4000], seed=42)


def test_static_scratch_rejects_oversize(dev):
    import __graft_entry__
    __graft_entry__.build()
    import trainable_block_sparse_infllm_gb300 as T
    import torch
    # 16 tokens for 80 groups: enough tiles that no cluster splits them, so the
    # selection keeps one score per (token, head, kernel) in scratch:
    # 1280 units x 16 heads x 1024 kernels x 4 bytes = 80 MiB > 8 MiB.
    p = T.make_params(40, 2, 16384, 16, True)
    assert T.workspace_size(p, 16, T.OP_SELECT) > 8 << 20
    q = torch.zeros((40, 16, 32, 128), dtype=torch.bfloat16, device=dev)
    kc = T.alloc_kc(p, dev)
    lens = torch.full((40,), 16384, dtype=torch.int32, device=dev)
    idx = torch.empty((40, 2, 16, 16), dtype=torch.int32, device=dev)
    n = torch.empty((40, 2, 16), dtype=torch.int32, device=dev)
    with pytest.raises(T.InfLLMv2Error) as ei:
        T.select_blocks_static(p, q, kc, lens, idx, n)
    assert ei.value.code == 3 and "built-in scratch" in str(ei.value)
