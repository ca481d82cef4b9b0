"""Host-side checks of the C ABI (no GPU needed).

The library must build, load, and export every function that
include/infllmv2.h declares; argument errors must come back as return codes
before anything touches the device.  Fake pointers used here are never
dereferenced: every call below fails validation first.
"""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from trainable_block_sparse_infllm_gb300 import _lib
    return _lib


def _declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(infllmv2_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_four_stages():
    names = _declared_functions()
    for n in ("infllmv2_compress_keys", "infllmv2_select_blocks", "infllmv2_sparse_attn_decode",
              "infllmv2_sparse_attn_prefill"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (infllmv2_\w+)", out))
    missing = [n for n in _declared_functions() if n not in exported]
    assert not missing, missing
    for n in _declared_functions():
        getattr(L.lib, n)


def _params(L, **kw):
    p = L.Params()
    L.lib.infllmv2_default_params(ctypes.byref(p), kw.pop("batch", 2), kw.pop("hkv", 2),
                                  kw.pop("lmax", 4096), kw.pop("topk", 16), kw.pop("inc", 1))
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_default_params_and_sizes(L):
    p = _params(L)
    assert (p.group_size, p.head_dim, p.block_size, p.kernel_size, p.kernel_stride) == (16, 128, 64, 32, 16)
    assert (p.n_init_blocks, p.n_local_blocks) == (1, 2)
    assert abs(p.score_scale - 128 ** -0.5) < 1e-7 and abs(p.attn_scale - 128 ** -0.5) < 1e-7
    assert L.lib.infllmv2_num_kernels(ctypes.byref(p)) == 255
    assert L.lib.infllmv2_max_selected(ctypes.byref(p)) == 16
    p2 = _params(L, inc=0)
    assert L.lib.infllmv2_max_selected(ctypes.byref(p2)) == 19
    ws1 = L.lib.infllmv2_workspace_size(ctypes.byref(p), 1, L.OP_SELECT)
    ws8 = L.lib.infllmv2_workspace_size(ctypes.byref(p), 8, L.OP_SELECT)
    assert 0 < ws1 < ws8
    assert L.lib.infllmv2_workspace_size(ctypes.byref(p), 100, L.OP_SELECT) == 0
    assert L.lib.infllmv2_workspace_size(ctypes.byref(p), 1, L.OP_DECODE) == 0   # merged on chip
    assert L.lib.infllmv2_workspace_size(ctypes.byref(p), 100, L.OP_PREFILL) == 0
    assert L.lib.infllmv2_workspace_size(ctypes.byref(p), 100, L.OP_DECODE) == 0
    assert L.lib.infllmv2_workspace_size(ctypes.byref(p), 1, 99) == 0


FAKE = ctypes.c_void_p(0x7F0000000000)
FAKE_ODD = ctypes.c_void_p(0x7F0000000008)


def _attn(L, p, nq=1, q=FAKE, ws=None, ws_bytes=0, fn="infllmv2_sparse_attn_decode", out=FAKE):
    return getattr(L.lib, fn)(ctypes.byref(p), q, nq, FAKE, FAKE, FAKE, FAKE, FAKE, out, None, ws,
                              ws_bytes, None)


def test_argument_errors_return_codes(L):
    p = _params(L)
    assert L.lib.infllmv2_compress_keys(None, FAKE, FAKE, 0, -1, FAKE, None) == L.INVALID_ARGUMENT
    assert L.lib.infllmv2_compress_keys(ctypes.byref(p), None, FAKE, 0, -1, FAKE, None) == L.INVALID_ARGUMENT
    assert L.lib.infllmv2_compress_keys(ctypes.byref(p), FAKE_ODD, FAKE, 0, -1, FAKE, None) == L.UNSUPPORTED
    assert b"aligned" in L.lib.infllmv2_last_error()
    for field, value in (("head_dim", 64), ("group_size", 8), ("block_size", 128), ("kernel_size", 64),
                         ("kernel_stride", 32)):
        bad = _params(L, **{field: value})
        assert _attn(L, bad) == L.UNSUPPORTED, field
    assert _attn(L, _params(L, topk=2)) == L.INVALID_ARGUMENT           # topk < forced
    assert _attn(L, _params(L, score_scale=float("nan"))) == L.INVALID_ARGUMENT
    assert _attn(L, p, nq=0) == L.INVALID_ARGUMENT
    assert _attn(L, p, nq=5000) == L.INVALID_ARGUMENT                    # > max_kv_len
    assert _attn(L, p, nq=17) == L.INVALID_ARGUMENT                      # decode takes n_q <= 16
    assert _attn(L, p, q=FAKE_ODD) == L.UNSUPPORTED
    assert _attn(L, p, out=None) == L.INVALID_ARGUMENT
    rc = L.lib.infllmv2_select_blocks(ctypes.byref(p), FAKE, 1, FAKE, FAKE, FAKE, FAKE, None, None, 0, None)
    assert rc == L.WORKSPACE_TOO_SMALL
    assert b"workspace" in L.lib.infllmv2_last_error()
    need = L.lib.infllmv2_workspace_size(ctypes.byref(p), 1, L.OP_SELECT)
    rc = L.lib.infllmv2_select_blocks(ctypes.byref(p), FAKE, 1, FAKE, FAKE, FAKE, FAKE, None, FAKE, need - 1, None)
    assert rc == L.WORKSPACE_TOO_SMALL
    rc = L.lib.infllmv2_select_blocks(ctypes.byref(p), FAKE, 1, None, FAKE, FAKE, FAKE, None, None, 0, None)
    assert rc == L.INVALID_ARGUMENT
    assert L.status_string(L.WORKSPACE_TOO_SMALL) == "INFLLMV2_WORKSPACE_TOO_SMALL"
    assert L.status_string(12345) == "INFLLMV2_UNKNOWN_STATUS"


def test_python_binding_rejects_cpu_tensors(L):
    import torch
    import trainable_block_sparse_infllm_gb300 as T
    p = T.make_params(1, 1, 256, 4)
    k = torch.zeros((1, 1, 256, 128), dtype=torch.bfloat16)
    with pytest.raises(T.InfLLMv2Error):
        T.compress_keys(p, k, torch.zeros(1, dtype=torch.int32), T.alloc_kc(p))


def test_coarse_lse_entry_points_validate_first(L):
    p = _params(L)
    sel = L.lib.infllmv2_select_blocks_coarse_lse
    # The decode path (n_q <= 16) has no coarse form.
    assert sel(ctypes.byref(p), FAKE, 1, FAKE, 64, FAKE, FAKE, FAKE, FAKE, None, None) == L.UNSUPPORTED
    assert b"prefill path" in L.lib.infllmv2_last_error()
    for bad in (0, 16, 33, 8192):
        assert sel(ctypes.byref(p), FAKE, 100, FAKE, bad, FAKE, FAKE, FAKE, FAKE, None, None) == L.INVALID_ARGUMENT
        assert L.lib.infllmv2_coarse_means(ctypes.byref(p), FAKE, FAKE, bad, FAKE, None) == L.INVALID_ARGUMENT
    assert sel(ctypes.byref(p), FAKE, 100, FAKE, 64, None, FAKE, FAKE, FAKE, None, None) == L.INVALID_ARGUMENT
    assert L.lib.infllmv2_coarse_means(ctypes.byref(p), FAKE_ODD, FAKE, 64, FAKE, None) == L.UNSUPPORTED


def test_append_and_backward_entry_points_validate_first(L):
    p = _params(L)
    app = L.lib.infllmv2_append_kv
    assert app(ctypes.byref(p), 1, None, FAKE, FAKE, FAKE, FAKE, None, None, None) == L.INVALID_ARGUMENT
    assert app(ctypes.byref(p), 1, FAKE_ODD, FAKE, FAKE, FAKE, FAKE, None, None, None) == L.UNSUPPORTED
    assert app(ctypes.byref(p), 0, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None) == L.INVALID_ARGUMENT
    assert app(ctypes.byref(p), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == L.INVALID_ARGUMENT  # q_src alone
    assert app(ctypes.byref(p), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE_ODD, FAKE, None) == L.UNSUPPORTED
    # The one-launch append + step: one token per sequence, every pointer but lse.
    ads = L.lib.infllmv2_append_decode_step
    args = [FAKE] * 9   # k_new, v_new, k_cache, v_cache, kv_lens, kc, block_idx, n_selected, out
    assert len(ads.argtypes) == 3 + len(args) + 2
    assert ads(ctypes.byref(p), FAKE, 1, None, *args[1:], None, None) == L.INVALID_ARGUMENT
    assert ads(ctypes.byref(p), FAKE, 2, *args, None, None) == L.UNSUPPORTED
    assert b"n_q = 1" in L.lib.infllmv2_last_error()
    assert ads(ctypes.byref(p), FAKE_ODD, 1, *args, None, None) == L.UNSUPPORTED
    bwd = L.lib.infllmv2_sparse_attn_backward
    # q, n_q, then k_cache, v_cache, kv_lens, block_idx, n_selected, out, lse, dout, dq, dk, dv
    ptrs = [FAKE] * 11
    no_lse = list(ptrs)
    no_lse[6] = None
    assert bwd(ctypes.byref(p), FAKE, 4, *no_lse, FAKE, 1 << 30, None) == L.INVALID_ARGUMENT
    assert bwd(ctypes.byref(p), FAKE, 4, *ptrs, None, 0, None) == L.WORKSPACE_TOO_SMALL
    need = L.lib.infllmv2_workspace_size(ctypes.byref(p), 4, 5)
    assert need > 0
    assert bwd(ctypes.byref(p), FAKE, 4, *ptrs, FAKE, need - 1, None) == L.WORKSPACE_TOO_SMALL
    assert bwd(ctypes.byref(p), FAKE_ODD, 4, *ptrs, FAKE, need, None) == L.UNSUPPORTED


def test_prefill_selection_capacity_bound(L):
    # Prefill selection (n_q > 16): 8 tokens' block scores on chip up to
    # 327,360 tokens of capacity (no workspace); past it they take one
    # workspace slot per SM, up to about 680K tokens; the coarse-LSE form
    # takes no workspace and keeps the on-chip bound.
    for lmax in (250_000, 327_360):
        ok = _params(L, batch=1, hkv=1, lmax=lmax)
        assert L.lib.infllmv2_workspace_size(ctypes.byref(ok), 100, L.OP_SELECT) == 0
    p = _params(L, batch=1, hkv=1, lmax=327_361)
    need = L.lib.infllmv2_workspace_size(ctypes.byref(p), 100, L.OP_SELECT)
    assert need >= 8 * ((327_361 + 63) // 64) * 4
    rc = L.lib.infllmv2_select_blocks(ctypes.byref(p), FAKE, 100, FAKE, FAKE, FAKE, FAKE, None, None, 0, None)
    assert rc == L.WORKSPACE_TOO_SMALL
    rc = L.lib.infllmv2_select_blocks_coarse_lse(ctypes.byref(p), FAKE, 100, FAKE, 64, FAKE, FAKE, FAKE, FAKE, None,
                                                 None)
    assert rc == L.UNSUPPORTED
    assert b"327360" in L.lib.infllmv2_last_error()
    big = _params(L, batch=1, hkv=1, lmax=1_000_000)
    rc = L.lib.infllmv2_select_blocks(ctypes.byref(big), FAKE, 100, FAKE, FAKE, FAKE, FAKE, None, None, 0, None)
    assert rc == L.UNSUPPORTED
    assert b"680K" in L.lib.infllmv2_last_error()
