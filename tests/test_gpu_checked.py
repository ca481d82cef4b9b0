"""The checked build (libinfllmv2_checked.so, built with INFLLMV2_CHECKED).

It stands in for a memory checker: every caller-given index is verified
before use and a violation sets INFLLMV2_DEVICE_BOUNDS; its bounded waits are
short, and its fault-injection hook makes one of them expire.  The cases run
in a child process that loads the checked library (INFLLMV2_LIBRARY=checked):
  * out-of-range block_idx entries and an out-of-range n_selected, given to
    the prefill, decode and backward kernels, set DEVICE_BOUNDS and the
    calls return; the units with valid rows still match the oracle;
  * a valid selection sets no status bit in any kernel (no false alarm);
  * with the hook armed, a fused decode step withholds one release of a ring
    stage: a bounded wait expires, DEVICE_TIMEOUT is set and the call
    returns; disarmed, the same context then gives the oracle's result.
No GPU fault is involved: every failure is a status word the host reads.
"""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import json, sys
import numpy as np, torch
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
import oracle as O
import synthetic_inputs as S
import trainable_block_sparse_infllm_gb300 as T
from helpers import DeviceRun, check_attention
assert T.is_checked_build()
dev = torch.device("cuda:0"); torch.cuda.set_device(dev)
res = {}
T.get_device_status(clear=True)

def sels_of(inp, st):
    return O.run_selection(inp, st)

# ---- prefill attention and backward: bad rows in two units
inp = S.make_random(batch=1, n_kv_heads=1, kv_len=700, n_q=100, topk=4, includes_forced=True, seed=11)
st = O.Settings(topk=4)
sels = sels_of(inp, st)
run = DeviceRun(inp, dev)
idx, nsel = run.upload_selection(sels)
run.attend(idx, nsel, prefill=True)
torch.cuda.synchronize()
res["prefill_clean"] = T.get_device_status(clear=True)
bad_idx, bad_n = idx.clone(), nsel.clone()
c50 = (700 - 100 + 50) // 64
bad_idx[0, 0, 50, 1] = c50 + 3            # a block in the query's future
bad_n[0, 0, 60] = run.kmax + 5            # a count past the row
run.attend(bad_idx, bad_n, prefill=True)
torch.cuda.synchronize()
res["prefill_bad"] = T.get_device_status(clear=True)
good = {u: v for u, v in O.run_attention(inp, st, {u: s.blocks for u, s in sels.items()}).items()
        if u[2] not in (50, 60)}
check_attention(run, good)
res["prefill_valid_units_match"] = True
dout = S.make_grad_out(inp.wl, seed=3)
run.attend(idx, nsel, prefill=True)
run.backward(idx, nsel, dout)
torch.cuda.synchronize()
res["backward_clean"] = T.get_device_status(clear=True)
run.backward(bad_idx, nsel, dout)
torch.cuda.synchronize()
res["backward_bad"] = T.get_device_status(clear=True)

# ---- decode attention (n_q = 2)
inp = S.make_random(batch=2, n_kv_heads=1, kv_len=3000, n_q=2, topk=8, seed=12, kv_lens=[3000, 2000])
st = O.Settings(topk=8)
sels = sels_of(inp, st)
run = DeviceRun(inp, dev)
idx, nsel = run.upload_selection(sels)
run.attend(idx, nsel, prefill=False)
torch.cuda.synchronize()
res["decode_clean"] = T.get_device_status(clear=True)
bad_idx = idx.clone()
bad_idx[1, 0, 0, 2] = -5
run.attend(bad_idx, nsel, prefill=False)
torch.cuda.synchronize()
res["decode_bad"] = T.get_device_status(clear=True)

# ---- fused decode step with the hook armed: a bounded wait expires
inp = S.make_random(batch=1, n_kv_heads=1, kv_len=80000, n_q=1, topk=16, seed=13)
st = O.Settings(topk=16)
run = DeviceRun(inp, dev)
run.blank_step_kernels()
run.step()
torch.cuda.synchronize()
res["step_clean"] = T.get_device_status(clear=True)
T.test_hooks(1)
run.step()
torch.cuda.synchronize()
res["step_hooked"] = T.get_device_status(clear=True)
T.test_hooks(0)
run.blank_step_kernels()
run.idx.fill_(-7)
run.out.fill_(float("nan"))
run.step()
torch.cuda.synchronize()
res["step_after"] = T.get_device_status(clear=True)
sel = O.run_selection(inp, st)
got = run.gpu_blocks(sel.keys())
res["step_after_selection_exact"] = all(np.array_equal(got[u], s.blocks) for u, s in sel.items())
check_attention(run, O.run_attention(inp, st, got))
res["step_after_matches_oracle"] = True
print("RESULT " + json.dumps(res))
'''


@pytest.fixture(scope="module")
def child_result():
    import __graft_entry__
    __graft_entry__.build()
    sys.path.insert(0, os.path.join(ROOT, "trainable_block_sparse_infllm_gb300"))
    from build_lib import build
    build(checked=True)
    env = dict(os.environ, INFLLMV2_LIBRARY="checked")
    r = subprocess.run([sys.executable, "-c", "ROOT = " + repr(ROOT) + "\n" + CHILD], env=env,
                       capture_output=True, text=True, timeout=900)
    lines = [x for x in r.stdout.splitlines() if x.startswith("RESULT ")]
    assert r.returncode == 0 and lines, r.stdout[-3000:] + r.stderr[-3000:]
    return json.loads(lines[-1][len("RESULT "):])


BOUNDS, TIMEOUT = 0x4, 0x2


def test_checked_build_reports_no_false_alarm(child_result):
    for k in ("prefill_clean", "backward_clean", "decode_clean", "step_clean"):
        assert child_result[k] == 0, (k, child_result[k])


def test_checked_build_flags_out_of_range_indices(child_result):
    for k in ("prefill_bad", "backward_bad", "decode_bad"):
        assert child_result[k] & BOUNDS, (k, child_result[k])
        assert not child_result[k] & TIMEOUT, (k, child_result[k])
    assert child_result["prefill_valid_units_match"]


def test_bounded_wait_expires_and_the_call_returns(child_result):
    assert child_result["step_hooked"] & TIMEOUT, child_result["step_hooked"]
    assert child_result["step_after"] == 0, child_result["step_after"]
    assert child_result["step_after_selection_exact"]
    assert child_result["step_after_matches_oracle"]
