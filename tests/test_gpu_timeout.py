"""The kernels' bounded waits running out, on the GPU, without faulting or hanging anything
(include/gdn_testing.h): one wait is made to wait for a barrier that nothing arrives on, with a
10 ms bound, and the tests check what the library promises then -- GDN_DEVERR_TIMEOUT in the
caller's error word, slots the call does not address untouched, the call ending in bounded
time, and the context still usable: the same call without the fault matches the oracle.

The prefill case is the one the CPU model of the state pass's failure path
(tests/test_pass_failure_model.py) found: compute warp 0 of the pass's first CTA gives up while
the next chunk's tiles are being copied in; the CTA must drain those copies before it frees its
tensor memory and exits. Every other (sequence, value head) is computed as usual and is checked
against the oracle; the failed one keeps its initial state.
"""
import time

import numpy as np
import pytest
import torch

import gated_deltanet_linear_gdn_gb300 as gdn
from gated_deltanet_linear_gdn_gb300 import inputs as gi

from _harness import Device, OracleRun, gpu_decode, gpu_prefill, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_gdn_gb300 import build
    build.build_library()
    import oracle
    oracle.lib()
    assert torch.cuda.is_available()


@pytest.fixture
def fault():
    yield gdn.gdn_testing_set_fault
    gdn.gdn_testing_set_fault(gdn.GDN_TEST_FAULT_NONE)


def test_decode_wait_runs_out_sets_timeout_and_leaves_other_slots(fault):
    inp = gi.decode_sweep(64, seed=31, num_slots=200)   # 1024 units: the persistent kernel
    d = Device(inp)
    ssm0, conv0 = d.ssm.clone(), d.conv_state.clone()
    fault(gdn.GDN_TEST_FAULT_DECODE_CONSUMER)
    t0 = time.monotonic()
    gpu_decode(d, out_f32=True)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    fault(gdn.GDN_TEST_FAULT_NONE)
    assert int(d.err.item()) & gdn.GDN_DEVERR_TIMEOUT
    assert elapsed < 30.0
    untouched = torch.from_numpy(np.setdiff1d(np.arange(inp.num_slots), inp.slot)).cuda()
    assert torch.equal(d.ssm[untouched], ssm0[untouched])
    assert torch.equal(d.conv_state[untouched], conv0[untouched])
    # the context is still usable: the same call, fault off, matches the oracle
    ref = OracleRun(inp)
    d2 = Device(inp)
    out = gpu_decode(d2, out_f32=True)
    torch.cuda.synchronize()
    assert int(d2.err.item()) == 0
    assert rel_err(out.cpu().numpy(), ref.out) <= 1e-3


def test_prefill_pass_wait_runs_out_drains_and_reports(fault):
    lens = [200, 150, 90]                                # sequence 0 is ranked first
    geo = gi.QWEN3_NEXT
    inp = gi.make_inputs(geo, lens, 10, seed=33)
    ref = OracleRun(inp)
    d = Device(inp)
    ssm0 = d.ssm.clone()
    fault(gdn.GDN_TEST_FAULT_PREFILL_PASS)
    t0 = time.monotonic()
    out = gpu_prefill(d, chunk=64, out_f32=True)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    fault(gdn.GDN_TEST_FAULT_NONE)
    assert int(d.err.item()) & gdn.GDN_DEVERR_TIMEOUT
    assert elapsed < 30.0
    ssm = d.ssm.cpu().numpy()
    s_fail = int(inp.slot[0])
    # the failed CTA (sequence 0, value head 0) stored no state
    assert np.array_equal(ssm[s_fail, 0], ssm0[s_fail, 0].cpu().numpy())
    # every other (sequence, value head): state and outputs as the oracle computes them
    for i, s in enumerate(inp.slot):
        k = int(np.nonzero(ref.sel == s)[0][0])
        heads = np.arange(geo.Hv) if i else np.arange(1, geo.Hv)
        assert rel_err(ssm[s][heads], ref.ssm[k][heads]) <= 5e-3
        bos, eos = inp.cu_seqlens[i], inp.cu_seqlens[i + 1]
        o = out[bos:eos].cpu().numpy()
        assert rel_err(o[:, heads], ref.out[bos:eos][:, heads]) <= 5e-3
    # the conv windows are written by their own kernel, unaffected
    conv = d.conv_state_host()
    for s in inp.slot:
        assert np.array_equal(conv[s], ref.conv[int(np.nonzero(ref.sel == s)[0][0])])
    untouched = np.setdiff1d(np.arange(inp.num_slots), inp.slot)
    assert np.array_equal(ssm[untouched], inp.ssm_state[untouched])
    # the context is still usable: the same call, fault off, matches the oracle
    d2 = Device(inp)
    out2 = gpu_prefill(d2, chunk=64, out_f32=True)
    torch.cuda.synchronize()
    assert int(d2.err.item()) == 0
    assert rel_err(out2.cpu().numpy(), ref.out) <= 5e-3
