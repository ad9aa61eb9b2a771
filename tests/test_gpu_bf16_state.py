"""bf16 recurrent-state storage (RL-Kernel PR #469 "C6: GDN decode-step goldens and
recurrent/conv state contract": Summary, state ABI -- fp32 arithmetic, the state rounded to its
storage dtype when written -- and Notes, "L1, and the bf16 recurrent state"): parity of decode
and prefill against the oracle in the same storage mode, and the page's fixed drift fixture
(B=8, 128 steps, seed 11) comparing an fp32-state run with a bf16-state run."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_gdn_gb300 import inputs as gi

from _harness import (Device, OracleRun, bf16_state_within, bits_to_torch, gpu_decode,
                      gpu_prefill, rel_err, ssm_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_gdn_gb300 import build
    build.build_library()
    import oracle
    oracle.lib()
    assert torch.cuda.is_available()


def check(inp, fn, tol, **kw):
    ref = OracleRun(inp)
    d = Device(inp)
    out = fn(d, out_f32=True, **kw)
    torch.cuda.synchronize()
    assert d.ssm.dtype == torch.bfloat16
    assert rel_err(out.cpu().numpy(), ref.out) <= tol
    got = ssm_host(d)
    act = ref.sel[1:]
    assert bf16_state_within(got[act], ref.ssm[1:], tol)
    untouched = np.setdiff1d(np.arange(inp.num_slots), act)
    assert np.array_equal(gi.f32_to_bf16_bits(got[untouched].astype(np.float32)),
                          inp.ssm_state[untouched])


@pytest.mark.parametrize("B", [1, 3, 64])
def test_decode_bf16_state(B):
    inp = gi.decode_sweep(B, seed=30 + B, num_slots=128, state_bf16=True)
    check(inp, gpu_decode, 1e-3)


def test_decode_bf16_state_tiny_and_f32_cache():
    check(gi.make_inputs(gi.TINY, [1] * 5, 9, seed=31, state_bf16=True), gpu_decode, 1e-3)
    check(gi.make_inputs(gi.TINY, [1] * 5, 9, seed=32, state_bf16=True, conv_f32=True,
                         conv_layout=1), gpu_decode, 1e-3)


@pytest.mark.parametrize("geo,chunk", [(gi.TINY, 16), (gi.Geometry(1, 2, 128, 128), 64),
                                       (gi.Geometry(1, 2, 128, 128), 16)])
def test_prefill_bf16_state(geo, chunk):
    inp = gi.make_inputs(geo, [1, 70, 5, 130], 10, seed=33, state_bf16=True,
                         has_init=[1, 1, 0, 1])
    check(inp, gpu_prefill, 5e-3, chunk=chunk)


def test_bf16_state_drift_fixture():
    """B=8, 128 decode steps, seed 11; gate inputs fixed, only the token changes. The bf16-state
    run drifts from the fp32-state run from the first step, stays within 5% relative, and the
    second half drifts at most twice the first half plus 1e-3 (the page's fixture bounds)."""
    geo = gi.QWEN3_NEXT
    B, steps = 8, 128
    base = gi.make_inputs(geo, [1] * B, 16, seed=11, state_bf16=True)
    d16 = Device(base)
    d32 = Device(base)
    d32.ssm = d16.ssm.float().clone()           # same (bf16-representable) starting state
    d32.conv_state = d16.conv_state.clone()
    rng = np.random.default_rng(11)
    drift = []
    slots = base.slot.astype(np.int64)
    for t in range(steps):
        x = gi.f32_to_bf16_bits(rng.standard_normal((B, geo.D), dtype=np.float32))
        d16.mixed = d32.mixed = bits_to_torch(x).cuda()
        gpu_decode(d16, out_f32=True)
        gpu_decode(d32, out_f32=True)
        s32 = d32.ssm[slots].double()
        s16 = d16.ssm[slots].double()
        drift.append(float((s16 - s32).abs().max() / s32.abs().max()))
    torch.cuda.synchronize()
    drift = np.array(drift)
    assert drift[0] > 0
    assert drift.max() < 0.05
    assert drift[steps // 2:].max() <= 2 * drift[:steps // 2].max() + 1e-3


def test_graph_replay_on_a_bf16_state_pool_equals_the_direct_call():
    """A captured decode step over a bf16 pool (gdn_decode_graph_create) replays bitwise like
    the direct call, state included."""
    import gated_deltanet_linear_gdn_gb300 as gdn
    from _harness import dims_of
    inp = gi.make_inputs(gi.QWEN3_NEXT, [1] * 8, 64, seed=41, state_bf16=True)
    dd, dg = Device(inp), Device(inp)
    want = gpu_decode(dd, out_f32=False)
    out = torch.empty_like(want)
    g = gdn.DecodeGraph(dg.mixed, dg.a, dg.b, dg.A_log, dg.dt_bias, dg.conv_w, dg.conv_b,
                        dg.conv_state, dg.ssm, dg.slot, out, dims_of(inp.geo), err=dg.err)
    g.launch()
    torch.cuda.synchronize()
    g.close()
    assert torch.equal(out, want)
    assert torch.equal(dg.ssm, dd.ssm) and torch.equal(dg.conv_state, dd.conv_state)
