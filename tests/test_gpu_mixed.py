"""Mixed decode + prefill steps (gdn_mixed_step), after the RL-Kernel PR #469 page's section "Not
reproducible from this branch: the mixed decode+prefill measurement": there, the decode rows
of a step that also holds a prefill went through another kernel and their results changed
with the step's composition. Here a mixed step must equal the separate decode and prefill calls
bitwise -- outputs, recurrent states and conv states -- for every composition, including the
page's case of one decode request in three different prefill-bearing steps."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_gdn_gb300 as gdn
from gated_deltanet_linear_gdn_gb300 import inputs as gi

from _harness import Device, OracleRun, bits_to_torch, dims_of, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_gdn_gb300 import build
    build.build_library()
    import oracle
    oracle.lib()
    assert torch.cuda.is_available()


def workspace(T, N, geo, chunk):
    nb = gdn.gdn_chunked_prefill_workspace_size(T, max(N, 1), dims_of(geo), chunk)
    return torch.empty(nb, dtype=torch.uint8, device="cuda")


def run_mixed(inp, nd, chunk, out_f32=True, gate=None):
    """One mixed call over a Device copy of inp (decode rows = its first nd sequences)."""
    geo = inp.geo
    d = Device(inp)
    T = inp.total_tokens - nd
    N = inp.slot.size - nd
    cu = torch.from_numpy((inp.cu_seqlens[nd:] - nd).astype(np.int32)).cuda()
    hi = None if d.has_init is None else d.has_init[nd:].contiguous()
    out = torch.empty(inp.total_tokens, geo.Hv, geo.dv,
                      dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    gdn.gdn_mixed_step(d.mixed, d.a, d.b, d.A_log, d.dt_bias, d.conv_w, d.conv_b, d.conv_state,
                       d.ssm, d.slot, nd, cu, hi, out, workspace(T, N, geo, chunk) if N else None,
                       dims_of(geo), chunk=chunk, silu=inp.silu, scale=inp.scale, gate=gate,
                       err=d.err)
    return d, out


def run_separate(inp, nd, chunk, out_f32=True, gate=None):
    """The same step as a decode call on rows [0, nd) and a prefill call on the rest."""
    geo = inp.geo
    d = Device(inp)
    dt = torch.float32 if out_f32 else torch.bfloat16
    out = torch.empty(inp.total_tokens, geo.Hv, geo.dv, dtype=dt, device="cuda")
    if nd:
        gd = None
        if gate is not None:
            gd = gdn.OutputGate(gate.z[:nd], gate.weight, weight_offset=gate._c.weight_offset,
                                eps=gate._c.eps, act="silu" if gate._c.act == 0 else "sigmoid")
        gdn.gdn_decode_step(d.mixed[:nd], d.a[:nd], d.b[:nd], d.A_log, d.dt_bias, d.conv_w,
                            d.conv_b, d.conv_state, d.ssm, d.slot[:nd], out[:nd], dims_of(geo),
                            silu=inp.silu, scale=inp.scale, gate=gd, err=d.err)
    T = inp.total_tokens - nd
    N = inp.slot.size - nd
    if N:
        gp = None
        if gate is not None:
            gp = gdn.OutputGate(gate.z[nd:], gate.weight, weight_offset=gate._c.weight_offset,
                                eps=gate._c.eps, act="silu" if gate._c.act == 0 else "sigmoid")
        cu = torch.from_numpy((inp.cu_seqlens[nd:] - nd).astype(np.int32)).cuda()
        hi = None if d.has_init is None else d.has_init[nd:].contiguous()
        gdn.gdn_chunked_prefill(d.mixed[nd:], d.a[nd:], d.b[nd:], d.A_log, d.dt_bias, d.conv_w,
                                d.conv_b, d.conv_state, d.ssm, cu, d.slot[nd:], hi, out[nd:],
                                workspace(T, N, geo, chunk), dims_of(geo), chunk=chunk,
                                silu=inp.silu, scale=inp.scale, gate=gp, err=d.err)
    return d, out


COMPOSITIONS = [
    ("decode-only", gi.QWEN3_NEXT, 8, [], 64, False),
    ("prefill-only", gi.QWEN3_NEXT, 0, [90, 200], 64, False),
    ("one-decode-one-prefill", gi.QWEN3_NEXT, 1, [300], 64, False),
    ("b64-three-prefills", gi.QWEN3_NEXT, 64, [130, 1, 77], 64, False),
    ("tiny-cuda-core-prefill", gi.TINY, 5, [40, 17], 16, False),
    ("b16-two-prefills-bf16-state", gi.QWEN3_NEXT, 16, [70, 129], 64, True),
    # prefills of few sequences and at least 16 chunks run in pieces; the decode rows then run
    # beside the last pass piece
    ("b32-pieced-prefill", gi.QWEN3_NEXT, 32, [1500], 64, False),
    ("b8-pieced-two-prefills-bf16-state", gi.QWEN3_NEXT, 8, [1100, 40], 64, True),
]


@pytest.mark.parametrize("name,geo,nd,lengths,chunk,sbf16", COMPOSITIONS,
                         ids=[c[0] for c in COMPOSITIONS])
def test_mixed_step_equals_separate_calls_bitwise(name, geo, nd, lengths, chunk, sbf16):
    inp = gi.make_inputs(geo, [1] * nd + lengths, 512 if geo is gi.QWEN3_NEXT else 32,
                         seed=700 + nd + len(lengths), state_bf16=sbf16,
                         has_init=[1] * nd + [1, 0, 1][:len(lengths)] if lengths else True)
    dm, om = run_mixed(inp, nd, chunk)
    ds, os_ = run_separate(inp, nd, chunk)
    torch.cuda.synchronize()
    assert int(dm.err.item()) == 0 and int(ds.err.item()) == 0
    assert torch.equal(om, os_)
    assert torch.equal(dm.ssm, ds.ssm)
    assert torch.equal(dm.conv_state, ds.conv_state)


def test_decode_rows_do_not_depend_on_the_step_composition():
    """The page's case: one decode request, fp32 state, in three prefill-bearing steps."""
    geo = gi.QWEN3_NEXT
    base = gi.make_inputs(geo, [1], 512, seed=801)
    results = []
    for lengths in ([257], [31, 64, 900], [5, 5, 5, 5]):
        rng = np.random.default_rng(sum(lengths))
        step = gi.make_inputs(geo, [1] + lengths, 512, seed=900 + len(lengths))
        # the decode row (row 0, its slot and every pool entry it reads) is the same in every step
        step.mixed[0] = base.mixed[0]
        step.a[0], step.b[0] = base.a[0], base.b[0]
        step.A_log, step.dt_bias = base.A_log, base.dt_bias
        step.conv_w, step.conv_b = base.conv_w, base.conv_b
        s0 = int(base.slot[0])
        others = [s for s in rng.permutation(np.arange(1, 512)) if s != s0][:len(lengths)]
        step.slot = np.array([s0] + others, dtype=np.int32)
        step.ssm_state[s0] = base.ssm_state[s0]
        step.conv_state[s0] = base.conv_state[s0]
        d, out = run_mixed(step, 1, 64, out_f32=False)
        torch.cuda.synchronize()
        results.append((out[0].clone(), d.ssm[s0].clone(), d.conv_state[s0].clone()))
    for r in results[1:]:
        assert all(torch.equal(x, y) for x, y in zip(results[0], r))


def test_mixed_step_matches_the_oracle():
    geo = gi.QWEN3_NEXT
    inp = gi.make_inputs(geo, [1] * 6 + [70, 129], 64, seed=811)
    ref = OracleRun(inp)
    d, out = run_mixed(inp, 6, 64)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert rel_err(o[:6], ref.out[:6]) <= 1e-3
    assert rel_err(o[6:], ref.out[6:]) <= 5e-3
    ssm = d.ssm.cpu().numpy()
    assert rel_err(ssm[ref.sel[1:]], ref.ssm[1:]) <= 5e-3


def test_gated_mixed_step_equals_separate_gated_calls():
    geo = gi.QWEN3_NEXT
    nd, lengths = 16, [100, 60]
    inp = gi.make_inputs(geo, [1] * nd + lengths, 128, seed=821)
    rng = np.random.default_rng(822)
    z = bits_to_torch(gi.f32_to_bf16_bits(rng.standard_normal((inp.total_tokens, geo.Hv, geo.dv),
                                                              dtype=np.float32))).cuda()
    w = torch.from_numpy(rng.standard_normal(geo.dv).astype(np.float32)).cuda()
    g = gdn.OutputGate(z, w, eps=1e-6)
    dm, om = run_mixed(inp, nd, 64, out_f32=False, gate=g)
    ds, os_ = run_separate(inp, nd, 64, out_f32=False, gate=g)
    torch.cuda.synchronize()
    assert torch.equal(om, os_) and torch.equal(dm.ssm, ds.ssm)
    assert torch.equal(dm.conv_state, ds.conv_state)
