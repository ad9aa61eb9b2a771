"""Output gate of the GDN block fused into the decode step (gated RMSNorm with z; RL-Kernel PR
#469 "C6: GDN decode-step goldens and recurrent/conv state contract", Summary by CodeRabbit and
Walkthrough on the stacked gated-RMSNorm PRs #466-#468: SiLU or sigmoid gating and a weight
offset). The gated call must leave every state exactly as the ungated call does, and its output
must be the gate applied to the same fp32 core output.

Bounds. The decode core output o carries the decode tolerance e = 1e-3 * max|o_ref| (absolute).
y = o / r * w' * act(z) with r = sqrt(mean(o^2) + eps) per head; perturbing o by at most e moves r
by at most e (r is 1-Lipschitz in the max norm), so |dy_i| <= |w'_i act(z_i)| * e * (1 + |o_i| / r)
/ r. The bf16 store adds half a ULP of y."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_gdn_gb300 as gdn
from gated_deltanet_linear_gdn_gb300 import inputs as gi

from _harness import (Device, OracleRun, bits_to_torch, dims_of, gpu_decode, ssm_host,
                      tensor_hash)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_gdn_gb300 import build
    build.build_library()
    import oracle
    oracle.lib()
    assert torch.cuda.is_available()


def gate_inputs(geo, B, seed, offset=0.0, eps=1e-6, act="silu"):
    rng = np.random.default_rng(seed)
    z = gi.f32_to_bf16_bits(rng.standard_normal((B, geo.Hv, geo.dv), dtype=np.float32) * 2)
    w = (rng.standard_normal(geo.dv) * 0.5 + (0.0 if offset else 1.0)).astype(np.float32)
    g = gdn.OutputGate(bits_to_torch(z).cuda(), torch.from_numpy(w).cuda(), weight_offset=offset,
                       eps=eps, act=act)
    return z, w, g


def gate_bound(o_ref, z, w, offset, eps, act, y_ref, bf16_out):
    zf = gi.bf16_bits_to_f32(z).astype(np.float64)
    sig = 1.0 / (1.0 + np.exp(-zf))
    actv = zf * sig if act == "silu" else sig
    r = np.sqrt(np.mean(o_ref * o_ref, axis=-1, keepdims=True) + eps)
    e = 1e-3 * np.abs(o_ref).max()
    bound = np.abs((w.astype(np.float64) + offset) * actv) * e * (1.0 + np.abs(o_ref) / r) / r
    bound += 1e-6 * np.abs(y_ref).max()
    if bf16_out:
        bound += np.ldexp(1.0, np.frexp(np.abs(y_ref))[1] - 9)
    return bound


def torch_gate_f32(o, z_bits, w, offset, eps, act):
    """Plain PyTorch fp32 reference of the gate (same op, same precision)."""
    zf = bits_to_torch(z_bits).float()
    ms = (o * o).mean(dim=-1, keepdim=True)
    g = torch.nn.functional.silu(zf) if act == "silu" else torch.sigmoid(zf)
    return o * torch.rsqrt(ms + eps) * (torch.from_numpy(w) + offset) * g


CASES = [
    ("tiny", gi.TINY, 5, 9, "silu", 0.0, False),
    ("tiny-sig-off", gi.TINY, 5, 9, "sigmoid", 1.0, False),
    ("qwen-b64", gi.QWEN3_NEXT, 64, 128, "silu", 0.0, False),
    ("qwen-b64-bf16state", gi.QWEN3_NEXT, 64, 128, "silu", 0.0, True),
    ("head64-r4", gi.Geometry(2, 8, 64, 64), 7, 16, "silu", 1.0, False),
]


@pytest.mark.parametrize("name,geo,B,ns,act,offset,sbf16", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out_f32", [True, False])
def test_decode_gated_matches_oracle_and_keeps_states(name, geo, B, ns, act, offset, sbf16,
                                                       out_f32):
    import oracle
    inp = gi.make_inputs(geo, [1] * B, ns, seed=400 + B, state_bf16=sbf16)
    inp.slot[1] = 0  # one inactive row
    z, w, g = gate_inputs(geo, B, seed=500 + B, offset=offset, act=act)
    ref = OracleRun(inp)
    y_ref = oracle.gated_rmsnorm(ref.out, z, w, offset=offset, eps=1e-6, act=act)
    y_ref[1] = 0.0

    dg, dp = Device(inp), Device(inp)
    y = gpu_decode(dg, out_f32=out_f32, gate=g)
    o = gpu_decode(dp, out_f32=True)
    torch.cuda.synchronize()
    assert int(dg.err.item()) == 0
    # the gate changes nothing but the output
    assert torch.equal(dg.ssm, dp.ssm) and torch.equal(dg.conv_state, dp.conv_state)
    yh = y.float().cpu().numpy().astype(np.float64)
    assert np.all(yh[1] == 0.0)
    bound = gate_bound(ref.out, z, w, offset, 1e-6, act, y_ref, not out_f32)
    assert np.all(np.abs(yh - y_ref) <= bound)
    # against a plain fp32 gate applied to this GPU's own ungated o (identical fp32 o)
    yt = torch_gate_f32(o.cpu(), z, w, offset, 1e-6, act).numpy()
    yt[1] = 0.0
    tol = 2e-6 * np.abs(yt).max() + (np.ldexp(1.0, np.frexp(np.abs(yt))[1] - 8) if not out_f32 else 0)
    assert np.all(np.abs(yh - yt) <= tol)


def test_decode_gated_bitwise_replay_and_graph():
    geo, B, ns = gi.QWEN3_NEXT, 16, 64
    inp = gi.make_inputs(geo, [1] * B, ns, seed=77)
    z, w, g = gate_inputs(geo, B, seed=78)
    hashes = set()
    for _ in range(3):
        d = Device(inp)
        y = gpu_decode(d, out_f32=False, gate=g)
        torch.cuda.synchronize()
        hashes.add((tensor_hash(y), tensor_hash(d.ssm), tensor_hash(d.conv_state)))
    assert len(hashes) == 1
    # a captured gated step replays bitwise like the direct call
    d = Device(inp)
    out = torch.empty(B, geo.Hv, geo.dv, dtype=torch.bfloat16, device="cuda")
    graph = gdn.DecodeGraph(d.mixed, d.a, d.b, d.A_log, d.dt_bias, d.conv_w, d.conv_b,
                            d.conv_state, d.ssm, d.slot, out, dims_of(geo), gate=g, err=d.err)
    graph.launch()
    torch.cuda.synchronize()
    assert (tensor_hash(out), tensor_hash(d.ssm), tensor_hash(d.conv_state)) in hashes
    graph.close()


PREFILL_CASES = [
    ("tiny-c16", gi.TINY, [1, 37, 0, 20], 16, "silu", 0.0, False),
    ("head128-c64", gi.Geometry(1, 2, 128, 128), [70, 5, 130], 64, "silu", 0.0, False),
    ("head128-c16-sig-bf16state", gi.Geometry(1, 2, 128, 128), [70, 130], 16, "sigmoid", 1.0, True),
]


@pytest.mark.parametrize("name,geo,lengths,chunk,act,offset,sbf16", PREFILL_CASES,
                         ids=[c[0] for c in PREFILL_CASES])
@pytest.mark.parametrize("out_f32", [True, False])
def test_prefill_gated_matches_oracle_and_keeps_states(name, geo, lengths, chunk, act, offset,
                                                        sbf16, out_f32):
    """The prefill gates o as stored in the output dtype (a bf16 output is rounded first), so
    the bf16 bound adds that rounding (half a ULP of each o) to the prefill tolerance."""
    import oracle
    from _harness import gpu_prefill
    inp = gi.make_inputs(geo, lengths, 12, seed=600 + len(lengths), state_bf16=sbf16)
    T = inp.total_tokens
    z, w, g = gate_inputs(geo, T, seed=601, offset=offset, act=act)
    ref = OracleRun(inp)
    y_ref = oracle.gated_rmsnorm(ref.out, z, w, offset=offset, eps=1e-6, act=act)

    dg, dp = Device(inp), Device(inp)
    y = gpu_prefill(dg, chunk=chunk, out_f32=out_f32, gate=g)
    o = gpu_prefill(dp, chunk=chunk, out_f32=out_f32)
    torch.cuda.synchronize()
    assert int(dg.err.item()) == 0
    assert torch.equal(dg.ssm, dp.ssm) and torch.equal(dg.conv_state, dp.conv_state)
    yh = y.float().cpu().numpy().astype(np.float64)
    # decode-style bound with the prefill tolerance, plus the bf16 rounding of o
    zf = gi.bf16_bits_to_f32(z).astype(np.float64)
    sig = 1.0 / (1.0 + np.exp(-zf))
    actv = zf * sig if act == "silu" else sig
    r = np.sqrt(np.mean(ref.out * ref.out, axis=-1, keepdims=True) + 1e-6)
    e = 5e-3 * np.abs(ref.out).max()
    if not out_f32:
        e = e + np.ldexp(1.0, np.frexp(np.abs(ref.out).max(axis=-1, keepdims=True))[1] - 9)
    bound = np.abs((w.astype(np.float64) + offset) * actv) * e * (1.0 + np.abs(ref.out) / r) / r
    bound = bound + 1e-6 * np.abs(y_ref).max()
    if not out_f32:
        bound = bound + np.ldexp(1.0, np.frexp(np.abs(y_ref))[1] - 9)
    assert np.all(np.abs(yh - y_ref) <= bound)
    # against a plain fp32 gate applied to this GPU's own ungated output (same stored o)
    yt = torch_gate_f32(o.float().cpu(), z, w, offset, 1e-6, act).numpy()
    tol = 2e-6 * np.abs(yt).max() + (np.ldexp(1.0, np.frexp(np.abs(yt))[1] - 8) if not out_f32 else 0)
    assert np.all(np.abs(yh - yt) <= tol)
