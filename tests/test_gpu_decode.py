"""GPU parity of the conv update and the fused decode step against the fp64 oracle,
through the C ABI, plus the slot contract, bitwise replay and batch invariance.

Bounds: conv state and slot bookkeeping bitwise; conv output within 1 bf16 ULP (bitwise
without SiLU, where the fp32 accumulation order is fixed on both sides); decode output
(f32 store) and state max|err| / max|ref| <= 1e-3; the bf16 output store is the RNE
rounding of the f32 output, bitwise, and so within 1e-3 max|ref| plus half a bf16 ULP of
the oracle elementwise.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_gdn_gb300 as gdn
from gated_deltanet_linear_gdn_gb300 import inputs as gi

from _harness import (Device, OracleRun, bf16_store_within, bf16_ulp_diff, bits_to_torch,
                      gpu_decode, rel_err, tensor_hash, torch_to_bits)

pytestmark = pytest.mark.gpu

DECODE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_gdn_gb300 import build
    build.build_library()
    import oracle
    oracle.lib()
    assert torch.cuda.is_available()


# --------------------------------------------------------------------------- conv update

@pytest.mark.parametrize("conv_f32", [False, True])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("bias,silu", [(True, True), (False, False), (True, False)])
def test_conv_update_parity(conv_f32, layout, bias, silu):
    import oracle
    geo = gi.QWEN3_NEXT
    B, ns = 17, 40
    inp = gi.make_inputs(geo, [1] * B, ns, seed=21, conv_f32=conv_f32, conv_layout=layout,
                         bias=bias, conv_w_std=0.5, slots=list(range(3, 3 + B - 2)) + [0, -1])
    d = Device(inp)
    out = torch.empty(B, geo.D, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_conv_update(d.mixed, d.conv_state, d.conv_w, d.conv_b, d.slot, out, silu=silu,
                        conv_layout=layout, err=d.err)
    torch.cuda.synchronize()
    ref_state = inp.conv_state.copy()
    ref_bits, _, err = oracle.conv_update(inp.mixed, ref_state, conv_f32, layout, inp.conv_w,
                                          inp.conv_b, silu, inp.slot, ns)
    assert err == 0 and int(d.err.item()) == 0
    assert np.array_equal(d.conv_state_host(), ref_state)          # roll: bitwise
    got = torch_to_bits(out)
    ulp = bf16_ulp_diff(got, ref_bits)
    if silu:
        assert ulp.max() <= 1
    else:
        assert ulp.max() == 0                                        # no SiLU: bitwise
    assert np.all(got[-2:] == 0)


def test_conv_update_out_of_range_slot_sets_error():
    geo = gi.TINY
    inp = gi.make_inputs(geo, [1, 1, 1], 6, seed=2, slots=[2, 6, 3])
    d = Device(inp)
    before = d.conv_state.clone()
    out = torch.full((3, geo.D), 7.0, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_conv_update(d.mixed, d.conv_state, d.conv_w, d.conv_b, d.slot, out, err=d.err)
    torch.cuda.synchronize()
    assert int(d.err.item()) & gdn.GDN_DEVERR_SLOT_RANGE
    assert torch.all(out[1] == 0)
    untouched = [0, 1, 4, 5]
    assert torch.equal(d.conv_state[untouched], before[untouched])


# --------------------------------------------------------------------------- decode

def check_decode(inp, out_bf16_too=True, head_mask=None):
    ref = OracleRun(inp, head_mask=head_mask)
    d = Device(inp)
    out32 = gpu_decode(d, out_f32=True)
    torch.cuda.synchronize()
    hm = np.ones(inp.geo.Hv, bool) if head_mask is None else np.asarray(head_mask, bool)
    got = out32.cpu().numpy()
    assert rel_err(got[:, hm], ref.out[:, hm]) <= DECODE_TOL
    ssm = d.ssm.cpu().numpy()
    act = ref.sel[1:]
    assert rel_err(ssm[act][:, hm], ref.ssm[1:][:, hm]) <= DECODE_TOL
    # slots the call does not touch keep their bits
    untouched = np.setdiff1d(np.arange(inp.num_slots), act)
    assert np.array_equal(ssm[untouched], inp.ssm_state[untouched])
    if inp.conv_state is not None:
        cs = d.conv_state_host()
        assert np.array_equal(cs[act], ref.conv[1:])
        assert np.array_equal(cs[untouched], inp.conv_state[untouched])
    if out_bf16_too:
        d2 = Device(inp)
        out16 = gpu_decode(d2, out_f32=False)
        torch.cuda.synchronize()
        bits = torch_to_bits(out16)
        assert np.array_equal(bits, torch_to_bits(out32.to(torch.bfloat16)))
        assert bf16_store_within(bits[:, hm], ref.out[:, hm], DECODE_TOL)
        assert torch.equal(d2.ssm, d.ssm)
    return ref, d


def test_decode_tiny():
    inp = gi.tiny_decode(seed=0)
    check_decode(inp)


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16, 64, 256])
def test_decode_qwen3_next_sweep(B):
    inp = gi.decode_sweep(B, seed=B)
    check_decode(inp)


@pytest.mark.parametrize("conv_f32,bias,silu", [(False, True, True), (True, True, True),
                                                (False, False, False), (True, False, True)])
def test_decode_batch_1024_over_2048_slots(conv_f32, bias, silu):
    inp = gi.decode_sweep(1024, seed=5, num_slots=2048, conv_f32=conv_f32, bias=bias, silu=silu)
    check_decode(inp, out_bf16_too=False, head_mask=np.arange(32) % 5 == 0)


@pytest.mark.parametrize("layout", [0, 1])
def test_decode_variants_tiny(layout):
    # conv bypass, direct gates, no L2 norm, tap-first conv layout, Hv/Hk = 1 and 4
    check_decode(gi.make_inputs(gi.TINY, [1] * 5, 9, seed=3, conv=False))
    check_decode(gi.make_inputs(gi.TINY, [1] * 5, 9, seed=4, gate_direct=True,
                                conv_layout=layout))
    inp = gi.make_inputs(gi.TINY, [1] * 5, 9, seed=5, conv_layout=layout)
    inp.qk_l2norm = False
    check_decode(inp)
    check_decode(gi.make_inputs(gi.Geometry(4, 4, 64, 64), [1] * 3, 5, seed=6,
                                conv_layout=layout))
    check_decode(gi.make_inputs(gi.Geometry(2, 8, 128, 128), [1] * 3, 5, seed=7,
                                conv_layout=layout, conv_f32=True))


def test_decode_slot_contract():
    inp = gi.make_inputs(gi.TINY, [1] * 5, 8, seed=9, slots=[0, 3, 8, -4, 5])
    d = Device(inp)
    before_ssm = d.ssm.clone()
    before_conv = d.conv_state.clone()
    out = gpu_decode(d, out_f32=True)
    torch.cuda.synchronize()
    assert int(d.err.item()) & gdn.GDN_DEVERR_SLOT_RANGE
    assert torch.all(out[[0, 2, 3]] == 0)
    keep = [0, 1, 2, 4, 6, 7]
    assert torch.equal(d.ssm[keep], before_ssm[keep])
    assert torch.equal(d.conv_state[keep], before_conv[keep])
    ref = OracleRun(inp)
    assert rel_err(out.cpu().numpy(), ref.out) <= DECODE_TOL


def test_decode_bitwise_replay():
    """Five runs from the same initial pools hash identically (outputs, conv, state)."""
    inp = gi.decode_sweep(64, seed=11)
    hashes = set()
    for _ in range(5):
        d = Device(inp)
        out = gpu_decode(d, out_f32=False)
        torch.cuda.synchronize()
        hashes.add((tensor_hash(out), tensor_hash(d.ssm), tensor_hash(d.conv_state)))
    assert len(hashes) == 1


def test_decode_batch_invariance():
    """Rows alone, sub-batches of 2 / 7 / 64 at offsets and a shuffled batch, with contiguous
    and shuffled cache blocks: outputs and state blocks bitwise equal to the full batch."""
    B, ns = 96, 200
    inp = gi.decode_sweep(B, seed=12, num_slots=ns)
    d = Device(inp)
    full = gpu_decode(d, out_f32=False)
    torch.cuda.synchronize()
    full_bits = torch_to_bits(full)
    full_ssm = d.ssm.cpu()
    full_conv = d.conv_state.cpu()
    rng = np.random.default_rng(0)
    subsets = [[0], [1], [31], [95], list(range(5, 7)), list(range(40, 47)), list(range(20, 84)),
               list(rng.permutation(B))]
    for rows in subsets:
        for shuffle_pool in (False, True):
            sub = gi.LayerInputs(**{**inp.__dict__})
            rows = np.asarray(rows)
            perm = (np.concatenate([[0], 1 + rng.permutation(ns - 1)]) if shuffle_pool
                    else np.arange(ns))  # slot 0 stays the null block
            inv = np.argsort(perm)
            sub.mixed, sub.a, sub.b = inp.mixed[rows], inp.a[rows], inp.b[rows]
            sub.slot = inv[inp.slot[rows]].astype(np.int32)
            sub.conv_state = np.ascontiguousarray(inp.conv_state[perm])
            sub.ssm_state = np.ascontiguousarray(inp.ssm_state[perm])
            sub.cu_seqlens = np.arange(rows.size + 1, dtype=np.int32)
            ds = Device(sub)
            o = gpu_decode(ds, out_f32=False)
            torch.cuda.synchronize()
            assert np.array_equal(torch_to_bits(o), full_bits[rows])
            sl = inp.slot[rows]
            assert torch.equal(ds.ssm.cpu()[inv[sl]], full_ssm[sl])
            assert torch.equal(ds.conv_state.cpu()[inv[sl]], full_conv[sl])


def test_decode_multi_step_chain():
    """Eight successive decode steps on the same slots stay within the bound."""
    import oracle
    inp = gi.tiny_decode(seed=1)
    geo = inp.geo
    d = Device(inp)
    ref = OracleRun(inp)  # step 0 on the oracle ...
    out = gpu_decode(d, out_f32=True)  # ... and on the GPU
    torch.cuda.synchronize()
    assert rel_err(out.cpu().numpy(), ref.out) <= DECODE_TOL
    for step in range(8):
        step_inp = gi.make_inputs(geo, [1, 1], 8, seed=100 + step, slots=inp.slot)
        d.mixed = bits_to_torch(step_inp.mixed).cuda()
        d.a = bits_to_torch(step_inp.a).cuda()
        d.b = bits_to_torch(step_inp.b).cuda()
        out = gpu_decode(d, out_f32=True)
        o, _, _ = oracle.layer(step_inp.mixed, step_inp.a, step_inp.b, False, inp.A_log,
                               inp.dt_bias, inp.conv_w, inp.conv_b, True, ref.conv, False, 0,
                               ref.ssm, np.arange(3, dtype=np.int32), ref.slot_c,
                               None, geo.Hk, geo.Hv, geo.dk, geo.dv)
        torch.cuda.synchronize()
        assert rel_err(out.cpu().numpy(), o) <= DECODE_TOL
    assert rel_err(d.ssm.cpu().numpy()[ref.sel[1:]], ref.ssm[1:]) <= DECODE_TOL
