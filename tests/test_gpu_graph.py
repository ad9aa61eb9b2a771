"""CUDA-graph decode buckets (gdn_decode_graph_create / gdn_graph_launch), after the Rocket
post "A reduction barrier makes Qwen GDN graph replay bit exact": per bucket c1..c16, a
replay equals the direct decode call bitwise; five replays from the same pools hash
identically; a c16 -> c1 transition zeroes the 15 inactive rows; slot 0 is never touched."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_gdn_gb300 as gdn
from gated_deltanet_linear_gdn_gb300 import inputs as gi

from _harness import bits_to_torch, dims_of, tensor_hash

pytestmark = pytest.mark.gpu

GEO = gi.QWEN3_NEXT
NS = 64


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_gdn_gb300 import build
    build.build_library()
    assert torch.cuda.is_available()


@pytest.fixture(scope="module")
def pools():
    inp = gi.make_inputs(GEO, [1] * 16, NS, seed=70)
    conv = bits_to_torch(inp.conv_state).cuda()
    ssm = torch.from_numpy(inp.ssm_state).cuda()
    w = bits_to_torch(inp.conv_w).cuda()
    cb = bits_to_torch(inp.conv_b).cuda()
    A_log = torch.from_numpy(inp.A_log).cuda()
    dt = torch.from_numpy(inp.dt_bias).cuda()
    return dict(conv=conv, ssm=ssm, w=w, cb=cb, A_log=A_log, dt=dt)


def step_inputs(rows, active, seed):
    """Inputs for a bucket of `rows` rows of which the first `active` are live."""
    st = gi.make_inputs(GEO, [1] * rows, NS, seed=seed, conv=False, state_pool=False)
    slot = np.zeros(rows, np.int32)
    slot[:active] = np.arange(1, active + 1) * 3  # distinct slots, never 0
    return (bits_to_torch(st.mixed).cuda(), bits_to_torch(st.a).cuda(),
            bits_to_torch(st.b).cuda(), torch.from_numpy(slot).cuda())


class Bucket:
    def __init__(self, rows, p):
        self.rows = rows
        self.x = torch.zeros(rows, GEO.D, dtype=torch.bfloat16, device="cuda")
        self.a = torch.zeros(rows, GEO.Hv, dtype=torch.bfloat16, device="cuda")
        self.b = torch.zeros(rows, GEO.Hv, dtype=torch.bfloat16, device="cuda")
        self.slot = torch.zeros(rows, dtype=torch.int32, device="cuda")
        self.out = torch.empty(rows, GEO.Hv, GEO.dv, dtype=torch.bfloat16, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.g = gdn.DecodeGraph(self.x, self.a, self.b, p["A_log"], p["dt"], p["w"], p["cb"],
                                 p["conv"], p["ssm"], self.slot, self.out, dims_of(GEO),
                                 err=self.err)

    def run(self, x, a, b, slot):
        self.x.copy_(x); self.a.copy_(a); self.b.copy_(b); self.slot.copy_(slot)
        self.g.launch()


def direct(p, x, a, b, slot, conv, ssm):
    out = torch.empty(x.shape[0], GEO.Hv, GEO.dv, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_step(x, a, b, p["A_log"], p["dt"], p["w"], p["cb"], conv, ssm, slot, out,
                        dims_of(GEO))
    return out


@pytest.mark.parametrize("rows", [1, 2, 4, 8, 16])
def test_replay_equals_direct_call_and_hashes_are_stable(pools, rows):
    p = pools
    conv0, ssm0 = p["conv"].clone(), p["ssm"].clone()
    bucket = Bucket(rows, p)
    x, a, b, slot = step_inputs(rows, rows, seed=rows)
    # direct call on copies of the pools
    conv_d, ssm_d = conv0.clone(), ssm0.clone()
    out_d = direct(p, x, a, b, slot, conv_d, ssm_d)
    hashes = set()
    for _ in range(5):
        p["conv"].copy_(conv0); p["ssm"].copy_(ssm0)
        bucket.run(x, a, b, slot)
        torch.cuda.synchronize()
        assert torch.equal(bucket.out, out_d)
        assert torch.equal(p["ssm"], ssm_d) and torch.equal(p["conv"], conv_d)
        hashes.add((tensor_hash(bucket.out), tensor_hash(p["ssm"]), tensor_hash(p["conv"])))
    assert len(hashes) == 1
    assert int(bucket.err.item()) == 0
    p["conv"].copy_(conv0); p["ssm"].copy_(ssm0)
    bucket.g.close()


def test_bucket_transition_clears_inactive_rows_and_keeps_slot0(pools):
    p = pools
    conv0, ssm0 = p["conv"].clone(), p["ssm"].clone()
    c16 = Bucket(16, p)
    x, a, b, slot = step_inputs(16, 16, seed=90)
    c16.run(x, a, b, slot)
    torch.cuda.synchronize()
    assert torch.all(c16.out.abs().sum(dim=(1, 2)) > 0)
    # one live row in the same graph: the other 15 rows become inactive (slot 0)
    x1, a1, b1, slot1 = step_inputs(16, 1, seed=91)
    ssm_before = p["ssm"].clone(); conv_before = p["conv"].clone()
    c16.run(x1, a1, b1, slot1)
    torch.cuda.synchronize()
    assert torch.all(c16.out[1:] == 0)
    assert torch.equal(p["ssm"][0], ssm0[0]) and torch.equal(p["conv"][0], conv0[0])
    changed = [s for s in range(NS) if not torch.equal(p["ssm"][s], ssm_before[s])]
    assert changed == [int(slot1[0])]
    # the live row matches a direct single-row call from the same pools
    conv_d, ssm_d = conv_before.clone(), ssm_before.clone()
    out_d = direct(p, x1[:1], a1[:1], b1[:1], slot1[:1], conv_d, ssm_d)
    assert torch.equal(c16.out[:1], out_d)
    assert torch.equal(p["ssm"], ssm_d)
    p["conv"].copy_(conv0); p["ssm"].copy_(ssm0)
    c16.g.close()


def test_graph_steps_chain_like_direct_calls(pools):
    """Three successive replays with new inputs equal three direct calls (state carried)."""
    p = pools
    conv0, ssm0 = p["conv"].clone(), p["ssm"].clone()
    c4 = Bucket(4, p)
    conv_d, ssm_d = conv0.clone(), ssm0.clone()
    for step in range(3):
        x, a, b, slot = step_inputs(4, 4, seed=200 + step)
        out_d = direct(p, x, a, b, slot, conv_d, ssm_d)
        c4.run(x, a, b, slot)
        torch.cuda.synchronize()
        assert torch.equal(c4.out, out_d)
    assert torch.equal(p["ssm"], ssm_d) and torch.equal(p["conv"], conv_d)
    p["conv"].copy_(conv0); p["ssm"].copy_(ssm0)
    c4.g.close()
