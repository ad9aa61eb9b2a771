"""CUDA-graph decode buckets (gdn_decode_graph_create / gdn_graph_launch), after the Rocket
post "A reduction barrier makes Qwen GDN graph replay bit exact": per bucket c1..c1024, a
replay equals the direct decode call bitwise and agrees with the fp64 oracle (on sampled
rows: each row depends only on its own inputs and slot); five replays from the same pools
hash identically; a c16 -> c1 transition zeroes the 15 inactive rows; slot 0 is never
touched.

The slot pool (1100 slots, Qwen3-Next geometry, 2.3 GB of fp32 state) is drawn on the
device; the oracle gets host copies of the slots a sampled row touches."""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_gdn_gb300 as gdn
from gated_deltanet_linear_gdn_gb300 import inputs as gi

from _harness import OracleRun, bf16_store_within, bits_to_torch, dims_of, rel_err, torch_to_bits

pytestmark = pytest.mark.gpu

GEO = gi.QWEN3_NEXT
NS = 1100
DECODE_TOL = 1e-3
ORACLE_ROWS = 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_gdn_gb300 import build
    build.build_library()
    import oracle
    oracle.lib()
    assert torch.cuda.is_available()


@pytest.fixture(scope="module")
def pools():
    prm = gi.make_inputs(GEO, [1], 2, seed=70, state_pool=False)
    g = torch.Generator(device="cuda")
    g.manual_seed(71)
    conv = torch.empty(NS, GEO.D, GEO.W - 1, dtype=torch.float32, device="cuda")
    conv.normal_(0.0, 1.0, generator=g)
    conv = conv.to(torch.bfloat16)
    ssm = gi.device_state_pool(NS, GEO, 0.05, seed=72)
    return dict(prm=prm, conv=conv, ssm=ssm, w=bits_to_torch(prm.conv_w).cuda(),
                cb=bits_to_torch(prm.conv_b).cuda(), A_log=torch.from_numpy(prm.A_log).cuda(),
                dt=torch.from_numpy(prm.dt_bias).cuda())


class Step:
    """Host and device inputs of one bucket step: `rows` rows, the first `active` live on
    distinct shuffled slots, the rest on slot 0."""

    def __init__(self, rows, active, seed):
        st = gi.make_inputs(GEO, [1] * rows, 2, seed=seed, conv=False, state_pool=False,
                            slots=[0] * rows)
        rng = np.random.default_rng(seed + 5000)
        slot = np.zeros(rows, np.int32)
        slot[:active] = 1 + rng.permutation(NS - 1)[:active]
        self.mixed, self.a, self.b, self.slot = st.mixed, st.a, st.b, slot
        self.x = bits_to_torch(st.mixed).cuda()
        self.ta = bits_to_torch(st.a).cuda()
        self.tb = bits_to_torch(st.b).cuda()
        self.tslot = torch.from_numpy(slot).cuda()


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

    def run(self, st: Step):
        self.x.copy_(st.x); self.a.copy_(st.ta); self.b.copy_(st.tb); self.slot.copy_(st.tslot)
        self.g.launch()


def direct(p, x, a, b, slot, conv, ssm):
    out = torch.empty(x.shape[0], GEO.Hv, GEO.dv, dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_step(x, a, b, p["A_log"], p["dt"], p["w"], p["cb"], conv, ssm, slot, out,
                        dims_of(GEO))
    return out


def digest(t: torch.Tensor) -> tuple:
    """Device-side digest of a tensor's bits (replays compare digests; equality of the
    tensors themselves is asserted separately)."""
    u = t.contiguous().flatten().view(torch.int32).to(torch.int64)
    idx = torch.arange(u.numel(), device=u.device, dtype=torch.int64)
    return int(u.sum()), int((u * (idx % 65521 + 1)).sum())


def oracle_check(p, st: Step, out, conv0, ssm0, conv1, ssm1, rows_idx):
    """Sampled rows of one step against the oracle, from host copies of their slots before
    the step (conv0, ssm0) and the GPU's state after it (conv1, ssm1)."""
    prm = p["prm"]
    sl = st.slot[rows_idx].astype(np.int64)
    tsl = torch.from_numpy(sl).cuda()
    n = sl.size
    ssm_c = np.zeros((n + 1, GEO.Hv, GEO.dv, GEO.dk), np.float32)
    ssm_c[1:] = ssm0[tsl].cpu().numpy()
    conv_c = np.zeros((n + 1, GEO.D, GEO.W - 1), np.uint16)
    conv_c[1:] = torch_to_bits(conv0[tsl])
    inp = gi.LayerInputs(GEO, st.mixed[rows_idx], st.a[rows_idx], st.b[rows_idx], False,
                         prm.A_log, prm.dt_bias, prm.conv_w, prm.conv_b, True, conv_c, False, 0,
                         ssm_c, np.arange(1, n + 1, dtype=np.int32),
                         np.arange(n + 1, dtype=np.int32), None, float(GEO.dk ** -0.5))
    ref = OracleRun(inp)
    bits = torch_to_bits(out[torch.from_numpy(rows_idx).cuda()])
    assert bf16_store_within(bits, ref.out, DECODE_TOL)
    assert rel_err(ssm1[tsl].cpu().numpy(), ref.ssm[1:]) <= DECODE_TOL
    assert np.array_equal(torch_to_bits(conv1[tsl]), ref.conv[1:])


@pytest.mark.parametrize("rows", [1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024])
def test_replay_equals_direct_call_and_the_oracle(pools, rows):
    p = pools
    conv0, ssm0 = p["conv"].clone(), p["ssm"].clone()
    bucket = Bucket(rows, p)
    st = Step(rows, rows, seed=rows)
    touched = torch.from_numpy(st.slot.astype(np.int64)).cuda()
    # direct call on copies of the pools
    conv_d, ssm_d = conv0.clone(), ssm0.clone()
    out_d = direct(p, st.x, st.ta, st.tb, st.tslot, conv_d, ssm_d)
    digests = set()
    for _ in range(5):
        p["conv"].copy_(conv0); p["ssm"].copy_(ssm0)
        bucket.run(st)
        torch.cuda.synchronize()
        assert torch.equal(bucket.out, out_d)
        assert torch.equal(p["ssm"], ssm_d) and torch.equal(p["conv"], conv_d)
        digests.add((digest(bucket.out), digest(p["ssm"][touched]), digest(p["conv"][touched])))
    assert len(digests) == 1
    assert int(bucket.err.item()) == 0
    rng = np.random.default_rng(rows)
    idx = (np.arange(rows) if rows <= ORACLE_ROWS
           else np.sort(rng.choice(rows, ORACLE_ROWS, replace=False)))
    oracle_check(p, st, bucket.out, conv0, ssm0, p["conv"], p["ssm"], idx)
    p["conv"].copy_(conv0); p["ssm"].copy_(ssm0)
    bucket.g.close()


def test_bucket_transition_clears_inactive_rows_and_keeps_slot0(pools):
    p = pools
    conv0, ssm0 = p["conv"].clone(), p["ssm"].clone()
    c16 = Bucket(16, p)
    c16.run(Step(16, 16, seed=90))
    torch.cuda.synchronize()
    assert torch.all(c16.out.abs().sum(dim=(1, 2)) > 0)
    # one live row in the same graph: the other 15 rows become inactive (slot 0)
    st1 = Step(16, 1, seed=91)
    ssm_before = p["ssm"].clone(); conv_before = p["conv"].clone()
    c16.run(st1)
    torch.cuda.synchronize()
    assert torch.all(c16.out[1:] == 0)
    assert torch.equal(p["ssm"][0], ssm0[0]) and torch.equal(p["conv"][0], conv0[0])
    diff = (p["ssm"] != ssm_before).flatten(1).any(dim=1)
    assert diff.nonzero().flatten().tolist() == [int(st1.slot[0])]
    # the live row matches a direct single-row call from the same pools, and the oracle
    conv_d, ssm_d = conv_before.clone(), ssm_before.clone()
    out_d = direct(p, st1.x[:1], st1.ta[:1], st1.tb[:1], st1.tslot[:1], conv_d, ssm_d)
    assert torch.equal(c16.out[:1], out_d)
    assert torch.equal(p["ssm"], ssm_d)
    oracle_check(p, st1, c16.out, conv_before, ssm_before, p["conv"], p["ssm"], np.array([0]))
    p["conv"].copy_(conv0); p["ssm"].copy_(ssm0)
    c16.g.close()


def test_graph_steps_chain_like_direct_calls(pools):
    """Three successive replays with new inputs equal three direct calls (state carried)."""
    p = pools
    conv0, ssm0 = p["conv"].clone(), p["ssm"].clone()
    c4 = Bucket(4, p)
    conv_d, ssm_d = conv0.clone(), ssm0.clone()
    for step in range(3):
        st = Step(4, 4, seed=200)   # the same slots every step
        st2 = Step(4, 4, seed=300 + step)
        st.x, st.ta, st.tb = st2.x, st2.ta, st2.tb
        out_d = direct(p, st.x, st.ta, st.tb, st.tslot, conv_d, ssm_d)
        c4.run(st)
        torch.cuda.synchronize()
        assert torch.equal(c4.out, out_d)
    assert torch.equal(p["ssm"], ssm_d) and torch.equal(p["conv"], conv_d)
    p["conv"].copy_(conv0); p["ssm"].copy_(ssm0)
    c4.g.close()
