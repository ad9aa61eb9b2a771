"""GPU parity of the chunked prefill against the fp64 token-by-token oracle, through
the C ABI: tiny and Qwen3-Next shapes, ragged lengths (1, 2, 3, lengths off the chunk
grid), chunk sizes 16/32/64, conv on and bypassed, initial states on and off, inactive,
invalid and empty sequences, the correlated-key adversarial case, bitwise replay and
packing invariance.

Bounds: output (f32 store) and final state max|err| / max|ref| <= 5e-3; final conv
state bitwise; bf16 output = RNE of the f32 output, bitwise.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_gdn_gb300 as gdn
from gated_deltanet_linear_gdn_gb300 import inputs as gi

from _harness import (Device, OracleRun, bf16_store_within, dims_of, gpu_prefill, rel_err,
                      tensor_hash, torch_to_bits)

pytestmark = pytest.mark.gpu

PREFILL_TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_gdn_gb300 import build
    build.build_library()
    import oracle
    oracle.lib()
    assert torch.cuda.is_available()


def check_prefill(inp, chunk=64, head_mask=None, bf16_too=True, tol=PREFILL_TOL):
    ref = OracleRun(inp, head_mask=head_mask)
    d = Device(inp)
    out = gpu_prefill(d, chunk=chunk, out_f32=True)
    torch.cuda.synchronize()
    assert int(d.err.item()) == (ref.err if ref.err else 0)
    hm = np.ones(inp.geo.Hv, bool) if head_mask is None else np.asarray(head_mask, bool)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got[:, hm]))
    assert rel_err(got[:, hm], ref.out[:, hm]) <= tol
    ssm = d.ssm.cpu().numpy()
    act = ref.sel[1:]
    if act.size:
        assert rel_err(ssm[act][:, hm], ref.ssm[1:][:, hm]) <= tol
    untouched = np.setdiff1d(np.arange(inp.num_slots), act)
    assert np.array_equal(ssm[untouched], inp.ssm_state[untouched])
    if inp.conv_state is not None:
        cs = d.conv_state_host()
        assert np.array_equal(cs[act], ref.conv[1:])
        assert np.array_equal(cs[untouched], inp.conv_state[untouched])
    if bf16_too:
        d2 = Device(inp)
        o16 = gpu_prefill(d2, chunk=chunk, out_f32=False)
        torch.cuda.synchronize()
        bits = torch_to_bits(o16)
        assert np.array_equal(bits, torch_to_bits(out.to(torch.bfloat16)))
        assert bf16_store_within(bits[:, hm], ref.out[:, hm], tol)
    return ref, d, out


def test_prefill_tiny_chunk16():
    check_prefill(gi.tiny_prefill(seed=0), chunk=16)


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("conv_f32", [False, True])
def test_prefill_ragged_tiny(chunk, conv_f32):
    lens = [1, 2, 3, 17, 64, 100, 5]
    inp = gi.make_inputs(gi.TINY, lens, 12, seed=chunk + conv_f32, conv_f32=conv_f32,
                         has_init=[1, 0, 1, 1, 0, 1, 1])
    check_prefill(inp, chunk=chunk)


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("conv_f32", [False, True])
def test_prefill_ragged_head128(chunk, conv_f32):
    """dk = dv = 128 (the tensor-core path): ragged lengths around and across the chunk
    grid, initial states on and off, several sequences packed."""
    lens = [1, 2, 3, 17, 64, 100, 5, 130]
    inp = gi.make_inputs(gi.Geometry(1, 2, 128, 128), lens, 12, seed=40 + chunk + conv_f32,
                         conv_f32=conv_f32, has_init=[1, 0, 1, 1, 0, 1, 1, 1])
    check_prefill(inp, chunk=chunk)


@pytest.mark.parametrize("layout", [0, 1])
def test_prefill_variants(layout):
    # conv bypass + direct gates; no L2 norm; Hv/Hk = 1 and 4; dk = 64 and 128
    check_prefill(gi.make_inputs(gi.TINY, [33, 7], 5, seed=1, conv=False, gate_direct=True))
    inp = gi.make_inputs(gi.TINY, [40, 9], 5, seed=2, conv_layout=layout)
    inp.qk_l2norm = False
    check_prefill(inp, chunk=16)
    check_prefill(gi.make_inputs(gi.Geometry(4, 4, 64, 64), [70, 3], 5, seed=3,
                                 conv_layout=layout), chunk=32)
    check_prefill(gi.make_inputs(gi.Geometry(2, 8, 128, 128), [130, 1], 5, seed=4,
                                 conv_layout=layout, conv_f32=True))


def test_prefill_slot_contract_and_empty_sequences():
    inp = gi.make_inputs(gi.TINY, [5, 0, 9, 4, 0, 6], 8, seed=5,
                         slots=[3, 5, 0, 8, 2, -1], has_init=[1, 0, 1, 1, 1, 1])
    ref, d, out = check_prefill(inp, chunk=16)
    assert int(d.err.item()) & gdn.GDN_DEVERR_SLOT_RANGE
    o = out.cpu().numpy()
    cu = inp.cu_seqlens
    for i in (2, 3, 5):   # inactive or invalid: zero outputs
        assert np.all(o[cu[i]:cu[i + 1]] == 0)
    # the empty sequence without an initial state (slot 5) ends with zero state and window
    assert np.all(d.ssm[5].cpu().numpy() == 0)
    assert np.all(d.conv_state_host()[5] == 0)


@pytest.mark.parametrize("geo", [gi.TINY, gi.Geometry(1, 2, 128, 128)], ids=["tiny", "head128"])
def test_prefill_more_sequences_than_ranked(geo):
    """1,100 sequences, more than the chunk-table kernel ranks by length (1,024): mostly 0..4
    tokens, a few longer ones, some inactive slots and some without an initial state."""
    rng = np.random.default_rng(1100)
    n = 1100
    lens = rng.integers(0, 5, n)
    lens[rng.choice(n, 6, replace=False)] = [40, 70, 129, 150, 64, 200]
    slots = rng.permutation(np.arange(1, 1201))[:n]
    slots[rng.choice(n, 20, replace=False)] = 0
    slots[rng.choice(n, 5, replace=False)] = -1
    inp = gi.make_inputs(geo, [int(x) for x in lens], 1201, seed=1101, slots=list(slots),
                         has_init=list(rng.integers(0, 2, n)))
    for chunk in (16, 64):
        check_prefill(inp, chunk=chunk, bf16_too=False)


@pytest.mark.parametrize("chunk", [32, 64])
def test_prefill_pieces_with_empty_and_short_sequences(chunk):
    """A call of few (sequence, value head) pairs and enough chunks runs in pieces: here two
    empty sequences (one with an initial state, one without), a 3-token one that ends in the
    first piece, and two that carry their state across pieces."""
    lens = [0, 1500, 3, 0, 700]
    inp = gi.make_inputs(gi.Geometry(1, 2, 128, 128), lens, 8, seed=1500 + chunk,
                         has_init=[1, 0, 1, 0, 1])
    m = (sum(lens) + len(lens) * (chunk - 1)) // chunk
    assert len(lens) * 2 <= 64 and m >= 16        # the piece rule applies
    ref, d, out = check_prefill(inp, chunk=chunk)
    s_empty = int(inp.slot[3])                    # empty, no initial state: zero state and window
    assert np.all(d.ssm[s_empty].cpu().numpy() == 0)
    assert np.all(d.conv_state_host()[s_empty] == 0)


def test_prefill_bad_cu_seqlens_sets_error():
    inp = gi.make_inputs(gi.TINY, [5, 6], 4, seed=6)
    d = Device(inp)
    d.cu = torch.tensor([0, 7, 6], dtype=torch.int32, device="cuda")   # decreasing
    before = d.ssm.clone()
    gpu_prefill(d, chunk=16)
    torch.cuda.synchronize()
    assert int(d.err.item()) & gdn.GDN_DEVERR_SEQLENS
    assert torch.equal(d.ssm, before)


def test_prefill_single_sequence_4096():
    """One sequence of 4096 tokens, chunk 64, conv bypassed, k L2-normalised at the input,
    zero initial state (Qwen3-Next geometry)."""
    check_prefill(gi.prefill_single(4096, seed=0), chunk=64, bf16_too=False)


def test_prefill_varlen_32k_sampled_heads():
    """Eight sequences of lengths ~U[1, 8192] (~32k tokens), conv on, random initial states
    in shuffled slots; outputs and states compared on every fifth value head."""
    inp = gi.prefill_varlen(8, 8192, seed=0)
    check_prefill(inp, chunk=64, head_mask=np.arange(32) % 5 == 0, bf16_too=False)


@pytest.mark.parametrize("chunk", [16, 64])
def test_prefill_correlated_keys(chunk):
    """64 tokens of correlated keys, beta = 0.9, g = 0, zero state, all 32 heads: finite and
    within the bound (the case where a 3-round bf16 Newton-Schulz inverse fails)."""
    check_prefill(gi.correlated_keys(64, seed=0), chunk=chunk)


def test_prefill_bitwise_replay():
    inp = gi.prefill_varlen(4, 700, seed=3, num_slots=16)
    hashes = set()
    for _ in range(5):
        d = Device(inp)
        out = gpu_prefill(d, chunk=64, out_f32=False)
        torch.cuda.synchronize()
        hashes.add((tensor_hash(out), tensor_hash(d.ssm), tensor_hash(d.conv_state)))
    assert len(hashes) == 1


@pytest.mark.parametrize("geo,chunk,lens", [
    (gi.TINY, 16, [37, 64, 1, 150, 9]),
    # dk = dv = 128, the tensor-core path: the intra kernel packs 128 / C chunks into one
    # 128-row MMA tile, so odd chunk counts move every later sequence's chunks to another
    # tile position between compositions
    (gi.QWEN3_NEXT, 64, [37, 64, 1, 150, 9, 200]),
    (gi.QWEN3_NEXT, 16, [37, 64, 1, 150, 9, 200]),
])
def test_prefill_packing_invariance(geo, chunk, lens):
    """Each sequence alone, packed with the others, and packed in another order (with
    shuffled cache blocks) gives bitwise the same outputs, final recurrent states and final
    conv windows."""
    inp = gi.make_inputs(geo, lens, 16, seed=8)
    d = Device(inp)
    full = gpu_prefill(d, chunk=chunk, out_f32=False)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    full_bits = torch_to_bits(full)
    cu = inp.cu_seqlens
    rng = np.random.default_rng(1)
    orders = ([[i] for i in range(len(lens))] + [list(rng.permutation(len(lens)))]
              + [list(rng.permutation(len(lens)))[:3]])
    for order in orders:
        perm = np.concatenate([[0], 1 + rng.permutation(inp.num_slots - 1)])  # 0 stays null
        inv = np.argsort(perm)
        toks = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in order]).astype(np.int64)
        sub = gi.LayerInputs(**{**inp.__dict__})
        sub.mixed, sub.a, sub.b = inp.mixed[toks], inp.a[toks], inp.b[toks]
        sub.slot = inv[inp.slot[order]].astype(np.int32)
        sub.cu_seqlens = np.concatenate([[0], np.cumsum([lens[i] for i in order])]).astype(np.int32)
        sub.conv_state = np.ascontiguousarray(inp.conv_state[perm])
        sub.ssm_state = np.ascontiguousarray(inp.ssm_state[perm])
        ds = Device(sub)
        o = gpu_prefill(ds, chunk=chunk, out_f32=False)
        torch.cuda.synchronize()
        assert int(ds.err.item()) == 0
        assert np.array_equal(torch_to_bits(o), full_bits[toks])
        sl = inp.slot[order]
        assert torch.equal(ds.ssm.cpu()[inv[sl]], d.ssm.cpu()[sl])
        assert torch.equal(ds.conv_state.cpu()[inv[sl]], d.conv_state.cpu()[sl])


def _pieces_alone_equals_packed(geo, lens, chunk, state_bf16, seed):
    """The first sequence alone (in pieces) against the whole list packed (one piece): outputs,
    final state and conv window bitwise. Returns the alone call's inputs."""
    inp = gi.make_inputs(geo, lens, 64, seed=seed, state_bf16=state_bf16)
    d = Device(inp)
    full = gpu_prefill(d, chunk=chunk, out_f32=False)
    torch.cuda.synchronize()
    assert int(d.err.item()) == 0
    full_bits = torch_to_bits(full)
    sub = gi.LayerInputs(**{**inp.__dict__})
    n0 = lens[0]
    sub.mixed, sub.a, sub.b = inp.mixed[:n0], inp.a[:n0], inp.b[:n0]
    sub.slot = inp.slot[:1].copy()
    sub.cu_seqlens = np.array([0, n0], np.int32)
    sub.has_init = None if inp.has_init is None else inp.has_init[:1].copy()
    ds = Device(sub)
    o = gpu_prefill(ds, chunk=chunk, out_f32=False)
    torch.cuda.synchronize()
    assert int(ds.err.item()) == 0
    assert np.array_equal(torch_to_bits(o), full_bits[:n0])
    s0 = int(inp.slot[0])
    assert torch.equal(ds.ssm.cpu()[s0], d.ssm.cpu()[s0])
    assert torch.equal(ds.conv_state.cpu()[s0], d.conv_state.cpu()[s0])
    return sub


@pytest.mark.parametrize("chunk,state_bf16", [(64, False), (32, False), (64, True)])
def test_prefill_pieces_bitwise(chunk, state_bf16):
    """A long sequence alone runs its chunks in pieces (its intra kernel beside its state pass,
    the fp32 state handed from piece to piece); packed with 44 other sequences it runs in one
    piece. Its outputs, final state and conv window are bitwise the same either way (with a
    bf16 state too: the state crosses piece boundaries unrounded)."""
    _pieces_alone_equals_packed(gi.QWEN3_NEXT, [4096, 37, 150, 9, 200] + [5] * 40, chunk,
                                state_bf16, seed=12)


def test_prefill_pieces_bitwise_four_value_heads_per_k_head():
    """Hv / Hk = 4: alone, the sequence's first intra piece splits its CTAs four ways by value
    head; packed with 14 others (120 sequence-head pairs) nothing is split. Bitwise the same,
    and the alone call matches the oracle."""
    geo = gi.Geometry(2, 8, 128, 128)
    sub = _pieces_alone_equals_packed(geo, [1500, 37, 150, 9, 200] + [5] * 10, 64, False,
                                      seed=13)
    check_prefill(sub, chunk=64, bf16_too=False)


def test_prefill_then_decode_continues_the_state():
    """A prefill followed by decode steps equals the oracle run over the whole stream."""
    import oracle
    geo = gi.TINY
    inp = gi.make_inputs(geo, [45], 4, seed=9, slots=[2])
    ref = OracleRun(inp)
    d = Device(inp)
    gpu_prefill(d, chunk=16)
    for step in range(4):
        st = gi.make_inputs(geo, [1], 4, seed=50 + step, slots=[2])
        from _harness import bits_to_torch, gpu_decode
        d.mixed = bits_to_torch(st.mixed).cuda()
        d.a, d.b = bits_to_torch(st.a).cuda(), bits_to_torch(st.b).cuda()
        d.inp = gi.LayerInputs(**{**inp.__dict__, "slot": st.slot, "cu_seqlens": st.cu_seqlens})
        out = gpu_decode(d, out_f32=True)
        o, _, _ = oracle.layer(st.mixed, st.a, st.b, False, inp.A_log, inp.dt_bias, inp.conv_w,
                               inp.conv_b, True, ref.conv, False, 0, ref.ssm,
                               np.array([0, 1], np.int32), ref.slot_c, None, geo.Hk, geo.Hv,
                               geo.dk, geo.dv)
        torch.cuda.synchronize()
        assert rel_err(out.cpu().numpy(), o) <= PREFILL_TOL
