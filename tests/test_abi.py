"""The C-ABI library loads and exports every symbol include/gdn.h and include/gdn_testing.h
declare, and its
host-side logic (argument checks, workspace sizing, slot validation, status strings)
behaves as documented. No call here reaches a kernel launch: every argument error
returns before any CUDA call, so these run without a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import gated_deltanet_linear_gdn_gb300 as gdn
from gated_deltanet_linear_gdn_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build_library()
    return gdn.lib()


def declared_functions(header="gdn.h"):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"gdn_conv_update", "gdn_decode_step", "gdn_chunked_prefill",
            "gdn_chunked_prefill_workspace_size", "gdn_validate_slots",
            "gdn_status_string"} <= set(names)
    for n in names:
        assert hasattr(L, n), n
    testing = declared_functions("gdn_testing.h")
    assert testing == ["gdn_testing_set_fault"]
    assert hasattr(L, testing[0])


def test_testing_fault_rejects_unknown_modes(L):
    """An unknown mode is refused before any CUDA call (so this runs without a GPU)."""
    assert L.gdn_testing_set_fault(3) == gdn.GDN_ERR_INVALID_ARG
    assert L.gdn_testing_set_fault(-1) == gdn.GDN_ERR_INVALID_ARG


def test_status_strings(L):
    for s in range(4):
        assert gdn.status_string(s).startswith(["GDN_OK", "GDN_ERR_INVALID_ARG",
                                                "GDN_ERR_UNSUPPORTED", "GDN_ERR_CUDA"][s])


def test_validate_slots(L):
    assert gdn.gdn_validate_slots([1, 2, 0, -1, 0, 3], 4) == 0
    assert gdn.gdn_validate_slots([1, 4], 4) == 1
    assert gdn.gdn_validate_slots([3, 0, 3], 4) == 2
    assert gdn.gdn_validate_slots([], 1) == 0


def test_workspace_size_monotone(L):
    d = gdn.Dims(16, 32, 128, 128)
    a = gdn.gdn_chunked_prefill_workspace_size(4096, 1, d, 64)
    b = gdn.gdn_chunked_prefill_workspace_size(8192, 1, d, 64)
    c = gdn.gdn_chunked_prefill_workspace_size(4096, 8, d, 64)
    e = gdn.gdn_chunked_prefill_workspace_size(4096, 1, d, 16)
    assert 0 < a < b and a < c and e > 0
    assert gdn.gdn_chunked_prefill_workspace_size(4096, 1, d, 48) == 0
    assert gdn.gdn_chunked_prefill_workspace_size(0, 0, d, 64) > 0


P = ctypes.c_void_p
FAKE = P(0x10000)  # never dereferenced: every call below fails its checks first


def _conv(L, **kw):
    args = dict(x=FAKE, state=FAKE, dt=0, layout=0, w=FAKE, bias=None, silu=1, slot=FAKE, B=2,
                D=64, W=4, ns=4, out=FAKE)
    args.update(kw)
    return L.gdn_conv_update(args["x"], args["state"], args["dt"], args["layout"], args["w"],
                             args["bias"], args["silu"], args["slot"], args["B"], args["D"],
                             args["W"], args["ns"], args["out"], None, None)


def test_conv_update_argument_errors(L):
    assert _conv(L, B=0) == gdn.GDN_OK            # empty batch: no-op
    assert _conv(L, x=None) == gdn.GDN_ERR_INVALID_ARG
    assert _conv(L, slot=None) == gdn.GDN_ERR_INVALID_ARG
    assert _conv(L, B=-1) == gdn.GDN_ERR_INVALID_ARG
    assert _conv(L, dt=7) == gdn.GDN_ERR_INVALID_ARG
    assert _conv(L, layout=5) == gdn.GDN_ERR_INVALID_ARG
    assert _conv(L, W=3) == gdn.GDN_ERR_UNSUPPORTED
    assert _conv(L, D=60) == gdn.GDN_ERR_UNSUPPORTED
    assert _conv(L, x=P(0x10002)) == gdn.GDN_ERR_INVALID_ARG  # misaligned


def _decode(L, dims=None, **kw):
    d = dims or gdn.Dims(2, 4, 32, 32)
    args = dict(mixed=FAKE, a=FAKE, b=FAKE, gm=0, A=FAKE, dt=FAKE, cw=None, cb=None, silu=1,
                cs=None, cdt=0, lay=0, ssm=FAKE, slot=FAKE, B=2, ns=8, scale=0.1, l2=1,
                gate=None, out=FAKE, odt=1)
    args.update(kw)
    return L.gdn_decode_step(args["mixed"], args["a"], args["b"], args["gm"], args["A"],
                             args["dt"], args["cw"], args["cb"], args["silu"], args["cs"],
                             args["cdt"], args["lay"], args["ssm"], args["slot"], args["B"],
                             args["ns"], d.c(), args["scale"], args["l2"], args["gate"],
                             args["out"], args["odt"], None, None)


def test_decode_argument_errors(L):
    assert _decode(L, B=0) == gdn.GDN_OK
    assert _decode(L, ssm=None) == gdn.GDN_ERR_INVALID_ARG
    assert _decode(L, A=None) == gdn.GDN_ERR_INVALID_ARG          # fused gates need A_log
    assert _decode(L, cw=FAKE, cs=None) == gdn.GDN_ERR_INVALID_ARG  # conv needs its state
    assert _decode(L, ns=0) == gdn.GDN_ERR_INVALID_ARG
    assert _decode(L, dims=gdn.Dims(3, 4, 32, 32)) == gdn.GDN_ERR_INVALID_ARG  # Hv % Hk
    assert _decode(L, dims=gdn.Dims(2, 4, 48, 48)) == gdn.GDN_ERR_UNSUPPORTED
    assert _decode(L, dims=gdn.Dims(2, 4, 32, 64)) == gdn.GDN_ERR_UNSUPPORTED
    assert _decode(L, dims=gdn.Dims(1, 8, 32, 32)) == gdn.GDN_ERR_UNSUPPORTED
    assert _decode(L, cw=FAKE, cs=FAKE, dims=gdn.Dims(2, 4, 32, 32, 3)) == gdn.GDN_ERR_UNSUPPORTED
    assert _decode(L, mixed=P(0x10008)) == gdn.GDN_ERR_INVALID_ARG  # misaligned
    assert _decode(L, odt=9) == gdn.GDN_ERR_INVALID_ARG


def _gate_struct(z=FAKE, w=FAKE, off=0.0, eps=1e-6, act=0):
    g = gdn.gdn_output_gate(z, w, off, eps, act)
    return ctypes.byref(g), g


def test_output_gate_argument_errors(L):
    """Every call here fails a host check before anything is launched."""
    for kw, want in [(dict(z=None), gdn.GDN_ERR_INVALID_ARG),
                     (dict(w=None), gdn.GDN_ERR_INVALID_ARG),
                     (dict(z=P(0x10008)), gdn.GDN_ERR_INVALID_ARG),   # z not 16-byte aligned
                     (dict(w=P(0x10004)), gdn.GDN_ERR_INVALID_ARG),   # weight not 16-byte aligned
                     (dict(act=2), gdn.GDN_ERR_INVALID_ARG),
                     (dict(eps=-1.0), gdn.GDN_ERR_INVALID_ARG),
                     (dict(eps=float("nan")), gdn.GDN_ERR_INVALID_ARG),
                     (dict(eps=float("inf")), gdn.GDN_ERR_INVALID_ARG),
                     (dict(off=float("nan")), gdn.GDN_ERR_INVALID_ARG)]:
        ref, _keep = _gate_struct(**kw)
        assert _decode(L, gate=ref) == want, kw
    ref, _keep = _gate_struct()
    assert _decode(L, gate=ref, out=P(0x10004)) == gdn.GDN_ERR_INVALID_ARG  # gated out 16 B
    assert _decode(L, gate=ref, ssm=None) == gdn.GDN_ERR_INVALID_ARG  # layer checks come first


def test_prefill_argument_errors(L):
    d = gdn.Dims(2, 4, 32, 32)

    def call(**kw):
        args = dict(cu=FAKE, slot=FAKE, N=1, T=8, chunk=16, ws=FAKE, nbytes=1 << 30, mixed=FAKE,
                    gate=None)
        args.update(kw)
        return L.gdn_chunked_prefill(args["mixed"], FAKE, FAKE, 0, FAKE, FAKE, None, None, 1,
                                     None, 0, 0, FAKE, args["cu"], args["slot"], None, args["N"],
                                     args["T"], 8, d.c(), 0.1, 1, args["chunk"], args["gate"],
                                     FAKE, 1, args["ws"], args["nbytes"], None, None)

    assert call(N=0, T=0) == gdn.GDN_OK
    assert call(N=0, T=5) == gdn.GDN_ERR_INVALID_ARG
    assert call(chunk=48) == gdn.GDN_ERR_UNSUPPORTED
    assert call(cu=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(ws=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(nbytes=16) == gdn.GDN_ERR_INVALID_ARG
    assert call(mixed=None) == gdn.GDN_ERR_INVALID_ARG


def test_prefill_bf16_output_alignment(L):
    """The dk = dv = 128 state pass stores a bf16 output 16 bytes at a time."""
    d = gdn.Dims(16, 32, 128, 128)

    def call(out, out_dtype):
        return L.gdn_chunked_prefill(FAKE, FAKE, FAKE, 0, FAKE, FAKE, None, None, 1, None, 0, 0,
                                     FAKE, FAKE, FAKE, None, 1, 8, 8, d.c(), 0.1, 1, 64, None,
                                     out, out_dtype, FAKE, 1 << 40, None, None)

    assert call(P(0x10004), 0) == gdn.GDN_ERR_INVALID_ARG   # bf16, 4-byte aligned


def test_mixed_step_argument_errors(L):
    """The mixed step's own checks, then each part's, all before any launch."""
    d = gdn.Dims(2, 4, 32, 32)

    def call(**kw):
        args = dict(nd=1, nseq=1, T=8, cu=FAKE, slot=FAKE, ssm=FAKE, chunk=16, ws=FAKE,
                    nbytes=1 << 30)
        args.update(kw)
        return L.gdn_mixed_step(FAKE, FAKE, FAKE, 0, FAKE, FAKE, None, None, 1, None, 0, 0,
                                args["ssm"], args["slot"], args["nd"], args["cu"], None,
                                args["nseq"], args["T"], 8, d.c(), 0.1, 1, args["chunk"], None,
                                FAKE, 1, args["ws"], args["nbytes"], None, None)

    assert call(nd=0, nseq=0, T=0) == gdn.GDN_OK              # nothing to do
    assert call(nd=-1) == gdn.GDN_ERR_INVALID_ARG
    assert call(nseq=-1) == gdn.GDN_ERR_INVALID_ARG
    assert call(nseq=0, T=4) == gdn.GDN_ERR_INVALID_ARG       # tokens without sequences
    assert call(ssm=None) == gdn.GDN_ERR_INVALID_ARG          # the decode part's check
    assert call(nseq=0, T=0, slot=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(nd=0, cu=None) == gdn.GDN_ERR_INVALID_ARG     # the prefill part's checks
    assert call(nd=0, ws=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(chunk=48) == gdn.GDN_ERR_UNSUPPORTED


def test_noalloc_prefill_argument_errors(L):
    """Size checks of the fixed-scratch entry point: all before it looks up its array."""
    d = gdn.Dims(16, 32, 128, 128)

    def call(N=1, T=8, chunk=64, mixed=FAKE, cu=FAKE):
        return L.gdn_chunked_prefill_noalloc(mixed, FAKE, FAKE, 0, FAKE, FAKE, None, None, 1,
                                             None, 0, 0, FAKE, cu, FAKE, None, N, T, 8, d.c(),
                                             0.1, 1, chunk, None, FAKE, 1, None, None)

    assert call(N=-1) == gdn.GDN_ERR_INVALID_ARG
    # sizes that fit the scratch, but a null pointer: refused before the array's look-up
    # (no CUDA call, so this runs without a GPU)
    assert call(mixed=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(cu=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(N=0, T=0) == gdn.GDN_OK                        # the ordinary no-op
    assert call(T=-1) == gdn.GDN_ERR_INVALID_ARG
    assert call(T=200_000) == gdn.GDN_ERR_SCRATCH_LIMIT       # ~13 GB of workspace > 64 MiB
    assert call(chunk=48) == gdn.GDN_ERR_UNSUPPORTED          # the ordinary entry point's verdict


def test_graph_create_argument_errors(L):
    d = gdn.Dims(2, 4, 32, 32)
    h = ctypes.c_void_p(0x1234)

    def call(batch=1, out=True):
        return L.gdn_decode_graph_create(FAKE, FAKE, FAKE, 0, FAKE, FAKE, None, None, 1, None, 0,
                                         0, FAKE, FAKE, batch, 8, d.c(), 0.1, 1, None, FAKE, 1,
                                         None, ctypes.byref(h) if out else None)

    assert call(out=False) == gdn.GDN_ERR_INVALID_ARG
    assert call(batch=0) == gdn.GDN_ERR_INVALID_ARG
    assert h.value is None                                     # cleared on failure


def test_binding_refuses_missing_library(monkeypatch, tmp_path):
    """No CPU fallback: without the shared library every entry point raises."""
    monkeypatch.setattr(gdn, "_lib", None)
    monkeypatch.setattr(gdn, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError):
        gdn.gdn_validate_slots(np.array([1], np.int32), 2)
