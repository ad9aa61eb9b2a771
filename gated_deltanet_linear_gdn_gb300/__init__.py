"""GB300-native Gated DeltaNet (GDN) layer hot path.

A thin ctypes binding over ``libgdn.so`` (the C ABI of ``include/gdn.h``):
the functions below carry the C entry points' names and only marshal
arguments -- torch tensors in, device pointers and sizes out. Every step of
the layer runs in the library's CUDA kernels; there is no Python or CPU
fallback. If the library is missing or fails to load, every call raises.

torch is used only for device memory, streams and dtypes.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA = 0, 1, 2, 3
GDN_ERR_SCRATCH_LIMIT = 4
GDN_NOALLOC_SCRATCH_BYTES = 64 << 20
GDN_BF16, GDN_F32 = 0, 1
GDN_CONV_DIM_FIRST, GDN_CONV_TAP_FIRST = 0, 1
GDN_GATE_FUSED, GDN_GATE_DIRECT = 0, 1
GDN_DEVERR_SLOT_RANGE, GDN_DEVERR_SEQLENS, GDN_DEVERR_TIMEOUT = 1, 2, 4
GDN_TEST_FAULT_NONE, GDN_TEST_FAULT_DECODE_CONSUMER, GDN_TEST_FAULT_PREFILL_PASS = 0, 1, 2
GDN_ACT_SILU, GDN_ACT_SIGMOID = 0, 1


class GDNError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class gdn_dims(ctypes.Structure):
    _fields_ = [("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_k_dim", ctypes.c_int32), ("head_v_dim", ctypes.c_int32),
                ("conv_width", ctypes.c_int32), ("state_bf16", ctypes.c_int32)]


@dataclass(frozen=True)
class Dims:
    Hk: int
    Hv: int
    dk: int
    dv: int
    W: int = 4

    @property
    def D(self) -> int:
        return 2 * self.Hk * self.dk + self.Hv * self.dv

    def c(self, state_bf16: bool = False) -> gdn_dims:
        return gdn_dims(self.Hk, self.Hv, self.dk, self.dv, self.W, int(bool(state_bf16)))


class gdn_output_gate(ctypes.Structure):
    _fields_ = [("z", ctypes.c_void_p), ("weight", ctypes.c_void_p),
                ("weight_offset", ctypes.c_float), ("eps", ctypes.c_float),
                ("act", ctypes.c_int32)]


class OutputGate:
    """The GDN block's output gate (include/gdn.h, gdn_output_gate): out = o / rms(o) *
    (weight + weight_offset) * act(z) per value head. z: bf16 [tokens, Hv, dv] on the device;
    weight: f32 [dv] on the device; act "silu" or "sigmoid"."""

    def __init__(self, z, weight, *, weight_offset=0.0, eps=1e-6, act="silu"):
        if z.dtype != torch.bfloat16 or weight.dtype != torch.float32:
            raise ValueError("z must be bfloat16 and weight float32")
        self.z, self.weight = z, weight
        self._c = gdn_output_gate(_ptr(z), _ptr(weight), float(weight_offset), float(eps),
                                  {"silu": GDN_ACT_SILU, "sigmoid": GDN_ACT_SIGMOID}[act])

    def ref(self):
        return ctypes.byref(self._c)


def _gate(gate):
    return None if gate is None else gate.ref()


def _sdims(dims: "Dims", ssm_state) -> gdn_dims:
    """dims for a call: the state storage type follows the pool tensor's dtype."""
    if ssm_state.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("the recurrent state pool must be float32 or bfloat16")
    return dims.c(ssm_state.dtype == torch.bfloat16)


_lib = None


def lib():
    """Load libgdn.so (raises if it is absent: build it with build.build_library())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: the CUDA library must be built "
                               "(gated_deltanet_linear_gdn_gb300.build.build_library())")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        L.gdn_conv_update.restype = I32
        L.gdn_conv_update.argtypes = [P, P, I32, I32, P, P, I32, P, I32, I32, I32, I32, P, P, P]
        L.gdn_decode_step.restype = I32
        L.gdn_decode_step.argtypes = [P, P, P, I32, P, P, P, P, I32, P, I32, I32, P, P, I32, I32,
                                      gdn_dims, F, I32, P, P, I32, P, P]
        L.gdn_chunked_prefill_workspace_size.restype = ctypes.c_size_t
        L.gdn_chunked_prefill_workspace_size.argtypes = [I32, I32, gdn_dims, I32]
        L.gdn_chunked_prefill.restype = I32
        L.gdn_chunked_prefill.argtypes = [P, P, P, I32, P, P, P, P, I32, P, I32, I32, P, P, P, P,
                                          I32, I32, I32, gdn_dims, F, I32, I32, P, P, I32, P,
                                          ctypes.c_size_t, P, P]
        L.gdn_chunked_prefill_noalloc.restype = I32
        L.gdn_chunked_prefill_noalloc.argtypes = [P, P, P, I32, P, P, P, P, I32, P, I32, I32, P,
                                                  P, P, P, I32, I32, I32, gdn_dims, F, I32, I32,
                                                  P, P, I32, P, P]
        L.gdn_mixed_step.restype = I32
        L.gdn_mixed_step.argtypes = [P, P, P, I32, P, P, P, P, I32, P, I32, I32, P, P, I32, P, P,
                                     I32, I32, I32, gdn_dims, F, I32, I32, P, P, I32, P,
                                     ctypes.c_size_t, P, P]
        L.gdn_decode_graph_create.restype = I32
        L.gdn_decode_graph_create.argtypes = [P, P, P, I32, P, P, P, P, I32, P, I32, I32, P, P,
                                              I32, I32, gdn_dims, F, I32, P, P, I32, P,
                                              ctypes.POINTER(ctypes.c_void_p)]
        L.gdn_graph_launch.restype = I32
        L.gdn_graph_launch.argtypes = [P, P]
        L.gdn_graph_destroy.restype = None
        L.gdn_graph_destroy.argtypes = [P]
        L.gdn_validate_slots.restype = I32
        L.gdn_validate_slots.argtypes = [P, I32, I32]
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_status_string.argtypes = [I32]
        L.gdn_testing_set_fault.restype = I32
        L.gdn_testing_set_fault.argtypes = [I32]
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        if t.numel() and not t.is_cuda:
            raise ValueError("device tensors expected")
        if t.numel() and not t.is_contiguous():
            raise ValueError("contiguous tensors expected")
        return ctypes.c_void_p(t.data_ptr()) if t.numel() else None
    return ctypes.c_void_p(int(t))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dt(t) -> int:
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def _check(status: int):
    if status != GDN_OK:
        raise GDNError(status, lib().gdn_status_string(status).decode())


def status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


# --------------------------------------------------------------------------- entry points

def gdn_conv_update(x, conv_state, weight, bias, slot, out, *, silu=True,
                    conv_layout=GDN_CONV_DIM_FIRST, err=None, stream=None):
    """Decode conv update (in place on conv_state). x, out: [B, D] bf16."""
    B, D = x.shape
    _check(lib().gdn_conv_update(_ptr(x), _ptr(conv_state), _dt(conv_state), int(conv_layout),
                                 _ptr(weight), _ptr(bias), int(bool(silu)), _ptr(slot), B, D,
                                 weight.shape[1], conv_state.shape[0], _ptr(out), _ptr(err),
                                 _stream(stream)))


def _gate_mode(a):
    return GDN_GATE_DIRECT if a.dtype == torch.float32 else GDN_GATE_FUSED


def gdn_decode_step(mixed_qkv, a, b, A_log, dt_bias, conv_weight, conv_bias, conv_state,
                    ssm_state, slot, out, dims: Dims, *, silu=True,
                    conv_layout=GDN_CONV_DIM_FIRST, scale=None, qk_l2norm=True, gate=None,
                    err=None, stream=None):
    """One fused decode step (conv state and ssm_state updated in place).

    a, b: bf16 [B, Hv] (fused gates with A_log, dt_bias) or f32 g, beta (direct).
    gate: an OutputGate, or None for the plain core output."""
    B = mixed_qkv.shape[0]
    scale = dims.dk ** -0.5 if scale is None else scale
    conv_dt = _dt(conv_state) if conv_state is not None else GDN_BF16
    _check(lib().gdn_decode_step(
        _ptr(mixed_qkv), _ptr(a), _ptr(b), _gate_mode(a), _ptr(A_log), _ptr(dt_bias),
        _ptr(conv_weight), _ptr(conv_bias), int(bool(silu)), _ptr(conv_state), conv_dt,
        int(conv_layout), _ptr(ssm_state), _ptr(slot), B, ssm_state.shape[0],
        _sdims(dims, ssm_state), float(scale), int(bool(qk_l2norm)), _gate(gate), _ptr(out),
        _dt(out), _ptr(err), _stream(stream)))


def gdn_chunked_prefill_workspace_size(total_tokens, num_seqs, dims: Dims, chunk=64) -> int:
    return int(lib().gdn_chunked_prefill_workspace_size(int(total_tokens), int(num_seqs),
                                                        dims.c(), int(chunk)))


def gdn_chunked_prefill(mixed_qkv, a, b, A_log, dt_bias, conv_weight, conv_bias, conv_state,
                        ssm_state, cu_seqlens, slot, has_initial_state, out, workspace,
                        dims: Dims, *, chunk=64, silu=True, conv_layout=GDN_CONV_DIM_FIRST,
                        scale=None, qk_l2norm=True, gate=None, err=None, stream=None):
    """Chunked prefill over packed sequences (states updated in place by slot)."""
    T = mixed_qkv.shape[0]
    N = slot.shape[0]
    scale = dims.dk ** -0.5 if scale is None else scale
    conv_dt = _dt(conv_state) if conv_state is not None else GDN_BF16
    _check(lib().gdn_chunked_prefill(
        _ptr(mixed_qkv), _ptr(a), _ptr(b), _gate_mode(a), _ptr(A_log), _ptr(dt_bias),
        _ptr(conv_weight), _ptr(conv_bias), int(bool(silu)), _ptr(conv_state), conv_dt,
        int(conv_layout), _ptr(ssm_state), _ptr(cu_seqlens), _ptr(slot),
        _ptr(has_initial_state), N, T, ssm_state.shape[0], _sdims(dims, ssm_state),
        float(scale), int(bool(qk_l2norm)), int(chunk), _gate(gate), _ptr(out), _dt(out),
        _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err), _stream(stream)))


def gdn_chunked_prefill_noalloc(mixed_qkv, a, b, A_log, dt_bias, conv_weight, conv_bias,
                                conv_state, ssm_state, cu_seqlens, slot, has_initial_state, out,
                                dims: Dims, *, chunk=64, silu=True,
                                conv_layout=GDN_CONV_DIM_FIRST, scale=None, qk_l2norm=True,
                                gate=None, err=None, stream=None):
    """gdn_chunked_prefill without a caller workspace, for callers that cannot allocate device
    memory: the library's fixed GDN_NOALLOC_SCRATCH_BYTES array serves as the workspace.
    Raises GDNError(GDN_ERR_SCRATCH_LIMIT) when the call needs more than that. Calls that may
    overlap on the GPU share the array and race; make the first call on a device before any
    stream capture."""
    T = mixed_qkv.shape[0]
    N = slot.shape[0]
    scale = dims.dk ** -0.5 if scale is None else scale
    conv_dt = _dt(conv_state) if conv_state is not None else GDN_BF16
    _check(lib().gdn_chunked_prefill_noalloc(
        _ptr(mixed_qkv), _ptr(a), _ptr(b), _gate_mode(a), _ptr(A_log), _ptr(dt_bias),
        _ptr(conv_weight), _ptr(conv_bias), int(bool(silu)), _ptr(conv_state), conv_dt,
        int(conv_layout), _ptr(ssm_state), _ptr(cu_seqlens), _ptr(slot),
        _ptr(has_initial_state), N, T, ssm_state.shape[0], _sdims(dims, ssm_state),
        float(scale), int(bool(qk_l2norm)), int(chunk), _gate(gate), _ptr(out), _dt(out),
        _ptr(err), _stream(stream)))


def gdn_mixed_step(mixed_qkv, a, b, A_log, dt_bias, conv_weight, conv_bias, conv_state,
                   ssm_state, slot, num_decode, cu_seqlens, has_initial_state, out, workspace,
                   dims: Dims, *, chunk=64, silu=True, conv_layout=GDN_CONV_DIM_FIRST,
                   scale=None, qk_l2norm=True, gate=None, err=None, stream=None):
    """A step of num_decode decode rows followed by prefill sequences, packed in one token
    array (include/gdn.h, gdn_mixed_step). slot: decode rows' slots then one per prefill
    sequence; cu_seqlens: offsets within the prefill part; workspace: the prefill part's."""
    nd = int(num_decode)
    N = slot.shape[0] - nd
    T = mixed_qkv.shape[0] - nd
    scale = dims.dk ** -0.5 if scale is None else scale
    conv_dt = _dt(conv_state) if conv_state is not None else GDN_BF16
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().gdn_mixed_step(
        _ptr(mixed_qkv), _ptr(a), _ptr(b), _gate_mode(a), _ptr(A_log), _ptr(dt_bias),
        _ptr(conv_weight), _ptr(conv_bias), int(bool(silu)), _ptr(conv_state), conv_dt,
        int(conv_layout), _ptr(ssm_state), _ptr(slot), nd, _ptr(cu_seqlens),
        _ptr(has_initial_state), N, T, ssm_state.shape[0], _sdims(dims, ssm_state),
        float(scale), int(bool(qk_l2norm)), int(chunk), _gate(gate), _ptr(out), _dt(out),
        _ptr(workspace), ws_bytes, _ptr(err), _stream(stream)))


class DecodeGraph:
    """A captured decode step over fixed buffers (gdn_decode_graph_create). The tensors passed
    at creation are kept referenced here: write each step's inputs into them, then launch()."""

    def __init__(self, mixed_qkv, a, b, A_log, dt_bias, conv_weight, conv_bias, conv_state,
                 ssm_state, slot, out, dims: Dims, *, silu=True, conv_layout=GDN_CONV_DIM_FIRST,
                 scale=None, qk_l2norm=True, gate=None, err=None):
        self._keep = (mixed_qkv, a, b, A_log, dt_bias, conv_weight, conv_bias, conv_state,
                      ssm_state, slot, out, err, gate)
        B = mixed_qkv.shape[0]
        scale = dims.dk ** -0.5 if scale is None else scale
        conv_dt = _dt(conv_state) if conv_state is not None else GDN_BF16
        h = ctypes.c_void_p()
        _check(lib().gdn_decode_graph_create(
            _ptr(mixed_qkv), _ptr(a), _ptr(b), _gate_mode(a), _ptr(A_log), _ptr(dt_bias),
            _ptr(conv_weight), _ptr(conv_bias), int(bool(silu)), _ptr(conv_state), conv_dt,
            int(conv_layout), _ptr(ssm_state), _ptr(slot), B, ssm_state.shape[0],
            _sdims(dims, ssm_state), float(scale), int(bool(qk_l2norm)), _gate(gate), _ptr(out),
            _dt(out), _ptr(err), ctypes.byref(h)))
        self._h = h

    def launch(self, stream=None):
        _check(lib().gdn_graph_launch(self._h, _stream(stream)))

    def close(self):
        if getattr(self, "_h", None):
            lib().gdn_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def gdn_testing_set_fault(mode: int) -> None:
    """Test hook (include/gdn_testing.h): make one bounded wait of the kernels run out."""
    _check(lib().gdn_testing_set_fault(int(mode)))


def gdn_validate_slots(host_slot, num_slots) -> int:
    """Host-side duplicate / range check of a host slot table (0 ok, 1 range, 2 repeat)."""
    import numpy as np
    s = np.ascontiguousarray(host_slot, dtype=np.int32)
    return int(lib().gdn_validate_slots(s.ctypes.data_as(ctypes.c_void_p), s.size,
                                        int(num_slots)))
