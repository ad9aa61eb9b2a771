"""fp64 CPU oracle of the GDN layer hot path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package. It wraps ``gdn_oracle.c`` (plain sequential C, fp64)
through ctypes and shares no code with the CUDA library.

Every array argument is a numpy array; bf16 data travels as ``uint16`` bit
patterns, fp32 as ``float32`` and the recurrent state pool as ``float64``.
Each function names the page section it follows in ``gdn_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "libgdn_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into libgdn_oracle.so beside it (gcc, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["cc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC,
             "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        _lib.gdn_ref_round_bf16.restype = ctypes.c_uint16
        _lib.gdn_ref_round_bf16.argtypes = [D]
        _lib.gdn_ref_softplus.restype = D
        _lib.gdn_ref_softplus.argtypes = [D]
        _lib.gdn_ref_sigmoid.restype = D
        _lib.gdn_ref_sigmoid.argtypes = [D]
        _lib.gdn_ref_recurrent_head.restype = None
        _lib.gdn_ref_recurrent_head.argtypes = [P, P, P, P, P, P, I, I, I, P]
        _lib.gdn_ref_chunked_head.restype = None
        _lib.gdn_ref_chunked_head.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P]
        _lib.gdn_ref_unit_lower_inverse.restype = None
        _lib.gdn_ref_unit_lower_inverse.argtypes = [P, I, P]
        _lib.gdn_ref_validate_slots.restype = I
        _lib.gdn_ref_validate_slots.argtypes = [P, I, I]
        _lib.gdn_ref_conv_update.restype = I
        _lib.gdn_ref_conv_update.argtypes = [P, P, I, I, P, P, I, P, I, I, I, I, P, P, P]
        _lib.gdn_ref_layer.restype = I
        _lib.gdn_ref_layer.argtypes = [P, P, P, I, P, P, P, P, I, P, I, I, P, P, P, P, I, I, I,
                                       I, I, I, I, I, D, I, P, P, P, I, P, I]
        _lib.gdn_ref_gated_rmsnorm.restype = None
        _lib.gdn_ref_gated_rmsnorm.argtypes = [P, P, P, D, D, I, ctypes.c_int64, I, P]
        _lib.gdn_ref_recurrent_head_batch_dependent.restype = None
        _lib.gdn_ref_recurrent_head_batch_dependent.argtypes = [P, P, P, P, P, P, I, I, I, I, P]
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    if a is None:
        return None
    out = np.ascontiguousarray(a, dtype=dtype)
    return out


# --------------------------------------------------------------------------- scalars

def round_bf16(x: float) -> int:
    """bf16 bits of one round-to-nearest-even rounding of the fp64 value x."""
    return int(lib().gdn_ref_round_bf16(float(x)))


def round_bf16_array(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64).ravel()
    f = lib().gdn_ref_round_bf16
    return np.array([f(float(v)) for v in x], dtype=np.uint16)


def softplus(x: float) -> float:
    return float(lib().gdn_ref_softplus(float(x)))


def sigmoid(x: float) -> float:
    return float(lib().gdn_ref_sigmoid(float(x)))


# --------------------------------------------------------------------------- one head

def recurrent_head(q, k, v, g, beta, S0):
    """Token-by-token gated delta rule for one head; returns (o [T,dv], S [dv,dk])."""
    q = _c(q, np.float64); k = _c(k, np.float64); v = _c(v, np.float64)
    g = _c(g, np.float64); beta = _c(beta, np.float64)
    S = np.array(S0, dtype=np.float64, copy=True, order="C")
    T, dk = q.shape
    dv = v.shape[1]
    o = np.zeros((T, dv), dtype=np.float64)
    lib().gdn_ref_recurrent_head(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S), T, dk, dv, _p(o))
    return o, S


def recurrent_head_batch_dependent(q, k, v, g, beta, S0, batch):
    """The planted batch-dependent variant (negative control only)."""
    q = _c(q, np.float64); k = _c(k, np.float64); v = _c(v, np.float64)
    g = _c(g, np.float64); beta = _c(beta, np.float64)
    S = np.array(S0, dtype=np.float64, copy=True, order="C")
    T, dk = q.shape
    dv = v.shape[1]
    o = np.zeros((T, dv), dtype=np.float64)
    lib().gdn_ref_recurrent_head_batch_dependent(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S),
                                                 T, dk, dv, int(batch), _p(o))
    return o, S


def chunked_head(q, k, v, g, beta, S0, chunk, inverse_mode=0):
    """Chunked (UT/WY) form for one head; inverse_mode 0 = exact, n>0 = n-round bf16 NS."""
    q = _c(q, np.float64); k = _c(k, np.float64); v = _c(v, np.float64)
    g = _c(g, np.float64); beta = _c(beta, np.float64)
    S = np.array(S0, dtype=np.float64, copy=True, order="C")
    T, dk = q.shape
    dv = v.shape[1]
    o = np.zeros((T, dv), dtype=np.float64)
    lib().gdn_ref_chunked_head(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(S), T, dk, dv,
                               int(chunk), int(inverse_mode), _p(o))
    return o, S


def unit_lower_inverse(A):
    """(I + A)^-1 for strictly lower-triangular A (fp64 forward substitution)."""
    A = _c(A, np.float64)
    n = A.shape[0]
    T = np.zeros((n, n), dtype=np.float64)
    lib().gdn_ref_unit_lower_inverse(_p(A), n, _p(T))
    return T


def gated_rmsnorm(o, z_bits, w, offset=0.0, eps=1e-6, act="silu"):
    """Output gate of the GDN block (gdn_oracle.c, gdn_ref_gated_rmsnorm): for each vector
    o[..., :] over the value-head dim, y = o / sqrt(mean(o^2) + eps) * (w + offset) * act(z),
    act = SiLU or sigmoid. o: fp64 [..., dv]; z_bits: bf16 bits of the same shape; w: fp32 [dv].
    Returns fp64 y."""
    o = np.ascontiguousarray(o, dtype=np.float64)
    dv = o.shape[-1]
    z_bits = np.ascontiguousarray(z_bits, dtype=np.uint16).reshape(o.shape)
    w = np.ascontiguousarray(w, dtype=np.float32)
    assert w.shape == (dv,)
    y = np.empty_like(o)
    L = lib()
    L.gdn_ref_gated_rmsnorm(_p(o), _p(z_bits), _p(w), ctypes.c_double(offset), ctypes.c_double(eps),
                            ctypes.c_int({"silu": 0, "sigmoid": 1}[act]),
                            ctypes.c_int64(o.size // dv), ctypes.c_int(dv), _p(y))
    return y


def validate_slots(slot, num_slots) -> int:
    s = _c(slot, np.int32)
    return int(lib().gdn_ref_validate_slots(_p(s), s.size, int(num_slots)))


# --------------------------------------------------------------------------- layer

def conv_update(x_bits, conv_state, cache_f32, layout, w_bits, bias_bits, silu, slot, num_slots):
    """Decode conv update. conv_state (uint16 or float32 pool) is updated IN PLACE.

    Returns (out_bits [B, D] uint16, out_act [B, D] fp64 before rounding, err)."""
    x = _c(x_bits, np.uint16)
    w = _c(w_bits, np.uint16)
    bias = _c(bias_bits, np.uint16)
    slot = _c(slot, np.int32)
    assert conv_state.flags["C_CONTIGUOUS"]
    assert conv_state.dtype == (np.float32 if cache_f32 else np.uint16)
    B, D = x.shape
    W = w.shape[1]
    out = np.zeros((B, D), dtype=np.uint16)
    act = np.zeros((B, D), dtype=np.float64)
    err = np.zeros(1, dtype=np.int32)
    lib().gdn_ref_conv_update(_p(x), _p(conv_state), int(cache_f32), int(layout), _p(w),
                              _p(bias), int(silu), _p(slot), B, D, W, int(num_slots), _p(out),
                              _p(act), _p(err))
    return out, act, int(err[0])


def layer(mixed_bits, a, b, gate_direct, A_log, dt_bias, conv_w_bits, conv_b_bits, silu,
          conv_state, conv_f32, conv_layout, ssm_state, cu_seqlens, slot, has_init,
          Hk, Hv, dk, dv, W=4, scale=None, qk_l2norm=True, head_mask=None, nthreads=1,
          state_bf16=False):
    """Packed-sequence GDN layer (decode = every sequence of length 1).

    state_bf16: the recurrent state is stored in bf16 (values in the fp64 pool are then
    bf16-representable; each call's final state is rounded once, RNE).

    conv_state (uint16/float32 pool) and ssm_state (float64 pool
    [num_slots, Hv, dv, dk]) are updated IN PLACE. Returns
    (out fp64 [Ttot, Hv, dv], out_bits uint16 [Ttot, Hv, dv], err)."""
    x = _c(mixed_bits, np.uint16)
    Ttot, D = x.shape
    assert D == 2 * Hk * dk + Hv * dv
    if gate_direct:
        a = _c(a, np.float32); b = _c(b, np.float32)
    else:
        a = _c(a, np.uint16); b = _c(b, np.uint16)
    A_log = _c(A_log, np.float32)
    dt_bias = _c(dt_bias, np.float32)
    w = _c(conv_w_bits, np.uint16)
    cb = _c(conv_b_bits, np.uint16)
    cu = _c(cu_seqlens, np.int32)
    slot = _c(slot, np.int32)
    hi = None if has_init is None else _c(has_init, np.uint8)
    hm = None if head_mask is None else _c(head_mask, np.uint8)
    assert ssm_state.dtype == np.float64 and ssm_state.flags["C_CONTIGUOUS"]
    num_slots = ssm_state.shape[0]
    if conv_state is not None:
        assert conv_state.flags["C_CONTIGUOUS"]
    N = slot.size
    if scale is None:
        scale = dk ** -0.5
    out = np.zeros((Ttot, Hv, dv), dtype=np.float64)
    out_bits = np.zeros((Ttot, Hv, dv), dtype=np.uint16)
    err = np.zeros(1, dtype=np.int32)
    rc = lib().gdn_ref_layer(_p(x), _p(a), _p(b), int(gate_direct), _p(A_log), _p(dt_bias),
                             _p(w), _p(cb), int(silu), _p(conv_state), int(conv_f32),
                             int(conv_layout), _p(ssm_state), _p(cu), _p(slot), _p(hi), N, Ttot,
                             num_slots, Hk, Hv, dk, dv, W, float(scale), int(bool(qk_l2norm)),
                             _p(out), _p(out_bits), _p(hm), int(nthreads), _p(err),
                             int(bool(state_bf16)))
    if rc != 0:
        raise ValueError("oracle rejected the layer arguments")
    return out, out_bits, int(err[0])


def decode_step(mixed_bits, a, b, gate_direct, A_log, dt_bias, conv_w_bits, conv_b_bits, silu,
                conv_state, conv_f32, conv_layout, ssm_state, slot, Hk, Hv, dk, dv, W=4,
                scale=None, qk_l2norm=True, head_mask=None, nthreads=1, state_bf16=False):
    """One decode step over B rows (each row a length-1 sequence starting from its slot)."""
    B = np.asarray(slot).size
    cu = np.arange(B + 1, dtype=np.int32)
    out, out_bits, err = layer(mixed_bits, a, b, gate_direct, A_log, dt_bias, conv_w_bits,
                               conv_b_bits, silu, conv_state, conv_f32, conv_layout, ssm_state,
                               cu, slot, None, Hk, Hv, dk, dv, W, scale, qk_l2norm, head_mask,
                               nthreads, state_bf16)
    return out, out_bits, err
