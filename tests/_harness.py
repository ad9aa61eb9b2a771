"""Shared test plumbing: seeded inputs -> device tensors -> the C-ABI path, and
the same inputs -> the fp64 oracle. Comparison helpers.

The oracle runs on a compacted slot pool (only the slots a call touches, plus
a dummy slot 0), so that large pools do not need fp64 copies on the host.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import gated_deltanet_linear_gdn_gb300 as gdn
from gated_deltanet_linear_gdn_gb300 import inputs as gi

NTHREADS = max(1, min(32, os.cpu_count() or 1))


def bits_to_torch(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def torch_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def dims_of(geo: gi.Geometry) -> gdn.Dims:
    return gdn.Dims(geo.Hk, geo.Hv, geo.dk, geo.dv, geo.W)


class Device:
    """Device copies of a LayerInputs."""

    def __init__(self, inp: gi.LayerInputs, dev="cuda"):
        self.inp = inp
        f = lambda x: None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to(dev)
        fb = lambda x: None if x is None else bits_to_torch(x).to(dev)
        self.mixed = fb(inp.mixed)
        if inp.gate_direct:
            self.a, self.b = f(inp.a), f(inp.b)
        else:
            self.a, self.b = fb(inp.a), fb(inp.b)
        self.A_log, self.dt_bias = f(inp.A_log), f(inp.dt_bias)
        self.conv_w, self.conv_b = fb(inp.conv_w), fb(inp.conv_b)
        if inp.conv_state is None:
            self.conv_state = None
        elif inp.conv_f32:
            self.conv_state = f(inp.conv_state)
        else:
            self.conv_state = fb(inp.conv_state)
        self.ssm = fb(inp.ssm_state) if inp.state_bf16 else f(inp.ssm_state)
        self.slot = f(inp.slot)
        self.cu = f(inp.cu_seqlens)
        self.has_init = f(inp.has_init)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    def conv_state_host(self):
        if self.conv_state is None:
            return None
        if self.inp.conv_f32:
            return self.conv_state.cpu().numpy()
        return torch_to_bits(self.conv_state)


def gpu_decode(d: Device, out_f32=True, silu=None, stream=None, gate=None):
    inp = d.inp
    geo = inp.geo
    B = inp.slot.size
    out = torch.empty(B, geo.Hv, geo.dv, dtype=torch.float32 if out_f32 else torch.bfloat16,
                      device=d.mixed.device)
    gdn.gdn_decode_step(d.mixed, d.a, d.b, d.A_log, d.dt_bias, d.conv_w, d.conv_b, d.conv_state,
                        d.ssm, d.slot, out, dims_of(geo),
                        silu=inp.silu if silu is None else silu, conv_layout=inp.conv_layout,
                        scale=inp.scale, qk_l2norm=inp.qk_l2norm, gate=gate, err=d.err,
                        stream=stream)
    return out


def gpu_prefill(d: Device, chunk=64, out_f32=True, workspace=None, stream=None, gate=None):
    inp = d.inp
    geo = inp.geo
    T = inp.total_tokens
    N = inp.slot.size
    out = torch.empty(T, geo.Hv, geo.dv, dtype=torch.float32 if out_f32 else torch.bfloat16,
                      device=d.mixed.device)
    if workspace is None:
        nb = gdn.gdn_chunked_prefill_workspace_size(T, N, dims_of(geo), chunk)
        workspace = torch.empty(nb, dtype=torch.uint8, device=d.mixed.device)
    gdn.gdn_chunked_prefill(d.mixed, d.a, d.b, d.A_log, d.dt_bias, d.conv_w, d.conv_b,
                            d.conv_state, d.ssm, d.cu, d.slot, d.has_init, out, workspace,
                            dims_of(geo), chunk=chunk, silu=inp.silu,
                            conv_layout=inp.conv_layout, scale=inp.scale,
                            qk_l2norm=inp.qk_l2norm, gate=gate, err=d.err, stream=stream)
    return out


class OracleRun:
    """Oracle result on a compacted pool. sel[i] = original slot of compact slot i."""

    def __init__(self, inp: gi.LayerInputs, head_mask=None, nthreads=NTHREADS):
        import oracle

        self.inp = inp
        geo = inp.geo
        ns = inp.num_slots
        active = sorted({int(s) for s in inp.slot if 0 < s < ns})
        self.sel = np.array([0] + active, dtype=np.int64)
        mp = {s: i + 1 for i, s in enumerate(active)}
        nsc = len(self.sel)
        slot_c = np.array([mp[int(s)] if 0 < s < ns else (int(s) if s <= 0 else nsc)
                           for s in inp.slot], dtype=np.int32)
        self.slot_c = slot_c
        pool = inp.ssm_state[self.sel]
        if inp.state_bf16:
            pool = gi.bf16_bits_to_f32(pool)
        self.ssm = np.ascontiguousarray(pool.astype(np.float64))
        self.conv = (None if inp.conv_state is None
                     else np.ascontiguousarray(inp.conv_state[self.sel]))
        self.out, self.out_bits, self.err = oracle.layer(
            inp.mixed, inp.a, inp.b, inp.gate_direct, inp.A_log, inp.dt_bias, inp.conv_w,
            inp.conv_b, inp.silu, self.conv, inp.conv_f32, inp.conv_layout, self.ssm,
            inp.cu_seqlens, slot_c, inp.has_init, geo.Hk, geo.Hv, geo.dk, geo.dv, geo.W,
            inp.scale, inp.qk_l2norm, head_mask, nthreads, inp.state_bf16)


def rel_err(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    num = np.abs(x - ref).max()
    if den == 0:
        return float(num)
    return float(num / den)


def bf16_ulp_diff(a_bits, b_bits) -> np.ndarray:
    """|a - b| in bf16 ULPs (ordered-integer distance of the bit patterns)."""
    def key(x):
        x = np.asarray(x, dtype=np.uint16).astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return np.abs(key(a_bits) - key(b_bits))


def bf16_store_within(bits, ref, tol) -> bool:
    """A bf16 store of a value within tol * max|ref| of ref: |bf16 - ref| <= tol * max|ref|
    + half a bf16 ULP of |ref| (the rounding of the store itself), elementwise."""
    from gated_deltanet_linear_gdn_gb300.inputs import bf16_bits_to_f32
    got = bf16_bits_to_f32(bits).astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    half_ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 9)  # 2^(e-1-8): half ULP for |ref| in [2^(e-1), 2^e)
    bound = tol * np.abs(ref).max() + half_ulp + 1e-45
    return bool(np.all(np.abs(got - ref) <= bound))


def ssm_host(d: "Device") -> np.ndarray:
    """The device state pool as fp64 values (fp32 or bf16 storage)."""
    if d.ssm.dtype == torch.bfloat16:
        return gi.bf16_bits_to_f32(torch_to_bits(d.ssm)).astype(np.float64)
    return d.ssm.cpu().numpy().astype(np.float64)


def bf16_state_within(got, ref_rounded, tol) -> bool:
    """A bf16-stored state against the oracle's bf16-rounded state: elementwise within
    tol * max|ref| plus one bf16 ULP (the two fp roundings may land on either side of a
    rounding boundary)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref_rounded, np.float64)
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    return bool(np.all(np.abs(got - ref) <= tol * np.abs(ref).max() + ulp + 1e-45))


def tensor_hash(t: torch.Tensor) -> int:
    """64-bit digest of a tensor's bytes (replay checks compare digests across runs)."""
    import hashlib
    b = t.detach().cpu().contiguous().view(torch.uint8).numpy().tobytes()
    return int.from_bytes(hashlib.sha256(b).digest()[:8], "little")
