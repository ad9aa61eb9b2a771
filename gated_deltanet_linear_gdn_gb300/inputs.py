"""Seeded synthetic inputs for the GDN layer hot path.

Shared by the tests, the smoke check and the benchmark. This module only draws
random numbers and shapes them into the distributions of the Qwen3-Next-shaped
workloads (sizes, dtypes, slot tables, sequence-length mixes); it contains none
of the layer's arithmetic. bf16 data is produced as uint16 bit patterns by
round-to-nearest-even from fp32 draws.

Every generator takes an explicit seed and uses numpy's PCG64.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Geometry:
    Hk: int
    Hv: int
    dk: int
    dv: int
    W: int = 4

    @property
    def D(self) -> int:
        return 2 * self.Hk * self.dk + self.Hv * self.dv


QWEN3_NEXT = Geometry(Hk=16, Hv=32, dk=128, dv=128, W=4)
TINY = Geometry(Hk=2, Hv=4, dk=32, dv=32, W=4)


@dataclass
class LayerInputs:
    """Host arrays of one call (decode: one row per sequence of length 1)."""
    geo: Geometry
    mixed: np.ndarray            # [T, D] uint16 (bf16)
    a: np.ndarray                # [T, Hv] uint16 (fused) or float32 g (direct)
    b: np.ndarray                # [T, Hv] uint16 (fused) or float32 beta (direct)
    gate_direct: bool
    A_log: np.ndarray            # [Hv] float32
    dt_bias: np.ndarray          # [Hv] float32
    conv_w: np.ndarray | None    # [D, W] uint16
    conv_b: np.ndarray | None    # [D] uint16
    silu: bool
    conv_state: np.ndarray | None  # pool, uint16 or float32
    conv_f32: bool
    conv_layout: int             # 0: [slots, D, W-1], 1: [slots, W-1, D]
    ssm_state: np.ndarray        # [num_slots, Hv, dv, dk] float32
    slot: np.ndarray             # [N] int32
    cu_seqlens: np.ndarray       # [N+1] int32
    has_init: np.ndarray | None  # [N] uint8
    scale: float
    qk_l2norm: bool = True
    meta: dict = field(default_factory=dict)
    state_bf16: bool = False     # ssm_state holds bf16 bit patterns (uint16) when True

    @property
    def num_slots(self) -> int:
        return self.ssm_state.shape[0]

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])


def _conv_pool(rng, num_slots, geo, f32, layout, std=1.0):
    shape = (num_slots, geo.D, geo.W - 1) if layout == 0 else (num_slots, geo.W - 1, geo.D)
    vals = rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
    return vals if f32 else f32_to_bf16_bits(vals)


def shuffled_slots(rng, n, num_slots):
    """n distinct slots drawn from [1, num_slots-1] in shuffled order (slot 0 = null block)."""
    assert n <= num_slots - 1
    return (rng.permutation(num_slots - 1)[:n] + 1).astype(np.int32)


def make_inputs(geo: Geometry, lengths, num_slots: int, seed: int, *, conv=True, bias=True,
                silu=True, conv_f32=False, conv_layout=0, gate_direct=False,
                conv_w_std=0.02, conv_state_std=1.0, state_std=0.05, A_log_range=(0.0, 2.0),
                dt_bias_zero=True, has_init=True, slots=None, state_pool=True,
                normalise_k_input=False, state_bf16=False) -> LayerInputs:
    """Generic generator: sequences of the given lengths (decode = all ones).

    mixed q|k|v ~ N(0,1) bf16; a, b ~ N(0,1) bf16 (fused gates) with
    A_log ~ U(A_log_range) and dt_bias = 0; conv weight and bias ~ N(0, conv_w_std);
    conv state ~ N(0, conv_state_std); recurrent state ~ N(0, state_std) fp32.
    normalise_k_input scales each k head vector of the input to unit length.
    gate_direct draws g = -|N(0,1)| and beta ~ U(0,1) as f32 instead of a, b.
    state_bf16 stores the drawn state pool as bf16 bit patterns.
    """
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in lengths]
    N = len(lengths)
    T = int(sum(lengths))
    cu = np.zeros(N + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    mixed_f = rng.standard_normal((T, geo.D), dtype=np.float32)
    if normalise_k_input:
        kblk = mixed_f[:, geo.Hk * geo.dk: 2 * geo.Hk * geo.dk].reshape(T, geo.Hk, geo.dk)
        kblk /= np.linalg.norm(kblk, axis=-1, keepdims=True)
        mixed_f[:, geo.Hk * geo.dk: 2 * geo.Hk * geo.dk] = kblk.reshape(T, -1)
    mixed = f32_to_bf16_bits(mixed_f)
    if gate_direct:
        # direct gates: g = -|N(0,1)| (a decay in (0, 1]), beta ~ U(0, 1)
        a = (-np.abs(rng.standard_normal((T, geo.Hv)))).astype(np.float32)
        b = rng.uniform(0.0, 1.0, (T, geo.Hv)).astype(np.float32)
    else:
        a = f32_to_bf16_bits(rng.standard_normal((T, geo.Hv), dtype=np.float32))
        b = f32_to_bf16_bits(rng.standard_normal((T, geo.Hv), dtype=np.float32))
    lo, hi = A_log_range
    A_log = rng.uniform(lo, hi, geo.Hv).astype(np.float32)
    dt_bias = (np.zeros(geo.Hv, dtype=np.float32) if dt_bias_zero
               else rng.standard_normal(geo.Hv, dtype=np.float32))
    conv_w = conv_b = conv_state = None
    if conv:
        conv_w = f32_to_bf16_bits(rng.standard_normal((geo.D, geo.W), dtype=np.float32)
                                  * np.float32(conv_w_std))
        if bias:
            conv_b = f32_to_bf16_bits(rng.standard_normal(geo.D, dtype=np.float32)
                                      * np.float32(conv_w_std))
        conv_state = _conv_pool(rng, num_slots, geo, conv_f32, conv_layout, conv_state_std)
    if state_pool:
        ssm = (rng.standard_normal((num_slots, geo.Hv, geo.dv, geo.dk), dtype=np.float32)
               * np.float32(state_std))
    else:
        ssm = np.zeros((num_slots, geo.Hv, geo.dv, geo.dk), dtype=np.float32)
    slot = shuffled_slots(rng, N, num_slots) if slots is None else np.asarray(slots, np.int32)
    hi_arr = None
    if has_init is not True:
        hi_arr = (np.zeros(N, np.uint8) if has_init is False
                  else np.asarray(has_init, dtype=np.uint8))
    if state_bf16:
        ssm = f32_to_bf16_bits(ssm)
    return LayerInputs(geo, mixed, a, b, gate_direct, A_log, dt_bias, conv_w, conv_b, silu,
                       conv_state, conv_f32, conv_layout, ssm, slot, cu, hi_arr,
                       float(geo.dk ** -0.5), True, {"seed": seed, "lengths": lengths},
                       bool(state_bf16))


# --------------------------------------------------------------------------- named workloads

def tiny_decode(seed=0, **kw) -> LayerInputs:
    """Tiny geometry (Hk=2, Hv=4, dk=dv=32, W=4): batch 2 over 8 slots, fp32 state ~N(0, 0.1),
    conv weight/bias ~N(0, 0.02), gates from a, b ~N(0,1) with A_log = 0, dt_bias = 0."""
    kw.setdefault("state_std", 0.1)
    kw.setdefault("A_log_range", (0.0, 0.0))
    return make_inputs(TINY, [1, 1], 8, seed, **kw)


def tiny_prefill(seed=0, **kw) -> LayerInputs:
    """Tiny geometry, one 64-token sequence (chunk 16 splits it into 4 chunks)."""
    kw.setdefault("state_std", 0.1)
    kw.setdefault("A_log_range", (0.0, 0.0))
    return make_inputs(TINY, [64], 8, seed, **kw)


def decode_sweep(B, seed=0, num_slots=512, **kw) -> LayerInputs:
    """Qwen3-Next geometry decode step: B rows through a shuffled slot table over num_slots,
    conv weight ~N(0,0.02) with bias, bf16 conv cache ~N(0,1), fp32 state ~N(0,0.05)."""
    return make_inputs(QWEN3_NEXT, [1] * B, num_slots, seed, **kw)


def prefill_single(T=4096, seed=0, **kw) -> LayerInputs:
    """One sequence of T tokens, conv bypassed, k L2-normalised at the input, zero initial
    state; g = -exp(A_log ~ U(0,2)) softplus(a), a ~ N(0,1); beta = sigmoid(b), b ~ N(0,1)."""
    kw.setdefault("conv", False)
    kw.setdefault("normalise_k_input", True)
    kw.setdefault("has_init", False)
    kw.setdefault("state_pool", False)
    return make_inputs(QWEN3_NEXT, [T], kw.pop("num_slots", 4), seed, **kw)


def varlen_lengths(n=8, max_len=8192, seed=0):
    rng = np.random.default_rng(seed + 1000)
    return [int(x) for x in rng.integers(1, max_len + 1, n)]


def prefill_varlen(n=8, max_len=8192, seed=0, num_slots=64, **kw) -> LayerInputs:
    """n sequences with lengths ~ U[1, max_len] packed by cu_seqlens, conv on, random fp32
    initial states ~N(0,0.05) and bf16 conv states ~N(0,1) in shuffled slots."""
    return make_inputs(QWEN3_NEXT, varlen_lengths(n, max_len, seed), num_slots, seed, **kw)


def correlated_keys(T=64, seed=0, geo: Geometry = QWEN3_NEXT, eps=0.01) -> LayerInputs:
    """The adversarial prefill case: per k-head k_t = normalise(k0 + eps * e_t), q, v ~ N(0,1),
    beta = 0.9 and g = 0 given directly, zero initial state, conv bypassed."""
    rng = np.random.default_rng(seed)
    mixed_f = rng.standard_normal((T, geo.D), dtype=np.float32)
    k0 = rng.standard_normal((geo.Hk, geo.dk), dtype=np.float32)
    e = rng.standard_normal((T, geo.Hk, geo.dk), dtype=np.float32)
    kk = k0[None] + np.float32(eps) * e
    kk /= np.linalg.norm(kk, axis=-1, keepdims=True)
    mixed_f[:, geo.Hk * geo.dk: 2 * geo.Hk * geo.dk] = kk.reshape(T, -1)
    mixed = f32_to_bf16_bits(mixed_f)
    a = np.zeros((T, geo.Hv), dtype=np.float32)
    b = np.full((T, geo.Hv), 0.9, dtype=np.float32)
    ssm = np.zeros((2, geo.Hv, geo.dv, geo.dk), dtype=np.float32)
    cu = np.array([0, T], dtype=np.int32)
    return LayerInputs(geo, mixed, a, b, True, np.zeros(geo.Hv, np.float32),
                       np.zeros(geo.Hv, np.float32), None, None, False, None, False, 0, ssm,
                       np.array([1], np.int32), cu, np.zeros(1, np.uint8),
                       float(geo.dk ** -0.5), True, {"seed": seed, "lengths": [T]})


def device_state_pool(num_slots: int, geo: Geometry, std: float, seed: int, device="cuda",
                      dtype=None):
    """State pool [num_slots, Hv, dv, dk] ~ N(0, std) drawn on the device (seeded torch
    generator), fp32 unless dtype says otherwise: for benchmark pools too large to draw
    on the host quickly."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    pool = torch.empty((num_slots, geo.Hv, geo.dv, geo.dk), dtype=dtype or torch.float32,
                       device=device)
    pool.normal_(0.0, float(std), generator=g)
    return pool
