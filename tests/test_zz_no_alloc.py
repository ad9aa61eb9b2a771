"""The scratch-free prefill entry point (gdn_chunked_prefill_noalloc) against the
ordinary one (gdn_chunked_prefill with a caller workspace).

gdn_chunked_prefill_noalloc serves callers that cannot allocate device memory
(a thread that must not risk the device synchronisation an allocation can
cause, a plug-in whose host runtime owns all device memory, a process with a
fixed footprint): it keeps its workspace in a fixed array inside the library.
This file checks, through the C ABI, that two calls in a row -- different
shapes, so the second runs over whatever the first left in the shared array --
give bitwise the same outputs and final states as the ordinary entry point on
the same inputs (both run the same deterministic kernels), after a first call
whose inputs are NaN has filled the array with NaNs: a read of stale scratch
would show. A request larger than the fixed array is refused without touching
anything.

It sits in its own file, collected last, and builds what it needs itself, so
it runs the same alone in a fresh process or after the other tests.
"""
import numpy as np
import pytest
import torch

import gated_deltanet_linear_gdn_gb300 as gdn
from gated_deltanet_linear_gdn_gb300 import inputs as gi

from _harness import Device, dims_of, gpu_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_gdn_gb300 import build
    build.build_library()
    assert torch.cuda.is_available()


def noalloc_prefill(d: Device, chunk):
    inp = d.inp
    geo = inp.geo
    out = torch.empty(inp.total_tokens, geo.Hv, geo.dv, dtype=torch.float32, device="cuda")
    gdn.gdn_chunked_prefill_noalloc(d.mixed, d.a, d.b, d.A_log, d.dt_bias, d.conv_w, d.conv_b,
                                    d.conv_state, d.ssm, d.cu, d.slot, d.has_init, out,
                                    dims_of(geo), chunk=chunk, silu=inp.silu,
                                    conv_layout=inp.conv_layout, scale=inp.scale,
                                    qk_l2norm=inp.qk_l2norm, err=d.err)
    return out


def compare(inp, chunk):
    ref_d = Device(inp)
    ref_out = gpu_prefill(ref_d, chunk=chunk, out_f32=True)
    d = Device(inp)
    out = noalloc_prefill(d, chunk)
    torch.cuda.synchronize()
    assert int(d.err.item()) == int(ref_d.err.item()) == 0
    assert torch.equal(out, ref_out)
    assert torch.equal(d.ssm, ref_d.ssm)
    if d.conv_state is not None:
        assert torch.equal(d.conv_state, ref_d.conv_state)


def test_noalloc_prefill_two_calls_match_the_workspace_entry_point():
    # fill most of the scratch with NaNs: a prefill whose inputs and states are all NaN
    poison = gi.prefill_varlen(8, 250, seed=30, num_slots=12)   # ~60 MiB of the 64
    poison.mixed[:] = 0x7FC0
    poison.ssm_state[:] = np.nan
    poison.conv_state[:] = 0x7FC0
    assert (gdn.gdn_chunked_prefill_workspace_size(poison.total_tokens, poison.slot.size,
                                                   dims_of(poison.geo), 16)
            <= gdn.GDN_NOALLOC_SCRATCH_BYTES)
    dp = Device(poison)
    noalloc_prefill(dp, 16)
    torch.cuda.synchronize()
    first = gi.prefill_varlen(5, 200, seed=31, num_slots=16)                # ~0.5k tokens
    second = gi.make_inputs(gi.TINY, [64, 3, 150, 1], 10, seed=32, conv_f32=True)
    assert (gdn.gdn_chunked_prefill_workspace_size(first.total_tokens, first.slot.size,
                                                   dims_of(first.geo), 64)
            <= gdn.GDN_NOALLOC_SCRATCH_BYTES)
    compare(first, chunk=64)
    compare(second, chunk=16)


def test_noalloc_prefill_refuses_requests_beyond_its_scratch():
    inp = gi.prefill_single(2048, seed=33)
    assert (gdn.gdn_chunked_prefill_workspace_size(2048, 1, dims_of(inp.geo), 64)
            > gdn.GDN_NOALLOC_SCRATCH_BYTES)
    d = Device(inp)
    out = torch.full((2048, inp.geo.Hv, inp.geo.dv), 3.0, dtype=torch.float32, device="cuda")
    ssm_before = d.ssm.clone()
    with pytest.raises(gdn.GDNError) as ei:
        gdn.gdn_chunked_prefill_noalloc(d.mixed, d.a, d.b, d.A_log, d.dt_bias, None, None, None,
                                        d.ssm, d.cu, d.slot, d.has_init, out, dims_of(inp.geo),
                                        chunk=64, err=d.err)
    assert ei.value.status == gdn.GDN_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert torch.all(out == 3.0) and torch.equal(d.ssm, ssm_before)
