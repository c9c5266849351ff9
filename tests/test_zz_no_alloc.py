"""replayssm_decode_noalloc, the decode entry point for callers that cannot
allocate device memory (for example a plugin whose host engine plans all
device memory and passes it only inputs and outputs).  It keeps the
per-sequence arrival counters in the library's own fixed device array instead
of the caller's cache->arrive.

Checked through the C ABI against replayssm_decode on two calls in a row,
for the per-tile kernel and for the persistent serving-shape kernel, with the
second call a fused flush.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from ssm_decode_state_gb300 import inputs as gen
from tests.helpers import assert_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [
    gen.Mamba2Shape(batch=3, nheads=8, headdim=32, dstate=64, ngroups=2, L=2),        # per-tile kernel
    gen.Mamba2Shape(batch=32, nheads=128, headdim=64, dstate=128, ngroups=8, L=2),    # persistent kernel
], ids=["per_tile", "persistent"])
def test_noalloc_matches_decode_two_calls(shape):
    from ssm_decode_state_gb300 import replayssm as rs
    seed = 2024
    prm = gen.mamba2_params(shape, seed)
    h0 = gen.mamba2_random_state(shape, seed)
    dims = rs.mamba2_dims(shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L)
    A, D = torch.from_numpy(prm.A), torch.from_numpy(prm.D)
    ref = rs.mamba2_cache(dims, A, D, ckpt=to_dev(h0))
    new = rs.mamba2_cache(dims, A, D, ckpt=to_dev(h0))
    new.arrive = None                        # the no-alloc entry point needs no counters from us
    for step in range(2):                    # step 1 folds the ring (L = 2)
        st = gen.mamba2_step_inputs(shape, prm, seed, step)
        args = (to_dev(st.dt), to_dev(st.x, torch.bfloat16), to_dev(st.B, torch.bfloat16),
                to_dev(st.C, torch.bfloat16))
        y_ref = rs.decode(ref, *args)
        y_new = torch.empty_like(y_ref)
        cs = new.c_struct()
        code = rs._lib.replayssm_decode_noalloc(ctypes.byref(dims), ctypes.byref(cs),
                                                *(a.data_ptr() for a in args), y_new.data_ptr(),
                                                torch.cuda.current_stream().cuda_stream)
        assert code == 0, rs.status_string(code)
        torch.cuda.synchronize()
        # the same kernel with the same arithmetic: only where the counters live differs,
        # so outputs and checkpoints agree bit for bit (the tolerance gate is implied)
        assert_close(y_new.cpu().numpy(), y_ref.cpu().numpy(), f"noalloc y call {step}")
        np.testing.assert_array_equal(y_new.cpu().numpy(), y_ref.cpu().numpy())
        np.testing.assert_array_equal(new.ring_len.cpu().numpy(), ref.ring_len.cpu().numpy())
        np.testing.assert_array_equal(new.ring_head.cpu().numpy(), ref.ring_head.cpu().numpy())
        np.testing.assert_array_equal(new.ckpt.cpu().numpy(), ref.ckpt.cpu().numpy())
        assert int(new.err.item()) == 0
    assert new.ring_len.cpu().tolist() == [0] * shape.batch     # the second call flushed

