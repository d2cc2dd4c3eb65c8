"""The allocation-free entry point against the regular one.

moe_w4a8_forward_noalloc serves callers that cannot allocate device memory
when they run the layer (runtimes that own all device memory, hot paths
where cudaMalloc is not allowed): it keeps its intermediates in a fixed
array inside the library instead of a caller-supplied workspace.  Its
output must match moe_w4a8_forward's on the same inputs, call after call,
although every call reuses (and must fully re-initialise) the same array.

This file is collected last on purpose, so that a run stopping at its first
failure has run every other test already.
"""
import ctypes

import numpy as np
import pytest
import torch

from bit_moe_expert_router_gb300 import binding, synth

import _gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    binding._load()


def _same(out, ref, what):
    """The same kernels on the same inputs: the same bits."""
    assert np.array_equal(out, ref), f"{what}: no-alloc output differs from moe_w4a8_forward"


def _both(w, tok, bank_dev):
    w13, s13, w2, s2 = bank_dev
    d = gh.dims(w)
    x = [gh.to_dev(a) for a in (tok.x_q, tok.x_scale, tok.logits)]
    ref = torch.full((w.T, w.H), float("nan"), dtype=torch.float32, device="cuda:0")
    ws = binding.alloc_workspace(binding.moe_w4a8_workspace_size(d), "cuda:0")
    binding.moe_w4a8_forward(*x, w13, s13, w2, s2, d, ref, ws)
    out = torch.full((w.T, w.H), float("nan"), dtype=torch.float32, device="cuda:0")
    binding.moe_w4a8_forward_noalloc(*x, w13, s13, w2, s2, d, out)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ref.cpu().numpy()


def test_noalloc_matches_forward_on_consecutive_calls():
    w = synth.WORKLOADS["decode_t4"]
    bank_dev = gh.device_bank(w)
    # two calls in a row on different batches: the second must not see the first's leftovers
    for batch in (0, 1):
        out, ref = _both(w, synth.make_tokens(w, batch=batch), bank_dev)
        gh.assert_output_close(out, ref.astype(np.float64), f"batch {batch}")
        _same(out, ref, f"batch {batch}")
        # the status word of the built-in array (a timed-out device wait would show here)
        assert binding.moe_w4a8_device_status(None) == 0


def test_noalloc_matches_forward_after_a_larger_layer():
    # a larger batch first (more of the array in use), then a small one on another layer shape
    w_big = synth.WORKLOADS["decode_t4"].with_tokens(64)
    out, ref = _both(w_big, synth.make_tokens(w_big), gh.device_bank(w_big))
    gh.assert_output_close(out, ref.astype(np.float64), "T=64")
    _same(out, ref, "T=64")
    w_small = synth.WORKLOADS["tiny"]
    out, ref = _both(w_small, synth.make_tokens(w_small), gh.device_bank(w_small))
    gh.assert_output_close(out, ref.astype(np.float64), "tiny")
    _same(out, ref, "tiny")


def test_noalloc_rejects_layers_beyond_its_array():
    w = synth.WORKLOADS["decode_t4"].with_tokens(4096)
    d = gh.dims(w)
    assert binding.moe_w4a8_workspace_size(d) > binding.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x100000)  # rejected on the host before any pointer is used
    rc = binding._load().moe_w4a8_forward_noalloc(fake, fake, fake, fake, fake, fake, fake, ctypes.byref(d), fake,
                                                   None)
    assert rc == 3  # MOE_ERR_WORKSPACE_TOO_SMALL
