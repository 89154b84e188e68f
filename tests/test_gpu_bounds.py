"""The bounds checks of the -DLLAMA_DEBUG build on the GPU.

The self-test stores, through the checked path, to element 40 of a 64-element buffer that it
declares 32 elements long: the bounds-checking library skips the store and reports
LLAMA_ERR_BOUNDS; the release library performs it (inside the buffer, so no build faults).
Running the whole GPU suite with LLAMA_BLOCK_DEBUG=1 (after
`python -m llama_decoder_block_fwd_gb300._build --debug`) checks every kernel's stores and TMA
boxes on every parity case: each test reads the status word, and a check that fired fails it.
"""
import pytest

import llama_decoder_block_fwd_gb300 as L

pytestmark = pytest.mark.gpu


def test_bounds_selftest():
    import torch
    scratch = torch.zeros(64, dtype=torch.float32, device="cuda")
    assert L.llama_get_device_status() == 0
    L.llama_selftest_bounds(scratch)
    status = L.llama_get_device_status()
    if L.llama_build_info() & L.BUILD_BOUNDS_CHECKS:
        assert status == 7                                     # LLAMA_ERR_BOUNDS
        assert float(scratch[40]) == 0.0                        # the store was skipped
    else:
        assert status == 0
        assert float(scratch[40]) == 1.0
    assert L.llama_get_device_status() == 0                    # read and cleared
    x = torch.randn(4, 64, device="cuda")                       # the context is still usable
    y = torch.empty_like(x)
    L.llama_rmsnorm(L.dims_of(1, 4, 64, 1, 1, 64, 128, 1e4, 1e-5), L.F32, x, torch.ones(64, device="cuda"), y)
    torch.cuda.synchronize()
    assert L.llama_get_device_status() == 0
    assert torch.allclose(y, x * torch.rsqrt((x * x).mean(-1, keepdim=True) + 1e-5), rtol=1e-5, atol=1e-5)
