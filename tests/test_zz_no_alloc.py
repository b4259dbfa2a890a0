"""The no-allocation fake-quant entry point against the allocating one.

nvfp4_fake_quant_noalloc serves callers that cannot hand the library device
scratch (a framework that owns all device memory through its own pool, or a
loop that must not call cudaMalloc/cudaFree).  It keeps the per-tensor amax in
a fixed array inside the library.  This test calls both entry points through
the C ABI on the same inputs, twice in a row with different inputs (the
second call must not see the first call's amax values), and checks that the
outputs agree bit for bit (fake-quant parity is bit-exact).  It lives in a
file of its own that pytest collects last.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _inputs(seed, nt, rows, cols, scale):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((nt, rows, cols), generator=g) * scale).to(torch.bfloat16).to("cuda:0")


def test_noalloc_fake_quant_matches_allocating_entry_point():
    import nvfp4_precision_moe_gb300 as nv

    L = nv.load(build=True)
    stream = torch.cuda.current_stream().cuda_stream
    # first call: large values; second call: more tensors, much smaller values
    for seed, nt, rows, cols, scale in [(1, 3, 256, 512, 8.0), (2, 5, 128, 1536, 0.01)]:
        w = _inputs(seed, nt, rows, cols, scale)
        ref = torch.empty_like(w)
        got = torch.empty_like(w)
        gs_ref = torch.zeros(nt, dtype=torch.float32, device="cuda:0")
        gs_got = torch.zeros(nt, dtype=torch.float32, device="cuda:0")
        amax_ws = torch.zeros(2 * nt + 1, dtype=torch.float32, device="cuda:0")
        status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        assert L.nvfp4_fake_quant(w.data_ptr(), nt, rows, cols, ref.data_ptr(), gs_ref.data_ptr(),
                                  amax_ws.data_ptr(), status.data_ptr(), stream) == 0
        assert L.nvfp4_fake_quant_noalloc(w.data_ptr(), nt, rows, cols, got.data_ptr(), gs_got.data_ptr(),
                                          status.data_ptr(), stream) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(gs_got, gs_ref)


def test_noalloc_without_optional_outputs():
    """gs_out and dev_status are optional: the same w_hat comes out without them."""
    import nvfp4_precision_moe_gb300 as nv

    L = nv.load(build=True)
    stream = torch.cuda.current_stream().cuda_stream
    nt, rows, cols = 2, 64, 256
    w = _inputs(3, nt, rows, cols, 3.0)
    ref = torch.empty_like(w)
    got = torch.empty_like(w)
    amax_ws = torch.zeros(2 * nt + 1, dtype=torch.float32, device="cuda:0")
    assert L.nvfp4_fake_quant(w.data_ptr(), nt, rows, cols, ref.data_ptr(), None, amax_ws.data_ptr(), None,
                              stream) == 0
    assert L.nvfp4_fake_quant_noalloc(w.data_ptr(), nt, rows, cols, got.data_ptr(), None, None, stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_noalloc_rejects_more_tensors_than_its_array():
    import nvfp4_precision_moe_gb300 as nv

    L = nv.load(build=True)
    w = torch.zeros((1, 32, 32), dtype=torch.bfloat16, device="cuda:0")
    st = L.nvfp4_fake_quant_noalloc(w.data_ptr(), 4097, 32, 32, w.data_ptr(), None, None,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == 2  # NVFP4_ERR_UNSUPPORTED, nothing launched
    assert b"4096" in L.nvfp4_last_error()
