"""The allocation-free entry point, exl3_linear_into_noalloc, for callers that
cannot allocate device memory (no cudaMalloc and no workspace to hand in): it
must give the same projection as exl3_linear_into with a workspace, within the
per-row tolerance the other tests use, on two calls in a row.  The second call
reuses the library's fixed scratch array as the first call left it.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic as syn
from tests._util import as_f64, assert_rows_close, dev

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_gemm_exl3_gb300")
NAN_BF16 = 0x7FC1


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_gemm_exl3_gb300 import build
    build.build()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_noalloc(x, code, K, sc, out, col0):
    """Straight through the C ABI: raw pointers, sizes, the current stream."""
    IC, OC = code.shape[0] * 16, code.shape[1] * 16
    st = m.lib().exl3_linear_into_noalloc(
        _ptr(x), x.shape[0], IC, _ptr(code), OC, K, *(_ptr(v) for v in sc), _ptr(out),
        out.shape[1], col0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == m.EXL3_OK, m.lib().exl3_last_error()


@pytest.mark.parametrize("M,K", [(8, 2), (5, 3), (1, 4)])
def test_noalloc_matches_workspace_path_twice(M, K):
    IC, OC = 2048, 1536
    ldo = 2 * OC
    ws = m.workspace(m.exl3_linear_workspace_bytes(M, IC, OC))
    for call in range(2):                      # two calls in a row, different inputs
        x, sh = syn.linear_case(900 + 10 * call + M + K, M, IC, OC, K)
        xd = dev(x, torch.bfloat16)
        code = dev(sh.code, torch.int16)
        sc = [dev(v, torch.float16) for v in (sh.s_in, sh.rin, sh.rout, sh.s_out)]
        ref = torch.full((M, ldo), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        got = torch.full((M, ldo), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        m.exl3_linear_into(xd, code, K, *sc, ref, OC, ws)
        _call_noalloc(xd, code, K, sc, got, OC)
        torch.cuda.synchronize()
        assert_rows_close(as_f64(got)[:, OC:], as_f64(ref)[:, OC:])
        # columns outside the slice are left as they were
        assert torch.equal(got.view(torch.int16)[:, :OC],
                           torch.full((M, OC), NAN_BF16, dtype=torch.int16, device="cuda"))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    x, sh = syn.linear_case(950, 9, 256, 256, 2)    # M = 9 > 8
    out = torch.empty((9, 256), dtype=torch.bfloat16, device="cuda")
    sc = [dev(v, torch.float16) for v in (sh.s_in, sh.rin, sh.rout, sh.s_out)]
    code = dev(sh.code, torch.int16)
    IC, OC = 256, 256
    st = m.lib().exl3_linear_into_noalloc(
        _ptr(dev(x, torch.bfloat16)), 9, IC, _ptr(code), OC, 2, *(_ptr(v) for v in sc), _ptr(out), OC, 0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == m.EXL3_EINVAL
    assert b"M <= 8" in m.lib().exl3_last_error()


def test_noalloc_allocates_nothing():
    # after a warm-up call, a further call changes neither the device's free memory
    # nor what torch's caching allocator holds
    M, IC, OC, K = 8, 1024, 1024, 2
    x, sh = syn.linear_case(960, M, IC, OC, K)
    xd = dev(x, torch.bfloat16)
    code = dev(sh.code, torch.int16)
    sc = [dev(v, torch.float16) for v in (sh.s_in, sh.rin, sh.rout, sh.s_out)]
    out = torch.empty((M, OC), dtype=torch.bfloat16, device="cuda")
    _call_noalloc(xd, code, K, sc, out, 0)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    _call_noalloc(xd, code, K, sc, out, 0)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_reserved() == reserved0


@pytest.mark.parametrize("M,IC,OC,K", [(8, 32640, 8192, 2), (3, 4992, 8192, 3)])
def test_noalloc_matches_oracle_near_its_limits(M, IC, OC, K):
    # a wide input (IC near the 32768 limit, not a power of two) and many column
    # groups, so the split-K partition runs on the fixed slab; compared with the oracle
    import oracle
    x, sh = syn.linear_case(970 + K, M, IC, OC, K)
    out = torch.full((M, OC), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    _call_noalloc(dev(x, torch.bfloat16), dev(sh.code, torch.int16), K,
                  [dev(v, torch.float16) for v in (sh.s_in, sh.rin, sh.rout, sh.s_out)], out, 0)
    torch.cuda.synchronize()
    ref = oracle.linear_f64(x, sh.code, K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    assert_rows_close(as_f64(out), ref)
