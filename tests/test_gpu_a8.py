"""GPU parity of the 8-bit activation variant against the oracle, through the C ABI.

The codes are a floating-point decision: the device computes the pre-transform,
amax, As and u / As in fp32, the oracle in fp64.  They must agree exactly except
where the exact value u / As lies within the fp32 error of a rounding boundary
(x.5), and there by one step at most.  As agrees to fp32 rounding.  Outputs are
held to the per-row tolerance of the other linear tests against the oracle's
own (fp64) quantization and product, on every GEMM path.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._util import as_f64, assert_rows_close, dev

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_gemm_exl3_gb300")
NAN_BF16 = 0x7FC1
# |u / As| error of the fp32 device computation, in quantization steps: the
# pre-transform (7 butterfly stages, 3 products) and the division, each a few
# fp32 ulps of values up to 127.5, with a wide margin
BOUNDARY = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_gemm_exl3_gb300 import build
    build.build()
    m.lib()


def _dev_scales(sh):
    return [dev(v, torch.float16) for v in (sh.s_in, sh.rin, sh.rout, sh.s_out)]


def _check_codes(A_gpu, As_gpu, x, sh):
    """Codes equal the oracle's except within BOUNDARY of a rounding boundary (there by one)."""
    _, A_ref, As_ref = oracle.linear_a8_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out, nblk=0)
    np.testing.assert_allclose(As_gpu, As_ref, rtol=2e-6, atol=0)
    u = oracle.pretransform_f64(x, sh.s_in, sh.rin)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(As_ref[:, None] > 0, u / As_ref[:, None], 0.0)
    dq = A_gpu.astype(np.int64) - A_ref.astype(np.int64)
    assert np.all(np.abs(dq) <= 1), f"code off by {np.abs(dq).max()}"
    near = np.abs(np.abs(t) - np.floor(np.abs(t)) - 0.5) <= BOUNDARY
    bad = (dq != 0) & ~near
    assert not bad.any(), f"{bad.sum()} codes differ away from a rounding boundary"
    return int((dq != 0).sum())


@pytest.mark.parametrize("M,IC,seed", [(1, 128, 1), (37, 2048, 2), (5, 5120, 3), (3, 17408, 4)])
def test_quantize_codes_and_scales_match_oracle(M, IC, seed):
    x, sh = syn.linear_case(300 + seed, M, IC, 128, 2, outlier_frac=0.01)
    s_in, rin = dev(sh.s_in, torch.float16), dev(sh.rin, torch.float16)
    A, As = m.exl3_quantize_a8(dev(x, torch.bfloat16), s_in, rin)
    torch.cuda.synchronize()
    flips = _check_codes(A.cpu().numpy(), As.cpu().numpy().astype(np.float64), x, sh)
    assert flips <= max(2, M * IC // 1000)


def test_quantize_zero_rows_and_constant_row():
    M, IC = 4, 256
    x, sh = syn.linear_case(310, M, IC, 128, 2)
    x = x.copy()
    x[1] = 0                      # all-zero row: As = 0, every code 128
    x[3] = 0x3F80                 # a constant input row (1.0)
    A, As = m.exl3_quantize_a8(dev(x, torch.bfloat16), dev(sh.s_in, torch.float16), dev(sh.rin, torch.float16))
    torch.cuda.synchronize()
    A, As = A.cpu().numpy(), As.cpu().numpy().astype(np.float64)
    assert As[1] == 0 and np.all(A[1] == 128)
    q = A.astype(np.int64) - 128
    for r in (0, 2, 3):
        assert np.abs(q[r]).max() == 127        # the row maximum maps to the end of the range
    _check_codes(A, As, x, sh)


def _run_a8(x, sh, M, IC, OC, ldo=None, col0=0):
    ldo = ldo or OC
    out = torch.full((M, ldo), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    ws = m.workspace(m.exl3_linear_a8_workspace_bytes(M, IC, OC))
    s_in, rin, rout, s_out = _dev_scales(sh)
    m.exl3_linear_into_a8(dev(x, torch.bfloat16), dev(sh.code, torch.int16), sh.K, s_in, rin, rout, s_out,
                          out, col0, ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("M,K,path", [(1, 2, "rows"), (5, 3, "rows"), (8, 4, "rows"), (13, 2, "rows"),
                                      (40, 3, "decode"), (64, 2, "fused"), (100, 4, "fused"),
                                      (150, 3, "prefill"), (200, 2, "rows")])
def test_linear_a8_matches_oracle_every_path(M, K, path, pin_gemm_path):
    pin_gemm_path(path)
    IC, OC = 1024, 768
    x, sh = syn.linear_case(320 + M + K, M, IC, OC, K, outlier_frac=0.01)
    out = _run_a8(x, sh, M, IC, OC, ldo=OC + 256, col0=128)
    y_ref, _, _ = oracle.linear_a8_f64(x, sh.code, K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    got = out.view(torch.int16)
    assert_rows_close(as_f64(out)[:, 128:128 + OC], y_ref)
    # columns outside the slice keep their poison
    assert torch.all(got[:, :128] == NAN_BF16) and torch.all(got[:, 128 + OC:] == NAN_BF16)


@pytest.mark.parametrize("M", [1, 8])
def test_linear_a8_gate_up_full_size_every_column(M):
    # the 5120 -> 17408 projection at K = 2 and 3 on the codes path: every row and
    # every column against the oracle
    IC, OC = 5120, 17408
    for K in (2, 3):
        x, sh = syn.linear_case(340 + K + M, M, IC, OC, K)
        out = _run_a8(x, sh, M, IC, OC)
        y_ref, _, _ = oracle.linear_a8_f64(x, sh.code, K, sh.s_in, sh.rin, sh.rout, sh.s_out)
        assert_rows_close(as_f64(out), y_ref)


@pytest.mark.parametrize("M,path", [(3, "rows"), (8, "rows"), (24, "rows"), (64, "fused"), (160, "prefill")])
def test_gemm_a8_into_equals_linear_into_a8(M, path, pin_gemm_path):
    # the split entry (quantize, then GEMM on the codes) gives the one-call result bit for bit
    pin_gemm_path(path)
    IC, OC, K = 2048, 1024, 3
    x, sh = syn.linear_case(360 + M, M, IC, OC, K)
    one = _run_a8(x, sh, M, IC, OC)
    s_in, rin, rout, s_out = _dev_scales(sh)
    A, As = m.exl3_quantize_a8(dev(x, torch.bfloat16), s_in, rin)
    two = torch.full((M, OC), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    ws = m.workspace(m.exl3_linear_a8_workspace_bytes(M, IC, OC))
    m.exl3_gemm_a8_into(A, As, dev(sh.code, torch.int16), K, rout, s_out, two, 0, ws)
    torch.cuda.synchronize()
    assert torch.equal(one.view(torch.int16), two.view(torch.int16))


def test_linear_a8_zero_rows_give_zero_output():
    M, IC, OC, K = 6, 512, 256, 2
    x, sh = syn.linear_case(370, M, IC, OC, K)
    x = x.copy()
    x[2] = 0
    x[5] = 0
    out = _run_a8(x, sh, M, IC, OC)
    got = as_f64(out)
    assert np.all(got[2] == 0) and np.all(got[5] == 0)
    y_ref, _, _ = oracle.linear_a8_f64(x, sh.code, K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    assert_rows_close(got[[0, 1, 3, 4]], y_ref[[0, 1, 3, 4]])


def test_a8_errors_and_empty_calls():
    L = m.lib()
    IC, OC, K = 256, 256, 2
    x, sh = syn.linear_case(380, 2, IC, OC, K)
    xd = dev(x, torch.bfloat16)
    code = dev(sh.code, torch.int16)
    s_in, rin, rout, s_out = _dev_scales(sh)
    out = torch.empty((2, OC), dtype=torch.bfloat16, device="cuda")
    ws = m.workspace(m.exl3_linear_a8_workspace_bytes(2, IC, OC))
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = torch.cuda.current_stream().cuda_stream
    # M = 0: nothing to do, success
    assert L.exl3_linear_into_a8(p(xd), 0, IC, p(code), OC, K, p(s_in), p(rin), p(rout), p(s_out), p(out), OC, 0,
                                 p(ws), ws.numel(), st) == m.EXL3_OK
    # a workspace one byte short
    assert L.exl3_linear_into_a8(p(xd), 2, IC, p(code), OC, K, p(s_in), p(rin), p(rout), p(s_out), p(out), OC, 0,
                                 p(ws), ws.numel() - 1, st) == m.EXL3_EWORKSPACE
    # null As
    A = torch.empty((2, IC), dtype=torch.uint8, device="cuda")
    assert L.exl3_gemm_a8_into(p(A), None, 2, IC, p(code), OC, K, p(rout), p(s_out), p(out), OC, 0,
                               p(ws), ws.numel(), st) == m.EXL3_EINVAL
    # a row wider than shared memory holds
    assert L.exl3_quantize_a8(p(xd), 1, 65536, p(s_in), p(rin), p(A), p(A), st) == m.EXL3_EUNSUPPORTED
    assert b"shared memory" in L.exl3_last_error()
    # workspace sizes never shrink as M grows
    sizes = [m.exl3_linear_a8_workspace_bytes(M, 5120, 17408) for M in (1, 8, 9, 16, 17, 128, 129, 8192)]
    assert sizes == sorted(sizes) and sizes[0] > 0


def _shard_sets(shards, col0s):
    return [(dev(s.code, torch.int16), s.K, *_dev_scales(s), c) for s, c in zip(shards, col0s)]


@pytest.mark.parametrize("M,path", [(1, "rows"), (6, "rows"), (13, "rows"), (40, "decode"), (64, "fused"),
                                    (150, "prefill")])
def test_shards_a8_match_oracle_per_shard(M, path, pin_gemm_path):
    # three shards with their own (s_in, rin), different K and OC, in one call: each
    # shard's columns against the oracle's 8-bit projection of that shard
    pin_gemm_path(path)
    IC = 1024
    g = syn.rng(400 + M)
    shards = [syn.make_shard(g, IC, OC, K) for OC, K in ((384, 2), (640, 3), (256, 4))]
    x = syn.normal_bf16(g, M, IC, outlier_frac=0.01)
    col0s = [0, 384 + 64, 384 + 64 + 640]
    ldo = col0s[-1] + 256 + 64
    sets = _shard_sets(shards, col0s)
    out = torch.full((M, ldo), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    ws = m.workspace(m.exl3_linear_shards_a8_workspace_bytes(M, IC, sets))
    m.exl3_linear_into_shards_a8(dev(x, torch.bfloat16), sets, out, ws)
    torch.cuda.synchronize()
    got = as_f64(out)
    for s, c in zip(shards, col0s):
        y_ref, _, _ = oracle.linear_a8_f64(x, s.code, s.K, s.s_in, s.rin, s.rout, s.s_out)
        assert_rows_close(got[:, c:c + s.OC], y_ref)
    gaps = out.view(torch.int16)
    assert torch.all(gaps[:, 384:384 + 64] == NAN_BF16) and torch.all(gaps[:, ldo - 64:] == NAN_BF16)


@pytest.mark.parametrize("M,Ks,IC,OC", [(1, (2, 3), 1024, 0), (8, (4, 2), 1024, 0), (8, (2, 3), 5120, 17408)])
def test_paired_shards_a8_every_column(M, Ks, IC, OC):
    # two shards of one width (OC = 0: 5/8 as many column groups per shard as the
    # GPU has SMs; the last case is the merged 5120 -> 2 x 17408 gate/up layer),
    # on the decode path's paired CTAs, on the 8-bit codes: every column against
    # the oracle's 8-bit projection, and the split entry (quantize, then the GEMM
    # on the codes) bit for bit equal to the one-call result
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    OC = OC or 128 * (sms * 5 // 8)
    g = syn.rng(440 + M)
    shards = [syn.make_shard(g, IC, OC, K) for K in Ks]
    x = syn.normal_bf16(g, M, IC, outlier_frac=0.01)
    sets = _shard_sets(shards, [0, OC])
    ws = m.workspace(m.exl3_linear_shards_a8_workspace_bytes(M, IC, sets))
    xd = dev(x, torch.bfloat16)
    one = torch.full((M, 2 * OC), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    m.exl3_linear_into_shards_a8(xd, sets, one, ws)
    A = torch.empty((2, M, IC), dtype=torch.uint8, device="cuda")
    As = torch.empty((2, M), dtype=torch.float32, device="cuda")
    for i, st in enumerate(sets):
        m.exl3_quantize_a8(xd, st[2], st[3], A=A[i], As=As[i])
    two = torch.empty((M, 2 * OC), dtype=torch.bfloat16, device="cuda")
    m.exl3_gemm_a8_into_shards(A, As, sets, two, ws)
    torch.cuda.synchronize()
    assert torch.equal(one.view(torch.int16), two.view(torch.int16))
    got = as_f64(one)
    for i, s in enumerate(shards):
        y_ref, _, _ = oracle.linear_a8_f64(x, s.code, s.K, s.s_in, s.rin, s.rout, s.s_out)
        assert_rows_close(got[:, i * OC:(i + 1) * OC], y_ref)


@pytest.mark.parametrize("M,path", [(5, "rows"), (20, "rows"), (96, "fused"), (140, "prefill")])
def test_gemm_a8_into_shards_equals_linear_into_shards_a8(M, path, pin_gemm_path):
    pin_gemm_path(path)
    IC = 2048
    g = syn.rng(420 + M)
    shards = [syn.make_shard(g, IC, OC, K) for OC, K in ((512, 2), (768, 3))]
    x = syn.normal_bf16(g, M, IC)
    sets = _shard_sets(shards, [0, 512])
    ws = m.workspace(m.exl3_linear_shards_a8_workspace_bytes(M, IC, sets))
    one = torch.empty((M, 1280), dtype=torch.bfloat16, device="cuda")
    two = torch.empty((M, 1280), dtype=torch.bfloat16, device="cuda")
    xd = dev(x, torch.bfloat16)
    m.exl3_linear_into_shards_a8(xd, sets, one, ws)
    A = torch.empty((2, M, IC), dtype=torch.uint8, device="cuda")
    As = torch.empty((2, M), dtype=torch.float32, device="cuda")
    for i, st in enumerate(sets):
        m.exl3_quantize_a8(xd, st[2], st[3], A=A[i], As=As[i])
    m.exl3_gemm_a8_into_shards(A, As, sets, two, ws)
    torch.cuda.synchronize()
    assert torch.equal(one.view(torch.int16), two.view(torch.int16))
