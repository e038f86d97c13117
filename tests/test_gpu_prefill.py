"""GPU parity of the prefill (large-M, tensor-core) EXL3 linear against the oracle.

Rows above the decode threshold go through tcgen05 GEMM tiles of 128 rows x 256
columns; the cases cover ragged row counts (M not a multiple of 128), an output
width that ends in half a tile (OC % 256 == 128), and the prefill-shaped
5120 -> 17408 linear at M = 8192 with 1 % outlier channels, checked on sampled
rows against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._util import as_f64, assert_rows_close, bits, dev

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_gemm_exl3_gb300")
NAN_BF16 = 0x7FC1


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_gemm_exl3_gb300 import build
    build.build()


def run(x, sh, out=None, col0=0):
    M = x.shape[0]
    ws = m.workspace(m.exl3_linear_workspace_bytes(M, sh.IC, sh.OC))
    code = dev(sh.code, torch.int16)
    sc = [dev(v, torch.float16) for v in (sh.s_in, sh.rin, sh.rout, sh.s_out)]
    if out is None:
        out = torch.empty((M, sh.OC), dtype=torch.bfloat16, device="cuda")
    m.exl3_linear_into(dev(x, torch.bfloat16), code, sh.K, *sc, out, col0, ws)
    torch.cuda.synchronize()
    assert m.exl3_workspace_error(ws) == 0
    return out


@pytest.mark.parametrize("M,OC,K", [(161, 384, 2), (300, 640, 3), (1000, 256, 4), (129, 1152, 2)])
def test_prefill_ragged(M, OC, K):
    x, sh = syn.linear_case(500 + M, M, 1024, OC, K, outlier_frac=0.01)
    y = run(x, sh)
    assert_rows_close(as_f64(y), oracle.linear_f64(x, sh.code, K, sh.s_in, sh.rin, sh.rout, sh.s_out))


def test_prefill_column_slice_isolation():
    x, sh = syn.linear_case(510, 200, 512, 384, 3)
    ldo = 384 + 128
    out = torch.full((200, ldo), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    run(x, sh, out=out, col0=64)
    b = bits(out)
    assert np.all(b[:, :64] == NAN_BF16) and np.all(b[:, 64 + 384:] == NAN_BF16)
    assert_rows_close(as_f64(out)[:, 64:64 + 384],
                      oracle.linear_f64(x, sh.code, 3, sh.s_in, sh.rin, sh.rout, sh.s_out))


@pytest.mark.parametrize("K", (2, 3, 4))
def test_prefill_full_shape_every_column_sampled_rows(K):
    # the benchmarked prefill shape: every output column, on rows in the first and last
    # 128-row tiles, around a tile boundary and in the middle
    x, sh = syn.prefill(2, M=8192, K=K)
    y = run(x, sh)
    got = as_f64(y)
    assert np.all(np.isfinite(got))
    rows = np.array([0, 1, 127, 128, 4095, 5000, 8190, 8191])
    ref = oracle.linear_f64(np.ascontiguousarray(x[rows]), sh.code, K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    assert_rows_close(got[rows], ref)
