"""GPU parity of the int8 output head (the int8 table as the output projection,
vllm-quantpack exl3/embedding.py, Exl3EmbeddingMethod.apply) against the oracle,
through the C ABI: per-row tolerance 2e-2 * rms plus half a bf16 ulp, on the
streaming path (up to 32 rows) and the tensor-core path (more rows, the table in
fp16 chunks)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._util import as_f64, assert_rows_close, dev

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_gemm_exl3_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_gemm_exl3_gb300 import build
    build.build()
    m.lib()


def _case(seed, M, V, H):
    q, s, _ = syn.embedding(seed, V=V, H=H, N=1)
    x = syn.normal_bf16(syn.rng(seed + 1), M, H)
    return x, q, s


def _run(x, q, s, ws=None):
    M, H = x.shape
    V = q.shape[0]
    if ws is None:
        ws = m.workspace(m.exl3_lm_head_workspace_bytes(M, H, V))
    y = m.exl3_lm_head_int8(dev(x, torch.bfloat16), dev(q, torch.int8), dev(s, torch.float16), ws)
    torch.cuda.synchronize()
    return as_f64(y), ws


@pytest.mark.parametrize("M,V", [(1, 1000), (5, 1021), (8, 4096), (17, 3000), (32, 777)])
def test_streaming_path(M, V):
    x, q, s = _case(20 + M, M, V, 512)
    got, _ = _run(x, q, s)
    assert_rows_close(got, oracle.lm_head_f64(x, q, s))


@pytest.mark.parametrize("M,V", [(33, 2000), (200, 20000)])
def test_tensor_core_path_chunks_and_partial_columns(M, V):
    # V = 20000 spans two converted chunks and ends inside a 128-column block
    x, q, s = _case(30 + M, M, V, 768)
    got, ws = _run(x, q, s)
    rows = np.unique(np.array([0, 1, M // 2, M - 1]))
    ref = oracle.lm_head_f64(np.ascontiguousarray(x[rows]), q, s)
    assert_rows_close(got[rows], ref)
    assert m.exl3_workspace_error(ws) == 0


@pytest.mark.parametrize("M", (1, 8, 300))
def test_full_vocabulary(M):
    # the 248,320 x 5120 table of the benchmarked gather, used as the head; vocabulary
    # windows at both ends and the middle, rows at both ends
    V, H = 248320, 5120
    q, s, _ = syn.embedding(5, V=V, H=H, N=1)
    x = syn.normal_bf16(syn.rng(40 + M), M, H)
    got, ws = _run(x, q, s)
    rows = np.unique(np.array([0, M - 1]))
    for v0 in (0, 123456, V - 3000):
        ref = oracle.lm_head_f64(np.ascontiguousarray(x[rows]), q, s, v0=v0, nv=3000)
        assert_rows_close(got[rows, v0:v0 + 3000], ref)
    assert m.exl3_workspace_error(ws) == 0


def test_repeated_calls_identical():
    # tiles go to warps in whatever order they ask; each tile is computed by one warp
    x, q, s = _case(50, 8, 30000, 1024)
    a, ws = _run(x, q, s)
    b, _ = _run(x, q, s, ws)
    assert np.array_equal(a, b)


def test_rejects_bad_sizes():
    x, q, s = _case(60, 2, 100, 256)
    ws = m.workspace(m.exl3_lm_head_workspace_bytes(2, 256, 100))
    with pytest.raises(m.Exl3Error):
        m.exl3_lm_head_int8(dev(x[:, :200], torch.bfloat16), dev(q[:, :200], torch.int8), dev(s, torch.float16), ws)
    assert m.exl3_lm_head_workspace_bytes(2, 200, 100) == 0
