"""exl3_linear_projections: a layer's projections in one call on one workspace
must equal the same projections called one by one (bit for bit: the same
kernels on the same transformed activations), on every GEMM path, including
a projection whose input is an earlier projection's output and projections
that share an input transform; and match the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._util import as_f64, assert_rows_close, bits, dev

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_gemm_exl3_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_gemm_exl3_gb300 import build
    build.build()
    m.lib()


def _dev_shard(sh, col0):
    return (dev(sh.code, torch.int16), sh.K, *(dev(v, torch.float16) for v in (sh.s_in, sh.rin, sh.rout, sh.s_out)),
            col0)


@pytest.mark.parametrize("M", (1, 8, 24, 200))
def test_layer_call_equals_separate_calls(M):
    g = syn.rng(600 + M)
    IC, I = 512, 1024
    # q/k/v share the input and (as given) one pre-scale pair; gate/up share the
    # input with their own pairs; down reads gate_up's output columns as its input
    qkv = [syn.make_shard(g, IC, 256, K) for K in (4, 3, 3)]
    qkv[1].s_in, qkv[1].rin = qkv[0].s_in, qkv[0].rin
    gu = [syn.make_shard(g, IC, I, K) for K in (2, 3)]
    down = syn.make_shard(g, I, IC, 3)
    x = dev(syn.normal_bf16(g, M, IC), torch.bfloat16)
    sq = [_dev_shard(sh, 256 * i) for i, sh in enumerate(qkv)]
    sq[1] = (sq[1][0], sq[1][1], sq[0][2], sq[0][3], *sq[1][4:])   # the same pointers as shard 0
    sg = [_dev_shard(sh, I * i) for i, sh in enumerate(gu)]
    sd = [_dev_shard(down, 0)]
    def outs():
        return (torch.empty((M, 768), dtype=torch.bfloat16, device="cuda"),
                torch.empty((M, 2 * I), dtype=torch.bfloat16, device="cuda"),
                torch.empty((M, IC), dtype=torch.bfloat16, device="cuda"))
    o1 = outs()
    # down reads a contiguous [M][I] copy of gate_up's first half (made between two calls)
    xin = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    projs = [(x, sq, o1[0]), (x, sg, o1[1]), (xin, sd, o1[2])]
    ws = m.workspace(m.exl3_projections_workspace_bytes(M, projs))
    m.exl3_linear_projections(projs[:2], ws)
    xin.copy_(o1[1][:, :I])
    m.exl3_linear_projections(projs[2:], ws)
    torch.cuda.synchronize()
    # the same projections one by one
    o2 = outs()
    wsl = m.workspace(max(m.exl3_linear_shards_workspace_bytes(M, IC, sq), m.exl3_linear_shards_workspace_bytes(M, IC, sg),
                          m.exl3_linear_shards_workspace_bytes(M, I, sd)))
    m.exl3_linear_into_shards(x, sq, o2[0], wsl)
    m.exl3_linear_into_shards(x, sg, o2[1], wsl)
    m.exl3_linear_into_shards(xin, sd, o2[2], wsl)
    torch.cuda.synchronize()
    for a, b in zip(o1, o2):
        assert np.array_equal(bits(a), bits(b))
    assert m.exl3_workspace_error(ws) == 0
    # and the oracle, on the first projection
    xs = bits(x)
    ref = np.concatenate([oracle.linear_f64(xs, sh.code, sh.K, qkv[0].s_in if i == 1 else sh.s_in,
                                            qkv[0].rin if i == 1 else sh.rin, sh.rout, sh.s_out)
                          for i, sh in enumerate(qkv)], axis=1)
    assert_rows_close(as_f64(o1[0]), ref)


def test_chained_input_in_one_call():
    # a projection may read what an earlier projection of the same call wrote
    M, IC = 8, 256
    g = syn.rng(650)
    a = syn.make_shard(g, IC, IC, 3)
    b2 = syn.make_shard(g, IC, 384, 2)
    x = dev(syn.normal_bf16(g, M, IC), torch.bfloat16)
    mid = torch.empty((M, IC), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((M, 384), dtype=torch.bfloat16, device="cuda")
    projs = [(x, [_dev_shard(a, 0)], mid), (mid, [_dev_shard(b2, 0)], out)]
    ws = m.workspace(m.exl3_projections_workspace_bytes(M, projs))
    m.exl3_linear_projections(projs, ws)
    torch.cuda.synchronize()
    ref_mid = oracle.linear_f64(bits(x), a.code, a.K, a.s_in, a.rin, a.rout, a.s_out)
    assert_rows_close(as_f64(mid), ref_mid)
    ref = oracle.linear_f64(bits(mid), b2.code, b2.K, b2.s_in, b2.rin, b2.rout, b2.s_out)
    assert_rows_close(as_f64(out), ref)


def test_rejects_bad_plans():
    assert m.lib().exl3_projections_workspace_bytes(8, None, 0) == 0
