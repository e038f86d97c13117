"""GPU parity of the int8 embedding gather (vllm-quantpack exl3/embedding.py,
embedding()): bit-exact against the oracle, including the 248,320 x 5120 table."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._util import bits, dev

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_gemm_exl3_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_gemm_exl3_gb300 import build
    build.build()


def test_gather_small_with_bad_ids():
    q, s, ids = syn.embedding(1, V=3000, H=208, N=513)
    ids[[0, 100, 512]] = [-5, 3000, 2 ** 30]
    nb = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = m.exl3_embed_int8_gather(dev(q, torch.int8), dev(s, torch.float16), dev(ids, torch.int32), n_bad=nb)
    ref, bad = oracle.gather(q, s, ids)
    assert np.array_equal(bits(out), ref)
    assert int(nb.item()) == bad == 3


def test_gather_full_vocab():
    q, s, ids = syn.embedding(5)
    out = m.exl3_embed_int8_gather(dev(q, torch.int8), dev(s, torch.float16), dev(ids, torch.int32))
    ref, bad = oracle.gather(q, s, ids)
    assert bad == 0
    assert np.array_equal(bits(out), ref)


def test_gather_empty():
    q, s, _ = syn.embedding(2, V=10, H=16, N=1)
    out = torch.empty((0, 16), dtype=torch.bfloat16, device="cuda")
    m.exl3_embed_int8_gather(dev(q, torch.int8), dev(s, torch.float16),
                             torch.empty(0, dtype=torch.int32, device="cuda"), out=out)
