"""GPU parity of the grouped EXL3 MoE layer against the CPU oracle, through the C ABI.

Expert bank layout from bank.py (w13 = [w1 | w3] per K-sorted slot, w2, fp16
suh/svh vectors); SiLU-gated FFN; top-k routing with softmax weights.  Outputs
must satisfy max|y - y_ref| <= 2e-2 * rms(y_ref) per token.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests._util import as_f64, assert_rows_close, bits, dev

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_gemm_exl3_gb300")

_DT = dict(w13=torch.int16, w2=torch.int16, off_w1=torch.int64, off_w3=torch.int64, off_w2=torch.int64,
           perm=torch.int32, k_gu=torch.int32, k_d=torch.int32, w13_suh=torch.float16,
           w13_svh=torch.float16, w2_suh=torch.float16, w2_svh=torch.float16)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_gemm_exl3_gb300 import build
    build.build()


def bank_dev(bank):
    return {k: dev(v, _DT[k]) for k, v in bank.items()}


def run_moe(x, ids, w, bank_d, E, H, I, ws=None):
    T, topk = ids.shape
    if ws is None:
        ws = m.workspace(m.exl3_moe_workspace_bytes(T, H, I, E, topk))
    y = m.exl3_moe_grouped(dev(x, torch.bfloat16), dev(ids, torch.int32), dev(w, torch.float32), bank_d, ws)
    torch.cuda.synchronize()
    return y, ws


def test_topk_softmax_matches_oracle():
    g = np.random.default_rng(3)
    logits = g.standard_normal((300, 128)).astype(np.float32)
    logits[7, [3, 90, 17]] = 9.0                 # ties: lower expert id first
    ids, w = m.exl3_moe_topk_softmax(dev(logits, torch.float32), 8)
    torch.cuda.synchronize()
    rid, rw = oracle.topk_softmax(logits, 8)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T", (1, 5, 20, 40))
def test_moe_small_bank_mixed_k(T):
    E, H, I, topk = 6, 256, 128, 3
    bank = syn.moe_bank(11, E=E, H=H, I=I, distinct_down_k=True)
    x, logits = syn.moe_tokens(12 + T, T, H=H, E=E)
    ids, w = oracle.topk_softmax(logits, topk)
    y, ws = run_moe(x, ids, w, bank_dev(bank), E, H, I)
    assert_rows_close(as_f64(y), oracle.moe_f64(x, ids, w, bank))
    assert m.exl3_workspace_error(ws) == 0


@pytest.mark.parametrize("T,topk", ((16, 4), (40, 4), (16, 2)))
def test_moe_skewed_routing_splits_entries(T, topk):
    # every token picks the same experts: each gets T rows, more than one row block
    # (16 tokens x 2 routes: the one-warp routing of at most 32 pairs, two blocks per slot)
    E, H, I = 16, 256, 128
    bank = syn.moe_bank(21, E=E, H=H, I=I, distinct_down_k=True)
    x, logits = syn.moe_tokens(30 + T, T, H=H, E=E)
    logits[:, [2, 7, 11, 13][:topk]] += 50.0
    ids, w = oracle.topk_softmax(logits, topk)
    assert len(np.unique(ids)) == topk
    y, ws = run_moe(x, ids, w, bank_dev(bank), E, H, I)
    assert_rows_close(as_f64(y), oracle.moe_f64(x, ids, w, bank))
    assert m.exl3_workspace_error(ws) == 0


@pytest.fixture(scope="module")
def full_bank():
    bank = syn.moe_bank(3)           # E = 128, H = 2048, I = 768, K per expert in {2, 3, 4}
    return bank, bank_dev(bank)


@pytest.mark.parametrize("T", (1, 16))
def test_moe_full_geometry(full_bank, T):
    bank, bank_d = full_bank
    x, logits = syn.moe_tokens(20 + T, T)
    ids, w = m.exl3_moe_topk_softmax(dev(logits, torch.float32), 8)
    ids, w = ids.cpu().numpy(), w.cpu().numpy()
    y, ws = run_moe(x, ids, w, bank_d, 128, 2048, 768)
    assert_rows_close(as_f64(y), oracle.moe_f64(x, ids, w, bank))
    assert m.exl3_workspace_error(ws) == 0


def test_moe_full_geometry_512_tokens_sampled(full_bank):
    bank, bank_d = full_bank
    T = 512
    x, logits = syn.moe_tokens(40, T)
    ids, w = oracle.topk_softmax(logits, 8)
    y, ws = run_moe(x, ids, w, bank_d, 128, 2048, 768)
    got = as_f64(y)
    assert np.all(np.isfinite(got))
    sample = np.array([0, 1, 77, 200, 311, 450, 510, 511])
    ref = oracle.moe_f64(np.ascontiguousarray(x[sample]), np.ascontiguousarray(ids[sample]),
                         np.ascontiguousarray(w[sample]), bank)
    assert_rows_close(got[sample], ref)


@pytest.mark.parametrize("E,T,topk", ((160, 40, 4), (16, 1200, 8)))
def test_moe_routing_paths_sampled(E, T, topk):
    # E above the per-warp ranking table (one warp ranks every pair) and more
    # pairs than the register-resident ranking holds (ranking through memory)
    H, I = 256, 128
    bank = syn.moe_bank(50 + E, E=E, H=H, I=I, distinct_down_k=True)
    x, logits = syn.moe_tokens(51 + T, T, H=H, E=E)
    ids, w = oracle.topk_softmax(logits, topk)
    y, ws = run_moe(x, ids, w, bank_dev(bank), E, H, I)
    assert m.exl3_workspace_error(ws) == 0
    got = as_f64(y)
    assert np.all(np.isfinite(got))
    sample = np.unique(np.array([0, 1, T // 3, T // 2, T - 2, T - 1]))
    ref = oracle.moe_f64(np.ascontiguousarray(x[sample]), np.ascontiguousarray(ids[sample]),
                         np.ascontiguousarray(w[sample]), bank)
    assert_rows_close(got[sample], ref)
    y2, _ = run_moe(x, ids, w, bank_dev(bank), E, H, I, ws)
    assert np.array_equal(bits(y), bits(y2))


def test_moe_long_call_runs_in_passes(full_bank):
    # more tokens than one pass serves (the column groups of a pass must fit the
    # workspace's arrival counters): the layer runs in passes over the token rows
    bank, bank_d = full_bank
    T = 4100
    x, logits = syn.moe_tokens(42, T)
    ids, w = oracle.topk_softmax(logits, 8)
    y, ws = run_moe(x, ids, w, bank_d, 128, 2048, 768)
    assert m.exl3_workspace_error(ws) == 0
    got = as_f64(y)
    assert np.all(np.isfinite(got))
    sample = np.array([0, 1, 3966, 3967, 4099])
    ref = oracle.moe_f64(np.ascontiguousarray(x[sample]), np.ascontiguousarray(ids[sample]),
                         np.ascontiguousarray(w[sample]), bank)
    assert_rows_close(got[sample], ref)
    # every row is written by exactly one pass: the same tokens as two calls of 3967
    # and 133 tokens on the same workspace give the identical output
    y1, _ = run_moe(np.ascontiguousarray(x[:3967]), np.ascontiguousarray(ids[:3967]),
                    np.ascontiguousarray(w[:3967]), bank_d, 128, 2048, 768, ws)
    y2, _ = run_moe(np.ascontiguousarray(x[3967:]), np.ascontiguousarray(ids[3967:]),
                    np.ascontiguousarray(w[3967:]), bank_d, 128, 2048, 768, ws)
    assert np.array_equal(bits(y), np.concatenate([bits(y1), bits(y2)]))


def test_moe_deterministic(full_bank):
    bank, bank_d = full_bank
    x, logits = syn.moe_tokens(41, 37)
    ids, w = oracle.topk_softmax(logits, 8)
    y1, ws = run_moe(x, ids, w, bank_d, 128, 2048, 768)
    y2, _ = run_moe(x, ids, w, bank_d, 128, 2048, 768, ws)
    assert np.array_equal(bits(y1), bits(y2))


def test_moe_invalid_expert_id_is_recorded_and_skipped():
    E, H, I, topk = 6, 256, 128, 2
    bank = syn.moe_bank(13, E=E, H=H, I=I)
    x, logits = syn.moe_tokens(14, 4, H=H, E=E)
    ids, w = oracle.topk_softmax(logits, topk)
    bad = ids.copy()
    bad[2, 1] = 99
    y, ws = run_moe(x, bad, w, bank_dev(bank), E, H, I)
    assert m.exl3_workspace_error(ws) == 2            # an expert id outside [0, E)
    # the invalid route contributes nothing: same as a valid id with weight 0
    w0 = w.copy()
    w0[2, 1] = 0.0
    assert_rows_close(as_f64(y), oracle.moe_f64(x, ids, w0, bank))


@pytest.mark.parametrize("T", (4, 20))
def test_moe_token_without_a_valid_route_gets_zeros(T):
    # T = 4: the one-warp routing (8 pairs); T = 20: the CTA-wide routing (40 pairs)
    E, H, I, topk = 6, 256, 128, 2
    bank = syn.moe_bank(17, E=E, H=H, I=I)
    x, logits = syn.moe_tokens(18 + T, T, H=H, E=E)
    ids, w = oracle.topk_softmax(logits, topk)
    bad = ids.copy()
    bad[1, :] = [99, -3]
    y, ws = run_moe(x, bad, w, bank_dev(bank), E, H, I)
    assert m.exl3_workspace_error(ws) == 2
    got = as_f64(y)
    assert np.all(got[1] == 0.0)
    keep = np.array([t for t in range(T) if t != 1])
    ref = oracle.moe_f64(np.ascontiguousarray(x[keep]), np.ascontiguousarray(ids[keep]),
                         np.ascontiguousarray(w[keep]), bank)
    assert_rows_close(got[keep], ref)


def test_moe_zero_tokens_is_a_no_op():
    E, H, I = 6, 256, 128
    bank = syn.moe_bank(15, E=E, H=H, I=I)
    ws = m.workspace(1 << 20)
    y = torch.empty((0, H), dtype=torch.bfloat16, device="cuda")
    m.exl3_moe_grouped(torch.empty((0, H), dtype=torch.bfloat16, device="cuda"),
                       torch.empty((0, 2), dtype=torch.int32, device="cuda"),
                       torch.empty((0, 2), dtype=torch.float32, device="cuda"), bank_dev(bank), ws, y=y)


# ---------------------------------------------------------------- FC1 / FC2 on the fused tensor-core GEMM

@pytest.mark.parametrize("T", (1, 5, 20, 40))
def test_moe_small_bank_fused_gemm(T, pin_gemm_path):
    # rows-mode fused GEMM over the device-built entry lists, mixed K, one to 40 tokens
    pin_gemm_path("fused")
    E, H, I, topk = 6, 256, 128, 3
    bank = syn.moe_bank(11, E=E, H=H, I=I, distinct_down_k=True)
    x, logits = syn.moe_tokens(12 + T, T, H=H, E=E)
    ids, w = oracle.topk_softmax(logits, topk)
    y, ws = run_moe(x, ids, w, bank_dev(bank), E, H, I)
    assert_rows_close(as_f64(y), oracle.moe_f64(x, ids, w, bank))
    assert m.exl3_workspace_error(ws) == 0


def test_moe_full_geometry_fused_gemm_16_tokens(full_bank, pin_gemm_path):
    pin_gemm_path("fused")
    bank, bank_d = full_bank
    x, logits = syn.moe_tokens(36, 16)
    ids, w = oracle.topk_softmax(logits, 8)
    y, ws = run_moe(x, ids, w, bank_d, 128, 2048, 768)
    assert_rows_close(as_f64(y), oracle.moe_f64(x, ids, w, bank))
    assert m.exl3_workspace_error(ws) == 0


def test_moe_fused_gemm_deterministic(full_bank, pin_gemm_path):
    pin_gemm_path("fused")
    bank, bank_d = full_bank
    x, logits = syn.moe_tokens(42, 300)
    ids, w = oracle.topk_softmax(logits, 8)
    y1, ws = run_moe(x, ids, w, bank_d, 128, 2048, 768)
    y2, _ = run_moe(x, ids, w, bank_d, 128, 2048, 768, ws)
    assert np.array_equal(bits(y1), bits(y2))
    assert m.exl3_workspace_error(ws) == 0


@pytest.mark.parametrize("T", (1, 4, 16, 512))
def test_moe_forward_back_to_back_bitwise_stable(full_bank, T):
    # Layers issued back to back on one workspace without a host sync give identical
    # bits (T = 512 runs FC1 and FC2 on the tensor-core GEMM in rows mode, whose code
    # ring is filled by bulk copies and must not be overwritten before it is read).
    n = 24
    bank, bank_d = full_bank
    x, logits = syn.moe_tokens(80 + T, T)
    xd, ld = dev(x, torch.bfloat16), dev(logits, torch.float32)
    ws = m.workspace(m.exl3_moe_workspace_bytes(T, 2048, 768, 128, 8))
    ys = torch.empty((n, T, 2048), dtype=torch.bfloat16, device="cuda")
    for i in range(n):
        m.exl3_moe_forward(xd, ld, 8, bank_d, ws, y=ys[i])
    o = ys.view(torch.int16)
    bad = (o != o[:1]).view(n, -1).any(dim=1)
    assert not bool(bad.any()), f"calls {torch.nonzero(bad).flatten().tolist()} differ from the first"
    assert m.exl3_workspace_error(ws) == 0


@pytest.mark.parametrize("T", (1, 16, 64, 65, 512))
def test_moe_forward_equals_topk_then_grouped(full_bank, T):
    # the one-call layer from logits (top-k inside the routing launch for small T)
    # returns the router's ids and weights and the grouped layer's output, bit for bit
    bank, bank_d = full_bank
    x, logits = syn.moe_tokens(60 + T, T)
    ld = dev(logits, torch.float32)
    xd = dev(x, torch.bfloat16)
    ids_ref, w_ref = m.exl3_moe_topk_softmax(ld, 8)
    ws = m.workspace(m.exl3_moe_workspace_bytes(T, 2048, 768, 128, 8))
    y_ref = m.exl3_moe_grouped(xd, ids_ref, w_ref, bank_d, ws)
    y, ids, w = m.exl3_moe_forward(xd, ld, 8, bank_d, ws)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids_ref)
    assert torch.equal(w, w_ref)
    assert np.array_equal(bits(y), bits(y_ref))


def test_moe_forward_small_bank_matches_oracle():
    E, H, I, topk, T = 6, 256, 128, 3, 9
    bank = syn.moe_bank(15, E=E, H=H, I=I, distinct_down_k=True)
    x, logits = syn.moe_tokens(16, T, H=H, E=E)
    ws = m.workspace(m.exl3_moe_workspace_bytes(T, H, I, E, topk))
    y, ids, w = m.exl3_moe_forward(dev(x, torch.bfloat16), dev(logits, torch.float32), topk, bank_dev(bank), ws)
    torch.cuda.synchronize()
    rid, rw = oracle.topk_softmax(logits, topk)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=1e-7)
    assert_rows_close(as_f64(y), oracle.moe_f64(x, rid, rw, bank))
