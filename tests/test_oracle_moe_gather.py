"""Pins the oracle's MoE routing, grouped expert FFN and int8 gather.

bank.py (one layer's EXL3 expert bank): w13 = [w1 | w3] per slot, w2, fp16
w13_suh [E,2,H], w13_svh [E,2,I], w2_suh [E,I], w2_svh [E,H], experts in
K-sorted physical slots.  Each projection is the EXL3 chain
Had(Had(x*suh) @ W) * svh (vllm-quantpack linear.py: "input suh sign-flip +
Hadamard-128, direct trellis GEMM, output svh + Hadamard-128" in the vLLM PR
#190 description).  vllm-quantpack exl3/embedding.py, embedding(): int8 rows
dequantized on the gathered rows, q[ids] * s[ids].
"""
import numpy as np
import scipy.linalg
import scipy.special
import torch

import oracle
import synthetic as syn


def f16(a):
    return np.asarray(a, np.uint16).view(np.float16).astype(np.float64)


def bf16(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def hblk(n):
    H = scipy.linalg.hadamard(128).astype(np.float64) / np.sqrt(128.0)
    return scipy.linalg.block_diag(*([H] * (n // 128)))


def _slot_code(bank, which, p, H, I):
    k = int(bank["k_gu"][p] if which != "w2" else bank["k_d"][p])
    if which == "w2":
        n = I * H * k // 16
        o = int(bank["off_w2"][p])
        return bank["w2"][o:o + n].reshape(I // 16, H // 16, 16 * k), k
    off = bank["off_w1" if which == "w1" else "off_w3"][p]
    n = H * I * k // 16
    return bank["w13"][int(off):int(off) + n].reshape(H // 16, I // 16, 16 * k), k


def _dense_moe(x, ids, w, bank, H, I):
    """Dense-matrix formulation: each projection as one fp64 matrix product."""
    T, topk = ids.shape
    y = np.zeros((T, H))
    for t in range(T):
        for k in range(topk):
            p = int(bank["perm"][ids[t, k]])
            mats = {}
            for which in ("w1", "w3", "w2"):
                code, kk = _slot_code(bank, which, p, H, I)
                mats[which] = f16(oracle.reconstruct(code, kk))
            xt = bf16(x[t])
            g = ((xt * f16(bank["w13_suh"][p, 0])) @ hblk(H) @ mats["w1"] @ hblk(I)) \
                * f16(bank["w13_svh"][p, 0])
            u = ((xt * f16(bank["w13_suh"][p, 1])) @ hblk(H) @ mats["w3"] @ hblk(I)) \
                * f16(bank["w13_svh"][p, 1])
            h = g * scipy.special.expit(g) * u
            d = ((h * f16(bank["w2_suh"][p])) @ hblk(I) @ mats["w2"] @ hblk(H)) \
                * f16(bank["w2_svh"][p])
            y[t] += float(w[t, k]) * d
    return y


def _small_bank(seed=0, distinct=False):
    return syn.moe_bank(seed, E=6, H=256, I=128, Ks=(2, 3, 4), distinct_down_k=distinct)


def test_topk_matches_lexsort_and_softmax():
    g = np.random.default_rng(0)
    logits = g.standard_normal((40, 16)).astype(np.float32)
    logits[3, [2, 5, 9]] = 10.0                     # ties: lower id first
    ids, w = oracle.topk_softmax(logits, 4)
    for t in range(40):
        order = np.lexsort((np.arange(16), -logits[t].astype(np.float64)))[:4]
        assert list(ids[t]) == list(order)
        ref = scipy.special.softmax(logits[t, order].astype(np.float64))
        assert np.allclose(w[t], ref, rtol=1e-6, atol=0)
        assert abs(float(np.sum(w[t], dtype=np.float64)) - 1.0) < 1e-6
    assert list(ids[3][:3]) == [2, 5, 9]


def test_moe_matches_dense_formulation():
    H, I = 256, 128
    bank = _small_bank(1, distinct=True)
    x, logits = syn.moe_tokens(2, 5, H=H, E=6)
    ids, w = oracle.topk_softmax(logits, 3)
    y = oracle.moe_f64(x, ids, w, bank)
    ref = _dense_moe(x, ids, w, bank, H, I)
    assert np.max(np.abs(y - ref)) <= 1e-9 * np.max(np.abs(ref))


def test_moe_single_route_is_one_expert_chain():
    H, I = 256, 128
    bank = _small_bank(3)
    x, _ = syn.moe_tokens(4, 2, H=H, E=6)
    ids = np.array([[4], [1]], np.int32)
    w = np.ones((2, 1), np.float32)
    y = oracle.moe_f64(x, ids, w, bank)
    assert np.max(np.abs(y - _dense_moe(x, ids, w, bank, H, I))) <= 1e-9 * np.max(np.abs(y))


def _repack(bank, new_order, H, I):
    """Same experts in another physical slot order."""
    E = len(new_order)
    old_slot_of = {e: int(bank["perm"][e]) for e in range(E)}
    perm = np.empty(E, np.int32)
    w13, w2 = [], []
    off1, off3, off2 = np.zeros(E, np.int64), np.zeros(E, np.int64), np.zeros(E, np.int64)
    k_gu, k_d = np.zeros(E, np.int32), np.zeros(E, np.int32)
    suh, svh = np.zeros_like(bank["w13_suh"]), np.zeros_like(bank["w13_svh"])
    s2, v2 = np.zeros_like(bank["w2_suh"]), np.zeros_like(bank["w2_svh"])
    a13 = a2 = 0
    for p, e in enumerate(new_order):
        q = old_slot_of[e]
        perm[e] = p
        c1, k1 = _slot_code(bank, "w1", q, H, I)
        c3, _ = _slot_code(bank, "w3", q, H, I)
        c2, k2 = _slot_code(bank, "w2", q, H, I)
        k_gu[p], k_d[p] = k1, k2
        off1[p], off3[p] = a13, a13 + c1.size
        w13 += [c1.ravel(), c3.ravel()]
        a13 += c1.size + c3.size
        off2[p] = a2
        w2.append(c2.ravel())
        a2 += c2.size
        suh[p], svh[p], s2[p], v2[p] = (bank["w13_suh"][q], bank["w13_svh"][q],
                                        bank["w2_suh"][q], bank["w2_svh"][q])
    return dict(w13=np.concatenate(w13), w2=np.concatenate(w2), off_w1=off1, off_w3=off3,
                off_w2=off2, perm=perm, k_gu=k_gu, k_d=k_d, w13_suh=suh, w13_svh=svh,
                w2_suh=s2, w2_svh=v2)


def test_moe_invariant_to_slot_order():
    H, I = 256, 128
    bank = _small_bank(5, distinct=True)
    x, logits = syn.moe_tokens(6, 4, H=H, E=6)
    ids, w = oracle.topk_softmax(logits, 2)
    y = oracle.moe_f64(x, ids, w, bank)
    y2 = oracle.moe_f64(x, ids, w, _repack(bank, [5, 0, 3, 1, 4, 2], H, I))
    assert np.array_equal(y, y2)


def test_bank_slots_are_k_sorted():
    bank = syn.moe_bank(7, E=16, H=256, I=128, distinct_down_k=True)
    keys = list(zip(bank["k_gu"], bank["k_d"]))
    assert keys == sorted(keys)


def test_gather_matches_numpy_and_masks_bad_ids():
    q, s, ids = syn.embedding(0, V=1000, H=96, N=300)
    ids[[3, 77]] = [-1, 1000]
    out, bad = oracle.gather(q, s, ids)
    assert bad == 2
    ok = (ids >= 0) & (ids < 1000)
    prod = (q[ids[ok]].astype(np.float64) * f16(s)[ids[ok], None]).astype(np.float32)
    ref = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out[ok], ref)      # the product is exact in fp32: one rounding
    assert np.all(out[~ok] == 0)
