"""Pins the oracle's EXL3 linear chain.

radiance_escha.py, module docstring ("THE FORWARD"): y = Had128((x*s_in)*rin)
@ decode(code) -> Had128 -> *rout -> *s_out; rin is a pre-scale applied before
its Hadamard, rout a post-scale after its own; rin is applied exactly once; no
bias.  The Hadamard is blocked at 128 channels (create_weights / process_weights
"% _HAD").  These tests check the oracle against scipy's Hadamard, a dense
fp64 matrix formulation built with numpy, and algebraic invariants.
"""
import numpy as np
import pytest
import scipy.linalg

import oracle
import synthetic as syn


def f16(a):
    return np.asarray(a, np.uint16).view(np.float16).astype(np.float64)


def bf16(a):
    b = np.asarray(a, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def hblk(n):
    """Block-diagonal orthonormal Hadamard over blocks of 128 (scipy's Sylvester order)."""
    H = scipy.linalg.hadamard(128).astype(np.float64) / np.sqrt(128.0)
    return scipy.linalg.block_diag(*([H] * (n // 128)))


def dense_reference(x, shard):
    W = f16(oracle.reconstruct(shard.code, shard.K))
    Weff = (np.diag(f16(shard.s_in) * f16(shard.rin)) @ hblk(shard.IC) @ W @ hblk(shard.OC)
            @ np.diag(f16(shard.rout) * f16(shard.s_out)))
    return bf16(x) @ Weff


def test_hadamard_matches_scipy_and_is_orthogonal():
    H = oracle.hadamard128()
    assert np.array_equal(H, scipy.linalg.hadamard(128).astype(np.float64))
    assert np.array_equal(H @ H.T, 128.0 * np.eye(128))
    assert np.array_equal(H, H.T)


@pytest.mark.parametrize("K", (2, 3, 4))
def test_two_formulations_agree(K):
    x, shard = syn.linear_case(7 + K, 5, 256, 384, K)
    y = oracle.linear_f64(x, shard.code, K, shard.s_in, shard.rin, shard.rout, shard.s_out)
    ref = dense_reference(x, shard)
    assert np.max(np.abs(y - ref)) <= 1e-10 * np.max(np.abs(ref))


def test_single_linear_workload_two_formulations():
    x, shard = syn.single_linear(0)
    y = oracle.linear_f64(x, shard.code, shard.K, shard.s_in, shard.rin, shard.rout, shard.s_out)
    ref = dense_reference(x, shard)
    assert np.max(np.abs(y - ref)) <= 1e-10 * np.max(np.abs(ref))


def test_unit_scales_reduce_to_had_w_had():
    x, shard = syn.linear_case(11, 3, 256, 256, 2)
    one = np.full(256, 0x3C00, np.uint16)            # fp16 1.0
    y = oracle.linear_f64(x, shard.code, 2, one, one, one, one)
    W = f16(oracle.reconstruct(shard.code, 2))
    ref = ((bf16(x) @ hblk(256)) @ W) @ hblk(256)
    assert np.max(np.abs(y - ref)) <= 1e-10 * np.max(np.abs(ref))


def test_rin_is_a_pre_scale_not_a_post_scale():
    # moving rin after the input Hadamard (the "easy mistake") gives another answer
    x, shard = syn.linear_case(12, 4, 256, 256, 3)
    y = oracle.linear_f64(x, shard.code, 3, shard.s_in, shard.rin, shard.rout, shard.s_out)
    W = f16(oracle.reconstruct(shard.code, 3))
    post = np.diag(f16(shard.rout) * f16(shard.s_out))
    wrong = ((bf16(x) * f16(shard.s_in)) @ hblk(256) * f16(shard.rin)) @ W @ hblk(256) @ post
    right = ((bf16(x) * f16(shard.s_in) * f16(shard.rin)) @ hblk(256)) @ W @ hblk(256) @ post
    assert np.max(np.abs(y - right)) <= 1e-10 * np.max(np.abs(right))
    assert np.max(np.abs(y - wrong)) > 0.1 * np.sqrt(np.mean(right ** 2))
    # rout likewise belongs after the output Hadamard
    wrong_out = ((bf16(x) * f16(shard.s_in) * f16(shard.rin)) @ hblk(256)) @ W \
        @ np.diag(f16(shard.rout)) @ hblk(256) @ np.diag(f16(shard.s_out))
    assert np.max(np.abs(y - wrong_out)) > 0.1 * np.sqrt(np.mean(right ** 2))


def test_rin_applied_exactly_once():
    # doubling rin (exact in fp16) doubles y exactly: rin enters once, linearly
    x, shard = syn.linear_case(13, 2, 256, 128, 2)
    y1 = oracle.linear_f64(x, shard.code, 2, shard.s_in, shard.rin, shard.rout, shard.s_out)
    rin2 = (f16(shard.rin) * 2).astype(np.float16).view(np.uint16)
    y2 = oracle.linear_f64(x, shard.code, 2, shard.s_in, rin2, shard.rout, shard.s_out)
    assert np.array_equal(y2, 2 * y1)


def test_linearity_and_no_bias():
    g = np.random.default_rng(14)
    _, shard = syn.linear_case(14, 1, 256, 256, 4)
    # small integers: exact in bf16, and so are their sums
    a = g.integers(-8, 9, (3, 256)).astype(np.float32)
    b = g.integers(-8, 9, (3, 256)).astype(np.float32)
    fa, fb, fab = (oracle.linear_f64(syn.f32_to_bf16_bits(v), shard.code, 4, shard.s_in,
                                     shard.rin, shard.rout, shard.s_out) for v in (a, b, a + b))
    assert np.max(np.abs(fab - (fa + fb))) <= 1e-10 * np.max(np.abs(fab))
    zero = oracle.linear_f64(np.zeros((2, 256), np.uint16), shard.code, 4, shard.s_in,
                             shard.rin, shard.rout, shard.s_out)
    assert np.all(zero == 0.0)


def test_blocks_subset_equals_full():
    x, shard = syn.linear_case(15, 3, 256, 512, 2)
    full = oracle.linear_f64(x, shard.code, 2, shard.s_in, shard.rin, shard.rout, shard.s_out)
    part = oracle.linear_f64(x, shard.code, 2, shard.s_in, shard.rin, shard.rout, shard.s_out,
                             blk0=1, nblk=2)
    assert np.array_equal(part, full[:, 128:384])


def test_linear_into_column_slice_and_bf16_rounding():
    x, shards = syn.gate_up(16, M=3, IC=256, OC=256, Ks=(2, 3))
    ldo = 2 * 256 + 64
    out = np.full((3, ldo), 0x7FC1, np.uint16)        # NaN-poisoned
    col = 32
    for s in shards:
        oracle.linear_into(out, x, s.code, s.K, s.s_in, s.rin, s.rout, s.s_out, col)
        y = oracle.linear_f64(x, s.code, s.K, s.s_in, s.rin, s.rout, s.s_out)
        import torch
        ref = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
        # the product is computed in fp64 and rounded once; fp32 then bf16 may double-round,
        # so compare values within one bf16 ulp and require exact bits almost everywhere
        got = out[:, col:col + 256]
        assert np.mean(got == ref.numpy().view(np.uint16)) > 0.99
        col += 256
    assert np.all(out[:, :32] == 0x7FC1) and np.all(out[:, col:] == 0x7FC1)


def test_m_zero_is_a_no_op():
    _, shard = syn.linear_case(17, 1, 128, 128, 2)
    out = np.full((0, 128), 0x7FC1, np.uint16)
    oracle.linear_into(out, np.zeros((0, 128), np.uint16), shard.code, 2, shard.s_in,
                       shard.rin, shard.rout, shard.s_out, 0)


def test_pretransform_matches_dense_hadamard():
    x, shard = syn.linear_case(18, 3, 384, 128, 2)
    u = oracle.pretransform_f64(x, shard.s_in, shard.rin)
    ref = (bf16(x) * f16(shard.s_in) * f16(shard.rin)) @ hblk(384)
    assert np.max(np.abs(u - ref)) <= 1e-12 * np.max(np.abs(ref))
