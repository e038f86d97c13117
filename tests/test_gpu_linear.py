"""GPU parity of the EXL3 linear path against the CPU oracle, through the C ABI.

Decoded weights and the codebook must match the oracle bit for bit; outputs
must satisfy max|y - y_ref| <= 2e-2 * rms(y_ref) per row (fp32 accumulation).
Columns outside a shard's slice must keep their NaN poison (the vLLM PR #190
trellis-MoE validation used NaN-poisoned scratch the same way).
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
    m.lib()


def shard_dev(sh):
    return (dev(sh.code, torch.int16), *(dev(v, torch.float16) for v in (sh.s_in, sh.rin, sh.rout, sh.s_out)))


def shard_set(sh, col0):
    """(code, K, s_in, rin, rout, s_out, col0) on the device: one shard of a merged call."""
    c, *sc = shard_dev(sh)
    return (c, sh.K, *sc, col0)


def test_codebook_table_exhaustive():
    got = bits(m.exl3_codebook_table())
    assert np.array_equal(got, oracle.codebook_table())


@pytest.mark.parametrize("K", (2, 3, 4))
def test_reconstruct_bit_exact_small(K):
    g = syn.rng(40 + K)
    code = syn.uniform_code(g, (32, 48, 16 * K))     # IC = 512, OC = 768
    W = m.exl3_reconstruct(dev(code, torch.int16), K)
    assert np.array_equal(bits(W), oracle.reconstruct(code, K))


@pytest.mark.parametrize("K", (2, 3, 4))
def test_reconstruct_single_bit_tiles(K):
    # one tile per stream bit position class: pins the bit order, window and tail-biting on GPU
    n = 256 * K
    pos = list(range(0, n, max(1, n // 61))) + [0, 15, 16, n - 1]
    code = np.zeros((1, len(pos), 16 * K), np.uint16)
    for i, p in enumerate(pos):
        code[0, i, p // 16] = 1 << (15 - p % 16)
    code = code.view(np.int16)
    pad = (-len(pos)) % 8                             # OC multiple of 128 is not needed here
    code = np.concatenate([code, np.zeros((1, pad, 16 * K), np.int16)], axis=1)
    W = m.exl3_reconstruct(dev(code, torch.int16), K)
    assert np.array_equal(bits(W), oracle.reconstruct(code, K))


@pytest.mark.parametrize("K", (2, 3))
def test_reconstruct_bit_exact_full_gate_up_shards(K):
    # every tile of a 5120 x 17408 shard
    g = syn.rng(50 + K)
    code = syn.uniform_code(g, (320, 1088, 16 * K))
    W = bits(m.exl3_reconstruct(dev(code, torch.int16), K))
    for b0 in range(0, 17408, 4352):                   # oracle in column chunks (memory)
        assert np.array_equal(W[:, b0:b0 + 4352], oracle.reconstruct(code, K, b0, 4352))


def test_pretransform_matches_oracle():
    x, sh = syn.linear_case(60, 7, 1024, 128, 2, outlier_frac=0.01)
    u = m.exl3_pretransform(dev(x, torch.bfloat16), dev(sh.s_in, torch.float16), dev(sh.rin, torch.float16))
    ref = oracle.pretransform_f64(x, sh.s_in, sh.rin)
    got = as_f64(u)
    # fp16 output: within half an fp16 ulp of the fp64 value plus fp32 rounding
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -10 + 1e-6)


@pytest.mark.parametrize("M,IC", ((16000, 640), (2500, 5120)))
def test_pretransform_long_runs_matches_oracle(M, IC):
    # enough blocks for the four-block runs per warp, including a row whose last
    # run is short (IC / 128 = 5 blocks); rows sampled for the oracle
    x, sh = syn.linear_case(61, M, IC, 128, 2, outlier_frac=0.01)
    u = m.exl3_pretransform(dev(x, torch.bfloat16), dev(sh.s_in, torch.float16), dev(sh.rin, torch.float16))
    rows = np.array([0, 1, M // 2, M - 2, M - 1])
    ref = oracle.pretransform_f64(np.ascontiguousarray(x[rows]), sh.s_in, sh.rin)
    got = as_f64(u)[rows]
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -10 + 1e-6)


def run_linear(x, sh, ws=None):
    M = x.shape[0]
    if ws is None:
        ws = m.workspace(m.exl3_linear_workspace_bytes(M, sh.IC, sh.OC))
    y = m.exl3_linear(dev(x, torch.bfloat16), *shard_dev(sh)[:1], sh.K, *shard_dev(sh)[1:], ws)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("K", (2, 3, 4))
@pytest.mark.parametrize("M", (1, 3, 8, 13, 32, 33, 70))
def test_linear_parity_small(K, M):
    x, sh = syn.linear_case(100 + M + K, M, 512, 640, K)
    y = run_linear(x, sh)
    ref = oracle.linear_f64(x, sh.code, K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    assert_rows_close(as_f64(y), ref)


def sample_rows(M):
    """Every row for decode-sized calls; for larger M, rows at both ends and the middle
    (the split-K partition and the reduction depend on the column group, not the row)."""
    return np.arange(M) if M <= 16 else np.unique(np.array([0, 1, M // 2, M - 2, M - 1]))


def test_single_linear_workload():
    x, sh = syn.single_linear(0)
    y = run_linear(x, sh)
    ref = oracle.linear_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    assert_rows_close(as_f64(y), ref)


@pytest.mark.parametrize("M", (1, 8, 64))
def test_gate_up_full_size_per_shard_calls(M):
    # the decode-shaped merged gate (K=2) / up (K=3) layer into one out[M, 34816],
    # one exl3_linear_into call per shard; every column against the oracle
    x, shards = syn.gate_up(1, M=M)
    OC = 17408
    out = torch.full((M, 2 * OC), 0, dtype=torch.int16, device="cuda")
    out.fill_(NAN_BF16)
    out = out.view(torch.bfloat16)
    ws = m.workspace(m.exl3_linear_workspace_bytes(M, 5120, OC))
    xd = dev(x, torch.bfloat16)
    for i, sh in enumerate(shards):
        c, *sc = shard_dev(sh)
        m.exl3_linear_into(xd, c, sh.K, *sc, out, i * OC, ws)
    torch.cuda.synchronize()
    got = as_f64(out)
    assert np.all(np.isfinite(got)), "a column of the output was left unwritten"
    rows = sample_rows(M)
    xs = np.ascontiguousarray(x[rows])
    for i, sh in enumerate(shards):
        ref = oracle.linear_f64(xs, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
        assert_rows_close(got[rows, i * OC:(i + 1) * OC], ref)


@pytest.mark.parametrize("M", (1, 8, 16, 32, 64, 128))
def test_gate_up_one_call_full_size_every_column(M):
    # the benchmarked launch: both shards in one exl3_linear_into_shards call (decode
    # mode to M = 16, the fused tensor-core kernel above); every 128-column block of
    # both shards is compared with the oracle, on every row up to M = 16
    x, shards = syn.gate_up(1, M=M)
    OC = 17408
    out = torch.full((M, 2 * OC), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    sets = [shard_set(sh, i * OC) for i, sh in enumerate(shards)]
    ws = m.workspace(m.exl3_linear_shards_workspace_bytes(M, 5120, sets))
    m.exl3_linear_into_shards(dev(x, torch.bfloat16), sets, out, ws)
    torch.cuda.synchronize()
    got = as_f64(out)
    assert np.all(np.isfinite(got)), "a column of the output was left unwritten"
    rows = sample_rows(M)
    xs = np.ascontiguousarray(x[rows])
    for i, sh in enumerate(shards):
        ref = oracle.linear_f64(xs, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
        assert_rows_close(got[rows, i * OC:(i + 1) * OC], ref)
    assert m.exl3_workspace_error(ws) == 0


@pytest.mark.parametrize("M", (8, 8192))
def test_decoder_layer_full_size_every_column(M):
    # the five projections of the benchmarked decoder layer, launched as the bench
    # launches them (qkv, o, down alone; gate and up in one call on gate's input);
    # every output column of every projection, on all rows at M = 8 and on rows at
    # both ends and the middle at M = 8192
    projs = {n: (x, sh) for n, x, sh in syn.decoder_layer(4, M=M)}
    sets = [shard_set(projs[n][1], c) for n, c in (("gate", 0), ("up", 17408))]
    ws = m.workspace(max(m.exl3_linear_workspace_bytes(M, 17408, 17408),
                         m.exl3_linear_shards_workspace_bytes(M, 5120, sets)))
    rows = np.arange(M) if M <= 128 else np.array([0, 1, 127, 128, 4095, 8190, 8191])
    checks = []
    for name in ("qkv", "o", "down"):
        x, sh = projs[name]
        out = torch.full((M, sh.OC), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        c, *sc = shard_dev(sh)
        m.exl3_linear_into(dev(x, torch.bfloat16), c, sh.K, *sc, out, 0, ws)
        torch.cuda.synchronize()
        checks.append((x, sh, as_f64(out), 0))
    xg = projs["gate"][0]
    out = torch.full((M, 2 * 17408), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    m.exl3_linear_into_shards(dev(xg, torch.bfloat16), sets, out, ws)
    torch.cuda.synchronize()
    got_gu = as_f64(out)
    checks += [(xg, projs["gate"][1], got_gu, 0), (xg, projs["up"][1], got_gu, 17408)]
    for x, sh, got, col0 in checks:
        assert np.all(np.isfinite(got[:, col0:col0 + sh.OC]))
        xs = np.ascontiguousarray(x[rows])
        ref = oracle.linear_f64(xs, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
        assert_rows_close(got[rows, col0:col0 + sh.OC], ref)
    assert m.exl3_workspace_error(ws) == 0


def test_column_slice_isolation_and_merged_layer():
    x, shards = syn.gate_up(7, M=5, IC=512, OC=384, Ks=(2, 3))
    ldo = 2 * 384 + 64
    out = torch.full((5, ldo), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    ws = m.workspace(m.exl3_linear_workspace_bytes(5, 512, 384))
    xd = dev(x, torch.bfloat16)
    col = 32
    for sh in shards:
        c, *sc = shard_dev(sh)
        m.exl3_linear_into(xd, c, sh.K, *sc, out, col, ws)
        col += 384
    torch.cuda.synchronize()
    b = bits(out)
    assert np.all(b[:, :32] == NAN_BF16) and np.all(b[:, col:] == NAN_BF16)
    col = 32
    for sh in shards:
        ref = oracle.linear_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
        assert_rows_close(as_f64(out)[:, col:col + 384], ref)
        col += 384


def test_deterministic_and_batch_invariant():
    x, sh = syn.linear_case(8, 8, 1024, 1024, 3)
    y8a = bits(run_linear(x, sh))
    y8b = bits(run_linear(x, sh))
    assert np.array_equal(y8a, y8b)
    for r in (0, 5):
        y1 = bits(run_linear(x[r:r + 1], sh))
        assert np.array_equal(y1[0], y8a[r])


def test_graph_replay_equals_eager():
    x, sh = syn.linear_case(9, 4, 1024, 768, 2)
    ws = m.workspace(m.exl3_linear_workspace_bytes(4, 1024, 768))
    xd = dev(x, torch.bfloat16)
    c, *sc = shard_dev(sh)
    eager = bits(m.exl3_linear(xd, c, 2, *sc, ws))
    out = torch.empty((4, 768), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            m.exl3_linear(xd, c, 2, *sc, ws, out=out)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), eager)


def test_errors_are_reported_not_launched():
    x, sh = syn.linear_case(10, 2, 256, 256, 2)
    c, *sc = shard_dev(sh)
    xd = dev(x, torch.bfloat16)
    small = m.workspace(1 << 20)
    with pytest.raises(m.Exl3Error) as e:
        m.exl3_linear(xd, c, 2, *sc, small)
    assert e.value.status == m.EXL3_EWORKSPACE
    ws = m.workspace(m.exl3_linear_workspace_bytes(2, 256, 256))
    out = torch.empty((2, 300), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.Exl3Error) as e:
        m.exl3_linear_into(xd, c, 2, *sc, out, 100, ws)       # slice past ldo
    assert e.value.status == m.EXL3_EINVAL
    with pytest.raises(ValueError):
        m.exl3_linear(xd, c, 3, *sc, ws)                       # K disagrees with the code's shape
    # M == 0 is a no-op
    m.exl3_linear(xd[:0], c, 2, *sc, ws)
    assert m.exl3_workspace_error(ws) == 0


@pytest.mark.parametrize("M,Ks", [(1, (2, 3)), (5, (4, 2)), (8, (3, 3)), (8, (2, 4)), (12, (2, 3)), (16, (4, 3))])
def test_paired_shards_every_column_and_stable(M, Ks):
    # Two shards of one width with 5/8 as many column groups per shard as the GPU
    # has SMs: the decode path gives each 16-warp CTA one group of each shard,
    # one to each half of its warps (one 8-row block to M = 8, two to M = 16).
    # Every column against the oracle, and 20 back-to-back calls identical bit
    # for bit.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    IC, OC = 1024, 128 * (sms * 5 // 8)
    x, shards = syn.gate_up(120 + M, M=M, IC=IC, OC=OC, Ks=Ks)
    sets = [shard_set(sh, i * OC) for i, sh in enumerate(shards)]
    ws = m.workspace(m.exl3_linear_shards_workspace_bytes(M, IC, sets))
    xd = dev(x, torch.bfloat16)
    n = 20
    outs = torch.full((n, M, 2 * OC), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    for i in range(n):
        m.exl3_linear_into_shards(xd, sets, outs[i], ws)
    torch.cuda.synchronize()
    o = outs.view(torch.int16)
    assert bool((o == o[:1]).all()), "back-to-back calls differ"
    got = as_f64(outs[0])
    for i, sh in enumerate(shards):
        ref = oracle.linear_f64(x, sh.code, sh.K, sh.s_in, sh.rin, sh.rout, sh.s_out)
        assert_rows_close(got[:, i * OC:(i + 1) * OC], ref)
    assert m.exl3_workspace_error(ws) == 0


@pytest.mark.parametrize("M", (1, 8, 13))
def test_linear_into_shards_host_equals_device_call(M):
    # x and out in pinned host memory, read and written by the kernels through
    # their device mappings: the result equals the device-buffer call bit for
    # bit, and the columns outside the shards keep their poison
    x, shards = syn.gate_up(1, M=M)
    OC = 17408
    sets = [shard_set(sh, 64 + i * OC) for i, sh in enumerate(shards)]
    ws = m.workspace(m.exl3_linear_shards_workspace_bytes(M, 5120, sets))
    xd = dev(x, torch.bfloat16)
    ref = torch.full((M, 2 * OC + 128), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    m.exl3_linear_into_shards(xd, sets, ref, ws)
    xh = xd.cpu().pin_memory()
    oh = torch.full((M, 2 * OC + 128), NAN_BF16, dtype=torch.int16).pin_memory().view(torch.bfloat16)
    m.exl3_linear_into_shards_host(xh, sets, oh, ws)
    torch.cuda.synchronize()
    assert torch.equal(oh.view(torch.int16), ref.cpu().view(torch.int16))
    assert bool((oh.view(torch.int16)[:, :64] == NAN_BF16).all())
    assert m.exl3_workspace_error(ws) == 0


def test_linear_into_shards_host_refuses_unmapped_buffers():
    # pageable host memory and device memory are refused on the host, before any launch
    import ctypes
    L = m.lib()
    x, sh = syn.linear_case(12, 2, 256, 256, 2)
    sets = [shard_set(sh, 0)]
    arr = m._shard_array(sets, 256)
    ws = m.workspace(m.exl3_linear_shards_workspace_bytes(2, 256, sets))
    st = torch.cuda.current_stream().cuda_stream
    pageable = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    pinned_x = pageable.pin_memory()
    pinned_out = torch.empty((2, 256), dtype=torch.bfloat16).pin_memory()
    dev_out = torch.empty((2, 256), dtype=torch.bfloat16, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    r = L.exl3_linear_into_shards_host(p(pageable), 2, 256, arr, 1, p(pinned_out), 256, p(ws), ws.numel(), st)
    assert r == m.EXL3_EINVAL and b"x_host" in L.exl3_last_error()
    r = L.exl3_linear_into_shards_host(p(pinned_x), 2, 256, arr, 1, p(dev_out), 256, p(ws), ws.numel(), st)
    assert r == m.EXL3_EINVAL and b"out_host" in L.exl3_last_error()
    with pytest.raises(ValueError):
        m.exl3_linear_into_shards_host(pageable, sets, pinned_out, ws)


@pytest.mark.parametrize("M", (1, 8, 20, 40))
def test_shards_call_equals_per_shard_calls(M):
    # a merged layer in one call gives the per-shard result (three shards, different K and OC)
    g = syn.rng(70 + M)
    IC = 1024
    shards = [syn.make_shard(g, IC, OC, K) for OC, K in ((384, 2), (640, 3), (256, 4))]
    x = syn.normal_bf16(g, M, IC)
    ldo = sum(s.OC for s in shards) + 64
    xd = dev(x, torch.bfloat16)
    dsh = [(*shard_dev(s)[:1], s.K, *shard_dev(s)[1:]) for s in shards]
    ws = m.workspace(m.exl3_linear_shards_workspace_bytes(M, IC, dsh))
    got = torch.full((M, ldo), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    m.exl3_linear_into_shards(xd, dsh, got, ws)
    torch.cuda.synchronize()
    b = bits(got)
    assert np.all(b[:, ldo - 64:] == NAN_BF16)
    col = 0
    for s in shards:
        ref = oracle.linear_f64(x, s.code, s.K, s.s_in, s.rin, s.rout, s.s_out)
        assert_rows_close(as_f64(got)[:, col:col + s.OC], ref)
        col += s.OC


# ---------------------------------------------------------------- fused tensor-core path (8 < M <= 128)

@pytest.mark.parametrize("M", (9, 16, 17, 31, 64, 65, 100, 128))
def test_fused_parity_split_and_whole_groups(M, pin_gemm_path):
    # 160 column groups of 8 stages over one persistent grid: some groups are
    # reduced across CTAs through the split-K slab, others owned by one CTA;
    # M spans all four accumulator widths (16, 32, 64, 128 rows)
    pin_gemm_path("fused")
    K = 2 + M % 3
    x, sh = syn.linear_case(300 + M, M, 512, 20480, K)
    ws = m.workspace(m.exl3_linear_workspace_bytes(M, sh.IC, sh.OC))
    y = run_linear(x, sh, ws)
    ref = oracle.linear_f64(x, sh.code, K, sh.s_in, sh.rin, sh.rout, sh.s_out)
    assert_rows_close(as_f64(y), ref)
    assert m.exl3_workspace_error(ws) == 0


@pytest.mark.parametrize("mode", ("decode", "fused", "prefill"))
def test_forced_modes_agree_with_oracle(mode, pin_gemm_path):
    # every GEMM path serves the same M; each must match the oracle
    pin_gemm_path(mode)
    x, sh = syn.linear_case(77, 24, 1024, 768, 3)
    y = run_linear(x, sh)
    ref = oracle.linear_f64(x, sh.code, 3, sh.s_in, sh.rin, sh.rout, sh.s_out)
    assert_rows_close(as_f64(y), ref)


@pytest.mark.parametrize("M", (12, 96))
def test_gemm_into_fused_from_caller_activations(M, pin_gemm_path):
    # caller-supplied pre-transformed activations go straight to the fused GEMM
    pin_gemm_path("fused")
    x, sh = syn.linear_case(500 + M, M, 1024, 1280, 4)
    c, s_in, rin, rout, s_out = shard_dev(sh)
    u = m.exl3_pretransform(dev(x, torch.bfloat16), s_in, rin)
    out = torch.full((M, 1280 + 128), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    ws = m.workspace(m.exl3_linear_workspace_bytes(M, 1024, 1280))
    m.exl3_gemm_into(u, c, 4, rout, s_out, out, 128, ws)
    torch.cuda.synchronize()
    assert np.all(bits(out)[:, :128] == NAN_BF16)
    ref = oracle.linear_f64(x, sh.code, 4, sh.s_in, sh.rin, sh.rout, sh.s_out)
    assert_rows_close(as_f64(out)[:, 128:], ref)


def test_fused_repeated_calls_deterministic():
    # the split-K counters reset themselves: back-to-back calls give identical bits
    x, sh = syn.linear_case(91, 40, 512, 20480, 3)
    ws = m.workspace(m.exl3_linear_workspace_bytes(40, 512, 20480))
    a = bits(run_linear(x, sh, ws))
    b = bits(run_linear(x, sh, ws))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("M", (64, 96, 128))
def test_fused_back_to_back_calls_bitwise_stable(M):
    # Merged gate/up calls issued back to back on one workspace, no host sync in
    # between.  The split-K partials are summed in CTA order, so every call must
    # give identical bits.  A code-ring slot handed to the next TMA copy before
    # every decoder warp had read it showed up here as about one wrong split
    # column group per call.
    n = 60
    x, shards = syn.gate_up(1, M=M)
    OC = shards[0].code.shape[1] * 16
    sets = [shard_set(sh, i * OC) for i, sh in enumerate(shards)]
    ws = m.workspace(m.exl3_linear_shards_workspace_bytes(M, x.shape[1], sets))
    xd = dev(x, torch.bfloat16)
    outs = torch.empty((n, M, 2 * OC), dtype=torch.bfloat16, device="cuda")
    for i in range(n):
        m.exl3_linear_into_shards(xd, sets, outs[i], ws)
    o = outs.view(torch.int16)
    bad = (o != o[:1]).view(n, M, -1, 128).any(dim=3).any(dim=1)   # [call][column group]
    calls, groups = torch.nonzero(bad, as_tuple=True)
    assert calls.numel() == 0, f"calls {calls.unique().tolist()} differ in groups {groups.unique().tolist()}"
    assert m.exl3_workspace_error(ws) == 0


def test_fused_single_stage_segments(pin_gemm_path):
    # IC = 128: two stages per column group, so CTAs at group boundaries get
    # one-stage segments that only one of the two MMA issuers accumulates
    pin_gemm_path("fused")
    x, sh = syn.linear_case(93, 20, 128, 128 * 300, 2)
    y = run_linear(x, sh)
    ref = oracle.linear_f64(x, sh.code, 2, sh.s_in, sh.rin, sh.rout, sh.s_out)
    assert_rows_close(as_f64(y), ref)
