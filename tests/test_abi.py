"""The C-ABI library loads and exports every symbol include/exl3.h declares
(no compute call: this runs without a GPU)."""
import ctypes
import os
import re

import moe_gemm_exl3_gb300 as m
from moe_gemm_exl3_gb300 import build as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "exl3.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(exl3_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    b.build()
    lib = ctypes.CDLL(m.LIB_PATH)
    names = declared_symbols()
    assert len(names) >= 14
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(m.EXPORTS) == names


def test_host_side_queries_without_gpu():
    b.build()
    L = m.lib()
    assert m.exl3_version().startswith("exl3-gb300")
    # workspace sizes are pure host arithmetic
    assert m.exl3_linear_workspace_bytes(8, 5120, 17408) > 0
    assert m.exl3_linear_workspace_bytes(8, 5000, 17408) == 0      # IC not a multiple of 128
    assert m.exl3_linear_workspace_bytes(8, 5120, 17400) == 0
    assert m.exl3_linear_workspace_bytes(-1, 5120, 17408) == 0
    # invalid sizes are rejected on the host before any CUDA call
    st = L.exl3_linear_into(None, 4, 500, None, 512, 2, None, None, None, None, None, 512, 0,
                            None, 0, None)
    assert st == m.EXL3_EINVAL
    assert b"multiples of 128" in L.exl3_last_error()
    st = L.exl3_linear_into(None, 4, 512, None, 512, 5, None, None, None, None, None, 512, 0,
                            None, 0, None)
    assert st == m.EXL3_EUNSUPPORTED
    st = L.exl3_embed_int8_gather(None, None, 10, 24, None, 3, None, None, None)
    assert st == m.EXL3_EINVAL


def test_workspace_sizes_never_shrink_as_the_call_grows():
    # a workspace sized for the largest call serves every smaller one
    b.build()
    L = m.lib()
    prev = 0
    for M in range(0, 300):
        v = L.exl3_linear_workspace_bytes(M, 5120, 17408)
        assert v >= prev, (M, prev, v)
        prev = v
    for H, I, E, topk in ((2048, 768, 128, 8), (1024, 512, 8, 2), (512, 256, 64, 4)):
        prev = 0
        for T in list(range(0, 1100, 3)) + [4000, 9000, 20000, 70000]:
            v = L.exl3_moe_workspace_bytes(T, H, I, E, topk)
            assert v >= prev, (H, I, E, topk, T, prev, v)
            prev = v


def test_long_moe_calls_run_in_passes_of_bounded_workspace():
    # past the tokens one pass serves (its column groups must fit the workspace's
    # arrival counters) the call runs in passes: the workspace stops growing
    b.build()
    L = m.lib()
    sizes = [L.exl3_moe_workspace_bytes(T, 2048, 768, 128, 8) for T in (3000, 3967, 3968, 8000, 100000, 2097152)]
    assert sizes[0] <= sizes[1]
    assert max(sizes[2:]) <= sizes[1] * 1.01 and min(sizes[2:]) > 0
    # a geometry whose column groups exceed the counters even for one token is refused on the host
    assert L.exl3_moe_workspace_bytes(1, 128 * 40000, 128, 8, 2) == 0
    st = L.exl3_moe_grouped(None, 1, 128 * 40000, 128, 8, 2, None, None, None, None, None, 0, None)
    assert st == m.EXL3_EINVAL and b"counters" in L.exl3_last_error()


def test_struct_layouts_match_the_binding(tmp_path):
    # the ctypes mirrors of exl3_shard and exl3_projection have the C layout
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "exl3.h"\n'
                   'int main(void) { printf("%zu %zu %zu %zu %zu\\n", sizeof(exl3_shard), '
                   'offsetof(exl3_shard, col0), offsetof(exl3_shard, codebook), sizeof(exl3_projection), '
                   'offsetof(exl3_projection, ldo)); return 0; }\n')
    exe = tmp_path / "layout"
    import subprocess
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    want = [ctypes.sizeof(m.Shard), m.Shard.col0.offset, m.Shard.codebook.offset, ctypes.sizeof(m.Projection),
            m.Projection.ldo.offset]
    assert got == want


def test_marked_codebooks_are_rejected_before_any_launch():
    # a shard carrying the MCG or MUL1 marker fails validation on the host (its
    # decode constants are not part of this build); an unknown value is invalid
    b.build()
    L = m.lib()
    for cb, st_want, word in ((1, m.EXL3_EUNSUPPORTED, b"MCG"), (2, m.EXL3_EUNSUPPORTED, b"MUL1"),
                              (7, m.EXL3_EINVAL, b"codebook = 7")):
        sh = (m.Shard * 1)()
        sh[0] = m.Shard(4096, 4096, 4096, 4096, 4096, 256, 2, 0, cb, 0)   # never dereferenced
        st = L.exl3_linear_into_shards(4096, 1, 256, sh, 1, 8192, 256, 16384, 1 << 20, None)
        assert st == st_want
        assert word in L.exl3_last_error()
