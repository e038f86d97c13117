"""Python binding of the GB300 EXL3 trellis library (``include/exl3.h``).

Argument marshalling only: every function checks dtypes, shapes and devices of
torch tensors, passes raw device pointers and the current CUDA stream to the
C ABI of ``libexl3_gb300.so`` (built in-tree by ``moe_gemm_exl3_gb300.build``)
and raises :class:`Exl3Error` on a non-zero status.  All compute runs in the
library's CUDA kernels; there is no host fallback.  Function names match the
C entry points.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libexl3_gb300.so")

EXL3_OK, EXL3_EINVAL, EXL3_EWORKSPACE, EXL3_ECUDA, EXL3_EUNSUPPORTED, EXL3_EDEVICE = range(6)
STATUS_NAMES = {0: "EXL3_OK", 1: "EXL3_EINVAL", 2: "EXL3_EWORKSPACE", 3: "EXL3_ECUDA",
                4: "EXL3_EUNSUPPORTED", 5: "EXL3_EDEVICE"}

# Every symbol include/exl3.h declares.
EXPORTS = ("exl3_last_error", "exl3_version", "exl3_linear_workspace_bytes", "exl3_workspace_init",
           "exl3_workspace_error", "exl3_set_gemm_path", "exl3_linear_into", "exl3_linear", "exl3_gemm_into", "exl3_linear_into_noalloc",
           "exl3_linear_shards_workspace_bytes", "exl3_linear_into_shards", "exl3_gemm_into_shards", "exl3_pretransform",
           "exl3_reconstruct", "exl3_codebook_table", "exl3_moe_topk_softmax",
           "exl3_moe_workspace_bytes", "exl3_moe_grouped", "exl3_embed_int8_gather",
           "exl3_lm_head_workspace_bytes", "exl3_lm_head_int8", "exl3_projections_workspace_bytes",
           "exl3_linear_projections", "exl3_linear_a8_workspace_bytes", "exl3_quantize_a8",
           "exl3_linear_into_a8", "exl3_gemm_a8_into", "exl3_linear_shards_a8_workspace_bytes",
           "exl3_linear_into_shards_a8", "exl3_gemm_a8_into_shards", "exl3_moe_forward",
           "exl3_linear_into_shards_host")


class Exl3Error(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


CODEBOOKS = {"3inst": 0, "mcg": 1, "mul1": 2}


class Shard(ctypes.Structure):
    """exl3_shard: one source tensor of a merged layer."""
    _fields_ = [("code", ctypes.c_void_p), ("s_in", ctypes.c_void_p), ("rin", ctypes.c_void_p),
                ("rout", ctypes.c_void_p), ("s_out", ctypes.c_void_p), ("OC", ctypes.c_int32),
                ("K", ctypes.c_int32), ("col0", ctypes.c_int64), ("codebook", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class Projection(ctypes.Structure):
    """exl3_projection: one projection of a layer (input, shards, output)."""
    _fields_ = [("x", ctypes.c_void_p), ("IC", ctypes.c_int32), ("n_shards", ctypes.c_int32),
                ("shards", ctypes.POINTER(Shard)), ("out", ctypes.c_void_p), ("ldo", ctypes.c_int64)]


class MoeBank(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w13", "w2", "off_w1", "off_w3", "off_w2", "perm", "k_gu", "k_d",
                 "w13_suh", "w13_svh", "w2_suh", "w2_svh")]


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Load the in-tree library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"EXL3 CUDA library missing ({LIB_PATH}); build it with "
                                   "moe_gemm_exl3_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            sig = {
                "exl3_last_error": ([], ctypes.c_char_p),
                "exl3_version": ([], ctypes.c_char_p),
                "exl3_linear_workspace_bytes": ([i64, i32, i32], sz),
                "exl3_workspace_init": ([vp, sz, vp], ctypes.c_int),
                "exl3_workspace_error": ([vp, sz, ctypes.POINTER(ctypes.c_int32), vp], ctypes.c_int),
                "exl3_set_gemm_path": ([i32], ctypes.c_int),
                "exl3_linear_into": ([vp, i64, i32, vp, i32, i32, vp, vp, vp, vp, vp, i64, i64, vp, sz,
                                      vp], ctypes.c_int),
                "exl3_linear": ([vp, i64, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp],
                                ctypes.c_int),
                "exl3_linear_into_noalloc": ([vp, i64, i32, vp, i32, i32, vp, vp, vp, vp, vp, i64, i64,
                                              vp], ctypes.c_int),
                "exl3_linear_shards_workspace_bytes": ([i64, i32, ctypes.POINTER(Shard), i32], sz),
                "exl3_linear_into_shards": ([vp, i64, i32, ctypes.POINTER(Shard), i32, vp, i64, vp, sz, vp],
                                            ctypes.c_int),
                "exl3_gemm_into_shards": ([vp, i64, i32, ctypes.POINTER(Shard), i32, vp, i64, vp, sz, vp],
                                          ctypes.c_int),
                "exl3_gemm_into": ([vp, i64, i32, vp, i32, i32, vp, vp, vp, i64, i64, vp, sz, vp],
                                   ctypes.c_int),
                "exl3_pretransform": ([vp, i64, i32, vp, vp, vp, vp], ctypes.c_int),
                "exl3_reconstruct": ([vp, i32, i32, i32, vp, vp], ctypes.c_int),
                "exl3_codebook_table": ([vp, vp], ctypes.c_int),
                "exl3_moe_topk_softmax": ([vp, i32, i32, i32, vp, vp, vp], ctypes.c_int),
                "exl3_moe_workspace_bytes": ([i32, i32, i32, i32, i32], sz),
                "exl3_moe_grouped": ([vp, i32, i32, i32, i32, i32, vp, vp, ctypes.POINTER(MoeBank), vp,
                                      vp, sz, vp], ctypes.c_int),
                "exl3_moe_forward": ([vp, vp, i32, i32, i32, i32, i32, ctypes.POINTER(MoeBank), vp, vp, vp, vp,
                                      sz, vp], ctypes.c_int),
                "exl3_embed_int8_gather": ([vp, vp, i64, i32, vp, i64, vp, vp, vp], ctypes.c_int),
                "exl3_lm_head_workspace_bytes": ([i64, i32, i64], sz),
                "exl3_projections_workspace_bytes": ([i64, ctypes.POINTER(Projection), i32], sz),
                "exl3_linear_projections": ([ctypes.POINTER(Projection), i32, i64, vp, sz, vp], ctypes.c_int),
                "exl3_lm_head_int8": ([vp, i64, i32, vp, vp, i64, vp, i64, vp, sz, vp], ctypes.c_int),
                "exl3_linear_a8_workspace_bytes": ([i64, i32, i32], sz),
                "exl3_quantize_a8": ([vp, i64, i32, vp, vp, vp, vp, vp], ctypes.c_int),
                "exl3_linear_into_a8": ([vp, i64, i32, vp, i32, i32, vp, vp, vp, vp, vp, i64, i64, vp, sz,
                                         vp], ctypes.c_int),
                "exl3_gemm_a8_into": ([vp, vp, i64, i32, vp, i32, i32, vp, vp, vp, i64, i64, vp, sz, vp],
                                      ctypes.c_int),
                "exl3_linear_shards_a8_workspace_bytes": ([i64, i32, ctypes.POINTER(Shard), i32], sz),
                "exl3_linear_into_shards_host": ([vp, i64, i32, ctypes.POINTER(Shard), i32, vp, i64, vp, sz, vp],
                                                 ctypes.c_int),
                "exl3_linear_into_shards_a8": ([vp, i64, i32, ctypes.POINTER(Shard), i32, vp, i64, vp, sz, vp],
                                               ctypes.c_int),
                "exl3_gemm_a8_into_shards": ([vp, vp, i64, i32, ctypes.POINTER(Shard), i32, vp, i64, vp, sz, vp],
                                             ctypes.c_int),
            }
            for name, (args, res) in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device=None) -> int:
    """The current CUDA stream of device (its raw handle)."""
    if _raw_stream is not None:
        # the handle without building a Stream object (a few microseconds a call)
        if device is None or device.index is None:
            return _raw_stream(torch.cuda.current_device())
        return _raw_stream(device.index)
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _check(st: int, fn: str):
    if st != EXL3_OK:
        raise Exl3Error(st, fn, lib().exl3_last_error().decode(errors="replace"))


def exl3_version() -> str:
    return lib().exl3_version().decode()


GEMM_PATHS = {"rows": 0, "decode": 1, "fused": 2, "prefill": 3}


def exl3_set_gemm_path(path) -> None:
    """Pin the GEMM path of every linear call ("rows" restores the choice by M);
    a test and measurement hook.  Size workspaces after pinning."""
    _check(lib().exl3_set_gemm_path(GEMM_PATHS.get(path, path)), "exl3_set_gemm_path")


# ---------------------------------------------------------------- workspace
def exl3_linear_workspace_bytes(max_M: int, max_IC: int, max_OC: int) -> int:
    return int(lib().exl3_linear_workspace_bytes(max_M, max_IC, max_OC))


def exl3_moe_workspace_bytes(T: int, H: int, I: int, E: int, topk: int) -> int:
    return int(lib().exl3_moe_workspace_bytes(T, H, I, E, topk))


def exl3_workspace_init(ws: torch.Tensor) -> None:
    _check(lib().exl3_workspace_init(_ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(ws.device)),
           "exl3_workspace_init")


def exl3_workspace_error(ws: torch.Tensor) -> int:
    flag = ctypes.c_int32(0)
    _check(lib().exl3_workspace_error(_ptr(ws, torch.uint8, "ws"), ws.numel(), ctypes.byref(flag),
                                      _stream(ws.device)), "exl3_workspace_error")
    return int(flag.value)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Allocate (through torch) and prepare a workspace of at least nbytes."""
    if nbytes <= 0:
        raise ValueError("workspace size must be positive (did the size query reject the shape?)")
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + nbytes]
    exl3_workspace_init(ws)
    return ws


# ---------------------------------------------------------------- linear
def _linear_shapes(x, code, K):
    if code.dim() != 3 or code.shape[2] != 16 * K:
        raise ValueError(f"code must be [IC/16, OC/16, 16*K] with K={K}, got {tuple(code.shape)}")
    IC, OC = code.shape[0] * 16, code.shape[1] * 16
    if x.shape[-1] != IC:
        raise ValueError(f"x has {x.shape[-1]} channels, code expects IC={IC}")
    return IC, OC


def exl3_linear_into(x: torch.Tensor, code: torch.Tensor, K: int, s_in, rin, rout, s_out,
                     out: torch.Tensor, col0: int, ws: torch.Tensor) -> None:
    """Write one EXL3 projection into out[:, col0:col0+OC] (bf16 [M, ldo])."""
    IC, OC = _linear_shapes(x, code, K)
    M = x.numel() // IC
    ldo = out.shape[-1]
    _check(lib().exl3_linear_into(
        _ptr(x, torch.bfloat16, "x"), M, IC, _ptr(code, torch.int16, "code"), OC, K,
        _ptr(s_in, torch.float16, "s_in"), _ptr(rin, torch.float16, "rin"),
        _ptr(rout, torch.float16, "rout"), _ptr(s_out, torch.float16, "s_out"),
        _ptr(out, torch.bfloat16, "out"), ldo, col0, _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _stream(x.device)), "exl3_linear_into")


def exl3_linear_into_noalloc(x: torch.Tensor, code: torch.Tensor, K: int, s_in, rin, rout, s_out,
                             out: torch.Tensor, col0: int) -> None:
    """exl3_linear_into with no workspace: scratch is the library's fixed device array
    (M <= 8, IC <= 32768, OC <= 65536).  For callers that cannot allocate device memory;
    calls that overlap on the GPU race on that array."""
    IC, OC = _linear_shapes(x, code, K)
    M = x.numel() // IC
    _check(lib().exl3_linear_into_noalloc(
        _ptr(x, torch.bfloat16, "x"), M, IC, _ptr(code, torch.int16, "code"), OC, K,
        _ptr(s_in, torch.float16, "s_in"), _ptr(rin, torch.float16, "rin"),
        _ptr(rout, torch.float16, "rout"), _ptr(s_out, torch.float16, "s_out"),
        _ptr(out, torch.bfloat16, "out"), out.shape[-1], col0, _stream(x.device)),
        "exl3_linear_into_noalloc")


def _shard_array(shards, IC):
    arr = (Shard * len(shards))()
    col = 0
    for i, sh in enumerate(shards):
        code, K, s_in, rin, rout, s_out = sh[:6]
        col0 = sh[6] if len(sh) > 6 and sh[6] is not None else col
        codebook = CODEBOOKS[sh[7]] if len(sh) > 7 else 0
        if code.dim() != 3 or code.shape[2] != 16 * K or code.shape[0] * 16 != IC:
            raise ValueError(f"shard {i}: code {tuple(code.shape)} does not match K={K}, IC={IC}")
        OC = code.shape[1] * 16
        arr[i] = Shard(_ptr(code, torch.int16, "code"), _ptr(s_in, torch.float16, "s_in"),
                       _ptr(rin, torch.float16, "rin"), _ptr(rout, torch.float16, "rout"),
                       _ptr(s_out, torch.float16, "s_out"), OC, K, col0, codebook, 0)
        col = col0 + OC
    return arr


def exl3_linear_shards_workspace_bytes(max_M: int, IC: int, shards) -> int:
    """shards: sequence of (code, K, s_in, rin, rout, s_out[, col0[, codebook]]); codebook "3inst" (default), "mcg" or "mul1"."""
    arr = _shard_array(shards, IC)
    return int(lib().exl3_linear_shards_workspace_bytes(max_M, IC, arr, len(shards)))


def exl3_linear_into_shards(x: torch.Tensor, shards, out: torch.Tensor, ws: torch.Tensor) -> None:
    """A merged layer in one call: shard i = (code, K, s_in, rin, rout, s_out[, col0]) writes
    out[:, col0:col0+OC_i]; col0 defaults to the running sum of the previous shards' OC."""
    IC = x.shape[-1]
    M = x.numel() // IC
    arr = _shard_array(shards, IC)
    _check(lib().exl3_linear_into_shards(_ptr(x, torch.bfloat16, "x"), M, IC, arr, len(shards),
                                         _ptr(out, torch.bfloat16, "out"), out.shape[-1],
                                         _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(x.device)),
           "exl3_linear_into_shards")


def exl3_linear_into_shards_host(x: torch.Tensor, shards, out: torch.Tensor, ws: torch.Tensor) -> None:
    """exl3_linear_into_shards with x and out in pinned host memory: the kernels read x
    and write out through their device mappings (see include/exl3.h)."""
    for t, name in ((x, "x"), (out, "out")):
        if t.is_cuda or not t.is_pinned():
            raise ValueError(f"{name} must be a pinned host tensor")
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor")
    IC = x.shape[-1]
    M = x.numel() // IC
    arr = _shard_array(shards, IC)
    _check(lib().exl3_linear_into_shards_host(x.data_ptr(), M, IC, arr, len(shards), out.data_ptr(), out.shape[-1],
                                              _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(ws.device)),
           "exl3_linear_into_shards_host")


def _projection_array(projs):
    """projs: sequence of (x [M][IC] bf16, shards, out [M][ldo] bf16); keeps the shard arrays alive."""
    arr = (Projection * len(projs))()
    keep = []
    for i, (x, shards, out) in enumerate(projs):
        IC = x.shape[-1]
        sa = _shard_array(shards, IC)
        keep.append(sa)
        arr[i] = Projection(_ptr(x, torch.bfloat16, "x"), IC, len(shards), sa, _ptr(out, torch.bfloat16, "out"),
                            out.shape[-1])
    return arr, keep


def exl3_projections_workspace_bytes(max_M: int, projs) -> int:
    arr, keep = _projection_array(projs)
    return int(lib().exl3_projections_workspace_bytes(max_M, arr, len(projs)))


def exl3_linear_projections(projs, ws: torch.Tensor) -> None:
    """Several projections of one layer in one call (see include/exl3.h): projs is a
    sequence of (x, shards, out); inputs read by several projections are transformed once."""
    arr, keep = _projection_array(projs)
    M = projs[0][0].shape[0]
    _check(lib().exl3_linear_projections(arr, len(projs), M, _ptr(ws, torch.uint8, "ws"), ws.numel(),
                                         _stream(projs[0][0].device)), "exl3_linear_projections")


def exl3_gemm_into_shards(u: torch.Tensor, shards, out: torch.Tensor, ws: torch.Tensor) -> None:
    """Grouped trellis GEMM + output transform of per-shard pre-transformed u [n][M][IC]."""
    IC = u.shape[-1]
    M = u.shape[-2]
    arr = _shard_array(shards, IC)
    _check(lib().exl3_gemm_into_shards(_ptr(u, torch.float16, "u"), M, IC, arr, len(shards),
                                       _ptr(out, torch.bfloat16, "out"), out.shape[-1],
                                       _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(u.device)),
           "exl3_gemm_into_shards")


def exl3_linear(x, code, K, s_in, rin, rout, s_out, ws, out=None) -> torch.Tensor:
    IC, OC = _linear_shapes(x, code, K)
    M = x.numel() // IC
    if out is None:
        out = torch.empty((M, OC), dtype=torch.bfloat16, device=x.device)
    _check(lib().exl3_linear(
        _ptr(x, torch.bfloat16, "x"), M, IC, _ptr(code, torch.int16, "code"), OC, K,
        _ptr(s_in, torch.float16, "s_in"), _ptr(rin, torch.float16, "rin"),
        _ptr(rout, torch.float16, "rout"), _ptr(s_out, torch.float16, "s_out"),
        _ptr(out, torch.bfloat16, "out"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _stream(x.device)), "exl3_linear")
    return out


def exl3_gemm_into(u: torch.Tensor, code: torch.Tensor, K: int, rout, s_out, out: torch.Tensor,
                   col0: int, ws: torch.Tensor) -> None:
    """Trellis GEMM + output transform of pre-transformed fp16 activations u into a slice."""
    IC, OC = _linear_shapes(u, code, K)
    M = u.numel() // IC
    _check(lib().exl3_gemm_into(
        _ptr(u, torch.float16, "u"), M, IC, _ptr(code, torch.int16, "code"), OC, K,
        _ptr(rout, torch.float16, "rout"), _ptr(s_out, torch.float16, "s_out"),
        _ptr(out, torch.bfloat16, "out"), out.shape[-1], col0, _ptr(ws, torch.uint8, "ws"),
        ws.numel(), _stream(u.device)), "exl3_gemm_into")


def exl3_pretransform(x, s_in, rin, u=None) -> torch.Tensor:
    IC = x.shape[-1]
    M = x.numel() // IC
    if u is None:
        u = torch.empty((M, IC), dtype=torch.float16, device=x.device)
    _check(lib().exl3_pretransform(_ptr(x, torch.bfloat16, "x"), M, IC,
                                   _ptr(s_in, torch.float16, "s_in"), _ptr(rin, torch.float16, "rin"),
                                   _ptr(u, torch.float16, "u"), _stream(x.device)),
           "exl3_pretransform")
    return u


# ------------------------------------------------------ 8-bit activations
def exl3_linear_a8_workspace_bytes(max_M: int, max_IC: int, max_OC: int) -> int:
    return int(lib().exl3_linear_a8_workspace_bytes(max_M, max_IC, max_OC))


def exl3_quantize_a8(x, s_in, rin, A=None, As=None):
    """Pre-transform and quantize x per row: (A uint8 [M, IC] codes q + 128, As fp32 [M])."""
    IC = x.shape[-1]
    M = x.numel() // IC
    if A is None:
        A = torch.empty((M, IC), dtype=torch.uint8, device=x.device)
    if As is None:
        As = torch.empty((M,), dtype=torch.float32, device=x.device)
    _check(lib().exl3_quantize_a8(_ptr(x, torch.bfloat16, "x"), M, IC, _ptr(s_in, torch.float16, "s_in"),
                                  _ptr(rin, torch.float16, "rin"), _ptr(A, torch.uint8, "A"),
                                  _ptr(As, torch.float32, "As"), _stream(x.device)), "exl3_quantize_a8")
    return A, As


def exl3_linear_into_a8(x: torch.Tensor, code: torch.Tensor, K: int, s_in, rin, rout, s_out,
                        out: torch.Tensor, col0: int, ws: torch.Tensor) -> None:
    """exl3_linear_into with the activations quantized to 8 bits per row."""
    IC, OC = _linear_shapes(x, code, K)
    M = x.numel() // IC
    _check(lib().exl3_linear_into_a8(
        _ptr(x, torch.bfloat16, "x"), M, IC, _ptr(code, torch.int16, "code"), OC, K,
        _ptr(s_in, torch.float16, "s_in"), _ptr(rin, torch.float16, "rin"),
        _ptr(rout, torch.float16, "rout"), _ptr(s_out, torch.float16, "s_out"),
        _ptr(out, torch.bfloat16, "out"), out.shape[-1], col0, _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _stream(x.device)), "exl3_linear_into_a8")


def exl3_gemm_a8_into(A: torch.Tensor, As: torch.Tensor, code: torch.Tensor, K: int, rout, s_out,
                      out: torch.Tensor, col0: int, ws: torch.Tensor) -> None:
    """Trellis GEMM + output transform of 8-bit activations (A, As from exl3_quantize_a8)."""
    IC, OC = _linear_shapes(A, code, K)
    M = A.numel() // IC
    if As.numel() != M:
        raise ValueError(f"As has {As.numel()} entries, A has {M} rows")
    _check(lib().exl3_gemm_a8_into(
        _ptr(A, torch.uint8, "A"), _ptr(As, torch.float32, "As"), M, IC, _ptr(code, torch.int16, "code"), OC, K,
        _ptr(rout, torch.float16, "rout"), _ptr(s_out, torch.float16, "s_out"),
        _ptr(out, torch.bfloat16, "out"), out.shape[-1], col0, _ptr(ws, torch.uint8, "ws"),
        ws.numel(), _stream(A.device)), "exl3_gemm_a8_into")


def exl3_linear_shards_a8_workspace_bytes(max_M: int, IC: int, shards) -> int:
    return int(lib().exl3_linear_shards_a8_workspace_bytes(max_M, IC, _shard_array(shards, IC), len(shards)))


def exl3_linear_into_shards_a8(x: torch.Tensor, shards, out: torch.Tensor, ws: torch.Tensor) -> None:
    """exl3_linear_into_shards with 8-bit activations (each shard quantized with its own s_in, rin)."""
    IC = x.shape[-1]
    M = x.numel() // IC
    arr, n = _shard_array(shards, IC), len(shards)
    _check(lib().exl3_linear_into_shards_a8(_ptr(x, torch.bfloat16, "x"), M, IC, arr, n,
                                            _ptr(out, torch.bfloat16, "out"), out.shape[-1],
                                            _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(x.device)),
           "exl3_linear_into_shards_a8")


def exl3_gemm_a8_into_shards(A: torch.Tensor, As: torch.Tensor, shards, out: torch.Tensor, ws: torch.Tensor) -> None:
    """Grouped GEMM on 8-bit activations A uint8 [n, M, IC], As fp32 [n, M]."""
    IC = A.shape[-1]
    arr, n = _shard_array(shards, IC), len(shards)
    M = A.numel() // (IC * n)
    if As.numel() != n * M:
        raise ValueError(f"As has {As.numel()} entries, A has {n} x {M} rows")
    _check(lib().exl3_gemm_a8_into_shards(_ptr(A, torch.uint8, "A"), _ptr(As, torch.float32, "As"), M, IC, arr, n,
                                          _ptr(out, torch.bfloat16, "out"), out.shape[-1],
                                          _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(A.device)),
           "exl3_gemm_a8_into_shards")


def exl3_reconstruct(code: torch.Tensor, K: int, W=None) -> torch.Tensor:
    IC, OC = code.shape[0] * 16, code.shape[1] * 16
    if W is None:
        W = torch.empty((IC, OC), dtype=torch.float16, device=code.device)
    _check(lib().exl3_reconstruct(_ptr(code, torch.int16, "code"), IC, OC, K,
                                  _ptr(W, torch.float16, "W"), _stream(code.device)),
           "exl3_reconstruct")
    return W


def exl3_codebook_table(out=None, device="cuda") -> torch.Tensor:
    if out is None:
        out = torch.empty(65536, dtype=torch.float16, device=device)
    _check(lib().exl3_codebook_table(_ptr(out, torch.float16, "table"), _stream(out.device)),
           "exl3_codebook_table")
    return out


# ---------------------------------------------------------------- MoE
def exl3_moe_topk_softmax(logits: torch.Tensor, topk: int, ids=None, w=None):
    T, E = logits.shape
    if ids is None:
        ids = torch.empty((T, topk), dtype=torch.int32, device=logits.device)
    if w is None:
        w = torch.empty((T, topk), dtype=torch.float32, device=logits.device)
    _check(lib().exl3_moe_topk_softmax(_ptr(logits, torch.float32, "logits"), T, E, topk,
                                       _ptr(ids, torch.int32, "ids"), _ptr(w, torch.float32, "w"),
                                       _stream(logits.device)), "exl3_moe_topk_softmax")
    return ids, w


_BANK_DTYPES = dict(w13=torch.int16, w2=torch.int16, off_w1=torch.int64, off_w3=torch.int64,
                    off_w2=torch.int64, perm=torch.int32, k_gu=torch.int32, k_d=torch.int32,
                    w13_suh=torch.float16, w13_svh=torch.float16, w2_suh=torch.float16,
                    w2_svh=torch.float16)


def moe_bank_struct(bank: dict) -> MoeBank:
    """C view of a dict of device tensors laid out as in include/exl3.h."""
    return MoeBank(**{k: _ptr(bank[k], dt, k) for k, dt in _BANK_DTYPES.items()})


def exl3_moe_grouped(x, ids, w, bank: dict, ws, y=None) -> torch.Tensor:
    T, H = x.shape
    topk = ids.shape[1]
    E = bank["perm"].shape[0]
    I = bank["w2_suh"].shape[1]
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    b = moe_bank_struct(bank)
    _check(lib().exl3_moe_grouped(_ptr(x, torch.bfloat16, "x"), T, H, I, E, topk,
                                  _ptr(ids, torch.int32, "ids"), _ptr(w, torch.float32, "w"),
                                  ctypes.byref(b), _ptr(y, torch.bfloat16, "y"),
                                  _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(x.device)),
           "exl3_moe_grouped")
    return y


def exl3_moe_forward(x, logits, topk: int, bank: dict, ws, y=None, ids=None, w=None):
    """The MoE layer from router logits [T, E]: returns (y, ids, w), the routing the layer used."""
    T, H = x.shape
    E = bank["perm"].shape[0]
    I = bank["w2_suh"].shape[1]
    if logits.shape != (T, E):
        raise ValueError(f"logits must be [{T}, {E}], got {tuple(logits.shape)}")
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    if ids is None:
        ids = torch.empty((T, topk), dtype=torch.int32, device=x.device)
    if w is None:
        w = torch.empty((T, topk), dtype=torch.float32, device=x.device)
    b = moe_bank_struct(bank)
    _check(lib().exl3_moe_forward(_ptr(x, torch.bfloat16, "x"), _ptr(logits, torch.float32, "logits"), T, H, I, E,
                                  topk, ctypes.byref(b), _ptr(ids, torch.int32, "ids"), _ptr(w, torch.float32, "w"),
                                  _ptr(y, torch.bfloat16, "y"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
                                  _stream(x.device)), "exl3_moe_forward")
    return y, ids, w


# ---------------------------------------------------------------- embedding
def exl3_embed_int8_gather(q: torch.Tensor, scale: torch.Tensor, ids: torch.Tensor, out=None,
                           n_bad=None) -> torch.Tensor:
    V, H = q.shape
    N = ids.numel()
    if out is None:
        out = torch.empty((N, H), dtype=torch.bfloat16, device=q.device)
    _check(lib().exl3_embed_int8_gather(_ptr(q, torch.int8, "q"), _ptr(scale, torch.float16, "scale"),
                                        V, H, _ptr(ids, torch.int32, "ids"), N,
                                        _ptr(out, torch.bfloat16, "out"),
                                        _ptr(n_bad, torch.int32, "n_bad"), _stream(q.device)),
           "exl3_embed_int8_gather")
    return out


# ---------------------------------------------------------------- output head
def exl3_lm_head_workspace_bytes(max_M: int, H: int, V: int) -> int:
    return int(lib().exl3_lm_head_workspace_bytes(max_M, H, V))


def exl3_lm_head_int8(x: torch.Tensor, q: torch.Tensor, scale: torch.Tensor, ws: torch.Tensor,
                      out=None) -> torch.Tensor:
    """out[m][v] = bf16(scale[v] * sum_h x[m][h] q[v][h]): the int8 table as the output projection."""
    M, H = x.shape
    V = q.shape[0]
    if q.shape[1] != H:
        raise ValueError(f"q is {tuple(q.shape)}, x has {H} channels")
    if out is None:
        out = torch.empty((M, V), dtype=torch.bfloat16, device=x.device)
    _check(lib().exl3_lm_head_int8(_ptr(x, torch.bfloat16, "x"), M, H, _ptr(q, torch.int8, "q"),
                                   _ptr(scale, torch.float16, "scale"), V, _ptr(out, torch.bfloat16, "out"),
                                   out.stride(0), _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(x.device)),
           "exl3_lm_head_int8")
    return out
