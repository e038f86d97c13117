"""CPU oracle for the EXL3 trellis linear, MoE, int8 gather and int8 output head.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg call this module; the product package never
imports it.  The arithmetic lives in ``exl3_oracle.c`` (plain C, fp64, built
with gcc); this file only marshals numpy arrays.  It shares no code with the
CUDA path.

Parity of the trellis bit layout and codebook (readings documented in
``exl3_oracle.c``) against real exllamav3 checkpoints: unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "exl3_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile exl3_oracle.c into liboracle.so (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(t):
    return ctypes.POINTER(t)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u16, i16, i32, i64, f64, f32, i8 = (ctypes.c_uint16, ctypes.c_int16, ctypes.c_int32,
                                                ctypes.c_int64, ctypes.c_double, ctypes.c_float,
                                                ctypes.c_int8)
            L.exl3o_f16_to_f64.argtypes = [u16]
            L.exl3o_f16_to_f64.restype = f64
            L.exl3o_bf16_to_f64.argtypes = [u16]
            L.exl3o_bf16_to_f64.restype = f64
            L.exl3o_f16_from_f64.argtypes = [f64]
            L.exl3o_f16_from_f64.restype = u16
            L.exl3o_bf16_from_f64.argtypes = [f64]
            L.exl3o_bf16_from_f64.restype = u16
            L.exl3o_codebook.argtypes = [ctypes.c_uint32]
            L.exl3o_codebook.restype = u16
            L.exl3o_state.argtypes = [_P(i16), ctypes.c_int, ctypes.c_int]
            L.exl3o_state.restype = ctypes.c_uint32
            L.exl3o_decode_tile.argtypes = [_P(i16), ctypes.c_int, _P(u16)]
            L.exl3o_reconstruct_cols.argtypes = [_P(i16)] + [ctypes.c_int] * 5 + [_P(u16)]
            L.exl3o_reconstruct_cols.restype = ctypes.c_int
            L.exl3o_hadamard128.argtypes = [_P(f64)]
            L.exl3o_pretransform_f64.argtypes = [_P(u16), ctypes.c_long, ctypes.c_int, _P(u16),
                                                 _P(u16), _P(f64)]
            L.exl3o_pretransform_f64.restype = ctypes.c_int
            L.exl3o_linear_f64.argtypes = [_P(u16), ctypes.c_long, ctypes.c_int, _P(i16),
                                           ctypes.c_int, ctypes.c_int, _P(u16), _P(u16), _P(u16),
                                           _P(u16), ctypes.c_int, ctypes.c_int, _P(f64)]
            L.exl3o_linear_f64.restype = ctypes.c_int
            L.exl3o_linear_into.argtypes = [_P(u16), ctypes.c_long, ctypes.c_int, _P(i16),
                                            ctypes.c_int, ctypes.c_int, _P(u16), _P(u16),
                                            _P(u16), _P(u16), _P(u16), ctypes.c_long,
                                            ctypes.c_long]
            L.exl3o_linear_into.restype = ctypes.c_int
            L.exl3o_linear_a8_f64.argtypes = [_P(u16), ctypes.c_long, ctypes.c_int, _P(i16), ctypes.c_int,
                                              ctypes.c_int, _P(u16), _P(u16), _P(u16), _P(u16), ctypes.c_int,
                                              ctypes.c_int, _P(f64), _P(ctypes.c_uint8), _P(f64)]
            L.exl3o_linear_a8_f64.restype = ctypes.c_int
            L.exl3o_lm_head_f64.argtypes = [_P(u16), ctypes.c_long, ctypes.c_int, _P(i8), _P(u16), ctypes.c_long,
                                            ctypes.c_long, ctypes.c_long, _P(f64)]
            L.exl3o_lm_head_f64.restype = ctypes.c_int
            L.exl3o_topk_softmax.argtypes = [_P(f32), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             _P(i32), _P(f32)]
            L.exl3o_topk_softmax.restype = ctypes.c_int
            L.exl3o_moe.argtypes = ([_P(u16)] + [ctypes.c_int] * 5 + [_P(i32), _P(f32), _P(i16),
                                    _P(i16), _P(i64), _P(i64), _P(i64), _P(i32), _P(i32),
                                    _P(i32), _P(u16), _P(u16), _P(u16), _P(u16), _P(f64)])
            L.exl3o_moe.restype = ctypes.c_int
            L.exl3o_gather.argtypes = [_P(i8), _P(u16), ctypes.c_long, ctypes.c_int, _P(i32),
                                       ctypes.c_long, _P(u16), _P(ctypes.c_long)]
            L.exl3o_gather.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype in (np.float16,):
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (status {rc})")


# ----------------------------------------------------------------- conversions
def f16_to_f64(bits: int) -> float:
    return lib().exl3o_f16_to_f64(int(bits))


def bf16_to_f64(bits: int) -> float:
    return lib().exl3o_bf16_to_f64(int(bits))


def f16_from_f64(v: float) -> int:
    return int(lib().exl3o_f16_from_f64(float(v)))


def bf16_from_f64(v: float) -> int:
    return int(lib().exl3o_bf16_from_f64(float(v)))


def bf16_bits_from_f64_array(y: np.ndarray) -> np.ndarray:
    """Round an fp64 array once to bf16 (nearest even); returns uint16 bits."""
    f = lib().exl3o_bf16_from_f64
    flat = np.ascontiguousarray(y, dtype=np.float64).ravel()
    return np.fromiter((f(float(v)) for v in flat), dtype=np.uint16,
                       count=flat.size).reshape(y.shape)


# ---------------------------------------------------------------- trellis
def codebook(state: int) -> int:
    """fp16 bits of the weight a 16-bit trellis state decodes to."""
    return int(lib().exl3o_codebook(int(state) & 0xFFFF))


def codebook_table() -> np.ndarray:
    """All 65,536 codebook entries as fp16 bits, indexed by state."""
    f = lib().exl3o_codebook
    return np.fromiter((f(s) for s in range(65536)), dtype=np.uint16, count=65536)


def state(tile: np.ndarray, K: int, t: int) -> int:
    tile = np.ascontiguousarray(tile, dtype=np.int16)
    assert tile.size == 16 * K
    return int(lib().exl3o_state(_ptr(tile, ctypes.c_int16), K, t))


def decode_tile(tile: np.ndarray, K: int) -> np.ndarray:
    """256 fp16 weight bits of one tile in trellis order t = 16r + c."""
    tile = np.ascontiguousarray(tile, dtype=np.int16)
    assert tile.size == 16 * K
    out = np.empty(256, np.uint16)
    lib().exl3o_decode_tile(_ptr(tile, ctypes.c_int16), K, _ptr(out, ctypes.c_uint16))
    return out


def reconstruct(code: np.ndarray, K: int, oc0: int = 0, noc: int | None = None) -> np.ndarray:
    """Dense fp16 weight bits W[IC][noc] of a code tensor [IC/16][OC/16][16K]."""
    code = np.ascontiguousarray(code, dtype=np.int16)
    IC, OC = code.shape[0] * 16, code.shape[1] * 16
    assert code.shape[2] == 16 * K, "K is implied by the code tensor's last dim / 16"
    noc = OC - oc0 if noc is None else noc
    W = np.empty((IC, noc), np.uint16)
    _check(lib().exl3o_reconstruct_cols(_ptr(code, ctypes.c_int16), IC, OC, K, oc0, noc,
                                        _ptr(W, ctypes.c_uint16)), "reconstruct")
    return W


def hadamard128() -> np.ndarray:
    H = np.empty((128, 128), np.float64)
    lib().exl3o_hadamard128(_ptr(H, ctypes.c_double))
    return H


# ---------------------------------------------------------------- linear
def pretransform_f64(x, s_in, rin) -> np.ndarray:
    """fp64 u[M][IC] = Had128((x * s_in) * rin) blockwise."""
    x = _u16(x)
    M, IC = x.shape
    u = np.empty((M, IC), np.float64)
    _check(lib().exl3o_pretransform_f64(_ptr(x, ctypes.c_uint16), M, IC,
                                        _ptr(_u16(s_in), ctypes.c_uint16),
                                        _ptr(_u16(rin), ctypes.c_uint16),
                                        _ptr(u, ctypes.c_double)), "pretransform")
    return u


def linear_f64(x, code, K, s_in, rin, rout, s_out, blk0=0, nblk=None) -> np.ndarray:
    """fp64 y[M][nblk*128] of output blocks [blk0, blk0+nblk) (unrounded)."""
    x = _u16(x)
    code = np.ascontiguousarray(code, dtype=np.int16)
    M, IC = x.shape
    OC = code.shape[1] * 16
    assert code.shape[0] * 16 == IC and code.shape[2] == 16 * K
    nblk = OC // 128 - blk0 if nblk is None else nblk
    y = np.empty((M, nblk * 128), np.float64)
    _check(lib().exl3o_linear_f64(_ptr(x, ctypes.c_uint16), M, IC, _ptr(code, ctypes.c_int16),
                                  OC, K, _ptr(_u16(s_in), ctypes.c_uint16),
                                  _ptr(_u16(rin), ctypes.c_uint16),
                                  _ptr(_u16(rout), ctypes.c_uint16),
                                  _ptr(_u16(s_out), ctypes.c_uint16), blk0, nblk,
                                  _ptr(y, ctypes.c_double)), "linear")
    return y


def linear_a8_f64(x, code, K, s_in, rin, rout, s_out, blk0=0, nblk=None):
    """The 8-bit activation variant (see exl3_oracle.c): fp64 y[M][nblk*128] (unrounded),
    the activation codes A uint8 [M][IC] (q + 128) and the row scales As [M]."""
    x = _u16(x)
    code = np.ascontiguousarray(code, dtype=np.int16)
    M, IC = x.shape
    OC = code.shape[1] * 16
    assert code.shape[0] * 16 == IC and code.shape[2] == 16 * K
    nblk = OC // 128 - blk0 if nblk is None else nblk
    y = np.empty((M, nblk * 128), np.float64)
    A = np.empty((M, IC), np.uint8)
    As = np.empty(M, np.float64)
    _check(lib().exl3o_linear_a8_f64(_ptr(x, ctypes.c_uint16), M, IC, _ptr(code, ctypes.c_int16), OC, K,
                                     _ptr(_u16(s_in), ctypes.c_uint16), _ptr(_u16(rin), ctypes.c_uint16),
                                     _ptr(_u16(rout), ctypes.c_uint16), _ptr(_u16(s_out), ctypes.c_uint16),
                                     blk0, nblk, _ptr(y, ctypes.c_double), _ptr(A, ctypes.c_uint8),
                                     _ptr(As, ctypes.c_double)), "linear_a8")
    return y, A, As


def linear_into(out: np.ndarray, x, code, K, s_in, rin, rout, s_out, col0: int) -> None:
    """Write bf16 bits of one shard into out[:, col0:col0+OC] (uint16 [M][ldo])."""
    x = _u16(x)
    assert out.dtype == np.uint16 and out.flags["C_CONTIGUOUS"]
    code = np.ascontiguousarray(code, dtype=np.int16)
    M, IC = x.shape
    OC = code.shape[1] * 16
    _check(lib().exl3o_linear_into(_ptr(x, ctypes.c_uint16), M, IC, _ptr(code, ctypes.c_int16),
                                   OC, K, _ptr(_u16(s_in), ctypes.c_uint16),
                                   _ptr(_u16(rin), ctypes.c_uint16),
                                   _ptr(_u16(rout), ctypes.c_uint16),
                                   _ptr(_u16(s_out), ctypes.c_uint16),
                                   _ptr(out, ctypes.c_uint16), out.shape[1], col0),
           "linear_into")


# ---------------------------------------------------------------- MoE
def topk_softmax(logits: np.ndarray, topk: int):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    ids = np.empty((T, topk), np.int32)
    w = np.empty((T, topk), np.float32)
    _check(lib().exl3o_topk_softmax(_ptr(logits, ctypes.c_float), T, E, topk,
                                    _ptr(ids, ctypes.c_int32), _ptr(w, ctypes.c_float)),
           "topk_softmax")
    return ids, w


def moe_f64(x, ids, w, bank: dict) -> np.ndarray:
    """fp64 y[T][H] of the grouped MoE over an expert bank (see exl3_oracle.c)."""
    x = _u16(x)
    T, H = x.shape
    ids = np.ascontiguousarray(ids, np.int32)
    w = np.ascontiguousarray(w, np.float32)
    topk = ids.shape[1]
    E = bank["perm"].shape[0]
    I = bank["w2_suh"].shape[1]
    y = np.empty((T, H), np.float64)
    a = {k: np.ascontiguousarray(v) for k, v in bank.items()}
    _check(lib().exl3o_moe(_ptr(x, ctypes.c_uint16), T, H, I, E, topk,
                           _ptr(ids, ctypes.c_int32), _ptr(w, ctypes.c_float),
                           _ptr(a["w13"], ctypes.c_int16), _ptr(a["w2"], ctypes.c_int16),
                           _ptr(a["off_w1"], ctypes.c_int64), _ptr(a["off_w3"], ctypes.c_int64),
                           _ptr(a["off_w2"], ctypes.c_int64), _ptr(a["perm"], ctypes.c_int32),
                           _ptr(a["k_gu"], ctypes.c_int32), _ptr(a["k_d"], ctypes.c_int32),
                           _ptr(_u16(a["w13_suh"]), ctypes.c_uint16),
                           _ptr(_u16(a["w13_svh"]), ctypes.c_uint16),
                           _ptr(_u16(a["w2_suh"]), ctypes.c_uint16),
                           _ptr(_u16(a["w2_svh"]), ctypes.c_uint16),
                           _ptr(y, ctypes.c_double)), "moe")
    return y


# ---------------------------------------------------------------- gather
def gather(q: np.ndarray, s, ids: np.ndarray):
    """bf16 bits out[N][H] = q[ids] * s[ids], and the number of out-of-range ids."""
    q = np.ascontiguousarray(q, np.int8)
    s = _u16(s)
    ids = np.ascontiguousarray(ids, np.int32)
    V, H = q.shape
    N = ids.shape[0]
    out = np.empty((N, H), np.uint16)
    bad = ctypes.c_long(0)
    _check(lib().exl3o_gather(_ptr(q, ctypes.c_int8), _ptr(s, ctypes.c_uint16), V, H,
                              _ptr(ids, ctypes.c_int32), N, _ptr(out, ctypes.c_uint16),
                              ctypes.byref(bad)), "gather")
    return out, int(bad.value)


# ---------------------------------------------------------------- int8 output head
def lm_head_f64(x, q: np.ndarray, s, v0: int = 0, nv: int | None = None) -> np.ndarray:
    """fp64 y[M][nv] = s[v] * sum_h x[m][h] * q[v][h] for vocabulary rows [v0, v0 + nv) (unrounded)."""
    x = _u16(x)
    q = np.ascontiguousarray(q, np.int8)
    s = _u16(s)
    M, H = x.shape
    V = q.shape[0]
    assert q.shape[1] == H
    nv = V - v0 if nv is None else nv
    y = np.empty((M, nv), np.float64)
    _check(lib().exl3o_lm_head_f64(_ptr(x, ctypes.c_uint16), M, H, _ptr(q, ctypes.c_int8),
                                   _ptr(s, ctypes.c_uint16), V, v0, nv, _ptr(y, ctypes.c_double)), "lm_head")
    return y
