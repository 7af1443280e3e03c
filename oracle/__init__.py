"""fp64 CPU oracle for the DCP LSE merge -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it, and this package imports nothing from
the product path.  The arithmetic lives in ``dcp_oracle.c`` (plain C, fp64);
this module compiles it with gcc on first use and wraps it with ctypes over
numpy arrays.

Every operand is a numpy array *view*; its strides (in bytes) are turned into
element strides for the C code, so strided and interleaved layouts are
described exactly as the pages describe them (a payload view plus an fp32
word view of the same buffer).  bf16 arrays are carried as ``uint16`` and
fp8 (e4m3) arrays as ``uint8``.

Pins: ``tests/test_oracle.py`` checks every function here against what the
pages and mathematics fix (identity at N=1, neutral empty ranks, shift
invariance, base-2/base-e agreement, closed forms, brute-force split
attention equal to unsplit attention, round-robin partition invariants,
numpy's own fp16/bf16 decoding and index maps); ``tests/test_oracle_mutants.py``
shows that 28 planted slips in ``dcp_oracle.c`` each make one of those pins fail.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dcp_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "f64": 3, "fp8": 4}
BASES = {"e": 0, "2": 1}
SANITIZE_O = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile dcp_oracle.c into a shared library with gcc (host compiler only)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # DCP_ORACLE_LIB points the oracle at another build of dcp_oracle.c:
        # the planted-mistake test (tests/test_oracle_mutants.py) runs the
        # pins against deliberately broken copies this way.
        lib = ctypes.CDLL(os.environ.get("DCP_ORACLE_LIB") or build())
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_pack.restype = i32
        lib.oracle_pack.argtypes = ([i32] * 6 + [vp, i64, i64, i64] + [vp, i64, i64, i64]
                                    + [vp, i64, i64, i64, i64] + [vp, i64, i64, i64, i64])
        lib.oracle_combine.restype = i32
        lib.oracle_combine.argtypes = ([i32] * 6 + [vp, i64, i64, i64, i64]
                                       + [vp, i64, i64, i64, i64] + [vp, vp, i32, ctypes.c_uint])
        lib.oracle_unpack_combine.restype = i32
        lib.oracle_unpack_combine.argtypes = ([i32] * 6 + [vp, i64, i64, i64, i64]
                                              + [vp, vp, i32, ctypes.c_uint])
        lib.oracle_dcp_lens.restype = i64
        lib.oracle_dcp_lens.argtypes = [i64, i32, i32]
        lib.oracle_split_attention.restype = None
        lib.oracle_split_attention.argtypes = [i32, i32, i32, ctypes.c_double, vp, vp, vp, i32,
                                               vp, vp]
        lib.oracle_split_attention_mla.restype = None
        lib.oracle_split_attention_mla.argtypes = [i32, i32, i32, i32, ctypes.c_double, vp, vp, i32,
                                                   vp, vp]
        lib.oracle_lse_pack_dim.restype = i32
        lib.oracle_lse_pack_dim.argtypes = [i32]
        lib.oracle_decode_elem.restype = ctypes.c_double
        lib.oracle_decode_elem.argtypes = [i32, vp, i64]
        _lib = lib
        return lib


def _estrides(a: np.ndarray) -> list[int]:
    out = []
    for s in a.strides:
        if s % a.itemsize:
            raise ValueError("stride is not a whole number of elements")
        out.append(s // a.itemsize)
    return out


def _ptr(a: np.ndarray) -> int:
    return a.__array_interface__["data"][0]


def _check_payload(a: np.ndarray, dtype: str) -> None:
    want = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "f64": np.float64,
            "fp8": np.uint8}[dtype]
    if a.dtype != want:
        raise TypeError(f"{dtype} payload must be a numpy {np.dtype(want)} array, got {a.dtype}")
    if a.shape and a.shape[-1] > 1 and a.strides[-1] != a.itemsize:
        raise ValueError("innermost (D) stride must be 1 element")


def lse_pack_dim(dtype: str) -> int:
    return _load().oracle_lse_pack_dim(DTYPES.get(dtype, 99))


def decode(dtype: str, a: np.ndarray) -> np.ndarray:
    """Decode a contiguous payload array into float64 with the oracle's own decoder."""
    a = np.ascontiguousarray(a)
    lib = _load()
    flat = a.reshape(-1)
    return np.array([lib.oracle_decode_elem(DTYPES[dtype], _ptr(flat), i)
                     for i in range(flat.size)], dtype=np.float64).reshape(a.shape)


def pack(dtype: str, N: int, o: np.ndarray, lse: np.ndarray,
         dst_o: np.ndarray, dst_lse: np.ndarray) -> None:
    """Scatter O [G,B,H,D] and LSE [G,B,H] into dst_o [G,N,B,H/N,D] and dst_lse [G,N,B,H/N].

    Writes through the views in place (they may share one buffer, as in the
    interleaved send layout)."""
    _check_payload(o, dtype)
    _check_payload(dst_o, dtype)
    if lse.dtype != np.float32 or dst_lse.dtype != np.float32:
        raise TypeError("LSE views must be float32")
    G, B, H, D = o.shape
    rc = _load().oracle_pack(DTYPES[dtype], N, B, H, D, G,
                             _ptr(o), *[_estrides(o)[i] for i in (0, 1, 2)],
                             _ptr(lse), *_estrides(lse),
                             _ptr(dst_o), *[_estrides(dst_o)[i] for i in (0, 1, 2, 3)],
                             _ptr(dst_lse), *_estrides(dst_lse))
    if rc != 0:
        raise ValueError(f"oracle_pack rejected its arguments (H={H} not a multiple of N={N}?)")


def combine(dtype: str, o: np.ndarray, lse: np.ndarray, base: str = "e",
            sanitize: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Merge O [G,N,B,Hc,D] with LSE [G,N,B,Hc]; returns (out [G,B,Hc,D], lse [G,B,Hc]) in fp64."""
    _check_payload(o, dtype)
    if lse.dtype != np.float32:
        raise TypeError("LSE view must be float32")
    G, N, B, Hc, D = o.shape
    out = np.empty((G, B, Hc, D), dtype=np.float64)
    out_lse = np.empty((G, B, Hc), dtype=np.float64)
    so = _estrides(o)
    rc = _load().oracle_combine(DTYPES[dtype], N, B, Hc, D, G,
                                _ptr(o), so[0], so[1], so[2], so[3],
                                _ptr(lse), *_estrides(lse),
                                _ptr(out), _ptr(out_lse), BASES[base],
                                SANITIZE_O if sanitize else 0)
    if rc != 0:
        raise ValueError("oracle_combine rejected its arguments")
    return out, out_lse


def unpack_combine(dtype: str, recv: np.ndarray, D: int, base: str = "e",
                   sanitize: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Merge an interleaved receive view [G,N,B,Hpr,D+lpd] (payload dtype)."""
    _check_payload(recv, dtype)
    G, N, B, Hpr, W = recv.shape
    if W != D + lse_pack_dim(dtype):
        raise ValueError("row width must be D + lpd")
    out = np.empty((G, B, Hpr, D), dtype=np.float64)
    out_lse = np.empty((G, B, Hpr), dtype=np.float64)
    sr = _estrides(recv)
    rc = _load().oracle_unpack_combine(DTYPES[dtype], N, B, Hpr, D, G,
                                       _ptr(recv), sr[0], sr[1], sr[2], sr[3],
                                       _ptr(out), _ptr(out_lse), BASES[base],
                                       SANITIZE_O if sanitize else 0)
    if rc != 0:
        raise ValueError("oracle_unpack_combine rejected its arguments")
    return out, out_lse


def dcp_lens(L: int, n: int, r: int) -> int:
    return int(_load().oracle_dcp_lens(L, n, r))


def split_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, n: int, scale: float,
                    base: str = "e") -> tuple[np.ndarray, np.ndarray]:
    """Per-rank (O [n,D], lse [n]) of single-query attention under round-robin KV ownership."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    L, D = K.shape
    O = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    _load().oracle_split_attention(L, D, n, float(scale), _ptr(q), _ptr(K), _ptr(V),
                                   BASES[base], _ptr(O), _ptr(lse))
    return O, lse


def split_attention_mla(q: np.ndarray, KV: np.ndarray, Dv: int, n: int, scale: float,
                        base: str = "e") -> tuple[np.ndarray, np.ndarray]:
    """Per-rank (O [n,Dv], lse [n]) of single-query attention over a latent
    cache KV [L, Dk] whose value is each row's first Dv elements (absorbed
    MLA), under round-robin KV ownership."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    KV = np.ascontiguousarray(KV, dtype=np.float64)
    L, Dk = KV.shape
    if q.shape != (Dk,) or not 0 < Dv <= Dk:
        raise ValueError("q must have Dk elements and 0 < Dv <= Dk")
    O = np.empty((n, Dv), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    _load().oracle_split_attention_mla(L, Dk, Dv, n, float(scale), _ptr(q), _ptr(KV),
                                       BASES[base], _ptr(O), _ptr(lse))
    return O, lse
