"""Plain CPU reference (oracle) of the ZipCCL BF16 exponent-coding path.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use it.  The product library never imports, links or calls
anything here, and this package imports nothing from the product.

The arithmetic lives in ``zipccl_oracle.c`` (single-threaded C, built with gcc
without fast-math or FP contraction).  This module only builds it and marshals
numpy arrays through ctypes.

Every function follows a passage of "ZipCCL: Efficient Lossless Data
Compression of Communication Collectives for Accelerating LLM Training": the
abstract (exponent coding of near-Gaussian BF16 tensors without online
statistics), the key-design paragraph of the shd-paper summary (frequent
exponents get short codes, from the Gaussian density), the Fig. 6 caption
(about 11 bits per value) and the Fig. 3 / Fig. 5 captions (ReduceScatter:
decompress and reduce).  Readings where the pages are silent are stated in
the C source beside the code that takes them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zipccl_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libzipccl_oracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_CORRUPT, ERR_VERSION = 0, 1, 2, 3, 4
TILE = 32768
SEGS = 64
ROW = 512
LANE_ELEMS = 8
NSYM = 16
ESC = 15
LMAX = 10


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build (plain -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    deps = [_SRC, os.path.join(_HERE, "zo_frozen_tables.h")]
    if force or not os.path.exists(_LIB_PATH) or any(
            os.path.exists(d) and os.path.getmtime(_LIB_PATH) < os.path.getmtime(d) for d in deps):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u64p = ctypes.POINTER(ctypes.c_uint64)
            L.zo_exponent_pmf.argtypes = [ctypes.c_double, ctypes.POINTER(ctypes.c_double)]
            L.zo_exponent_pmf.restype = None
            L.zo_entropy_bits.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.c_int]
            L.zo_entropy_bits.restype = ctypes.c_double
            L.zo_package_merge.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.c_int, ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_int)]
            L.zo_package_merge.restype = ctypes.c_int
            L.zo_phase_table.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
            L.zo_phase_table.restype = None
            L.zo_frozen_phase_table.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                                ctypes.POINTER(ctypes.c_int)]
            L.zo_frozen_phase_table.restype = None
            L.zo_select_q.argtypes = [ctypes.c_void_p, ctypes.c_uint64]
            L.zo_select_q.restype = ctypes.c_int
            L.zo_q_from_sigma.argtypes = [ctypes.c_double]
            L.zo_q_from_sigma.restype = ctypes.c_int
            L.zo_base_for_q.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
            L.zo_base_for_q.restype = ctypes.c_int
            L.zo_max_compressed_bytes.argtypes = [u64p, ctypes.c_uint32]
            L.zo_max_compressed_bytes.restype = ctypes.c_uint64
            L.zo_compress.argtypes = [ctypes.c_void_p, ctypes.c_uint64, u64p, ctypes.c_uint32,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint64, u64p]
            L.zo_compress.restype = ctypes.c_int
            L.zo_decompress.argtypes = [ctypes.c_void_p, u64p, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_uint64]
            L.zo_decompress.restype = ctypes.c_int
            L.zo_decompress_reduce.argtypes = [ctypes.POINTER(ctypes.c_void_p), u64p, ctypes.c_uint32,
                                               ctypes.c_uint64, ctypes.c_void_p]
            L.zo_decompress_reduce.restype = ctypes.c_int
            L.zo_float_to_bf16_rne.argtypes = [ctypes.c_float]
            L.zo_float_to_bf16_rne.restype = ctypes.c_uint16
            L.zo_format_version.argtypes = []
            L.zo_format_version.restype = ctypes.c_int
            L.zo_expected_exponent_bits.argtypes = [ctypes.c_double, ctypes.c_int]
            L.zo_expected_exponent_bits.restype = ctypes.c_double
            L.zo_predict_chunk_bytes.argtypes = [ctypes.c_uint64, ctypes.c_double, ctypes.POINTER(ctypes.c_double)]
            L.zo_predict_chunk_bytes.restype = ctypes.c_uint64
            _lib = L
    return _lib


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"oracle {what} failed with status {status}")
        self.status = status


def _u64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint64))


def _ptr_u64(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64))


# ---------------------------------------------------------------- coding theory
def exponent_pmf(sigma: float) -> np.ndarray:
    """Closed-form pmf of the biased BF16 exponent of X ~ N(0, sigma^2)."""
    p = np.zeros(256, dtype=np.float64)
    lib().zo_exponent_pmf(float(sigma), p.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return p


def entropy_bits(p) -> float:
    p = np.ascontiguousarray(np.asarray(p, dtype=np.float64))
    return float(lib().zo_entropy_bits(p.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), len(p)))


def package_merge(weights, limit: int) -> list[int]:
    w = np.ascontiguousarray(np.asarray(weights, dtype=np.float64))
    lens = (ctypes.c_int * len(w))()
    st = lib().zo_package_merge(w.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), len(w), int(limit), lens)
    if st != OK:
        raise OracleError(st, "package_merge")
    return list(lens)


def rebuilt_phase_table(r: int) -> tuple[int, list[int]]:
    """Phase r = q mod 16 rebuilt from the closed form: (window start - 127,
    code lengths of symbols 0..15), by the oracle's package-merge."""
    off = ctypes.c_int()
    lens = (ctypes.c_int * NSYM)()
    lib().zo_phase_table(int(r), ctypes.byref(off), lens)
    return off.value, list(lens)


def rebuilt_phase_tables() -> tuple[list[int], list[list[int]]]:
    offs, lens = [], []
    for r in range(16):
        o, l = rebuilt_phase_table(r)
        offs.append(o)
        lens.append(l)
    return offs, lens


def phase_table(r: int) -> tuple[int, list[int]]:
    """The frozen table of format v1 that the oracle's encoder uses for phase r."""
    off = ctypes.c_int()
    lens = (ctypes.c_int * NSYM)()
    lib().zo_frozen_phase_table(int(r), ctypes.byref(off), lens)
    return off.value, list(lens)


def phase_tables() -> tuple[list[int], list[list[int]]]:
    offs, lens = [], []
    for r in range(16):
        o, l = phase_table(r)
        offs.append(o)
        lens.append(l)
    return offs, lens


def select_q(x: np.ndarray) -> int:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    return int(lib().zo_select_q(x.ctypes.data, x.size))


def q_from_sigma(sigma: float) -> int:
    return int(lib().zo_q_from_sigma(float(sigma)))


def base_for_q(q: int) -> int:
    offs, _ = phase_tables()
    arr = (ctypes.c_int * 16)(*offs)
    return int(lib().zo_base_for_q(int(q), arr))


def expected_exponent_bits(sigma: float, q: int) -> float:
    """Expected code bits of one exponent of N(0, sigma^2) under the code for scale q."""
    return float(lib().zo_expected_exponent_bits(float(sigma), int(q)))


def predict_chunk_bytes(n: int, sigma: float) -> tuple[int, float]:
    """Predicted stream bytes of one chunk of n values from N(0, sigma^2) (sigma hint), and bits per value."""
    bits = ctypes.c_double()
    return int(lib().zo_predict_chunk_bytes(int(n), float(sigma), ctypes.byref(bits))), float(bits.value)


def float_to_bf16_rne(f: float) -> int:
    return int(lib().zo_float_to_bf16_rne(ctypes.c_float(f)))


def format_version() -> int:
    return int(lib().zo_format_version())


# ---------------------------------------------------------------- the path
def max_compressed_bytes(chunk_elems) -> int:
    ce = _u64(chunk_elems)
    return int(lib().zo_max_compressed_bytes(_ptr_u64(ce), len(ce)))


def compress(x: np.ndarray, chunk_elems=None, sigma_hint=None) -> tuple[bytes, np.ndarray]:
    """BF16 words (uint16) -> (stream bytes, chunk offsets[n_chunks + 1])."""
    x = np.ascontiguousarray(x, dtype=np.uint16).reshape(-1)
    if chunk_elems is None:
        chunk_elems = [x.size]
    ce = _u64(chunk_elems)
    cap = max_compressed_bytes(ce)
    out = np.zeros(max(cap, 16), dtype=np.uint8)
    offs = np.zeros(len(ce) + 1, dtype=np.uint64)
    hint_ptr = None
    if sigma_hint is not None:
        hint = np.ascontiguousarray(np.asarray(sigma_hint, dtype=np.float32))
        assert hint.size == ce.size
        hint_ptr = hint.ctypes.data
    st = lib().zo_compress(x.ctypes.data if x.size else None, x.size, _ptr_u64(ce), len(ce), hint_ptr,
                           out.ctypes.data, out.size, _ptr_u64(offs))
    if st != OK:
        raise OracleError(st, "compress")
    return out[: int(offs[-1])].tobytes(), offs


def decompress(stream: bytes, offsets, n: int) -> np.ndarray:
    buf = np.frombuffer(stream, dtype=np.uint8)
    if buf.size == 0:
        buf = np.zeros(16, dtype=np.uint8)
    buf = np.ascontiguousarray(buf)
    offs = _u64(offsets)
    out = np.zeros(max(int(n), 1), dtype=np.uint16)
    st = lib().zo_decompress(buf.ctypes.data, _ptr_u64(offs), len(offs) - 1, out.ctypes.data, int(n))
    if st != OK:
        raise OracleError(st, "decompress")
    return out[: int(n)]


def decompress_reduce(chunks: list[bytes], n: int) -> np.ndarray:
    bufs = [np.ascontiguousarray(np.frombuffer(c, dtype=np.uint8)) for c in chunks]
    ptrs = (ctypes.c_void_p * len(bufs))(*[b.ctypes.data for b in bufs])
    sizes = _u64([b.size for b in bufs])
    out = np.zeros(max(int(n), 1), dtype=np.uint16)
    st = lib().zo_decompress_reduce(ptrs, _ptr_u64(sizes), len(bufs), int(n), out.ctypes.data)
    if st != OK:
        raise OracleError(st, "decompress_reduce")
    return out[: int(n)]
