"""GB300 (sm_103a) ZipCCL BF16 exponent coding: Python binding of libzipccl.

"ZipCCL: Efficient Lossless Data Compression of Communication Collectives for
Accelerating LLM Training" (abstract; Fig. 3, 5, 6 captions): BF16 tensors are
compressed losslessly by entropy-coding their exponents with a code derived
from the Gaussian law; sign and mantissa stay raw; each destination rank's
chunk is a self-contained stream; the receive side of a reduce-scatter
decompresses k peer chunks and sums them.

This module only marshals arguments to the C ABI in ``include/zipccl.h``.
Every step of compression and decompression runs in the library's CUDA
kernels; there is no CPU path.  PyTorch provides device memory and streams.

Low-level names mirror the C ABI (``zipccl_compress`` ...) and take raw
pointers; ``compress`` / ``decompress`` / ``decompress_reduce`` are the same
calls on torch tensors.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = [
    "ZipcclError", "load", "library_path", "zipccl_format_version", "zipccl_status_string",
    "zipccl_max_compressed_bytes", "zipccl_compress_workspace_bytes", "zipccl_decompress_workspace_bytes",
    "zipccl_reduce_workspace_bytes", "zipccl_compress", "zipccl_compress_send", "zipccl_decompress",
    "zipccl_decompress_reduce",
    "zipccl_get_device_status", "zipccl_codebook_phase", "zipccl_codebook_rebuild_phase",
    "zipccl_decompress_reduce_noalloc",
    "zipccl_predict_chunk_bytes", "zipccl_choose_compressed", "zipccl_selftest_bounded_wait",
    "zipccl_profile_encode_events", "compress", "decompress", "decompress_reduce",
    "Compressed", "EXPORTED_SYMBOLS",
]

OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_CORRUPT, ERR_VERSION, ERR_TIMEOUT, ERR_CUDA = range(7)
EXPORTED_SYMBOLS = [
    "zipccl_format_version", "zipccl_status_string", "zipccl_max_compressed_bytes",
    "zipccl_compress_workspace_bytes", "zipccl_decompress_workspace_bytes", "zipccl_reduce_workspace_bytes",
    "zipccl_compress", "zipccl_compress_send", "zipccl_decompress", "zipccl_decompress_reduce",
    "zipccl_get_device_status", "zipccl_codebook_phase", "zipccl_codebook_rebuild_phase",
    "zipccl_decompress_reduce_noalloc",
    "zipccl_predict_chunk_bytes",
    "zipccl_choose_compressed", "zipccl_selftest_bounded_wait", "zipccl_profile_encode_events",
]

_lock = threading.Lock()
_lib = None


class ZipcclError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_status_name(status)} ({status})")
        self.status = status


def _status_name(st: int) -> str:
    try:
        return load().zipccl_status_string(int(st)).decode()
    except Exception:  # pragma: no cover - only when the library itself is unusable
        return "status"


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libzipccl.so (building it with nvcc when missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libzipccl is not built ({path}); run lossless_bf16_tensor_zipccl_gb300/build.py")
        L = ctypes.CDLL(path)
        u64, u32, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p
        u64p = ctypes.POINTER(ctypes.c_uint64)
        L.zipccl_format_version.restype = ctypes.c_int
        L.zipccl_format_version.argtypes = []
        L.zipccl_status_string.restype = ctypes.c_char_p
        L.zipccl_status_string.argtypes = [ctypes.c_int]
        for name in ("zipccl_max_compressed_bytes", "zipccl_compress_workspace_bytes"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [u64p, u32, u64p]
        L.zipccl_decompress_workspace_bytes.restype = ctypes.c_int
        L.zipccl_decompress_workspace_bytes.argtypes = [u64, u32, u64p]
        L.zipccl_reduce_workspace_bytes.restype = ctypes.c_int
        L.zipccl_reduce_workspace_bytes.argtypes = [u32, u64p]
        L.zipccl_compress.restype = ctypes.c_int
        L.zipccl_compress.argtypes = [vp, u64, u64p, u32, ctypes.POINTER(ctypes.c_float), vp, u64, vp, vp, u64, vp]
        L.zipccl_compress_send.restype = ctypes.c_int
        L.zipccl_compress_send.argtypes = [vp, u64, u64p, u32, ctypes.POINTER(ctypes.c_float), vp, u64, vp, vp, u64,
                                           vp, vp, u64, vp]
        L.zipccl_decompress.restype = ctypes.c_int
        L.zipccl_decompress.argtypes = [vp, vp, u32, vp, u64, vp, u64, vp]
        L.zipccl_decompress_reduce.restype = ctypes.c_int
        L.zipccl_decompress_reduce.argtypes = [ctypes.POINTER(vp), u64p, u32, u64, vp, vp, u64, vp]
        L.zipccl_get_device_status.restype = ctypes.c_int
        L.zipccl_get_device_status.argtypes = [vp, vp]
        L.zipccl_decompress_reduce_noalloc.restype = ctypes.c_int
        L.zipccl_decompress_reduce_noalloc.argtypes = [ctypes.POINTER(vp), u64p, u32, u64, vp,
                                                       ctypes.POINTER(vp), vp]
        for name in ("zipccl_codebook_phase", "zipccl_codebook_rebuild_phase"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_uint8)]
        dbl = ctypes.c_double
        L.zipccl_predict_chunk_bytes.restype = ctypes.c_int
        L.zipccl_predict_chunk_bytes.argtypes = [u64, ctypes.c_float, u64p, ctypes.POINTER(dbl)]
        L.zipccl_selftest_bounded_wait.restype = ctypes.c_int
        L.zipccl_selftest_bounded_wait.argtypes = [ctypes.c_int, vp, u64, vp]
        L.zipccl_profile_encode_events.restype = ctypes.c_int
        L.zipccl_profile_encode_events.argtypes = [vp, vp]
        L.zipccl_choose_compressed.restype = ctypes.c_int
        L.zipccl_choose_compressed.argtypes = [u64, ctypes.c_float, dbl, dbl, dbl, dbl, ctypes.POINTER(ctypes.c_int),
                                               ctypes.POINTER(dbl)]
        _lib = L
        return L


def _u64_array(vals):
    arr = (ctypes.c_uint64 * max(1, len(vals)))(*[int(v) for v in vals])
    return arr


def _check(st: int, what: str) -> None:
    if st != OK:
        raise ZipcclError(st, what)


# ------------------------------------------------------------------ C ABI mirrors
def zipccl_format_version() -> int:
    return int(load().zipccl_format_version())


def zipccl_status_string(status: int) -> str:
    return load().zipccl_status_string(int(status)).decode()


def zipccl_max_compressed_bytes(chunk_elems) -> int:
    out = ctypes.c_uint64()
    _check(load().zipccl_max_compressed_bytes(_u64_array(chunk_elems), len(chunk_elems), ctypes.byref(out)),
           "zipccl_max_compressed_bytes")
    return int(out.value)


def zipccl_compress_workspace_bytes(chunk_elems) -> int:
    out = ctypes.c_uint64()
    _check(load().zipccl_compress_workspace_bytes(_u64_array(chunk_elems), len(chunk_elems), ctypes.byref(out)),
           "zipccl_compress_workspace_bytes")
    return int(out.value)


def zipccl_decompress_workspace_bytes(n: int, n_chunks: int) -> int:
    out = ctypes.c_uint64()
    _check(load().zipccl_decompress_workspace_bytes(int(n), int(n_chunks), ctypes.byref(out)),
           "zipccl_decompress_workspace_bytes")
    return int(out.value)


def zipccl_reduce_workspace_bytes(k: int) -> int:
    out = ctypes.c_uint64()
    _check(load().zipccl_reduce_workspace_bytes(int(k), ctypes.byref(out)), "zipccl_reduce_workspace_bytes")
    return int(out.value)


def zipccl_compress(d_in: int, n: int, chunk_elems, sigma_hint, d_out: int, out_capacity: int,
                    d_chunk_offsets: int, d_ws: int, ws_bytes: int, stream: int) -> int:
    hint = None
    if sigma_hint is not None:
        hint = (ctypes.c_float * len(sigma_hint))(*[float(v) for v in sigma_hint])
    return int(load().zipccl_compress(d_in, n, _u64_array(chunk_elems), len(chunk_elems), hint, d_out,
                                      out_capacity, d_chunk_offsets, d_ws, ws_bytes, stream))


def zipccl_compress_send(d_in: int, n: int, chunk_elems, sigma_hint, d_out: int, out_capacity: int,
                         d_chunk_offsets: int, d_send: int, send_capacity: int, d_chunk_ready: int, d_ws: int,
                         ws_bytes: int, stream: int) -> int:
    hint = None
    if sigma_hint is not None:
        hint = (ctypes.c_float * len(sigma_hint))(*[float(v) for v in sigma_hint])
    return int(load().zipccl_compress_send(d_in, n, _u64_array(chunk_elems), len(chunk_elems), hint, d_out,
                                           out_capacity, d_chunk_offsets, d_send, send_capacity, d_chunk_ready,
                                           d_ws, ws_bytes, stream))


def zipccl_decompress(d_stream: int, d_chunk_offsets: int, n_chunks: int, d_out: int, n: int, d_ws: int,
                      ws_bytes: int, stream: int) -> int:
    return int(load().zipccl_decompress(d_stream, d_chunk_offsets, n_chunks, d_out, n, d_ws, ws_bytes, stream))


def _peer_arrays_match(d_peer_chunks, peer_chunk_bytes, k: int) -> bool:
    """The C call reads k entries of each host array: both must hold exactly k."""
    return int(k) == len(d_peer_chunks) == len(peer_chunk_bytes)


def zipccl_decompress_reduce(d_peer_chunks, peer_chunk_bytes, k: int, n: int, d_out: int, d_ws: int,
                             ws_bytes: int, stream: int) -> int:
    if not _peer_arrays_match(d_peer_chunks, peer_chunk_bytes, k):
        return ERR_INVALID_ARG
    ptrs = (ctypes.c_void_p * max(1, len(d_peer_chunks)))(*[int(p) for p in d_peer_chunks])
    return int(load().zipccl_decompress_reduce(ptrs, _u64_array(peer_chunk_bytes), k, n, d_out, d_ws, ws_bytes,
                                               stream))


def zipccl_get_device_status(d_ws: int, stream: int) -> int:
    return int(load().zipccl_get_device_status(d_ws, stream))


def zipccl_decompress_reduce_noalloc(d_peer_chunks, peer_chunk_bytes, k: int, n: int, d_out: int,
                                     stream: int) -> tuple[int, int]:
    """The no-allocation reduce call; returns (status, device address of its scratch)."""
    if not _peer_arrays_match(d_peer_chunks, peer_chunk_bytes, k):
        return ERR_INVALID_ARG, 0
    ptrs = (ctypes.c_void_p * max(1, len(d_peer_chunks)))(*[int(p) for p in d_peer_chunks])
    scratch = ctypes.c_void_p()
    st = load().zipccl_decompress_reduce_noalloc(ptrs, _u64_array(peer_chunk_bytes), k, n, d_out,
                                                 ctypes.byref(scratch), stream)
    return int(st), int(scratch.value or 0)


def zipccl_codebook_phase(phase: int) -> tuple[int, list[int]]:
    off = ctypes.c_int()
    lens = (ctypes.c_uint8 * 16)()
    _check(load().zipccl_codebook_phase(int(phase), ctypes.byref(off), lens), "zipccl_codebook_phase")
    return off.value, list(lens)


def zipccl_codebook_rebuild_phase(phase: int) -> tuple[int, list[int]]:
    """The phase table derived again from the closed form (for checking the frozen one)."""
    off = ctypes.c_int()
    lens = (ctypes.c_uint8 * 16)()
    _check(load().zipccl_codebook_rebuild_phase(int(phase), ctypes.byref(off), lens), "zipccl_codebook_rebuild_phase")
    return off.value, list(lens)


def zipccl_selftest_bounded_wait(which: int, ws_ptr: int, ws_bytes: int, stream_ptr: int) -> int:
    """Run one bounded wait that must give up (0: look-back, 1: mbarrier); returns the call's status."""
    return int(load().zipccl_selftest_bounded_wait(int(which), ws_ptr, int(ws_bytes), stream_ptr))


def zipccl_profile_encode_events(ev_before: int, ev_after: int) -> int:
    """Set (or, with two zeros, clear) the CUDA events every compress call records around its encode kernel."""
    return int(load().zipccl_profile_encode_events(ev_before or None, ev_after or None))


def zipccl_predict_chunk_bytes(n: int, sigma: float) -> tuple[int, float]:
    """Predicted stream bytes of one chunk of n values from N(0, sigma^2), and bits per value."""
    out = ctypes.c_uint64()
    bits = ctypes.c_double()
    _check(load().zipccl_predict_chunk_bytes(ctypes.c_uint64(int(n)), ctypes.c_float(sigma), ctypes.byref(out),
                                             ctypes.byref(bits)), "zipccl_predict_chunk_bytes")
    return int(out.value), float(bits.value)


def zipccl_choose_compressed(n: int, sigma: float, link_gbs: float, compress_gbs: float, decompress_gbs: float,
                             margin: float = 0.1) -> tuple[bool, float]:
    """(compress?, predicted speedup of the compressed exchange) under the sequential cost model."""
    use = ctypes.c_int()
    sp = ctypes.c_double()
    _check(load().zipccl_choose_compressed(ctypes.c_uint64(int(n)), ctypes.c_float(sigma), ctypes.c_double(link_gbs),
                                           ctypes.c_double(compress_gbs), ctypes.c_double(decompress_gbs),
                                           ctypes.c_double(margin), ctypes.byref(use), ctypes.byref(sp)),
           "zipccl_choose_compressed")
    return bool(use.value), float(sp.value)


# ------------------------------------------------------------------ torch level
class Compressed:
    """A compressed buffer: chunks back to back in ``data`` (uint8, device) and
    their byte offsets in ``offsets`` (int64 view of uint64, n_chunks + 1)."""

    def __init__(self, data, offsets, n: int, chunk_elems):
        self.data = data
        self.offsets = offsets
        self.n = int(n)
        self.chunk_elems = [int(c) for c in chunk_elems]

    @property
    def n_chunks(self) -> int:
        return len(self.chunk_elems)

    def nbytes(self) -> int:
        return int(self.offsets[-1].item())

    def chunk(self, c: int):
        o = self.offsets.cpu()
        return self.data[int(o[c]): int(o[c + 1])]


def _torch():
    import torch
    return torch


def _stream_ptr(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _words(x):
    torch = _torch()
    if x.dtype == torch.bfloat16:
        x = x.view(torch.int16)
    if x.dtype not in (torch.int16, torch.uint16):
        raise TypeError("expected a bfloat16 (or 16-bit word) tensor")
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return x.reshape(-1)


def _ws(nbytes: int, device, ws=None, stream=None):
    torch = _torch()
    if ws is not None and ws.numel() >= nbytes:
        return ws
    return _keep(torch.empty(max(256, nbytes), dtype=torch.uint8, device=device), stream)


def _keep(t, stream):
    """A tensor allocated here and used by work on `stream`: when that is not
    the current stream, the caching allocator must not hand its memory out
    again before the work on `stream` is done."""
    torch = _torch()
    if stream is not None and stream != torch.cuda.current_stream(t.device):
        t.record_stream(stream)
    return t


def compress(x, chunk_elems=None, sigma_hint=None, out=None, offsets=None, ws=None, stream=None,
             send=None, ready=None) -> Compressed:
    """Compress a BF16 CUDA tensor into per-chunk self-contained streams.  With
    ``send`` (a uint8 CUDA tensor of at least the worst-case size), the same
    kernel writes every chunk there too and posts each one as it completes;
    ``ready`` (int64 CUDA tensor of n_chunks + 1, optional) receives the post
    times (see zipccl_compress_send)."""
    torch = _torch()
    w = _words(x)
    n = w.numel()
    chunk_elems = [n] if chunk_elems is None else [int(c) for c in chunk_elems]
    cap = zipccl_max_compressed_bytes(chunk_elems)
    if out is None or out.numel() < cap:
        out = _keep(torch.empty(max(16, cap), dtype=torch.uint8, device=w.device), stream)
    if offsets is None:
        offsets = _keep(torch.empty(len(chunk_elems) + 1, dtype=torch.int64, device=w.device), stream)
    wsb = zipccl_compress_workspace_bytes(chunk_elems)
    ws = _ws(wsb, w.device, ws, stream)
    if send is None:
        st = zipccl_compress(w.data_ptr(), n, chunk_elems, sigma_hint, out.data_ptr(), out.numel(),
                             offsets.data_ptr(), ws.data_ptr(), ws.numel(), _stream_ptr(stream))
        _check(st, "zipccl_compress")
    else:
        st = zipccl_compress_send(w.data_ptr(), n, chunk_elems, sigma_hint, out.data_ptr(), out.numel(),
                                  offsets.data_ptr(), send.data_ptr(), send.numel(),
                                  0 if ready is None else ready.data_ptr(), ws.data_ptr(), ws.numel(),
                                  _stream_ptr(stream))
        _check(st, "zipccl_compress_send")
    return Compressed(out, offsets, n, chunk_elems)


def decompress(c: Compressed, out=None, ws=None, stream=None):
    """Decompress into a bfloat16 tensor of c.n elements (bit-identical)."""
    torch = _torch()
    if out is None:
        out = _keep(torch.empty(max(1, c.n), dtype=torch.bfloat16, device=c.data.device), stream)[: c.n]
    wsb = zipccl_decompress_workspace_bytes(c.n, c.n_chunks)
    ws = _ws(wsb, c.data.device, ws, stream)
    st = zipccl_decompress(c.data.data_ptr(), c.offsets.data_ptr(), c.n_chunks, out.data_ptr(), c.n,
                           ws.data_ptr(), ws.numel(), _stream_ptr(stream))
    _check(st, "zipccl_decompress")
    return out


def decompress_reduce(peer_chunks, n: int, out=None, ws=None, stream=None):
    """Receive side of a reduce-scatter: decode k peer chunks (uint8 CUDA
    tensors, rank order) and sum them in fp32 -> bfloat16[n]."""
    torch = _torch()
    k = len(peer_chunks)
    dev = peer_chunks[0].device
    if out is None:
        out = _keep(torch.empty(max(1, n), dtype=torch.bfloat16, device=dev), stream)[:n]
    wsb = zipccl_reduce_workspace_bytes(k)
    ws = _ws(wsb, dev, ws, stream)
    st = zipccl_decompress_reduce([p.data_ptr() for p in peer_chunks], [p.numel() for p in peer_chunks], k, n,
                                  out.data_ptr(), ws.data_ptr(), ws.numel(), _stream_ptr(stream))
    _check(st, "zipccl_decompress_reduce")
    return out
