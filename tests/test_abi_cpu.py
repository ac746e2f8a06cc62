"""The C ABI without a GPU: the library builds and loads, exports every symbol
include/zipccl.h declares, and its host-only calls behave -- argument and
capacity errors come back before any CUDA call, the worst-case bound and the
code tables agree with the oracle's."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

import lossless_bf16_tensor_zipccl_gb300 as zc
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "zipccl.h")).read()
    return sorted(set(re.findall(r"\b(zipccl_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = zc.load()
    names = declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(zc.EXPORTED_SYMBOLS) == names


def test_format_version_and_status_strings():
    assert zc.zipccl_format_version() == 1 == oracle.format_version()
    for s in range(7):
        assert zc.zipccl_status_string(s)
    assert zc.zipccl_status_string(99) == "unknown status"


def test_codebook_tables_match_oracle():
    # the frozen tables of format v1: the library's copy equals the oracle's copy
    offs, lens = oracle.phase_tables()
    for r in range(16):
        o, l = zc.zipccl_codebook_phase(r)
        assert o == offs[r] and l == lens[r], r
    with pytest.raises(zc.ZipcclError):
        zc.zipccl_codebook_phase(16)


def test_frozen_tables_equal_their_derivation():
    # each side's frozen copy still equals what its own builder derives from the
    # closed form: the library's exact dynamic program, the oracle's package-merge
    roffs, rlens = oracle.rebuilt_phase_tables()
    offs, lens = oracle.phase_tables()
    assert (roffs, rlens) == (offs, lens)
    for r in range(16):
        assert zc.zipccl_codebook_rebuild_phase(r) == zc.zipccl_codebook_phase(r), r
    with pytest.raises(zc.ZipcclError):
        zc.zipccl_codebook_rebuild_phase(-1)


@pytest.mark.parametrize("chunks", [[1], [0], [0, 5, 0], [32768], [32769, 1, 65536], [1 << 20] * 3,
                                    [12345678, 7]])
def test_max_bytes_matches_oracle(chunks):
    assert zc.zipccl_max_compressed_bytes(chunks) == oracle.max_compressed_bytes(chunks)


def test_workspace_sizes():
    assert zc.zipccl_compress_workspace_bytes([10, 0, 70000]) > 256
    assert zc.zipccl_decompress_workspace_bytes(70010, 3) >= 256 + 3 * 4096
    assert zc.zipccl_reduce_workspace_bytes(8) >= 256 + 8 * 4096
    with pytest.raises(zc.ZipcclError):
        zc.zipccl_reduce_workspace_bytes(17)
    with pytest.raises(zc.ZipcclError):
        zc.zipccl_compress_workspace_bytes([1 << 31])


FAKE = 1 << 20  # aligned non-null "device" addresses: never dereferenced, every call below fails validation first


def test_compress_argument_errors_return_before_launch():
    ok_ws = zc.zipccl_compress_workspace_bytes([100])
    cap = zc.zipccl_max_compressed_bytes([100])
    # sum of chunks != n
    assert zc.zipccl_compress(FAKE, 101, [100], None, FAKE, cap, FAKE, FAKE, ok_ws, 0) == zc.ERR_INVALID_ARG
    # misaligned input / output / workspace
    assert zc.zipccl_compress(FAKE + 2, 100, [100], None, FAKE, cap, FAKE, FAKE, ok_ws, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_compress(FAKE, 100, [100], None, FAKE + 8, cap, FAKE, FAKE, ok_ws, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_compress(FAKE, 100, [100], None, FAKE, cap, FAKE, FAKE + 16, ok_ws, 0) == zc.ERR_INVALID_ARG
    # null pointers, no chunks
    assert zc.zipccl_compress(0, 100, [100], None, FAKE, cap, FAKE, FAKE, ok_ws, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_compress(FAKE, 0, [], None, FAKE, cap, FAKE, FAKE, ok_ws, 0) == zc.ERR_INVALID_ARG
    # capacity and workspace too small
    assert zc.zipccl_compress(FAKE, 100, [100], None, FAKE, cap - 1, FAKE, FAKE, ok_ws, 0) == zc.ERR_CAPACITY
    assert zc.zipccl_compress(FAKE, 100, [100], None, FAKE, cap, FAKE, FAKE, ok_ws - 1, 0) == zc.ERR_CAPACITY
    # chunk too large
    assert zc.zipccl_compress(FAKE, 1 << 31, [1 << 31], None, FAKE, 1 << 40, FAKE, FAKE, 1 << 40, 0) == \
        zc.ERR_INVALID_ARG


def test_compress_send_argument_errors_return_before_launch():
    cap = zc.zipccl_max_compressed_bytes([100])
    ws = zc.zipccl_compress_workspace_bytes([100])
    SEND = FAKE + (1 << 20)

    def call(send, send_cap, out=FAKE):
        return zc.zipccl_compress_send(FAKE, 100, [100], None, out, cap, FAKE, send, send_cap, 0, FAKE, ws, 0)
    assert call(0, cap) == zc.ERR_INVALID_ARG              # no send buffer
    assert call(SEND + 8, cap) == zc.ERR_INVALID_ARG       # misaligned
    assert call(FAKE, cap) == zc.ERR_INVALID_ARG           # the output itself
    assert call(SEND, cap - 1) == zc.ERR_CAPACITY          # below the worst-case size
    assert zc.zipccl_compress_send(FAKE, 100, [100], None, FAKE, cap, FAKE, SEND, cap, FAKE + 4, FAKE, ws, 0) == \
        zc.ERR_INVALID_ARG                                   # misaligned ready array


def test_profile_hook_takes_both_events_or_none():
    # the measurement hook is host-side state: one event without the other is
    # refused, two nulls switch it off; nothing touches a device
    assert zc.zipccl_profile_encode_events(0x1000, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_profile_encode_events(0, 0x1000) == zc.ERR_INVALID_ARG
    assert zc.zipccl_profile_encode_events(0, 0) == zc.OK


def test_selftest_argument_errors_return_before_launch():
    assert zc.zipccl_selftest_bounded_wait(3, FAKE, 512, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_selftest_bounded_wait(2, FAKE, 335, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_selftest_bounded_wait(-1, FAKE, 512, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_selftest_bounded_wait(0, 0, 512, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_selftest_bounded_wait(0, FAKE + 16, 512, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_selftest_bounded_wait(1, FAKE, 271, 0) == zc.ERR_INVALID_ARG


def test_decompress_and_reduce_argument_errors():
    ws = zc.zipccl_decompress_workspace_bytes(100, 1)
    assert zc.zipccl_decompress(FAKE, FAKE, 0, FAKE, 100, FAKE, ws, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_decompress(FAKE + 4, FAKE, 1, FAKE, 100, FAKE, ws, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_decompress(FAKE, FAKE, 1, FAKE, 100, FAKE, ws - 1, 0) == zc.ERR_CAPACITY
    rws = zc.zipccl_reduce_workspace_bytes(2)
    assert zc.zipccl_decompress_reduce([FAKE, FAKE], [64, 64], 0, 10, FAKE, FAKE, rws, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_decompress_reduce([FAKE] * 17, [64] * 17, 17, 10, FAKE, FAKE, 1 << 30, 0) == \
        zc.ERR_INVALID_ARG
    assert zc.zipccl_decompress_reduce([FAKE, FAKE + 8], [64, 64], 2, 10, FAKE, FAKE, rws, 0) == \
        zc.ERR_INVALID_ARG
    assert zc.zipccl_decompress_reduce([FAKE, 0], [64, 64], 2, 10, FAKE, FAKE, rws, 0) == zc.ERR_INVALID_ARG
    assert zc.zipccl_decompress_reduce([FAKE, FAKE], [64, 64], 2, 10, FAKE, FAKE, rws - 1, 0) == zc.ERR_CAPACITY
    assert zc.zipccl_get_device_status(0, 0) == zc.ERR_INVALID_ARG


def test_product_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "lossless_bf16_tensor_zipccl_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src and "zipccl_oracle" not in src, f


# ----------------------------------------------------------------- size prediction / switch
@pytest.mark.parametrize("n", [0, 1, 1000, 32768, 32769, 70001, 1 << 20, 8388608])
@pytest.mark.parametrize("sigma", [1e-6, 1e-3, 0.02, 1.0, 100.0, 1e-39])
def test_predicted_chunk_bytes_match_oracle(n, sigma):
    s = float(np.float32(sigma))
    assert zc.zipccl_predict_chunk_bytes(n, s) == oracle.predict_chunk_bytes(n, s)


def test_choose_compressed_follows_the_cost_model():
    n, sigma = 1 << 26, 1e-3
    pred, _ = zc.zipccl_predict_chunk_bytes(n, sigma)
    for link in [10.0, 100.0, 900.0, 5000.0]:
        use, sp = zc.zipccl_choose_compressed(n, sigma, link, 1700.0, 2200.0, 0.1)
        t_raw = 2 * n / link
        t_zip = 2 * n / 1700.0 + pred / link + 2 * n / 2200.0
        assert sp == pytest.approx(t_raw / t_zip, rel=1e-12)
        assert use == (t_raw / t_zip > 1.1)
    assert zc.zipccl_choose_compressed(n, sigma, 10.0, 1700.0, 2200.0)[0]
    assert not zc.zipccl_choose_compressed(n, sigma, 5000.0, 1700.0, 2200.0)[0]
    # a margin larger than the predicted gain keeps the plain exchange
    sp = zc.zipccl_choose_compressed(n, sigma, 100.0, 1700.0, 2200.0, 0.0)[1]
    assert not zc.zipccl_choose_compressed(n, sigma, 100.0, 1700.0, 2200.0, sp)[0]


@pytest.mark.parametrize("args", [(1000, 0.0, 10.0, 1.0, 1.0, 0.1), (1000, -1.0, 10.0, 1.0, 1.0, 0.1),
                                  (1000, float("inf"), 10.0, 1.0, 1.0, 0.1), (1000, 1.0, 0.0, 1.0, 1.0, 0.1),
                                  (1000, 1.0, 10.0, 0.0, 1.0, 0.1), (1000, 1.0, 10.0, 1.0, -1.0, 0.1),
                                  (1000, 1.0, 10.0, 1.0, 1.0, -0.5), (1 << 40, 1.0, 10.0, 1.0, 1.0, 0.1)])
def test_switch_argument_errors(args):
    with pytest.raises(zc.ZipcclError) as ei:
        zc.zipccl_choose_compressed(*args)
    assert ei.value.status == zc.ERR_INVALID_ARG


def test_reduce_wrappers_reject_mismatched_peer_arrays():
    # k must equal the length of both host arrays, or the C call would read past them
    for call in (lambda p, b, k: zc.zipccl_decompress_reduce(p, b, k, 10, 16, 32, 4096, 0),
                 lambda p, b, k: zc.zipccl_decompress_reduce_noalloc(p, b, k, 10, 16, 0)[0]):
        assert call([16, 32], [100, 100], 3) == zc.ERR_INVALID_ARG
        assert call([16, 32], [100], 2) == zc.ERR_INVALID_ARG
        assert call([16], [100, 100], 1) == zc.ERR_INVALID_ARG
