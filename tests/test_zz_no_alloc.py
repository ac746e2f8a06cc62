"""zipccl_decompress_reduce_noalloc through the C ABI: argument errors come
back before any CUDA call (CPU), and on the GPU two calls in a row match the
workspace-taking zipccl_decompress_reduce and the oracle bit for bit, with a
clean device status read through the scratch address the call returns.

Collected last on purpose (file name), so the scratch's one-time set-up is
also exercised after every other test has run in the same process; each test
here passes on its own as well."""
from __future__ import annotations

import numpy as np
import pytest

import lossless_bf16_tensor_zipccl_gb300 as zc
import oracle
import workloads


def test_noalloc_argument_errors_before_any_cuda_call():
    zc.load()
    one = [16]
    assert zc.zipccl_decompress_reduce_noalloc([], one, 0, 10, 16, 0)[0] == zc.ERR_INVALID_ARG
    ptrs = [16] * 17
    assert zc.zipccl_decompress_reduce_noalloc(ptrs, [64] * 17, 17, 10, 16, 0)[0] == zc.ERR_INVALID_ARG
    assert zc.zipccl_decompress_reduce_noalloc([16], one, 1, 10, 0, 0)[0] == zc.ERR_INVALID_ARG


def test_noalloc_scratch_covers_the_maximum_peer_count():
    assert zc.zipccl_reduce_workspace_bytes(16) == 256 + 1024 + 16 * 4096


def _case(seed: int, k: int, n: int):
    rng = np.random.default_rng(seed)
    xs = [workloads.gaussian_bf16(n, 10.0 ** rng.uniform(-3, 1), seed, k, p) for p in range(k)]
    xs[0][:4] = np.array([0x7F80, 0xFF80, 0x7FC1, 0x8001], np.uint16)
    chunks = [oracle.compress(x)[0] for x in xs]
    return chunks, oracle.decompress_reduce(chunks, n)


@pytest.mark.gpu
def test_noalloc_matches_reduce_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zc.load()
    s = torch.cuda.current_stream().cuda_stream
    scratch_seen = []
    for seed, k, n in [(501, 8, 100000), (502, 3, 70001)]:
        chunks, ref = _case(seed, k, n)
        dev = [torch.from_numpy(np.frombuffer(c, dtype=np.uint8).copy()).cuda() for c in chunks]
        ptrs = [d.data_ptr() for d in dev]
        sizes = [len(c) for c in chunks]
        out_a = torch.full((n,), -1, dtype=torch.int16, device="cuda")
        out_b = torch.full((n,), -2, dtype=torch.int16, device="cuda")
        wsb = zc.zipccl_reduce_workspace_bytes(k)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        assert zc.zipccl_decompress_reduce(ptrs, sizes, k, n, out_a.data_ptr(), ws.data_ptr(), wsb, s) == zc.OK
        assert zc.zipccl_get_device_status(ws.data_ptr(), s) == zc.OK
        st, scratch = zc.zipccl_decompress_reduce_noalloc(ptrs, sizes, k, n, out_b.data_ptr(), s)
        assert st == zc.OK and scratch != 0 and scratch % 256 == 0
        assert zc.zipccl_get_device_status(scratch, s) == zc.OK
        scratch_seen.append(scratch)
        a = out_a.cpu().numpy().view(np.uint16)
        b = out_b.cpu().numpy().view(np.uint16)
        assert np.array_equal(b, a), "no-alloc reduce differs from zipccl_decompress_reduce"
        assert np.array_equal(b, ref), "no-alloc reduce differs from the oracle"
    assert scratch_seen[0] == scratch_seen[1], "one scratch per device"
