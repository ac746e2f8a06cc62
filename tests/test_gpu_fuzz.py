"""Randomised parity against the oracle, through the C ABI (seeded, bounded).

Each case draws a chunk layout (1 to ~300 chunks, empty, sub-tile, ragged and
multi-tile chunks, so chunk starts fall on any element offset) and a value
mix per chunk (Gaussian at scales from 1e-8 to 1e3, uniform 16-bit patterns
that force raw tiles, constant special values, heavy-tailed Student-t, and
Gaussian data with a share of random patterns), with special values spliced
in and optional sigma hints.  The GPU stream and offsets must equal the
oracle's byte for byte (plain compress or compress-and-send, whose send copy
must equal the stream), the GPU round trip must be bit-exact, and every
fourth case is a reduce of k random peers checked against the oracle's fold.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import lossless_bf16_tensor_zipccl_gb300 as zc  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402

SPECIALS = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x7FC1, 0xFFFF, 0x0001, 0x8001, 0x007F, 0x0080,
                     0x7F7F, 0xFF7F], dtype=np.uint16)
CASES = 200


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    zc.load()
    yield


def _values(rng, n):
    kind = rng.choice(["gauss", "raw", "const", "heavy", "mixed"], p=[.65, .08, .07, .1, .1])
    if n == 0:
        return np.empty(0, np.uint16)
    if kind == "gauss":
        x = workloads.f32_to_bf16_bits((rng.standard_normal(n) * 10.0 ** rng.uniform(-8, 3)).astype(np.float32))
    elif kind == "raw":
        x = rng.integers(0, 65536, size=n, dtype=np.uint16)
    elif kind == "const":
        x = np.full(n, rng.choice(SPECIALS), dtype=np.uint16)
    elif kind == "heavy":
        x = workloads.f32_to_bf16_bits((rng.standard_t(2, n) * 10.0 ** rng.uniform(-4, 1)).astype(np.float32))
    else:
        x = workloads.f32_to_bf16_bits((rng.standard_normal(n) * 10.0 ** rng.uniform(-5, 1)).astype(np.float32))
        m = rng.random(n) < rng.choice([0.001, 0.01, 0.2])
        x[m] = rng.integers(0, 65536, size=int(m.sum()), dtype=np.uint16)
    if rng.random() < 0.3:
        k = int(rng.integers(1, min(n, 64) + 1))
        x[rng.integers(0, n, size=k)] = rng.choice(SPECIALS, size=k)
    return x.astype(np.uint16)


def _layout(rng, budget):
    sizes = []
    for _ in range(int(np.exp(rng.uniform(0, np.log(300))))):
        r = rng.random()
        sizes.append(0 if r < 0.1 else int(rng.integers(1, 5000)) if r < 0.45 else
                     int(rng.integers(5000, 200000)) if r < 0.9 else int(rng.integers(200000, 2000000)))
    while sum(sizes) > budget:
        i = int(np.argmax(sizes))
        sizes[i] //= 2
    if sum(sizes) == 0:
        sizes[0] = int(rng.integers(1, 100000))
    return sizes


def _compress_case(rng):
    ce = _layout(rng, int(rng.choice([300_000, 2_000_000])))
    x = np.concatenate([_values(rng, n) for n in ce])
    hint = None
    if rng.random() < 0.3:
        hint = [0.0 if rng.random() < 0.4 else float(10.0 ** rng.uniform(-7, 2)) for _ in ce]
    d = torch.from_numpy(x.view(np.int16)).cuda()
    cap = zc.zipccl_max_compressed_bytes(ce)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    offs = torch.empty(len(ce) + 1, dtype=torch.int64, device="cuda")
    ws = torch.empty(zc.zipccl_compress_workspace_bytes(ce), dtype=torch.uint8, device="cuda")
    sp = torch.cuda.current_stream().cuda_stream
    send = None
    if rng.random() < 0.3:
        send = torch.empty(cap, dtype=torch.uint8, device="cuda")
        ready = torch.zeros(len(ce) + 1, dtype=torch.int64, device="cuda")
        st = zc.zipccl_compress_send(d.data_ptr(), x.size, ce, hint, out.data_ptr(), cap, offs.data_ptr(),
                                     send.data_ptr(), cap, ready.data_ptr(), ws.data_ptr(), ws.numel(), sp)
    else:
        st = zc.zipccl_compress(d.data_ptr(), x.size, ce, hint, out.data_ptr(), cap, offs.data_ptr(),
                                ws.data_ptr(), ws.numel(), sp)
    assert st == zc.OK and zc.zipccl_get_device_status(ws.data_ptr(), sp) == zc.OK
    o = offs.cpu().numpy().view(np.uint64)
    total = int(o[-1])
    so, oo = oracle.compress(x, ce, hint)
    assert np.array_equal(o, oo), "chunk offsets differ from the oracle"
    assert out[:total].cpu().numpy().tobytes() == so, "stream differs from the oracle"
    if send is not None:
        assert torch.equal(send[:total], out[:total]), "send buffer differs from the stream"
    wsd = torch.empty(zc.zipccl_decompress_workspace_bytes(x.size, len(ce)), dtype=torch.uint8, device="cuda")
    y = torch.empty(x.size, dtype=torch.int16, device="cuda")
    st = zc.zipccl_decompress(out.data_ptr(), offs.data_ptr(), len(ce), y.data_ptr(), x.size, wsd.data_ptr(),
                              wsd.numel(), sp)
    assert st == zc.OK and zc.zipccl_get_device_status(wsd.data_ptr(), sp) == zc.OK
    assert np.array_equal(y.cpu().numpy().view(np.uint16), x), "round trip differs from the input"


def _reduce_case(rng):
    k = int(rng.integers(1, 17))
    n = int(rng.integers(1, 400_000)) if rng.random() < 0.8 else int(rng.integers(1, 40000))
    chunks = [oracle.compress(_values(rng, n))[0] for _ in range(k)]
    ref = oracle.decompress_reduce(chunks, n)
    y = zc.decompress_reduce([torch.from_numpy(np.frombuffer(c, dtype=np.uint8).copy()).cuda() for c in chunks], n)
    torch.cuda.synchronize()
    assert np.array_equal(y.view(torch.int16).cpu().numpy().view(np.uint16), ref), f"reduce of {k} peers differs"


def test_randomised_parity():
    rng = np.random.default_rng(20261203)
    for i in range(1, CASES + 1):
        if i % 4 == 0:
            _reduce_case(rng)
        else:
            _compress_case(rng)
