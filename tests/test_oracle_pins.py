"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each check uses a library
routine (scipy's normal distribution, numpy float32 arithmetic, torch's BF16
cast), a closed form, an exhaustive optimum, an independent stream reader
(tests/zstream.py) or a figure printed on the pages.

Passages: "ZipCCL: Efficient Lossless Data Compression of Communication
Collectives for Accelerating LLM Training" -- abstract (exponent coding of
near-Gaussian tensors, no online statistics; lossless), shd-paper summary key
design (short codes for frequent exponents, from the Gaussian density),
Fig. 6 caption (about 11 bits per value, up to 31% smaller), Fig. 3 / Fig. 5
(ReduceScatter receive side: decompress then reduce).
"""
from __future__ import annotations

import heapq
import math
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle
import workloads
import zstream

HERE = os.path.dirname(os.path.abspath(__file__))


def golden(name):
    vals = {}
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    return (x.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------- pmf / entropy
def scipy_pmf(sigma):
    """P(biased exponent = e) for N(0, sigma^2) from scipy: 2 (Phi(b) - Phi(a)) on each binade,
    taken through scipy's erf below 1 standard deviation and its survival function above."""
    r2 = math.sqrt(2.0)
    p = np.zeros(256)
    p[0] = special.erf(2.0 ** -126 / sigma / r2)
    for e in range(1, 255):
        a, b = 2.0 ** (e - 127) / sigma, 2.0 ** (e - 126) / sigma
        if b < 1.0:
            p[e] = special.erf(b / r2) - special.erf(a / r2)
        else:
            p[e] = 2.0 * (stats.norm.sf(a) - stats.norm.sf(b))
    return p


@pytest.mark.parametrize("sigma", [1e-3, 0.02, 1.0, 1.37, 300.0, 2.0 ** -100])
def test_pmf_matches_scipy_normal(sigma):
    p = oracle.exponent_pmf(sigma)
    q = scipy_pmf(sigma)
    # erf differences: absolute accuracy ~1e-16 everywhere, relative 1e-9 on the bulk of the mass
    assert np.all(np.abs(p - q) < 1e-15)
    big = q > 1e-6
    assert np.allclose(p[big], q[big], rtol=1e-9, atol=0)
    assert abs(p.sum() - 1.0) < 1e-12


def test_entropy_is_scale_invariant_and_in_closed_form_band():
    # over the normal range the pmf only shifts with log2(sigma): H depends on the phase alone
    hs = []
    for r in range(64):
        s = 2.0 ** (r / 64)
        h = oracle.entropy_bits(oracle.exponent_pmf(s))
        h2 = oracle.entropy_bits(oracle.exponent_pmf(s * 2.0 ** -20))
        assert abs(h - h2) < 1e-9
        q = scipy_pmf(s)
        hq = -np.sum(q[q > 0] * np.log2(q[q > 0]))
        assert abs(h - hq) < 1e-8
        hs.append(h)
    assert 2.5420 < min(hs) and max(hs) < 2.5465
    h002 = oracle.entropy_bits(oracle.exponent_pmf(0.02))
    assert abs(h002 - 2.5453) < 1e-4
    p = oracle.exponent_pmf(0.02)
    assert int(np.argmax(p)) == 121 and abs(p[121] - 0.3165) < 1e-4


# ------------------------------------------------------------ code construction
def optimal_limited_cost(w, L):
    """Exact minimum of sum w_i l_i over all length vectors with Kraft <= 1, l_i <= L (DP)."""
    units = 1 << L
    INF = float("inf")
    dp = [INF] * (units + 1)
    dp[0] = 0.0
    for wi in w:
        nd = [INF] * (units + 1)
        for k in range(units + 1):
            if dp[k] == INF:
                continue
            for l in range(1, L + 1):
                k2 = k + (1 << (L - l))
                if k2 <= units and dp[k] + wi * l < nd[k2]:
                    nd[k2] = dp[k] + wi * l
        dp = nd
    return min(dp)


def huffman_cost(w):
    h = [(x, i) for i, x in enumerate(w)]
    heapq.heapify(h)
    cost, n = 0.0, len(w)
    while len(h) > 1:
        a, b = heapq.heappop(h), heapq.heappop(h)
        cost += a[0] + b[0]
        heapq.heappush(h, (a[0] + b[0], n))
        n += 1
    return cost


def kraft(lens, L=10):
    return sum(2 ** (L - l) for l in lens)


def test_phase_tables_complete_and_optimal():
    offs, tabs = oracle.phase_tables()
    for r in range(16):
        lens = tabs[r]
        assert len(lens) == 16 and all(1 <= l <= 10 for l in lens)
        assert kraft(lens) == 1024, "a complete prefix code"
        p = scipy_pmf(2.0 ** (r / 16))
        b = offs[r] + 127
        w = list(p[b:b + 15]) + [1.0 - p[b:b + 15].sum()]
        cost = sum(wi * li for wi, li in zip(w, lens))
        assert abs(cost - optimal_limited_cost(w, 10)) < 1e-12
        # window = 15 consecutive exponents of largest mass
        masses = [p[s:s + 15].sum() for s in range(0, 241)]
        assert b == int(np.argmax(masses))
        # the code sits within 0.06 bits of the entropy of the Gaussian exponent
        h = -np.sum(p[p > 0] * np.log2(p[p > 0]))
        assert 0 < cost + w[15] * 8 - h < 0.06


@pytest.mark.parametrize("seed", range(12))
def test_package_merge_optimal_on_random_weights(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 17))
    w = list(rng.dirichlet(np.full(n, 0.3)) + 1e-9)
    L = int(max(math.ceil(math.log2(n)), rng.integers(2, 8)))
    lens = oracle.package_merge(w, L)
    assert kraft(lens, L) <= (1 << L) and max(lens) <= L
    cost = sum(a * b for a, b in zip(w, lens))
    assert abs(cost - optimal_limited_cost(w, L)) < 1e-12
    big = oracle.package_merge(w, 16) if n <= 16 else None
    if big is not None and max(big) < 16:
        assert abs(sum(a * b for a, b in zip(w, big)) - huffman_cost(w)) < 1e-12


def test_phase_tables_robust_to_tiny_weight_perturbation():
    # the frozen lengths do not sit on a knife edge: 1e-9 relative noise in the pmf changes nothing
    offs, tabs = oracle.phase_tables()
    rng = np.random.default_rng(7)
    for r in range(16):
        p = oracle.exponent_pmf(2.0 ** (r / 16))
        b = offs[r] + 127
        w = np.array(list(p[b:b + 15]) + [1.0 - p[b:b + 15].sum()])
        for _ in range(5):
            wp = w * (1.0 + 1e-9 * rng.standard_normal(16))
            assert oracle.package_merge(wp, 10) == tabs[r]


# ------------------------------------------------------------ scale selection
def test_scale_constant_closed_form():
    # mean of floor(log2|Z|) over a uniform phase = E[log2|Z|] - 1/2, E[log2|Z|] = -(gamma + ln 2)/(2 ln 2)
    c0 = 0.5 + (np.euler_gamma + math.log(2)) / (2 * math.log(2))
    assert abs(c0 - 3541 / 2500) < 5e-5
    # and it matches the closed-form pmf averaged over the phase
    vals = []
    for r in range(32):
        s = 2.0 ** (r / 32)
        p = scipy_pmf(s)
        m = np.sum(np.arange(1, 255) * p[1:255]) / p[1:255].sum()
        vals.append(127 + math.log2(s) - m)
    assert abs(np.mean(vals) - c0) < 1e-4


@pytest.mark.parametrize("sigma", [1e-6, 1e-3, 0.02, 1.0, 7.0, 100.0])
def test_select_q_tracks_sigma(sigma):
    x = workloads.gaussian_bf16(1 << 18, sigma, 5, int(sigma * 1e6) % 1000)
    q = oracle.select_q(x)
    assert abs(q - 16 * math.log2(sigma)) <= 2.0
    assert oracle.q_from_sigma(sigma) == math.floor(16 * math.log2(sigma) + 0.5)


def test_select_q_small_and_special_chunks():
    assert oracle.select_q(np.zeros(100, np.uint16)) == 0          # nothing but zeros
    assert oracle.select_q(np.full(10, 0x7F80, np.uint16)) == 0    # nothing but inf
    x = np.full(7, 0x3F80, np.uint16)                              # 1.0: e = 127
    # q = round(16 (127 - 127 + c0)) = round(22.6624) = 23
    assert oracle.select_q(x) == 23


def _large_chunk_sample_input(n=100_003, a=120, e_other=200, shift_block=None, shift=0):
    """A chunk of n > 4096 values whose 64 sample blocks (64 values at floor(b n / 64), the
    rule of the scale select) hold exponents a and a + 1 and every other value exponent
    e_other.  214 sampled values hold a + 1: the first and last of every block and 86 more
    inside the blocks.  shift_block / shift: move that block's pattern by `shift` positions
    (the rule then reads one e_other value)."""
    x = np.full(n, e_other << 7, np.uint16)
    hi = set()
    for b in range(64):
        hi.update({(b, 0), (b, 63)})
    extra = 214 - len(hi)
    for b in range(64):
        for t in range(1, 63):
            if extra and (b, t) not in hi and t % 9 == 4:
                hi.add((b, t))
                extra -= 1
    assert len(hi) == 214
    for b in range(64):
        start = (b * n) // 64 + (shift if b == shift_block else 0)
        for t in range(64):
            x[start + t] = (a + ((b, t) in hi)) << 7
    return x


def test_select_q_large_chunk_samples_exactly_the_stated_blocks():
    # 4096 sampled exponents: 3882 x 120 and 214 x 121.  By hand:
    #   16 (mean - 127) + 16 c0 + 1/2 = 16 (120 - 127) + 16 * 214 / 4096 + 22.6624 + 0.5
    #                                 = -112 + 0.8359375 + 23.1624 = -88.0016625  ->  q = -89.
    # One value from outside the blocks (exponent 200) anywhere in the sample adds at least
    # 16 * 79 / 4096 = 0.31 and gives q >= -88.
    assert oracle.select_q(_large_chunk_sample_input()) == -89


@pytest.mark.parametrize("b", [0, 1, 17, 31, 32, 50, 62, 63])
@pytest.mark.parametrize("shift", [-1, 1])
def test_select_q_large_chunk_block_shift_changes_q(b, shift):
    # a block placed one position off the rule's start: the sample takes one exponent-200 value
    # in place of a 121 (and the sum rises by at least 79), so q leaves -89.
    if b == 0 and shift == -1:
        pytest.skip("block 0 starts at the first value")
    x = _large_chunk_sample_input(shift_block=b, shift=shift)
    assert oracle.select_q(x) != -89


def test_select_q_large_chunk_reads_the_whole_block():
    # the last value of every block becomes exponent 200 (was 121): by hand, the sample is
    # 64 x 200, 150 x 121 and 3882 x 120, so mean = 120 + (64 * 80 + 150) / 4096 = 121.28662 and
    #   16 (121.28662 - 127) + 23.1624 = -68.2517  ->  q = -69.
    # A block length of 63 would not see those values (q = -89); 65 would add more (q > -69).
    x = _large_chunk_sample_input()
    n = x.size
    for b in range(64):
        x[(b * n) // 64 + 63] = 200 << 7
    assert oracle.select_q(x) == -69


def test_base_clamped_to_valid_window():
    assert oracle.base_for_q(-32768) == 0
    assert oracle.base_for_q(32767) == 240
    offs, _ = oracle.phase_tables()
    assert oracle.base_for_q(0) == 127 + offs[0]
    assert oracle.base_for_q(-90) == math.floor(-90 / 16) + 127 + offs[(-90) % 16]


# ------------------------------------------------------------ round trips
def roundtrip(x, chunk_elems=None, hint=None, parse=True):
    s, offs = oracle.compress(x, chunk_elems, hint)
    y = oracle.decompress(s, offs, x.size)
    assert np.array_equal(y, x)
    if parse:
        chunks = zstream.parse_stream(s, offs)
        got = np.concatenate([c.values for c in chunks]) if chunks else np.zeros(0, np.uint16)
        assert np.array_equal(got, x), "independent reader disagrees with the input"
    assert len(s) <= oracle.max_compressed_bytes(chunk_elems or [x.size])
    return s, offs


def test_all_bf16_patterns_roundtrip():
    w = workloads.all_patterns()
    roundtrip(w.x)


def test_patterns_spliced_into_gaussian_take_the_escape():
    g = workloads.gaussian_bf16(1 << 20, 0.02, 11)
    pos = np.random.default_rng(3).choice(g.size, 65536, replace=False)
    g[pos] = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    s, offs = roundtrip(g, parse=False)
    ch = zstream.parse_chunk(s)
    assert all(t.mode == 0 for t in ch.tiles), "coded mode carries every exponent through ESC"
    assert sum(t.escapes for t in ch.tiles) > 30000
    assert np.array_equal(ch.values, g)


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 255, 256, 257, 2047, 32767, 32768, 32769, 65536 + 300])
def test_edge_sizes(n):
    x = workloads.gaussian_bf16(n, 0.5, 21, n)
    roundtrip(x)


@pytest.mark.parametrize("fill", [0x0000, 0x8000, 0x7FC0, 0xFFFF, 0x7F80, 0xFF80, 0x0001, 0x807F])
def test_constant_special_chunks(fill):
    x = np.full(40000, fill, np.uint16)
    roundtrip(x)


def test_denormal_only_chunk():
    rng = np.random.default_rng(4)
    x = rng.integers(0, 128, size=50000).astype(np.uint16) | (rng.integers(0, 2, 50000).astype(np.uint16) << 15)
    roundtrip(x)


@pytest.mark.parametrize("seed", range(6))
def test_random_ragged_chunk_mixes(seed):
    w = workloads.random_chunks(seed, n_chunks=int(3 + seed), max_elems=70000)
    hints = None
    if seed % 2:
        hints = [s if i % 2 else 0.0 for i, s in enumerate(w.sigma)]
    roundtrip(w.x, w.chunk_elems, hints)


def test_uniform_patterns_go_raw_with_bounded_expansion():
    x = np.random.default_rng(9).integers(0, 65536, size=100000, dtype=np.uint16)
    s, offs = roundtrip(x)
    ch = zstream.parse_chunk(s)
    assert all(t.mode == 1 for t in ch.tiles)
    assert len(s) <= 2 * x.size + 32 + 16 + 4 * 16 + 32 * len(ch.tiles)


# ------------------------------------------------------------ sizes and ratio
def test_size_identity_pr1():
    w = workloads.pr1()
    s, offs = oracle.compress(w.x)
    ch = zstream.parse_chunk(s)
    lens = ch.lens
    e = (w.x >> 7) & 0xFF
    sym = e.astype(np.int64) - ch.base
    sym[(sym < 0) | (sym > 14)] = 15
    Lx = np.array(lens)[sym] + np.where(sym == 15, 8, 0)
    for t, tile in enumerate(ch.tiles):
        assert tile.mode == 0
        seg = ((np.arange(tile.n) % zstream.ROW) // zstream.LANE)
        tl = Lx[t * 32768: t * 32768 + tile.n]
        for j in range(zstream.SEGS):
            # payload bits of a segment = sum of its code lengths + 8 per escape
            assert tile.seg_bits[j] == int(tl[seg == j].sum())
        assert tile.payload_words == (sum(tile.seg_bits) + 31) // 32
    # total = s/m plane + payload words + documented metadata
    expect = 32 + zstream.pad16(4 * len(ch.tiles))
    for tile in ch.tiles:
        expect += 16 + zstream.pad16(tile.n) + zstream.pad16(zstream.SEGTAB + 4 * tile.payload_words)
    assert len(s) == expect


def test_pr1_entropy_and_bits_per_value():
    w = workloads.pr1()
    e = ((w.x >> 7) & 0xFF).astype(np.int64)
    cnt = np.bincount(e, minlength=256) / e.size
    h_emp = -np.sum(cnt[cnt > 0] * np.log2(cnt[cnt > 0]))
    p = scipy_pmf(0.02)
    h = -np.sum(p[p > 0] * np.log2(p[p > 0]))
    assert abs(h_emp - h) / h < 0.01
    s, _ = oracle.compress(w.x)
    bpv = 8.0 * len(s) / w.n
    assert bpv <= 1.01 * (8.0 + h)
    g = golden("paper_figures.txt")
    assert bpv < g["bits_per_value_upper"]
    assert 100.0 * (1.0 - len(s) / (2 * w.n)) > g["size_reduction_percent"]


def test_moe_dispatch_within_one_percent_of_chunk_entropy():
    # Outlier-heavy activations routed to 64 expert chunks: the code built
    # from the Gaussian pmf of each chunk's sampled scale still comes within
    # 1% of 8 + the chunk's empirical exponent entropy (outliers escape).
    w = workloads.moe(tokens=1024)
    e = ((w.x >> 7) & 0xFF).astype(np.int64)
    bound, st = 0.0, 0
    for n in w.chunk_elems:
        if n:
            c = np.bincount(e[st:st + n], minlength=256)
            p = c[c > 0] / n
            bound += n * (8.0 - np.sum(p * np.log2(p)))
        st += n
    s, _ = oracle.compress(w.x, w.chunk_elems)
    assert 8.0 * len(s) <= 1.01 * bound


# ------------------------------------------------------------ decompress_reduce
def torch_bf16_rne(f32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_rne_matches_torch_cast():
    rng = np.random.default_rng(12)
    u = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    # force ties and near-overflow cases
    u[:2000] = (u[:2000] & 0xFFFF0000) | 0x8000
    u[2000:2100] = 0x7F7F8000 + np.arange(100, dtype=np.uint32)
    f = u.view(np.float32)
    ours = np.array([oracle.float_to_bf16_rne(float(v)) for v in f], dtype=np.uint16)
    ref = torch_bf16_rne(f)
    nan = np.isnan(f)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(ours[nan] == 0x7FC0)


def test_reduce_matches_numpy_float32_left_fold():
    rng = np.random.default_rng(13)
    k, n = 5, 40000
    xs = [workloads.gaussian_bf16(n, 10.0 ** rng.uniform(-3, 1), 77, p) for p in range(k)]
    xs[2][:50] = np.array([0x7F80, 0xFF80, 0x7FC1, 0x0001, 0x8001] * 10, np.uint16)
    chunks = [oracle.compress(x)[0] for x in xs]
    out = oracle.decompress_reduce(chunks, n)
    acc = bf16_to_f32(xs[0]).copy()
    for p in range(1, k):
        acc = (acc + bf16_to_f32(xs[p])).astype(np.float32)
    ref = torch_bf16_rne(acc)
    nan = np.isnan(acc)
    assert np.array_equal(out[~nan], ref[~nan])
    assert np.all(out[nan] == 0x7FC0)


def test_reduce_k1_is_decode_and_negation_cancels():
    x = workloads.gaussian_bf16(50000, 0.3, 31)
    s, _ = oracle.compress(x)
    assert np.array_equal(oracle.decompress_reduce([s], x.size), x)
    neg = x ^ np.uint16(0x8000)
    s2, _ = oracle.compress(neg)
    y = oracle.decompress_reduce([s, s2], x.size)
    assert np.all(y == 0)


# ----------------------------------------------------------------- size prediction
@pytest.mark.parametrize("sigma", [1e-3, 0.02, 1.0, 37.0])
def test_expected_exponent_bits_from_scipy_masses(sigma):
    # the predictor's E = sum_e p(e) L(e) with scipy's masses, the phase
    # table's lengths and window, an escape costing its codeword + 8 bits
    q = oracle.q_from_sigma(sigma)
    offs, lens = oracle.phase_tables()
    base = oracle.base_for_q(q)
    p = scipy_pmf(sigma)
    L = np.array([lens[q % 16][e - base] if 0 <= e - base < 15 else lens[q % 16][15] + 8 for e in range(256)])
    assert oracle.expected_exponent_bits(sigma, q) == pytest.approx(float((p * L).sum()), rel=1e-9)


@pytest.mark.parametrize("sigma,seed", [(0.02, 1), (1e-3, 2), (1.0, 3)])
def test_predicted_size_matches_compressed_gaussian(sigma, seed):
    # the model's size against a stream compressed from N(0, sigma^2) data:
    # sampling noise in the code lengths of 2^20 values is ~0.03%
    n = 1 << 20
    x = workloads.gaussian_bf16(n, sigma, 500 + seed)
    s, _ = oracle.compress(x, [n], [sigma])
    pred, bits = oracle.predict_chunk_bytes(n, sigma)
    assert abs(pred - len(s)) / len(s) < 2e-3
    assert bits == pytest.approx(8.0 * pred / n)


def test_predicted_bits_bounded_by_entropy():
    # 8 raw bits + the code's expected length: at least 8 + H(sigma), and
    # within the measured redundancy of the 10-bit-limited code (+ metadata)
    for sigma in [1e-5, 3e-3, 0.5, 20.0]:
        _, bits = oracle.predict_chunk_bytes(1 << 24, sigma)
        H = float(-(lambda p: (p[p > 0] * np.log2(p[p > 0])).sum())(scipy_pmf(sigma)))
        assert 8.0 + H <= bits <= 8.0 + H + 0.1
