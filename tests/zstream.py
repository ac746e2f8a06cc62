"""Independent reader of the v1 stream format, used only by tests.

Written from the format description (chunk header, tile table, tiles with a
sign/mantissa plane and a coded or raw exponent region), not from either
implementation.  It decodes with a dictionary of bit strings, so it shares no
decoding machinery with the oracle's canonical-range decoder or with the GPU
lookup tables.
"""
from __future__ import annotations

import struct
from dataclasses import dataclass, field

import numpy as np

MAGIC = 0x4C43435A
TILE = 32768
ROW = 512
LANE = 8
SEGS = 64
SEGTAB = 2 * SEGS


def pad16(x: int) -> int:
    return (x + 15) & ~15


def canonical_codes(lens: list[int]) -> dict[int, str]:
    """symbol -> codeword bit string (first transmitted bit first)."""
    order = sorted(range(len(lens)), key=lambda s: (lens[s], s))
    codes, code, prev = {}, 0, None
    for s in order:
        if prev is not None:
            code = (code + 1) << (lens[s] - prev)
        codes[s] = format(code, f"0{lens[s]}b")
        prev = lens[s]
    return codes


@dataclass
class Tile:
    mode: int
    n: int
    exp_bytes: int
    offset: int
    size: int
    seg_bits: list[int] = field(default_factory=list)
    payload_words: int = 0
    escapes: int = 0


@dataclass
class Chunk:
    n: int
    base: int
    q: int
    lens: list[int]
    tile_offsets: list[int]
    tiles: list[Tile]
    size: int
    values: np.ndarray


def _bits_lsb_first(words: bytes) -> str:
    return "".join(format(b, "08b")[::-1] for b in words)


def parse_chunk(buf: bytes) -> Chunk:
    magic, version, tile_log2, seg_log2, n, n_tiles, base, flags, q = struct.unpack_from("<IHBBQIBBh", buf, 0)
    assert magic == MAGIC and version == 1 and tile_log2 == 15 and seg_log2 == 9 and flags == 0
    lens = []
    for i in range(8):
        b = buf[24 + i]
        lens += [b & 15, b >> 4]
    assert n_tiles == (n + TILE - 1) // TILE
    toffs = list(struct.unpack_from(f"<{n_tiles}I", buf, 32)) if n_tiles else []
    assert all(v == 0 for v in buf[32 + 4 * n_tiles: 32 + pad16(4 * n_tiles)])
    codes = canonical_codes(lens)
    decode = {v: s for s, v in codes.items()}
    out = np.zeros(n, dtype=np.uint16)
    tiles = []
    pos = 32 + pad16(4 * n_tiles)
    for t in range(n_tiles):
        nt = TILE if t + 1 < n_tiles else n - t * TILE
        assert toffs[t] == pos, "tiles must be back to back"
        mode, tn, exp_bytes, zero = struct.unpack_from("<IIII", buf, pos)
        assert tn == nt and zero == 0 and mode in (0, 1)
        sm = np.frombuffer(buf, dtype=np.uint8, count=nt, offset=pos + 16).astype(np.uint16)
        assert all(v == 0 for v in buf[pos + 16 + nt: pos + 16 + pad16(nt)])
        ex = pos + 16 + pad16(nt)
        vals = ((sm & 0x80) << 8) | (sm & 0x7F)
        tile = Tile(mode, nt, exp_bytes, pos, 16 + pad16(nt) + pad16(exp_bytes))
        if mode == 1:
            assert exp_bytes == nt
            e = np.frombuffer(buf, dtype=np.uint8, count=nt, offset=ex).astype(np.uint16)
        else:
            segb = list(struct.unpack_from(f"<{SEGS}H", buf, ex))
            total = sum(segb)
            nwords = (total + 31) // 32
            assert exp_bytes == SEGTAB + 4 * nwords
            tile.seg_bits = segb
            tile.payload_words = nwords
            e = np.zeros(nt, dtype=np.uint16)
            bits = _bits_lsb_first(buf[ex + SEGTAB: ex + SEGTAB + 4 * nwords])
            k = 0
            for j in range(SEGS):
                end = k + segb[j]
                idx = [r + LANE * j + t8 for r in range(0, nt, ROW) for t8 in range(LANE) if r + LANE * j + t8 < nt]
                for i in idx:
                    cw = ""
                    while cw not in decode:
                        cw += bits[k]
                        k += 1
                    s = decode[cw]
                    if s == 15:
                        e[i] = int(bits[k:k + 8][::-1], 2)
                        k += 8
                        tile.escapes += 1
                    else:
                        e[i] = base + s
                assert k == end, "segment bit length must match its symbols"
            assert set(bits[k:]) <= {"0"}, "payload padding must be zero bits"
            assert len(bits) - k < 32
        assert all(v == 0 for v in buf[ex + exp_bytes: ex + pad16(exp_bytes)])
        out[t * TILE: t * TILE + nt] = vals | (e << 7)
        tiles.append(tile)
        pos += tile.size
    return Chunk(n, base, q, lens, toffs, tiles, pos, out)


def parse_stream(stream: bytes, offsets) -> list[Chunk]:
    chunks = []
    for c in range(len(offsets) - 1):
        a, b = int(offsets[c]), int(offsets[c + 1])
        ch = parse_chunk(stream[a:b])
        assert ch.size == b - a
        chunks.append(ch)
    return chunks
