"""Host-side checks of libnq.so that need no GPU: the library loads and
exports every symbol of include/nq.h, the host packer follows the layout in
the header and round-trips every code in every position, and bad arguments
are rejected."""
import os
import re

import numpy as np
import pytest

import quantized_weight_decode_gb300 as nqp
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session", autouse=True)
def built():
    nqp.build()
    return nqp.lib()


def test_exports_every_header_symbol():
    with open(os.path.join(ROOT, "include", "nq.h")) as f:
        hdr = f.read()
    declared = set(re.findall(r"\b(nq_[a-z_0-9]+)\s*\(", hdr))
    assert declared, "no declarations found"
    lib = nqp.lib()
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared == set(nqp.EXPORTED)
    assert nqp.layout_version() == 2


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_packed_bytes(bits):
    cb, sb = nqp.packed_bytes(5120, 34816, bits)
    assert cb == 34816 * 5120 * bits // 8
    assert sb == 34816 * 5120 // 64 * 2
    cb, sb = nqp.packed_bytes(64, 17, bits)          # padded to 2 row tiles
    assert cb == 2 * 128 * bits and sb == 2 * 32


def _spec_position(bits, lane, p, h):
    """(word, list of (bit in word, bit of code)) for code (lane, pair p, half h),
    written from the layout description in include/nq.h."""
    hs = 16 * h
    if bits == 4:
        return [(p // 4, 4 * (p % 4) + hs + m, m) for m in range(4)]
    if bits == 8:
        return [(p // 2, 8 * (p % 2) + hs + m, m) for m in range(8)]
    if bits == 5:
        if p < 15:
            return [(p // 3, 5 * (p % 3) + hs + m, m) for m in range(5)]
        return [(m, 15 + hs, m) for m in range(5)]
    if p < 12:
        return [(p // 2, 6 * (p % 2) + hs + m, m) for m in range(6)]
    d = p - 12
    out = [(d, 12 + hs + m, m) for m in range(4)]
    out += [(4 + d // 2, 12 + 2 * (d % 2) + hs + m, 4 + m) for m in range(2)]
    return out


def _word(packed, bits, blk, lane, w):
    base = blk * 128 * bits
    off = 16 * lane + 4 * w if w < 4 else 512 + 4 * (bits - 4) * lane + 4 * (w - 4)
    return int.from_bytes(bytes(packed[base + off: base + off + 4]), "little")


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_pack_matches_header_spec(bits):
    rng = synth.generator(0, 200, bits)
    N, K = 40, 128                                   # 3 row tiles (last padded), 2 groups
    codes = synth.uniform_codes(rng, N, K, bits)
    scales = rng.integers(0, 0x7C00, size=(N, K // 64), dtype=np.uint16)
    packed, sp = nqp.pack(codes, scales, bits)
    bias = 1 << (bits - 1)
    G = K // 64
    for rt in range(3):
        for g in range(G):
            blk = rt * G + g
            for lane in range(32):
                q, r = lane // 4, lane % 4
                for p in range(16):
                    j, i = p // 4, p % 4
                    for h in range(2):
                        row = q + 8 * (i % 2)
                        k = 16 * r + 4 * j + 2 * (i // 2) + h
                        n = rt * 16 + row
                        u_expect = (int(codes[n, g * 64 + k]) if n < N else 0) + bias
                        u = 0
                        for (w, bit, m) in _spec_position(bits, lane, p, h):
                            u |= ((_word(packed, bits, blk, lane, w) >> bit) & 1) << m
                        assert u == u_expect, (rt, g, lane, p, h)
            for row in range(16):
                n = rt * 16 + row
                want = scales[n, g] if n < N else 0
                assert sp[blk * 16 + 2 * (row % 8) + row // 8] == want


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_roundtrip_every_code_in_every_position(bits):
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1)) - 1
    vals = np.arange(lo, hi + 1, dtype=np.int8)
    N, K = 16, 64 * len(vals)
    # shift the value sequence per row so every value visits every (row, k)
    base = np.arange(K)[None, :] + np.arange(N)[:, None] * 7
    codes = vals[base % len(vals)]
    rng = synth.generator(0, 201, bits)
    scales = rng.integers(0, 0xFFFF, size=(N, K // 64), dtype=np.uint16)
    scales[(scales & 0x7C00) == 0x7C00] &= 0x83FF   # keep finite
    packed, sp = nqp.pack(codes, scales, bits)
    c2, s2 = nqp.unpack(packed, sp, K, N, bits)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)
    # every value appears in every (row, k mod 64) position across groups
    for v in (lo, hi, 0):
        assert (codes == v).any(axis=1).all()


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_roundtrip_ragged(bits):
    rng = synth.generator(0, 202, bits)
    for N, K in [(1, 64), (17, 192), (255, 512)]:
        codes = synth.uniform_codes(rng, N, K, bits)
        scales = rng.integers(0, 0x7C00, size=(N, K // 64), dtype=np.uint16)
        packed, sp = nqp.pack(codes, scales, bits)
        c2, s2 = nqp.unpack(packed, sp, K, N, bits)
        assert np.array_equal(c2, codes) and np.array_equal(s2, scales)


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_pack_rejects_out_of_range(bits):
    N, K = 16, 64
    codes = np.zeros((N, K), np.int8)
    scales = np.full((N, 1), 0x3C00, np.uint16)
    if bits < 8:                                    # every int8 is an 8-bit code
        codes[3, 5] = (1 << (bits - 1))             # one above the range
        with pytest.raises(nqp.NQError) as e:
            nqp.pack(codes, scales, bits)
        assert e.value.code == nqp.ERANGE
        codes[3, 5] = -(1 << (bits - 1)) - 1
        with pytest.raises(nqp.NQError):
            nqp.pack(codes, scales, bits)
        codes[3, 5] = 0
    for bad in (0x7C00, 0xFC00, 0x7E00):            # +inf, -inf, NaN
        s = scales.copy()
        s[2, 0] = bad
        with pytest.raises(nqp.NQError) as e:
            nqp.pack(codes, s, bits)
        assert e.value.code == nqp.ERANGE


def test_shape_validation():
    for K, N, bits in [(0, 16, 4), (65, 16, 4), (64, 0, 4), (64, 16, 3), (64, 16, 7), (-64, 16, 4)]:
        with pytest.raises(nqp.NQError) as e:
            nqp.packed_bytes(K, N, bits)
        assert e.value.code == nqp.EINVAL


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert nqp.status_string(code) and nqp.status_string(code) != "unknown status"
    assert nqp.status_string(-99) == "unknown status"


@pytest.mark.parametrize("bits", [4, 5, 6, 8])
def test_pack_gate_up_interleaves_rows(bits):
    """nq_pack_gate_up equals nq_pack of the row-interleaved matrix, and the
    unpacked rows are gate row 8 r + m at 16 r + m, up row 8 r + m at
    16 r + 8 + m."""
    rng = synth.generator(0, 810, bits)
    I, K = 40, 128
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1)) - 1
    cg = rng.integers(lo, hi + 1, (I, K)).astype(np.int8)
    cu = rng.integers(lo, hi + 1, (I, K)).astype(np.int8)
    sg = rng.integers(0, 0x7C00, (I, K // 64)).astype(np.uint16)
    su = rng.integers(0, 0x7C00, (I, K // 64)).astype(np.uint16)
    p, s = nqp.pack_gate_up(cg, sg, cu, su, bits)
    p2, s2 = nqp.pack(nqp.interleave_gate_up(cg, cu), nqp.interleave_gate_up(sg, su), bits)
    assert np.array_equal(p, p2) and np.array_equal(s, s2)
    codes, scales = nqp.unpack(p, s, K, 2 * I, bits)
    for n in range(2 * I):
        r, m, up = n // 16, n % 8, (n % 16) >= 8
        src_c, src_s = (cu, su) if up else (cg, sg)
        assert np.array_equal(codes[n], src_c[8 * r + m]) and np.array_equal(scales[n], src_s[8 * r + m])


def test_pack_gate_up_rejects_bad_arguments():
    cg = np.zeros((12, 64), np.int8)
    sg = np.zeros((12, 1), np.uint16)
    with pytest.raises(nqp.NQError) as e:          # I not a multiple of 8
        nqp.pack_gate_up(cg, sg, cg, sg, 4)
    assert e.value.code == nqp.EINVAL
    cg = np.zeros((8, 64), np.int8)
    sg = np.zeros((8, 1), np.uint16)
    bad = cg.copy()
    bad[3, 7] = 8                                   # outside [-8, 7]
    with pytest.raises(nqp.NQError) as e:
        nqp.pack_gate_up(cg, sg, bad, sg, 4)
    assert e.value.code == nqp.ERANGE


def test_row_tile_count_limit():
    """More than 2^31 - 1 row tiles is rejected (32-bit tile indices)."""
    nqp.packed_bytes(64, 16 * (2 ** 31 - 1), 4)
    with pytest.raises(nqp.NQError) as e:
        nqp.packed_bytes(64, 16 * (2 ** 31 - 1) + 1, 4)
    assert e.value.code == nqp.EINVAL
