"""Second, independent reading of the compressed bf16 stream format, in Python.

Used only to pin the C oracle: a decoder, and an encoder that takes the code
width k as an argument so that the choice of k can be brute-forced (encode at
every k, keep the shortest).  Written from the format definition, not from
the oracle's code.

Format (little endian):
  stream  = 64-byte header | u64 offset per chunk, zero-padded to 16 | chunks
  header  = magic "CCB1" u32, version u16 = 1, dtype u16 = 1 (bf16),
            chunk_elems u32 = 4096, u32 0, n_elems u64, n_chunks u64,
            total_bytes u64, 24 zero bytes
  chunk   = mode u8 (0 packed, 1 raw), k u8, base u8, u8 0, n_c u16,
            n_esc u16, chunk_bytes u32, u32 0, then the body, zero-padded
            to 16 bytes
  raw     = the n_c bf16 values
  packed  = 4096 sign+fraction bytes ((b >> 8) & 0x80 | b & 0x7F),
            k bit-planes of 128 u32 words, escape bytes (raw exponents of
            the elements whose code is the sentinel 2^k - 1, in bit-plane
            order: by word, then by bit)
  element i = 256 j + 8 l + s (j < 16, l < 32, s < 8) keeps bit p of its
  code in plane p, word 32 (j // 4) + l, bit 8 (s % 4) + 2 (j % 4) + s // 4.
"""

from __future__ import annotations

import struct

import numpy as np

CHUNK = 4096
MAGIC = 0x31424343


def _rup16(v: int) -> int:
    return -(-v // 16) * 16


def _element_slots():
    i = np.arange(CHUNK)
    j, l, s = i >> 8, (i >> 3) & 31, i & 7
    word = (j // 4) * 32 + l
    bit = 8 * (s % 4) + 2 * (j % 4) + s // 4
    return word, bit


WORD_OF, BIT_OF = _element_slots()


def split(x: np.ndarray):
    x = x.astype(np.uint32)
    expo = (x >> 7) & 0xFF
    sm = ((x >> 8) & 0x80) | (x & 0x7F)
    return expo, sm


def encode_chunk_at(x: np.ndarray, k: int | None, base: int | None = None) -> bytes | None:
    """Chunk bytes for a given width k (None = raw) and base (None: the
    minimum exponent); None if k cannot represent the chunk (k = 0 needs a
    single exponent, equal to the base).  Exponents outside
    [base, base + 2^k - 2] escape."""
    n_c = x.size
    if k is None:
        body = x.astype("<u2").tobytes()
        size = 16 + _rup16(len(body))
        hdr = struct.pack("<BBBBHHII", 1, 0, 0, 0, n_c, 0, size, 0)
        return (hdr + body).ljust(size, b"\0")
    assert n_c == CHUNK
    expo, sm = split(x)
    base = int(expo.min()) if base is None else int(base)
    off = expo.astype(np.int64) - base
    if k == 0:
        if off.min() != 0 or off.max() != 0:
            return None
        esc = b""
        planes = b""
    else:
        sent = (1 << k) - 1
        escaped = (off < 0) | (off >= sent)
        code = np.where(escaped, sent, off).astype(np.uint32)
        order = np.argsort(32 * WORD_OF + BIT_OF)  # elements in bit-plane order
        esc = expo[order][escaped[order]].astype(np.uint8).tobytes()
        words = np.zeros((k, 128), np.uint64)
        for p in range(k):
            bits = ((code >> p) & 1).astype(np.uint64) << BIT_OF.astype(np.uint64)
            np.add.at(words[p], WORD_OF, bits)
        planes = words.astype("<u4").tobytes()
    body = sm.astype(np.uint8).tobytes() + planes + esc
    size = 16 + _rup16(len(body))
    hdr = struct.pack("<BBBBHHII", 0, k, base, 0, n_c, len(esc), size, 0)
    return (hdr + body).ljust(size, b"\0")


def brute_force_chunk(x: np.ndarray) -> tuple[str, int | None, bytes]:
    """Encode at every candidate and keep the shortest; ties keep the smaller
    k, and raw wins every tie with a packed candidate."""
    raw = encode_chunk_at(x, None)
    if x.size != CHUNK:
        return "raw", None, raw
    best_k, best = None, None
    for k in range(8):
        enc = encode_chunk_at(x, k)
        if enc is not None and (best is None or len(enc) < len(best)):
            best_k, best = k, enc
    if best is None or len(best) >= len(raw):
        return "raw", None, raw
    return "packed", best_k, best


def encode_stream(x: np.ndarray) -> bytes:
    """Whole stream built from brute-forced chunks."""
    n = x.size
    nch = -(-n // CHUNK)
    start = 64 + _rup16(8 * nch)
    chunks = [brute_force_chunk(x[c * CHUNK:(c + 1) * CHUNK])[2] for c in range(nch)]
    offs, pos = [], start
    for ch in chunks:
        offs.append(pos)
        pos += len(ch)
    hdr = struct.pack("<IHHIIQQQ", MAGIC, 1, 1, CHUNK, 0, n, nch, pos).ljust(64, b"\0")
    table = struct.pack("<%dQ" % nch, *offs).ljust(start - 64, b"\0")
    return hdr + table + b"".join(chunks)


def window_table(x: np.ndarray):
    """Window-base variant: for every k, the escape count of every base
    (exponents outside [b, b + 2^k - 2]), counted directly; returns the
    chosen (k, base, n_esc) or None for raw, with the variant's tie rules."""
    e = split(x)[0].astype(np.int64)
    if e.min() == e.max():
        return 0, int(e.min()), 0
    best = None
    for k in range(1, 8):
        S = (1 << k) - 1
        b = np.arange(256)[:, None]
        n_esc = ((e[None, :] < b) | (e[None, :] >= b + S)).sum(1)
        bk = int(np.argmin(n_esc))  # first minimum: the smallest base
        size = 512 * k + _rup16(int(n_esc[bk]))
        if best is None or size < best[0]:
            best = (size, k, bk, int(n_esc[bk]))
    if best[0] >= 4096:
        return None
    return best[1], best[2], best[3]


def encode_stream_window(x: np.ndarray) -> bytes:
    """Whole version-2 stream from window_table's choices."""
    n = x.size
    nch = -(-n // CHUNK)
    start = 64 + _rup16(8 * nch)
    chunks = []
    for c in range(nch):
        xc = x[c * CHUNK:(c + 1) * CHUNK]
        choice = window_table(xc) if xc.size == CHUNK else None
        chunks.append(encode_chunk_at(xc, None) if choice is None else encode_chunk_at(xc, choice[0], choice[1]))
    offs, pos = [], start
    for ch in chunks:
        offs.append(pos)
        pos += len(ch)
    hdr = struct.pack("<IHHIIQQQ", MAGIC, 2, 1, CHUNK, 0, n, nch, pos).ljust(64, b"\0")
    table = struct.pack("<%dQ" % nch, *offs).ljust(start - 64, b"\0")
    return hdr + table + b"".join(chunks)


class Corrupt(ValueError):
    pass


def decode_chunk(buf: bytes, n_c: int) -> np.ndarray:
    mode, k, base, zero, nc, n_esc, size, zero2 = struct.unpack_from("<BBBBHHII", buf, 0)
    if nc != n_c or size != len(buf):
        raise Corrupt("chunk header")
    body = buf[16:]
    if mode == 1:
        return np.frombuffer(body[:2 * n_c], "<u2").astype(np.uint16)
    if mode != 0 or n_c != CHUNK or k > 7:
        raise Corrupt("mode")
    sm = np.frombuffer(body[:CHUNK], np.uint8).astype(np.uint32)
    words = np.frombuffer(body[CHUNK:CHUNK + 512 * k], "<u4").reshape(k, 128).astype(np.uint32)
    esc = np.frombuffer(body[CHUNK + 512 * k:CHUNK + 512 * k + n_esc], np.uint8).astype(np.uint32)
    code = np.zeros(CHUNK, np.uint32)
    for p in range(k):
        code |= ((words[p, WORD_OF] >> BIT_OF.astype(np.uint32)) & 1) << p
    expo = base + code
    if k > 0:
        order = np.argsort(32 * WORD_OF + BIT_OF)  # elements in bit-plane order
        where = order[code[order] == (1 << k) - 1]
        if where.size != n_esc:
            raise Corrupt("escape count")
        expo[where] = esc
    if expo.max() > 255:
        raise Corrupt("exponent range")
    return (((sm & 0x80) << 8) | (expo << 7) | (sm & 0x7F)).astype(np.uint16)


def decode_stream(s: bytes, n: int) -> np.ndarray:
    s = bytes(s)
    magic, ver, dt, ce, _, n_el, nch, total = struct.unpack_from("<IHHIIQQQ", s, 0)
    if (magic, dt, ce, n_el, nch) != (MAGIC, 1, CHUNK, n, -(-n // CHUNK)) or ver not in (1, 2):
        raise Corrupt("stream header")
    offs = list(struct.unpack_from("<%dQ" % nch, s, 64)) + [total]
    out = np.empty(n, np.uint16)
    for c in range(nch):
        n_c = min(CHUNK, n - c * CHUNK)
        out[c * CHUNK:c * CHUNK + n_c] = decode_chunk(s[offs[c]:offs[c + 1]], n_c)
    return out


def chunk_headers(s: bytes):
    """(offset, mode, k, base, n_c, n_esc, chunk_bytes) for every chunk."""
    s = bytes(s)
    nch, total = struct.unpack_from("<QQ", s, 24)
    offs = struct.unpack_from("<%dQ" % nch, s, 64)
    out = []
    for o in offs:
        mode, k, base, _, n_c, n_esc, size, _ = struct.unpack_from("<BBBBHHII", s, o)
        out.append((o, mode, k, base, n_c, n_esc, size))
    return out


# ---------------------------------------------------------------------------
# Element types.  dtype field 1 = bf16, 2 = fp16, 3 = fp32.  Per type: the
# exponent field (bits), where it sits (shift), and what a packed chunk's body
# holds before the exponent planes:
#   bf16  4096 bytes: sign << 7 | fraction bits 0..6
#   fp16  4096 bytes: fraction bits 0..7; then 3 bit-planes (same layout as
#         the code planes) holding fraction bit 8, fraction bit 9, sign
#   fp32  4096 bytes: sign << 7 | fraction bits 16..22; then the 4096 lower
#         halves (bits 0..15) as u16
# k runs 0..(exponent bits - 1); a chunk is packed only when
# 512 k + pad16(escapes) < 512 * exponent bits.  Raw chunks hold the values.
# ---------------------------------------------------------------------------
DTYPES = {1: dict(item=2, ebits=8, shift=7), 2: dict(item=2, ebits=5, shift=10), 3: dict(item=4, ebits=8, shift=23)}


def _planes_of(bits_list) -> bytes:
    """Bit-planes (128 u32 words each) of per-element 0/1 arrays."""
    out = b""
    for b in bits_list:
        words = np.zeros(128, np.uint64)
        np.add.at(words, WORD_OF, b.astype(np.uint64) << BIT_OF.astype(np.uint64))
        out += words.astype("<u4").tobytes()
    return out


def _plane_values(raw: bytes, count: int):
    words = np.frombuffer(raw, "<u4").reshape(count, 128).astype(np.uint32)
    return [(words[p, WORD_OF] >> BIT_OF.astype(np.uint32)) & 1 for p in range(count)]


def split_typed(dtype: int, x: np.ndarray):
    """(exponents, residual section bytes) of a full chunk."""
    d = DTYPES[dtype]
    v = x.astype(np.uint64)
    expo = ((v >> d["shift"]) & ((1 << d["ebits"]) - 1)).astype(np.int64)
    if dtype == 1:
        resid = (((v >> 8) & 0x80) | (v & 0x7F)).astype(np.uint8).tobytes()
    elif dtype == 2:
        resid = (v & 0xFF).astype(np.uint8).tobytes() + _planes_of([(v >> 8) & 1, (v >> 9) & 1, (v >> 15) & 1])
    else:
        hi = v >> 16
        resid = (((hi >> 8) & 0x80) | (hi & 0x7F)).astype(np.uint8).tobytes() + (v & 0xFFFF).astype("<u2").tobytes()
    return expo, resid


def encode_chunk_typed_at(dtype: int, x: np.ndarray, k: int | None, base: int | None = None) -> bytes | None:
    d = DTYPES[dtype]
    n_c = x.size
    if k is None:
        body = x.astype("<u%d" % d["item"]).tobytes()
        size = 16 + _rup16(len(body))
        return (struct.pack("<BBBBHHII", 1, 0, 0, 0, n_c, 0, size, 0) + body).ljust(size, b"\0")
    assert n_c == CHUNK
    expo, resid = split_typed(dtype, x)
    base = int(expo.min()) if base is None else int(base)
    off = expo - base
    if k == 0:
        if off.min() != 0 or off.max() != 0:
            return None
        esc, planes = b"", b""
    else:
        sent = (1 << k) - 1
        escaped = (off < 0) | (off >= sent)
        code = np.where(escaped, sent, off)
        order = np.argsort(32 * WORD_OF + BIT_OF)
        esc = expo[order][escaped[order]].astype(np.uint8).tobytes()
        planes = _planes_of([(code >> p) & 1 for p in range(k)])
    body = resid + planes + esc
    size = 16 + _rup16(len(body))
    return (struct.pack("<BBBBHHII", 0, k, base, 0, n_c, len(esc), size, 0) + body).ljust(size, b"\0")


def brute_force_chunk_typed(dtype: int, x: np.ndarray) -> bytes:
    """Every width tried; the shortest wins (ties: smaller k); raw unless the
    exponent part beats 512 * exponent bits."""
    d = DTYPES[dtype]
    raw = encode_chunk_typed_at(dtype, x, None)
    if x.size != CHUNK:
        return raw
    resid_len = len(split_typed(dtype, x)[1])
    best = None
    for k in range(d["ebits"]):
        enc = encode_chunk_typed_at(dtype, x, k)
        if enc is not None and (best is None or len(enc) < len(best)):
            best = enc
    if best is None or len(best) - 16 - resid_len >= 512 * d["ebits"]:
        return raw
    return best


def window_table_typed(dtype: int, x: np.ndarray):
    d = DTYPES[dtype]
    e = split_typed(dtype, x)[0]
    if e.min() == e.max():
        return 0, int(e.min())
    nsym = 1 << d["ebits"]
    best = None
    for k in range(1, d["ebits"]):
        S = (1 << k) - 1
        b = np.arange(nsym)[:, None]
        n_esc = ((e[None, :] < b) | (e[None, :] >= b + S)).sum(1)
        bk = int(np.argmin(n_esc))
        size = 512 * k + _rup16(int(n_esc[bk]))
        if best is None or size < best[0]:
            best = (size, k, bk)
    if best[0] >= 512 * d["ebits"]:
        return None
    return best[1], best[2]


def encode_stream_typed(dtype: int, x: np.ndarray, window: bool = False) -> bytes:
    n = x.size
    nch = -(-n // CHUNK)
    start = 64 + _rup16(8 * nch)
    chunks = []
    for c in range(nch):
        xc = x[c * CHUNK:(c + 1) * CHUNK]
        if not window:
            chunks.append(brute_force_chunk_typed(dtype, xc))
            continue
        choice = window_table_typed(dtype, xc) if xc.size == CHUNK else None
        chunks.append(encode_chunk_typed_at(dtype, xc, None) if choice is None
                      else encode_chunk_typed_at(dtype, xc, choice[0], choice[1]))
    offs, pos = [], start
    for ch in chunks:
        offs.append(pos)
        pos += len(ch)
    hdr = struct.pack("<IHHIIQQQ", MAGIC, 2 if window else 1, dtype, CHUNK, 0, n, nch, pos).ljust(64, b"\0")
    table = struct.pack("<%dQ" % nch, *offs).ljust(start - 64, b"\0")
    return hdr + table + b"".join(chunks)


def decode_chunk_typed(dtype: int, buf: bytes, n_c: int) -> np.ndarray:
    d = DTYPES[dtype]
    mode, k, base, _, nc, n_esc, size, _ = struct.unpack_from("<BBBBHHII", buf, 0)
    if nc != n_c or size != len(buf):
        raise Corrupt("chunk header")
    body = buf[16:]
    if mode == 1:
        return np.frombuffer(body[:d["item"] * n_c], "<u%d" % d["item"]).astype(np.uint64)
    if mode != 0 or n_c != CHUNK or k >= d["ebits"]:
        raise Corrupt("mode")
    resid_len = {1: 4096, 2: 4096 + 1536, 3: 4096 + 8192}[dtype]
    codes = _plane_values(body[resid_len:resid_len + 512 * k], k)
    code = np.zeros(CHUNK, np.int64)
    for p in range(k):
        code |= codes[p].astype(np.int64) << p
    expo = base + code
    if k > 0:
        order = np.argsort(32 * WORD_OF + BIT_OF)
        where = order[code[order] == (1 << k) - 1]
        if where.size != n_esc:
            raise Corrupt("escape count")
        expo[where] = np.frombuffer(body[resid_len + 512 * k:resid_len + 512 * k + n_esc], np.uint8)
    if expo.max() >= (1 << d["ebits"]):
        raise Corrupt("exponent range")
    e = expo.astype(np.uint64)
    b0 = np.frombuffer(body[:CHUNK], np.uint8).astype(np.uint64)
    if dtype == 1:
        return ((b0 & 0x80) << 8) | (e << 7) | (b0 & 0x7F)
    if dtype == 2:
        f8, f9, sg = _plane_values(body[CHUNK:CHUNK + 1536], 3)
        return b0 | (f8.astype(np.uint64) << 8) | (f9.astype(np.uint64) << 9) | (e << 10) | (sg.astype(np.uint64) << 15)
    lo = np.frombuffer(body[CHUNK:CHUNK + 8192], "<u2").astype(np.uint64)
    hi = ((b0 & 0x80) << 8) | (e << 7) | (b0 & 0x7F)
    return (hi << 16) | lo


def decode_stream_typed(dtype: int, s: bytes, n: int) -> np.ndarray:
    s = bytes(s)
    magic, ver, dt, ce, _, n_el, nch, total = struct.unpack_from("<IHHIIQQQ", s, 0)
    if (magic, dt, ce, n_el, nch) != (MAGIC, dtype, CHUNK, n, -(-n // CHUNK)) or ver not in (1, 2):
        raise Corrupt("stream header")
    offs = list(struct.unpack_from("<%dQ" % nch, s, 64)) + [total]
    out = np.empty(n, np.uint64)
    for c in range(nch):
        n_c = min(CHUNK, n - c * CHUNK)
        out[c * CHUNK:c * CHUNK + n_c] = decode_chunk_typed(dtype, s[offs[c]:offs[c + 1]], n_c)
    return out.astype(np.uint32 if DTYPES[dtype]["item"] == 4 else np.uint16)
