"""CPU oracle for the compressed expert tier's block codec.

TEST INFRASTRUCTURE ONLY (see oracle/moe.py for who may import the oracle). A plain, slow restatement of
the codec with pure-Python integers, written from its definition; it shares no code with the library.

Source: PR #651 "cuda: add experimental lossless compressed expert tier" keeps experts as independently
decodable 4096-byte ANS blocks. The codec itself is this project's own (the pages use DietGPU, which is
not available): range asymmetric numeral systems (rANS) over the nibbles of the packed bytes.

Definition:
  - symbols: the nibbles of the byte stream, low nibble then high nibble of each byte;
  - model: one table of 16 frequencies per stream, each >= 1, summing to M = 4096: f_s = 1 + floor(count_s
    (M - 16) / total), then the remainder handed out one at a time to the most frequent symbols (lowest
    symbol first among equals); c_s = f_0 + ... + f_{s-1};
  - blocks of 4096 bytes (the last one shorter), each coded on its own; in a block, symbol j goes to lane
    j mod 32, and each lane is an rANS coder with state x in [2^16, 2^32), starting at 2^16;
  - encoding a symbol s (a lane's symbols in reverse order): while x >= 2^20 f_s, emit the low 16 bits of x
    and shift x right by 16; then x <- floor(x / f_s) M + (x mod f_s) + c_s;
  - decoding (forward): slot = x mod M, s = the symbol with c_s <= slot < c_s + f_s,
    x <- f_s floor(x / M) + slot - c_s, and if x < 2^16, x <- 2^16 x + (the lane's next word).

Stream layout (little-endian): u32 magic 0x31413443, u32 4096, u64 n, u32 blocks, u32 0, u16 freq[16],
u32 offset[blocks + 1] (from the start of the block area), then per block u32 state[32], u16 words[32]
and the lanes' words, lane 0 first, each lane's words in decoding order, padded to 4 bytes.

Parity status: pinned by tests/test_oracle_pins.py (round trips, the entropy bound, a constant stream).
"""
from __future__ import annotations

import struct

M_BITS = 12
M = 1 << M_BITS
LOW = 1 << 16
BLOCK = 4096
MAGIC = 0x31413443


def nibbles(data: bytes):
    for b in data:
        yield b & 15
        yield b >> 4


def frequencies(data: bytes):
    count = [0] * 16
    for s in nibbles(data):
        count[s] += 1
    total = 2 * len(data)
    f = [1 + (count[s] * (M - 16) // total if total else (M - 16) // 16) for s in range(16)]
    while sum(f) < M:
        best = max(count)
        for s in range(16):
            if count[s] == best and sum(f) < M:
                f[s] += 1
    return f


def encode(data: bytes) -> bytes:
    n = len(data)
    f = frequencies(data)
    c = [sum(f[:s]) for s in range(16)]
    blocks = (n + BLOCK - 1) // BLOCK
    body, offsets = b"", []
    for b in range(blocks):
        chunk = data[b * BLOCK:(b + 1) * BLOCK]
        sym = list(nibbles(chunk))
        states, counts, streams = [], [], []
        for lane in range(32):
            x, out = LOW, []
            for s in reversed(sym[lane::32]):
                while x >= (1 << 20) * f[s]:
                    out.append(x & 0xFFFF)
                    x >>= 16
                x = (x // f[s]) * M + (x % f[s]) + c[s]
            states.append(x)
            counts.append(len(out))
            streams.extend(reversed(out))
        blk = struct.pack("<32I", *states) + struct.pack("<32H", *counts) + struct.pack(f"<{len(streams)}H", *streams)
        blk += b"\0" * (-len(blk) % 4)
        offsets.append(len(body))
        body += blk
    offsets.append(len(body))
    head = struct.pack("<IIQII16H", MAGIC, BLOCK, n, blocks, 0, *f)
    return head + struct.pack(f"<{blocks + 1}I", *offsets) + body


def decode(stream: bytes) -> bytes:
    magic, block, n, blocks, _ = struct.unpack_from("<IIQII", stream, 0)
    assert magic == MAGIC and block == BLOCK
    f = list(struct.unpack_from("<16H", stream, 24))
    c = [sum(f[:s]) for s in range(16)]
    offsets = struct.unpack_from(f"<{blocks + 1}I", stream, 56)
    area = 56 + 4 * (blocks + 1)
    out = bytearray()
    for b in range(blocks):
        m = min(BLOCK, n - b * BLOCK)
        base = area + offsets[b]
        states = list(struct.unpack_from("<32I", stream, base))
        counts = struct.unpack_from("<32H", stream, base + 128)
        words = struct.unpack_from(f"<{sum(counts)}H", stream, base + 192)
        start = [sum(counts[:lane]) for lane in range(32)]
        used = [0] * 32
        sym = [0] * (2 * m)
        for j in range(2 * m):
            lane = j % 32
            x = states[lane]
            slot = x % M
            s = max(t for t in range(16) if c[t] <= slot)
            x = f[s] * (x // M) + slot - c[s]
            if x < LOW:
                x = (x << 16) | words[start[lane] + used[lane]]
                used[lane] += 1
            states[lane] = x
            sym[j] = s
        assert all(x == LOW for x in states) and list(used) == list(counts), "inconsistent block"
        out += bytes(sym[2 * i] | (sym[2 * i + 1] << 4) for i in range(m))
    return bytes(out)
