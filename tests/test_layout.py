"""The expert blob layout, checked on the host with no GPU. The library repacks
canonical weights with moe_repack_expert. A decoder written here from the
layout's definition maps every blob byte back to its canonical tensor, row and
byte. The result must reproduce the canonical weights exactly, with every
byte of the blob read at most once and every unread byte zero.

Layout (one expert, sections 256-byte aligned, blob 1024-byte aligned):
  * K order within each weight row: per 128-element group, device position
    32q + 4s + i holds element 16s + 4q + i (s < 8, q < 4, i < 4).
  * FP32: gate [I,H], up [I,H], down [H,I] as given.
  * BF16: gate/up rows in blocks of 128 device rows, gate row u at
    128*(u // 64) + u % 64 and its up row 64 further; down rows in order.
  * NVFP4 / MXFP4: 16-row tiles. A gate/up tile t holds the gate rows of
    units 8t..8t+7 (tile rows 0-7) and their up rows (tile rows 8-15); down
    tile t holds rows 16t..16t+15. A tile is a run of chunks of up to 8
    groups, each chunk codes[16][ng*64 B] then scales[16][ng*sb B] (sb = 8
    NVFP4, 4 MXFP4). The 16-byte quarter q of group w of row r sits at
    r*ng*64 + 16*((4w + q) ^ x), with x = 4 for odd r when ng is even, else 0.
    The device K order on FP4 codes: byte 16q + 2s + b of a group's 64 bytes
    holds canonical byte 8s + 2q + b.
  * FP8: the same 16-row tiles of chunks of up to 8 groups, each chunk
    codes[16][ng*128 B] (one E4M3 byte per element, no block scales). Half
    hf of the 32-byte run of quad q of group w of row r sits at
    (r*ng + w)*128 + 16*((2q + hf) ^ (r & 1)); within a group the bytes are in
    the device K order above.
  * Then 4 fp32: the NVFP4 / FP8 per-tensor scales of gate, up, down and 1.0
    (all 1.0 for the other formats)."""
import numpy as np
import pytest

import expert_offload_softmax_b300 as moe
import synth


def _a(x, m):
    return (x + m - 1) // m * m


class Reader:
    def __init__(self, blob):
        self.blob = blob
        self.hits = np.zeros(blob.size, np.int32)

    def take(self, off, n):
        self.hits[off:off + n] += 1
        return self.blob[off:off + n]


def _canon_from_device_k(dev, elem_bytes):
    """Undo the device K order of one row (elements of elem_bytes bytes)."""
    K = dev.size
    out = np.empty_like(dev)
    j, p = np.divmod(np.arange(K), 128)
    q, rem = np.divmod(p, 32)
    s, i = np.divmod(rem, 4)
    out[j * 128 + 16 * s + 4 * q + i] = dev
    return out


def _fp4_row(rd, tile, r, K, sb):
    """Canonical codes (K/2 bytes) and scales (K/128*sb bytes) of tile row r."""
    G = K // 128
    dev = np.empty(K // 2, np.uint8)
    scales = np.empty(G * sb, np.uint8)
    for c in range((G + 7) // 8):
        ng = min(8, G - 8 * c)
        chunk = tile + 16 * 8 * c * (64 + sb)
        x = 4 if (r & 1) and ng % 2 == 0 else 0
        for w in range(ng):
            j = 8 * c + w
            for q in range(4):
                dev[64 * j + 16 * q:64 * j + 16 * q + 16] = rd.take(chunk + r * ng * 64 + 16 * ((4 * w + q) ^ x), 16)
            scales[j * sb:(j + 1) * sb] = rd.take(chunk + 16 * ng * 64 + r * ng * sb + w * sb, sb)
    canon = np.empty_like(dev)
    for j in range(G):
        for q in range(4):
            for s in range(8):
                for b in range(2):
                    canon[64 * j + 8 * s + 2 * q + b] = dev[64 * j + 16 * q + 2 * s + b]
    return canon, scales


def _fp8_row(rd, tile, r, K):
    """Canonical E4M3 codes (K bytes) of tile row r."""
    G = K // 128
    dev = np.empty(K, np.uint8)
    for c in range((G + 7) // 8):
        ng = min(8, G - 8 * c)
        chunk = tile + 16 * 8 * c * 128
        for w in range(ng):
            j = 8 * c + w
            for q in range(4):
                for hf in range(2):
                    dev[128 * j + 32 * q + 16 * hf:128 * j + 32 * q + 16 * hf + 16] = \
                        rd.take(chunk + (r * ng + w) * 128 + 16 * ((2 * q + hf) ^ (r & 1)), 16)
    return _canon_from_device_k(dev, 1)


def _decode(fmt, H, I, blob):
    rd = Reader(blob)
    out = {"gate": {}, "up": {}, "down": {}}
    if fmt == synth.FMT_FP32:
        n = I * H * 4
        out["gate"]["data"] = rd.take(0, n).view(np.float32).reshape(I, H)
        out["up"]["data"] = rd.take(n, n).view(np.float32).reshape(I, H)
        d = _a(2 * n, 256)
        out["down"]["data"] = rd.take(d, n).view(np.float32).reshape(H, I)
        gsc = _a(d + n, 256)
    elif fmt == synth.FMT_BF16:
        g = np.empty((I, H), np.uint16)
        u = np.empty((I, H), np.uint16)
        for row in range(I):
            for which, dst in ((0, g), (1, u)):
                dr = 128 * (row // 64) + 64 * which + row % 64
                dst[row] = _canon_from_device_k(rd.take(dr * H * 2, H * 2).view(np.uint16), 2)
        d = _a(2 * I * H * 2, 256)
        dn = np.empty((H, I), np.uint16)
        for row in range(H):
            dn[row] = _canon_from_device_k(rd.take(d + row * I * 2, I * 2).view(np.uint16), 2)
        out["gate"]["data"], out["up"]["data"], out["down"]["data"] = g, u, dn
        gsc = _a(d + H * I * 2, 256)
    elif fmt == synth.FMT_FP8:
        gu_tile, d_tile = 16 * H, 16 * I
        for name in ("gate", "up"):
            out[name]["codes"] = np.empty((I, H), np.uint8)
        for unit in range(I):
            for which, name in ((0, "gate"), (1, "up")):
                out[name]["codes"][unit] = _fp8_row(rd, (unit // 8) * gu_tile, 8 * which + unit % 8, H)
        d = _a((I // 8) * gu_tile, 256)
        out["down"]["codes"] = np.empty((H, I), np.uint8)
        for row in range(H):
            out["down"]["codes"][row] = _fp8_row(rd, d + (row // 16) * d_tile, row % 16, I)
        gsc = _a(d + (H // 16) * d_tile, 256)
    else:
        sb = 8 if fmt == synth.FMT_NVFP4 else 4
        gu_tile = 16 * (H // 128) * (64 + sb)
        d_tile = 16 * (I // 128) * (64 + sb)
        for name in ("gate", "up"):
            out[name]["codes"] = np.empty((I, H // 2), np.uint8)
            out[name]["scales"] = np.empty((I, H // 128 * sb), np.uint8)
        for unit in range(I):
            for which, name in ((0, "gate"), (1, "up")):
                c, s = _fp4_row(rd, (unit // 8) * gu_tile, 8 * which + unit % 8, H, sb)
                out[name]["codes"][unit], out[name]["scales"][unit] = c, s
        d = _a((I // 8) * gu_tile, 256)
        out["down"]["codes"] = np.empty((H, I // 2), np.uint8)
        out["down"]["scales"] = np.empty((H, I // 128 * sb), np.uint8)
        for row in range(H):
            c, s = _fp4_row(rd, d + (row // 16) * d_tile, row % 16, I, sb)
            out["down"]["codes"][row], out["down"]["scales"][row] = c, s
        gsc = _a(d + (H // 16) * d_tile, 256)
    out["gsc"] = rd.take(gsc, 16).view(np.float32).copy()
    assert blob.size == _a(gsc + 16, 1024)
    return out, rd.hits


@pytest.mark.parametrize("fmt,H,I", [
    (synth.FMT_FP32, 64, 32),
    (synth.FMT_BF16, 256, 128),
    (synth.FMT_NVFP4, 1152, 256),   # gate/up rows: a full 8-group chunk and a 1-group chunk
    (synth.FMT_MXFP4, 1152, 384),   # down rows: one 3-group chunk (odd ng: no swizzle)
    (synth.FMT_NVFP4, 256, 1152),
    (synth.FMT_FP8, 1152, 384),     # gate/up: an 8-group and a 1-group chunk; down: one 3-group chunk
])
def test_repacked_blob_decodes_to_the_canonical_weights(fmt, H, I):
    act = synth.ACT_FP32 if fmt == synth.FMT_FP32 else synth.ACT_BF16
    shape = synth.Shape("layout", L=1, E=4, k=2, H=H, I=I, fmt=fmt, act=act)
    w = synth.expert_weights(shape, 5, 0, 3)
    desc = moe.make_desc(1, 4, 2, H, I, fmt, act)
    blob = moe.moe_repack_expert(desc, w)
    assert blob.size == moe.moe_expert_bytes(desc)
    got, hits = _decode(fmt, H, I, blob)
    assert hits.max() == 1                      # no byte belongs to two places
    assert not blob[hits == 0].any()            # everything else is zero padding
    for name in ("gate", "up", "down"):
        for key in ("data", "codes", "scales"):
            if key in w[name]:
                np.testing.assert_array_equal(got[name][key], np.asarray(w[name][key]).reshape(got[name][key].shape))
    want = [1.0, 1.0, 1.0, 1.0]
    if fmt in (synth.FMT_NVFP4, synth.FMT_FP8):
        want = [w["gate"]["gscale"], w["up"]["gscale"], w["down"]["gscale"], 1.0]
    np.testing.assert_array_equal(got["gsc"], np.array(want, np.float32))


def test_repack_rejects_a_short_buffer():
    import ctypes
    shape = synth.Shape("layout", L=1, E=4, k=2, H=256, I=128, fmt=synth.FMT_MXFP4, act=synth.ACT_BF16)
    w = synth.expert_weights(shape, 5, 0, 0)
    desc = moe.make_desc(1, 4, 2, 256, 128, synth.FMT_MXFP4, synth.ACT_BF16)
    n = moe.moe_expert_bytes(desc)
    g, kg = moe._tensor(w["gate"])
    u, ku = moe._tensor(w["up"])
    d, kd = moe._tensor(w["down"])
    eh = moe.moe_expert_host(g, u, d)
    buf = np.zeros(n, np.uint8)
    assert moe.load().moe_repack_expert(ctypes.byref(desc), ctypes.byref(eh), buf.ctypes.data, n - 1) == moe.MOE_ERR_INVALID
    assert moe.load().moe_repack_expert(ctypes.byref(desc), ctypes.byref(eh), buf.ctypes.data, n) == moe.MOE_OK
    del kg, ku, kd
