"""Oracle: the packed weight layout (test infrastructure only).

The method packs the static weights once at load time into the layout the
matrix instruction reads, so that each lane's (here: each pipeline stage's)
slice is contiguous, and keeps the packed buffer at a fixed address for graph
replay ("Real-time VLA inference on AMD hardware", section "Packing around
the instruction").  The pages' map is for the CDNA3 MFMA; the layout here is
the one the GB300 kernels read, restated as a reshape/transpose in the same
style:

  * W is logical [K x N] (column n = output channel).  Packing stores W^T:
    one row of K elements per channel n, K contiguous, as bytes (1 byte per
    E4M3 element, 2 little-endian bytes per bf16 element).
  * Rows are padded with zeros to NB = ceil(N/128) groups of 128 channels,
    the K bytes to KB = ceil(K*esize/128) blocks of 128 bytes.
  * Tile (nb, kb) -- 128 channels x 128 bytes, 16 KiB -- sits at byte
    offset (nb * KB + kb) * 16384; channel r of the tile owns bytes
    [r * 128, r * 128 + 128) of it.
  * Inside a row, the 16-byte chunk c of the 128 K-bytes is stored at chunk
    position c XOR (r mod 8) (the 128-byte swizzle of the shared-memory
    operand), so a tile copied byte for byte into 1024-byte-aligned shared
    memory is already in the tensor core's swizzled K-major form.

The bf16 packing of fp32 weights rounds each weight to the nearest bf16 (ties
to even) first.
"""
import numpy as np

from . import bf16

TILE_ROWS = 128
TILE_BYTES = 128


def esize_of(kind):
    return {"e4m3": 1, "bf16": 2}[kind]


def packed_bytes(K, N, kind):
    """Size in bytes of the packed buffer of a K x N weight."""
    nb = -(-N // TILE_ROWS)
    kb = -(-(K * esize_of(kind)) // TILE_BYTES)
    return nb * kb * TILE_ROWS * TILE_BYTES


def _row_bytes(w, kind):
    """[K x N] element array -> [N x K*esize] byte array of W^T."""
    if kind == "e4m3":
        wt = np.ascontiguousarray(np.asarray(w, dtype=np.uint8).T)
        return wt
    wt = np.ascontiguousarray(np.asarray(w, dtype=np.uint16).T).astype("<u2")
    return wt.view(np.uint8).reshape(wt.shape[0], wt.shape[1] * 2)


def _swizzle_index():
    r = np.arange(TILE_ROWS)[:, None]
    c = np.arange(TILE_BYTES // 16)[None, :]
    return c ^ (r & 7)  # [128, 8]


def pack(w, kind):
    """Pack a [K x N] weight given as E4M3 bytes (kind 'e4m3', uint8) or bf16
    bit patterns (kind 'bf16', uint16) -> flat uint8 packed buffer."""
    w = np.asarray(w)
    K, N = w.shape
    es = esize_of(kind)
    nb = -(-N // TILE_ROWS)
    kb = -(-(K * es) // TILE_BYTES)
    rows = np.zeros((nb * TILE_ROWS, kb * TILE_BYTES), dtype=np.uint8)
    rows[:N, : K * es] = _row_bytes(w, kind)
    t = rows.reshape(nb, TILE_ROWS, kb, TILE_BYTES // 16, 16).transpose(0, 2, 1, 3, 4)
    # stored chunk p of row r holds logical chunk p XOR (r & 7)
    idx = _swizzle_index()[None, None, :, :, None]
    out = np.take_along_axis(t, np.broadcast_to(idx, t.shape), axis=3)
    return np.ascontiguousarray(out).reshape(-1)


def unpack(packed, K, N, kind):
    """Inverse of :func:`pack`: flat packed bytes -> [K x N] elements."""
    es = esize_of(kind)
    nb = -(-N // TILE_ROWS)
    kb = -(-(K * es) // TILE_BYTES)
    t = np.asarray(packed, dtype=np.uint8).reshape(nb, kb, TILE_ROWS, TILE_BYTES // 16, 16)
    idx = _swizzle_index()[None, None, :, :, None]  # logical chunk c is at c XOR (r & 7)
    logical = np.take_along_axis(t, np.broadcast_to(idx, t.shape), axis=3)
    rows = logical.transpose(0, 2, 1, 3, 4).reshape(nb * TILE_ROWS, kb * TILE_BYTES)
    rb = np.ascontiguousarray(rows[:N, : K * es])
    if kind == "e4m3":
        return np.ascontiguousarray(rb.T)
    return np.ascontiguousarray(rb.view("<u2").reshape(N, K).T).astype(np.uint16)


def pack_fp32_as_bf16(w_f32):
    """bf16 packing of fp32 weights: RNE to bf16, then :func:`pack`."""
    return pack(bf16.f32_to_bf16_bits(w_f32), "bf16")
