"""Chunks of the fp32 bit patterns for the exhaustive check of the router's
deterministic sigmoid, and the oracle's digest of one chunk.  Imports numpy and
the oracle only, so pool workers started with 'spawn' stay light."""
import hashlib

import numpy as np

import oracle

CHUNK = 1 << 23
_SUB = 1 << 18  # sub-chunk that keeps the oracle's temporaries in cache


def finite_chunks():
    """(first bit pattern, count) covering every finite fp32 value: 0x00000000 up to
    0x7F7FFFFF (+0, subnormals, normals up to the largest finite) and the same range
    with the sign bit set; infinities and NaNs are left out."""
    top = 0x7F800000  # first non-finite pattern of each sign
    out = []
    for base in (0, 0x80000000):
        for s in range(0, top, CHUNK):
            out.append((base + s, min(CHUNK, top - s)))
    return out


def oracle_chunk(start, n):
    z = np.arange(start, start + n, dtype=np.uint64).astype(np.uint32).view(np.float32)
    s = np.empty(n, dtype=np.float32)
    for i in range(0, n, _SUB):
        s[i:i + _SUB] = oracle.sigmoid_det_f32(z[i:i + _SUB])
    return s


def oracle_chunk_digest(start, n):
    return hashlib.sha256(oracle_chunk(start, n).view(np.uint8)).hexdigest()
