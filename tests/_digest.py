"""Per-chunk digests of the oracle's element converters over every float32
bit pattern, for the exhaustive GPU converter test (the library's test hook
computes the same digests from the kernels' converters on the device).

A chunk is 2^20 consecutive bit patterns. Its digest, one per converter, is
the sum modulo 2^64 of SplitMix64(key XOR salt) over the chunk's finite
inputs, key = (pattern << 32) | result: the E2M1 code (salt 1) and the
specified exponential's float bits (salt 3) of every finite input, the E4M3
scale code (salt 2) of +0 and every positive finite input. Equal digests
mean equal results up to a 2^-64 chance per chunk; the functions here are
test infrastructure only.
"""
import numpy as np

from oracle import nvfp4_moe_oracle as O

CHUNK_BITS = 20
SALTS = (np.uint64(0x243F6A8885A308D3), np.uint64(0x13198A2E03707344), np.uint64(0xA4093822299F31D0))


def splitmix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable
    pseudorandom number generators", 2014), uint64 arithmetic modulo 2^64."""
    z = z + np.uint64(0x9E3779B97F4A7C15)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def _digest(bits: np.ndarray, result: np.ndarray, salt) -> int:
    key = (bits.astype(np.uint64) << np.uint64(32)) | result.astype(np.uint64)
    return int(np.sum(splitmix64(key ^ salt), dtype=np.uint64))


def chunk_digests(chunks):
    """Digests (e2m1, e4m3, exp) of the oracle over each chunk index given."""
    out = []
    with np.errstate(over="ignore", invalid="ignore"):
        for c in chunks:
            b = np.arange(c << CHUNK_BITS, (c + 1) << CHUNK_BITS, dtype=np.uint64).astype(np.uint32)
            f = b.view(np.float32)
            fin = np.isfinite(f)
            bf, ff = b[fin], f[fin]
            pos = (ff > 0) | (bf == 0)
            out.append((_digest(bf, O.e2m1_rn(ff), SALTS[0]),
                        _digest(bf[pos], O.e4m3_rn_satfinite(ff[pos]), SALTS[1]),
                        _digest(bf, O.exp_spec(ff).view(np.uint32), SALTS[2])))
    return out
