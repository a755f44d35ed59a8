"""Round-to-nearest-even conversion of fp64 values to bfloat16.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

bfloat16 keeps the fp32 exponent and 7 explicit significand bits.  The KV
cache and the weights are stored in it ("Build a Speculative Decoding Engine
...", *KV Cache Management for Dual Models*: the caches are bf16 tensors).
The rounding below works on the fp64 bit pattern: it drops the low 45 of the
52 fraction bits with round-half-to-even, which is exact for every value in
the bf16 normal range (all values these tests produce).
"""
import numpy as np

_DROP = 45                      # 52 fp64 fraction bits - 7 bf16 fraction bits
_HALF = np.uint64((1 << (_DROP - 1)) - 1)
_MASK = np.uint64(~((1 << _DROP) - 1) & 0xFFFFFFFFFFFFFFFF)


def round_bf16(x) -> np.ndarray:
    """Nearest bf16 value (ties to even), returned as fp64."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    bits = x.view(np.uint64)
    lsb = (bits >> np.uint64(_DROP)) & np.uint64(1)
    r = ((bits + _HALF + lsb) & _MASK).view(np.float64)
    tiny = (np.abs(x) < 2.0 ** -126) & (x != 0)
    if np.any(tiny):
        raise ValueError("value below the bf16 normal range")
    return r.reshape(np.shape(x))


def to_bits(x) -> np.ndarray:
    """bf16 bit patterns (uint16) of values that are already bf16-exact."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def from_bits(b) -> np.ndarray:
    """fp64 values of bf16 bit patterns."""
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)
