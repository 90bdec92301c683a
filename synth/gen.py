"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no arithmetic of the decode step itself: it only produces
weights, token ids and test vectors from a counter-based generator, so that a
host (numpy) copy and a device (CUDA, ``synth/csrc/synth_gen.cu``) copy of the
same tensor are bit-identical.

Generator (written from the published SplitMix64 definition: Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014, and
Vigna's public-domain splitmix64 reference):

* ``mix64(z)``: the SplitMix64 output function (xor-shift 30, multiply,
  xor-shift 27, multiply, xor-shift 31).
* a tensor's stream key is ``mix64(seed * GOLDEN + tensor_id)``; its i-th
  64-bit word is ``mix64(key + (i + 1) * GOLDEN)`` (all mod 2**64), i.e. the
  i-th SplitMix64 output of a generator seeded with ``key``.

Derived values:

* ``normal_bf16``: the four 16-bit fields of a word are summed (Irwin-Hall of
  four uniforms, an exact integer in [0, 262140]), centred by subtracting
  131070, converted exactly to float32, multiplied once by the float32
  constant ``std / sigma_IH`` (sigma_IH = sqrt((65536**2 - 1) / 3)), then
  rounded to bfloat16 with round-to-nearest-even.  Every step is exact or a
  single IEEE rounding, so numpy and CUDA agree bit for bit.
* ``q4_packed``: byte i of a packed 4-bit tensor is byte (i mod 8) of word
  (i div 8); its nibbles are therefore uniform in 0..15 (values -8..7 after
  the +8 offset is removed).
* ``q4_scales``: scale = fp16_rne(float32(u16 + 49152) * float32(s0 / 65536))
  with u16 the low 16 bits of the word, so scales lie in [0.75, 1.75) * s0.
* ``uniform_ids``: ((word >> 32) * n) >> 32, an exact integer in [0, n).
"""
from __future__ import annotations

import math

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1

# standard deviation of the sum of four independent uniforms on {0..65535}
IH_SIGMA = math.sqrt((65536.0 ** 2 - 1.0) / 3.0)
IH_MEAN = 131070


def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (mod 2**64)."""
    z &= _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(_M1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int) -> int:
    return mix64_int((seed * GOLDEN + tensor_id) & _MASK)


def words(seed: int, tensor_id: int, start: int, n: int) -> np.ndarray:
    """Words ``start .. start+n-1`` of the tensor's stream (uint64)."""
    key = np.uint64(stream_key(seed, tensor_id))
    i = np.arange(start, start + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64_np(key + (i + np.uint64(1)) * np.uint64(GOLDEN))


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits, round to nearest even (inputs are finite)."""
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_scale_f32(std: float) -> np.float32:
    """The single float32 multiplier shared by host and device generators."""
    return np.float32(std / IH_SIGMA)


def normal_bf16(seed: int, tensor_id: int, n: int, std: float = 0.02, start: int = 0) -> np.ndarray:
    """``n`` bfloat16 (as uint16 bits) approximately N(0, std**2)."""
    w = words(seed, tensor_id, start, n)
    m = np.uint64(0xFFFF)
    s = (w & m) + ((w >> np.uint64(16)) & m) + ((w >> np.uint64(32)) & m) + (w >> np.uint64(48))
    centred = (s.astype(np.int64) - IH_MEAN).astype(np.float32)
    return f32_to_bf16_bits(centred * normal_scale_f32(std))


def q4_packed(seed: int, tensor_id: int, nbytes: int) -> np.ndarray:
    """Packed nibble bytes (uint8) of a 4-bit tensor."""
    nw = (nbytes + 7) // 8
    w = words(seed, tensor_id, 0, nw)
    return w.view(np.uint8)[:nbytes].copy()


Q4_SCALE_TID_OFFSET = 0x40000000


def q4_scale_mult_f32(s0: float) -> np.float32:
    return np.float32(s0 / 65536.0)


def q4_scales(seed: int, tensor_id: int, nblocks: int, s0: float) -> np.ndarray:
    """fp16 scales (as uint16 bits) of a 4-bit tensor, in [0.75, 1.75) * s0."""
    w = words(seed, tensor_id + Q4_SCALE_TID_OFFSET, 0, nblocks)
    u = (w & np.uint64(0xFFFF)).astype(np.int64) + 49152
    f = u.astype(np.float32) * q4_scale_mult_f32(s0)
    return f.astype(np.float16).view(np.uint16)


def uniform_ids(seed: int, tensor_id: int, n: int, upper: int, start: int = 0) -> np.ndarray:
    """``n`` integers uniform in [0, upper) (int32)."""
    w = words(seed, tensor_id, start, n)
    return (((w >> np.uint64(32)) * np.uint64(upper)) >> np.uint64(32)).astype(np.int32)


# scale s0 of the 4-bit weights: the RMS of a value uniform on {-8..7} is
# sqrt(21.25 + 0.25) ~ 4.637 and the mean scale is 1.25 * s0, so this s0 gives
# dequantised weights with RMS ~0.02, like the bfloat16 configurations
Q4_STD_NIBBLE = math.sqrt(((16 ** 2) - 1) / 12.0 + 0.25)
Q4_S0 = 0.02 / (1.25 * Q4_STD_NIBBLE)


# ------------------------------------------------------ synthetic cache state
# The generator behind hy_seq_fill_synthetic (a long context without replaying
# its prompt): value i of the stream keyed by `key` takes the word
# z = mix64(key + (i + 1) * GOLDEN), keeps its top 24 bits and maps them to
# (float32(z >> 40) * 2**-23 - 1) * scale, uniform in [-1, 1) * scale.  Every
# float32 step is exact but the last multiply, one IEEE rounding.

def fill_values(key: int, n: int, scale: float = 1.0) -> np.ndarray:
    """Values 0 .. n-1 (float32) of the cache-fill stream keyed by ``key``."""
    i = np.arange(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _mix64_np(np.uint64(key & _MASK) + (i + np.uint64(1)) * np.uint64(GOLDEN))
    u = (z >> np.uint64(40)).astype(np.float32)
    return (u * np.float32(2.0 ** -23) - np.float32(1.0)) * np.float32(scale)
