"""Per-token dynamic int8 activation quantization (oracle).

[CAS-blog] §2.1 item 3 and §2.2 (levels L2, L3) and the [CAS-paper] abstract
name 8-bit activation quantization as one of the switchable acceleration
strategies of a draft.  The pages give no formula; the plain reading used
here: symmetric, one scale per token (row), no zero point, codes in
[-127, 127]:

    amax = max_k |x_k|
    s    = amax / 127
    q_k  = clamp(round_half_even(x_k * (127 / amax)), -127, 127)
    x^_k = s * q_k                  (amax == 0  =>  x^ = 0)

The codes are an integer decision taken from floating point, so they are
computed in float32, the precision the GPU kernels use: x is rounded to
float32, 127/amax and amax/127 are IEEE float32 divisions, the product
x * (127/amax) is a float32 multiply, and rounding is half-to-even.
"""
import numpy as np

_F127 = np.float32(127.0)


def quantize_rows(x: np.ndarray):
    """Return (codes int32 [R, n], scale float32 [R]) for x [R, n]."""
    xf = np.asarray(x, dtype=np.float64).astype(np.float32)
    if xf.ndim == 1:
        xf = xf[None, :]
    amax = np.max(np.abs(xf), axis=1)
    codes = np.zeros(xf.shape, dtype=np.int32)
    scale = np.zeros(xf.shape[0], dtype=np.float32)
    for r in range(xf.shape[0]):
        if amax[r] == np.float32(0.0):
            continue
        inv = np.float32(_F127 / amax[r])
        prod = (xf[r] * inv).astype(np.float32)
        codes[r] = np.clip(np.rint(prod), -127, 127).astype(np.int32)
        scale[r] = np.float32(amax[r] / _F127)
    return codes, scale


def fake_quant_rows(x: np.ndarray) -> np.ndarray:
    """x^ = s * q per row, as float64 (the product of two float32 values is exact in float64)."""
    codes, scale = quantize_rows(x)
    out = codes.astype(np.float64) * scale.astype(np.float64)[:, None]
    return out.reshape(np.shape(x))
