"""Helpers for the GPU parity tests: strided device buffers with canaries.

Every output buffer is allocated with padding columns after each row, a
spare row above and below, and filled with a canary; after a call the
padding must still hold the canary (nothing written outside the output).
Source buffers can be given an arbitrary row pitch and a byte offset, so
that unaligned pointers and odd pitches take the library's non-bulk paths.
"""
import numpy as np
import torch

U8_CANARY = 0xA5
F32_CANARY = -12345.5


def device_image(img: np.ndarray, pitch_elems: int | None = None, offset_elems: int = 0, dev="cuda"):
    """Copy an (H, W, C) array to the GPU with the given row pitch and start offset (in elements)."""
    if img.ndim == 2:
        img = img[:, :, None]
    H, W, C = img.shape
    pitch = W * C if pitch_elems is None else pitch_elems
    assert pitch >= W * C
    flat = torch.zeros(offset_elems + H * pitch + 16, dtype=torch.from_numpy(img[:1, :1, :1].copy()).dtype, device=dev)
    view = torch.as_strided(flat, (H, W, C), (pitch, C, 1), offset_elems)
    view.copy_(torch.from_numpy(np.ascontiguousarray(img)).to(dev))
    return view, flat


class Canvas:
    """An (OH, OW, C) output view inside a canary-filled buffer."""

    def __init__(self, OH, OW, C, dtype, pad_elems=0, offset_elems=0, dev="cuda"):
        self.OH, self.OW, self.C = OH, OW, C
        self.pitch = OW * C + pad_elems
        self.off = offset_elems + self.pitch        # one spare row in front
        self.n = self.off + (OH + 1) * self.pitch + 8
        canary = U8_CANARY if dtype == torch.uint8 else F32_CANARY
        self.canary = canary
        self.flat = torch.full((self.n,), canary, dtype=dtype, device=dev)
        self.view = torch.as_strided(self.flat, (OH, OW, C), (self.pitch, C, 1), self.off)

    def result(self) -> np.ndarray:
        return self.view.cpu().numpy()

    def check_canary(self):
        flat = self.flat.cpu().numpy().copy()
        mask = np.ones(self.n, bool)
        idx = (self.off + np.arange(self.OH)[:, None] * self.pitch + np.arange(self.OW * self.C)[None, :]).ravel()
        mask[idx] = False
        outside = flat[mask]
        assert np.all(outside == np.array(self.canary, flat.dtype)), \
            f"{int((outside != np.array(self.canary, flat.dtype)).sum())} bytes written outside the output"


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0
