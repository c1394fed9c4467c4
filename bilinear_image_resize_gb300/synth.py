"""Seeded synthetic images for the resize workloads.

This module only draws pixels; it contains none of the resize arithmetic, so
both the CUDA library's callers and the CPU oracle's tests can use it.

Workloads (W x H, interleaved HWC):
  * ``tiny_gray``      u8, 1 channel, 64x48, i.i.d. uniform [0, 255], seed 0.
  * ``smooth_rgb``     u8 RGB, sum of 8 random 2-D sinusoids per channel around
                       128 (amplitudes U(8, 32), spatial frequencies
                       U(-1/64, 1/64) cycles/pixel, phases U(0, 2 pi)) plus
                       integer noise U{-16..16}, clipped to [0, 255]; 1920x1080
                       uses seed 2, 3840x2160 uses seed 3.
  * ``frames_rgb``     a batch of u8 RGB frames, i.i.d. uniform, seed 4
                       (64 frames of 1280x720 for the normalise workload).
  * ``float_gray``     f32, 1 channel, values uniform in [0, 255), seed 5
                       (8192x8192 for the filter workload).
  * ``filter_weights`` nine f32 weights, uniform [0, 1), normalised to sum 1
                       in float64 and then rounded to f32, seed 55.
"""
from __future__ import annotations

import functools

import numpy as np

# Per-channel normalisation constants of the batched workload.
NORM_MEAN = (0.485, 0.456, 0.406)
NORM_STD = (0.229, 0.224, 0.225)


@functools.lru_cache(maxsize=4)
def tiny_gray(seed: int = 0, w: int = 64, h: int = 48) -> np.ndarray:
    rng = np.random.default_rng(seed)
    img = rng.integers(0, 256, size=(h, w), dtype=np.uint8)
    img.setflags(write=False)
    return img


@functools.lru_cache(maxsize=4)
def smooth_rgb(w: int, h: int, seed: int) -> np.ndarray:
    """(h, w, 3) u8 smooth content; separable evaluation of each sinusoid."""
    rng = np.random.default_rng(seed)
    xs = np.arange(w, dtype=np.float64)
    ys = np.arange(h, dtype=np.float64)
    out = np.empty((h, w, 3), dtype=np.uint8)
    for c in range(3):
        acc = np.full((h, w), 128.0)
        for _ in range(8):
            amp = rng.uniform(8.0, 32.0)
            fx = rng.uniform(-1.0 / 64, 1.0 / 64)
            fy = rng.uniform(-1.0 / 64, 1.0 / 64)
            ph = rng.uniform(0.0, 2.0 * np.pi)
            ax = 2.0 * np.pi * fx * xs + ph
            ay = 2.0 * np.pi * fy * ys
            # sin(ax + ay) = sin(ax)cos(ay) + cos(ax)sin(ay)
            acc += amp * (np.outer(np.cos(ay), np.sin(ax)) + np.outer(np.sin(ay), np.cos(ax)))
        acc += rng.integers(-16, 17, size=(h, w))
        out[:, :, c] = np.clip(np.rint(acc), 0, 255).astype(np.uint8)
    out.setflags(write=False)
    return out


@functools.lru_cache(maxsize=2)
def frames_rgb(n: int = 64, w: int = 1280, h: int = 720, seed: int = 4) -> np.ndarray:
    rng = np.random.default_rng(seed)
    img = rng.integers(0, 256, size=(n, h, w, 3), dtype=np.uint8)
    img.setflags(write=False)
    return img


@functools.lru_cache(maxsize=2)
def float_gray(w: int = 8192, h: int = 8192, seed: int = 5) -> np.ndarray:
    rng = np.random.default_rng(seed)
    img = (rng.random((h, w), dtype=np.float64) * 255.0).astype(np.float32)
    img.setflags(write=False)
    return img


def filter_weights(seed: int = 55) -> np.ndarray:
    w = np.random.default_rng(seed).random(9)
    return (w / w.sum()).astype(np.float32)


def filter_weights_k(K: int, seed: int = 56) -> np.ndarray:
    """K x K positive weights summing to 1 (float32), the K x K analogue of filter_weights."""
    w = np.random.default_rng(seed + K).random((K, K))
    return (w / w.sum()).astype(np.float32)


def random_u8(shape, seed: int) -> np.ndarray:
    return np.random.default_rng(seed).integers(0, 256, size=shape, dtype=np.uint8)


def random_f32(shape, seed: int, scale: float = 255.0) -> np.ndarray:
    return (np.random.default_rng(seed).random(shape) * scale).astype(np.float32)
