"""Test-side helpers: layout conversions of library buffers and error norms.

These read the library's documented buffer layouts (include/moe.h) with
numpy index arithmetic of their own; they hold none of the layer's math.
"""
from __future__ import annotations

import numpy as np
import torch


def rel_frob(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def untile_scales(tiled, rows: int, K: int) -> np.ndarray:
    """Tiled scale bytes (512-byte atoms of 128 rows x 4 blocks) -> canonical [rows][K/32]."""
    t = np.asarray(tiled, dtype=np.uint8).reshape(-1)
    nb = K // 32
    r = np.arange(rows)[:, None]
    kb = np.arange(nb)[None, :]
    off = ((r // 128) * (K // 128) + kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    return t[off]


def tile_scales(canon, rows: int, K: int) -> np.ndarray:
    c = np.asarray(canon, dtype=np.uint8).reshape(rows, K // 32)
    out = np.zeros(rows * K // 32, np.uint8)
    r = np.arange(rows)[:, None]
    kb = np.arange(K // 32)[None, :]
    off = ((r // 128) * (K // 128) + kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    out[off] = c
    return out


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.uint8).numpy().copy()


def np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float32).numpy()


def np_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def bf16_tensor(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).to(device)


def gu_split(gu: np.ndarray, I: int) -> np.ndarray:
    """Saved g,u rows as [g | u]: the workspace keeps them interleaved per 32-column chunk
    (chunk j of a row holds g[32j..32j+31] then u[32j..32j+31])."""
    c = np.asarray(gu).reshape(gu.shape[0], I // 32, 2, 32)
    return np.concatenate([c[:, :, 0, :].reshape(gu.shape[0], I), c[:, :, 1, :].reshape(gu.shape[0], I)], axis=1)
