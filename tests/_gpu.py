"""Helpers of the GPU parity tests: device pools in the library's layout with
the same bits mirrored in the oracle's layout, and the comparison rules.

Tolerance (spec reading): verbatim parts and every byte the method
does not compute must be bit-exact; rotated and patched values must be
within 1 bf16 ulp of the oracle's fp64-rounded value (ordered-bit distance
<= 1), with an absolute floor of 1e-6 for results that cancel to near zero.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import position_independent_mla_gb300 as kv
import synth

SHAPES = {
    # name: (copy_dim, rot_heads, rot_head_dim, rope_base)
    "mla": (512, 1, 64, 10000.0),
    "gqa": (1024, 8, 128, 500000.0),
    "gqa4": (512, 4, 128, 1000000.0),
    "mha": (4096, 32, 128, 10000.0),
}


class DevPool:
    """A paged pool on the GPU (MLA: one fused [L][slots][576] tensor; GQA:
    separate V and K tensors) plus its oracle mirror."""

    def __init__(self, shape: str, L: int, slots: int, seed: int, block: int = 64,
                 pair_convention: int = 0):
        cd, H, d, base = SHAPES[shape]
        self.shape, self.cd, self.H, self.d, self.base, self.block = shape, cd, H, d, base, block
        copy = synth.bf16_normal((L, slots, cd), seed)
        rot = synth.bf16_normal((L, slots, H * d), seed + 1)
        if shape == "mla":
            self.fused = torch.cat([copy, rot], -1).cuda()
            self.copy_view = self.fused[..., :cd]
            self.rot_view = self.fused[..., cd:]
        else:
            self.copy_view = copy.cuda()
            self.rot_view = rot.cuda()
        self.desc = kv.pool_desc(self.copy_view, self.rot_view, block, H, base, pair_convention)
        self.orc = O.Pool(synth.bits(copy).copy(), synth.bits(rot).copy(), block, H, d, base,
                          pair_convention)

    def gpu_bits(self):
        torch.cuda.synchronize()
        return synth.bits(self.copy_view.cpu()), synth.bits(self.rot_view.cpu())


def ordered(b: np.ndarray) -> np.ndarray:
    b = b.astype(np.int64)
    return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_exact(gpu: np.ndarray, ref: np.ndarray, what: str) -> None:
    bad = np.argwhere(gpu != ref)
    assert len(bad) == 0, f"{what}: {len(bad)} values differ, first at {bad[:5].tolist()}"


def check_ulp(gpu: np.ndarray, ref: np.ndarray, what: str) -> dict:
    """<= 1 ulp (or |diff| <= 1e-6); NaN must meet NaN.  Returns statistics."""
    g, r = bf16_to_f64(gpu), bf16_to_f64(ref)
    nan_g, nan_r = np.isnan(g), np.isnan(r)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN pattern differs"
    fin = ~nan_r
    dist = np.abs(ordered(gpu) - ordered(ref))[fin]
    with np.errstate(invalid="ignore"):
        absd = np.abs(g - r)[fin]
    ok = (dist <= 1) | (absd <= 1e-6)
    n_bad = int((~ok).sum())
    assert n_bad == 0, f"{what}: {n_bad} values beyond 1 ulp (max dist {dist.max()})"
    return {"values": int(fin.sum()), "exact": int((dist == 0).sum()),
            "one_ulp": int((dist == 1).sum())}


def check_pool(dp: DevPool, what: str, rot_exact: bool = False, copy_exact: bool = True):
    gc, gr = dp.gpu_bits()
    if copy_exact:
        check_exact(gc, dp.orc.copy, what + " (verbatim part)")
    else:
        check_ulp(gc, dp.orc.copy, what + " (patched verbatim part)")
    if rot_exact:
        check_exact(gr, dp.orc.rot, what + " (rotary part)")
        return None
    return check_ulp(gr, dp.orc.rot, what + " (rotary part)")


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def i32(*v) -> torch.Tensor:
    return torch.tensor(v, dtype=torch.int32)


def resync(dp: DevPool) -> None:
    """Copy the GPU's current bits into the oracle mirror, so that the next
    operation is compared on identical inputs."""
    gc, gr = dp.gpu_bits()
    dp.orc.copy[...] = gc
    dp.orc.rot[...] = gr
