"""Parity bar shared by the GPU tests.

Per position (row): cosine(gpu, oracle) >= 0.99999 (the talker page's equality standard, cosine
to five nines plus a reported max|delta|) and max|delta| <= 5e-4 when the weights are stored f32,
<= 2e-3 * max|y| when they are stored bf16 (the oracle then uses the same bf16 values).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List

import numpy as np

COS_MIN = 0.99999
F32_ABS = 5e-4
BF16_REL = 2e-3


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


@dataclass
class Stats:
    worst_cos: float = 1.0
    worst_abs: float = 0.0
    worst_ratio: float = 0.0      # max|delta| / bound
    rows: int = 0
    notes: List[str] = field(default_factory=list)

    def line(self) -> str:
        return (f"rows={self.rows} worst_cos={self.worst_cos:.9f} "
                f"worst_max_abs={self.worst_abs:.3e} worst_abs/bound={self.worst_ratio:.3f}")


def check_rows(got: np.ndarray, want: np.ndarray, bf16: bool, stats: Stats = None,
               what: str = "") -> Stats:
    stats = stats or Stats()
    got = np.atleast_2d(np.asarray(got, np.float64))
    want = np.atleast_2d(np.asarray(want, np.float64))
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    for r in range(got.shape[0]):
        c = cosine(got[r], want[r])
        d = float(np.max(np.abs(got[r] - want[r])))
        bound = BF16_REL * float(np.max(np.abs(want[r]))) if bf16 else F32_ABS
        stats.rows += 1
        stats.worst_cos = min(stats.worst_cos, c)
        stats.worst_abs = max(stats.worst_abs, d)
        stats.worst_ratio = max(stats.worst_ratio, d / bound)
        assert c >= COS_MIN, f"{what} row {r}: cosine {c:.9f} < {COS_MIN}"
        assert d <= bound, f"{what} row {r}: max|delta| {d:.3e} > {bound:.3e}"
    return stats
