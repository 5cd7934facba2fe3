"""Seeded synthetic graphs and operands for the GIE zonal scatter.

This module only draws random inputs. It holds none of the scatter's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

The graphs stand in for the diamond-carbon frames that the deepmd-kit pull
request "fused Triton zonal scatter for the GIE head" measures (section
"Numbers": a 4096-atom frame with about 647k edges, C=32 radial channels), and
the 1000-atom / 158002-edge frames of the "SO(2) edge-cohort backward" pull
request. Those frames are not available; the generators reproduce their node
count, edge count, mean in-degree (about 158) and channel width.

Recipe (all draws from ``numpy.random.default_rng(seed)``, in this order):

1. per-source out-degrees (fixed, or Poisson(158) rescaled to sum exactly E);
2. destinations: uniform over the other N-1 nodes, or the Zipf recipe;
3. ``coup`` = U(-1, 1) of shape (E, 15), float32;
4. ``rad``  = N(0, 1) of shape (E, 3, C), float32;
5. ``grad_out`` = N(0, 1) of shape (N, 16, C), float32.

Sources are ascending, so destinations arrive unsorted.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

ROWS = 15            # zonal rows of the lmax=3 ladder (3 + 5 + 7)
SLOTS = 3            # radial slots, one per degree 1..3
D = 16               # padded node rows: scalar row + 15


@dataclasses.dataclass
class Workload:
    name: str
    N: int
    E: int
    C: int
    seed: int
    src: np.ndarray        # (E,) int32, ascending
    dst: np.ndarray        # (E,) int32
    coup: np.ndarray       # (E, 15) float32 ((E, D-1) for another ladder degree)
    rad: np.ndarray        # (E, 3, C) float32 ((E, lmax, C))
    grad_out: np.ndarray   # (N, 16, C) float32 ((N, D, C))

    def nbytes(self) -> int:
        return sum(a.nbytes for a in (self.dst, self.coup, self.rad, self.grad_out))


# name -> (N, E, degree model, destination model, seed)
CONFIGS = {
    "tiny": dict(N=64, E=2048, deg="fixed", dstm="uniform", seed=1),
    "n1000": dict(N=1000, E=158002, deg="poisson", dstm="uniform", seed=2),
    "n4096": dict(N=4096, E=647170, deg="poisson", dstm="uniform", seed=3),
    "zipf": dict(N=4096, E=647170, deg="poisson", dstm="zipf", seed=4),
    "large": dict(N=32768, E=5177344, deg="fixed", dstm="uniform", seed=5),
}
MEAN_DEGREE = 158
ZIPF_S = 1.1
ZIPF_EMPTY_FRACTION = 0.05


def poisson_degrees(rng: np.random.Generator, N: int, E: int, mean: float = MEAN_DEGREE) -> np.ndarray:
    """Poisson(mean) out-degrees rescaled to sum exactly to E.

    q_i = d_i * E / sum(d); take floor(q_i), then give +1 to the
    E - sum(floor) nodes with the largest fractional part (ties: lower index).
    """
    d = rng.poisson(mean, size=N).astype(np.float64)
    if d.sum() == 0:
        d[:] = 1.0
    q = d * (E / d.sum())
    fl = np.floor(q).astype(np.int64)
    short = int(E - fl.sum())
    frac = q - fl
    # stable sort on -frac keeps lower indices first among ties
    order = np.argsort(-frac, kind="stable")
    fl[order[:short]] += 1
    assert fl.sum() == E
    return fl


def fixed_degrees(N: int, E: int) -> np.ndarray:
    if E % N:
        raise ValueError("fixed degree model needs E divisible by N")
    return np.full(N, E // N, dtype=np.int64)


def uniform_dst(rng: np.random.Generator, src: np.ndarray, N: int) -> np.ndarray:
    """Uniform destination over the N-1 nodes other than the source."""
    u = rng.integers(0, N - 1, size=src.shape[0], dtype=np.int64)
    return (u + (u >= src)).astype(np.int32)


def zipf_dst(rng: np.random.Generator, src: np.ndarray, N: int,
             s: float = ZIPF_S, empty_fraction: float = ZIPF_EMPTY_FRACTION) -> np.ndarray:
    """Zipf(s) destinations over a random node permutation.

    The last ceil(empty_fraction*N) nodes of the permutation receive no edges.
    The others get weight (k+1)^-s by rank k; a destination is drawn by
    inverse CDF, and a draw equal to its source moves to the next rank
    (mod the number of eligible nodes).
    """
    perm = rng.permutation(N)
    n_empty = int(math.ceil(empty_fraction * N))
    M = N - n_empty
    w = (np.arange(M, dtype=np.float64) + 1.0) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = rng.random(size=src.shape[0])
    k = np.searchsorted(cdf, u, side="right")
    k = np.minimum(k, M - 1)
    d = perm[k]
    clash = d == src
    k = np.where(clash, (k + 1) % M, k)
    return perm[k].astype(np.int32)


def draw_operands(rng: np.random.Generator, N: int, E: int, C: int, lmax: int = 3):
    """coup (E, R) uniform(-1, 1), rad (E, lmax, C) and grad_out (N, D, C) standard
    normal, D = (lmax+1)^2, R = D - 1 (15 / 3 / 16 at lmax = 3)."""
    d = (lmax + 1) ** 2
    coup = (rng.random((E, d - 1), dtype=np.float32) * np.float32(2.0) - np.float32(1.0)).astype(np.float32)
    rad = rng.standard_normal((E, lmax, C), dtype=np.float32)
    grad_out = rng.standard_normal((N, d, C), dtype=np.float32)
    return coup, rad, grad_out


def make_workload(name: str, C: int = 32, seed: int | None = None, lmax: int = 3) -> Workload:
    """Build one of the named configurations (tiny, n1000, n4096, zipf, large);
    lmax picks the ladder of the operands (3: the pages' 3/5/7 rows)."""
    cfg = CONFIGS[name]
    N, E = cfg["N"], cfg["E"]
    rng = np.random.default_rng(cfg["seed"] if seed is None else seed)
    deg = poisson_degrees(rng, N, E) if cfg["deg"] == "poisson" else fixed_degrees(N, E)
    src = np.repeat(np.arange(N, dtype=np.int32), deg)
    if cfg["dstm"] == "zipf":
        dst = zipf_dst(rng, src, N)
    else:
        dst = uniform_dst(rng, src, N)
    coup, rad, grad_out = draw_operands(rng, N, E, C, lmax)
    return Workload(name, N, E, C, cfg["seed"] if seed is None else seed, src, dst, coup, rad, grad_out)


def make_random(N: int, E: int, C: int, seed: int, *, self_loops: bool = False,
                hot_node: int | None = None, hot_fraction: float = 0.0, lmax: int = 3) -> Workload:
    """Small ad-hoc graph: uniform destinations, optional self loops and a hot node.

    Used for edge cases (ragged sizes, odd channel counts, one heavy node,
    other ladder degrees lmax).
    """
    rng = np.random.default_rng(seed)
    src = np.sort(rng.integers(0, max(N, 1), size=E)).astype(np.int32) if N > 0 else np.zeros(E, np.int32)
    if N == 0:
        dst = np.zeros(E, np.int32)
    elif self_loops or N == 1:
        dst = rng.integers(0, N, size=E).astype(np.int32)
    else:
        dst = uniform_dst(rng, src, N)
    if hot_node is not None and E > 0:
        hot = rng.random(E) < hot_fraction
        dst = np.where(hot, np.int32(hot_node), dst).astype(np.int32)
    coup, rad, grad_out = draw_operands(rng, max(N, 0), E, C, lmax)
    tag = "" if lmax == 3 else f"_L{lmax}"
    return Workload(f"random_N{N}_E{E}_C{C}{tag}", N, E, C, seed, src, dst, coup, rad, grad_out)
