"""Seeded synthetic inputs: layer weight sets and token streams.

This module holds random-number generation, shapes and the data recipes only,
none of the FFN arithmetic.  The CUDA path (tests, benchmark) and the CPU oracle
both consume the arrays it returns, so both see identical, already-rounded
values.

Recipe (weights Gaussian with variance 1/fan-in, one bias channel):
  * tokens x in R^D: N(0,1) entries, except channel D-1 which is fixed to 1.0;
  * standard gate: W1, W3 in R^{H x D} with N(0, 1/D) entries, W2 in R^{D x H}
    with N(0, 1/H) entries; the bias column W1[:, D-1] holds the shift
    -Phi^{-1}(s), so a fraction ~(1-s) of ReLU gate units is live;
  * low-rank gate: V in R^{r x D} with N(0, 1/D) entries and U in R^{H' x r}
    with N(0, 1/r) entries; V's last column is e_{r-1} and V's last row is
    zero elsewhere, so t_{r-1} = (Vx)_{r-1} = x_{D-1} = 1 exactly; U's last
    column is the bias column and holds the shift;  W3 N(0,1/D), W2 N(0,1/H').
Values are drawn in float32 with numpy's PCG64 generator (platform independent)
and rounded once to the storage dtype (round-to-nearest-even for bfloat16).
Seeds: weights 1000*workload + set index, tokens 1000*workload + 500.
"""
from __future__ import annotations

import math
import statistics
from dataclasses import dataclass, field

import numpy as np
import torch

#: the shift the 90 %-sparsity workloads state literally
SHIFT_90 = -1.2816

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def shift_for_sparsity(s: float) -> float:
    """Bias that leaves a fraction ~(1-s) of gate units live: -Phi^{-1}(s)."""
    return -statistics.NormalDist().inv_cdf(s)


def _round(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Round a float32 array once to the storage dtype (RNE for bf16); CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DTYPES[dtype])


def _normal(rng, shape, std):
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(std)


@dataclass
class LayerWeights:
    """One layer's FFN weights as CPU tensors in the storage dtype, row-major.

    Standard gate: W1[H,D].  Low-rank gate: U[H,r], V[r,D] (W1 is None).
    Always: W3[H,D], W2[D,H].
    """
    D: int
    H: int
    r: int
    dtype: str
    W1: torch.Tensor | None
    U: torch.Tensor | None
    V: torch.Tensor | None
    W3: torch.Tensor
    W2: torch.Tensor
    meta: dict = field(default_factory=dict)

    def tensors(self):
        return {k: getattr(self, k) for k in ("W1", "U", "V", "W3", "W2")}


def standard_layer(D: int, H: int, *, dtype: str = "bf16", seed: int = 0,
                   shift: float = SHIFT_90) -> LayerWeights:
    rng = np.random.default_rng(seed)
    W1 = _normal(rng, (H, D), 1.0 / math.sqrt(D))
    W1[:, D - 1] = shift
    W3 = _normal(rng, (H, D), 1.0 / math.sqrt(D))
    W2 = _normal(rng, (D, H), 1.0 / math.sqrt(H))
    return LayerWeights(D, H, 0, dtype, _round(W1, dtype), None, None,
                        _round(W3, dtype), _round(W2, dtype),
                        {"seed": seed, "shift": shift})


def lopa_layer(D: int, Hp: int, r: int, *, dtype: str = "bf16", seed: int = 0,
               shift: float = SHIFT_90) -> LayerWeights:
    rng = np.random.default_rng(seed)
    V = _normal(rng, (r, D), 1.0 / math.sqrt(D))
    V[:, D - 1] = 0.0
    V[r - 1, :] = 0.0
    V[r - 1, D - 1] = 1.0
    U = _normal(rng, (Hp, r), 1.0 / math.sqrt(r))
    U[:, r - 1] = shift
    W3 = _normal(rng, (Hp, D), 1.0 / math.sqrt(D))
    W2 = _normal(rng, (D, Hp), 1.0 / math.sqrt(Hp))
    return LayerWeights(D, Hp, r, dtype, None, _round(U, dtype), _round(V, dtype),
                        _round(W3, dtype), _round(W2, dtype),
                        {"seed": seed, "shift": shift})


def tokens(n: int, D: int, *, dtype: str = "bf16", seed: int = 500) -> torch.Tensor:
    """n tokens x[n,D]: N(0,1) entries, channel D-1 fixed to 1.0 (CPU tensor)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, D), dtype=np.float32)
    x[:, D - 1] = 1.0
    return _round(x, dtype)


def oracle_view(t: torch.Tensor | None) -> np.ndarray | None:
    """The storage bits as numpy: float32 values, or bf16 bit patterns as uint16."""
    if t is None:
        return None
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(f"unsupported dtype {t.dtype}")


# Named workloads (the shapes and recipes of the paper's Fig. 2 layer and of the
# sparsity/batch sweep).  Seeds follow 1000*id + set.
WORKLOADS = {
    "tiny-f32-D384-H1024": dict(id=0, gate="standard", D=384, H=1024, r=0, dtype="f32",
                                B=1, tokens=64, sets=1, shift=SHIFT_90),
    "std-bf16-D2560-H7168-B1": dict(id=1, gate="standard", D=2560, H=7168, r=0, dtype="bf16",
                                    B=1, tokens=4096, sets=8, shift=SHIFT_90),
    "lopa-bf16-D2560-H9787-r400-B1": dict(id=2, gate="lopa", D=2560, H=9787, r=400, dtype="bf16",
                                          B=1, tokens=4096, sets=8, shift=SHIFT_90),
    "std-bf16-D2560-H7168-batched": dict(id=3, gate="standard", D=2560, H=7168, r=0, dtype="bf16",
                                         B=(4, 16, 64), tokens=4096, sets=8, shift=SHIFT_90),
    "sweep-bf16-D4096-H14336": dict(id=4, gate=("standard", "lopa"), D=4096, H=14336, r=640,
                                    Hp=19649, dtype="bf16", B=(1, 8, 32, 128),
                                    s=(0.5, 0.75, 0.9, 0.95), tokens=1024, sets=4),
}


def workload_layers(name: str, *, sets: int | None = None, gate: str | None = None,
                    s: float | None = None, full_form: bool = False):
    """The weight sets of a named workload (CPU tensors).

    full_form: the low-rank layer is meant for the full gate Gx + U RMSNorm(Vx).
    The tiled identity adds x_{i mod D} ~ N(0, 1) to every z_i, doubling the
    variance of the unshifted gate, so the shift is scaled by sqrt(2) to keep
    the same sparsity."""
    w = WORKLOADS[name]
    n = w["sets"] if sets is None else sets
    g = gate or (w["gate"] if isinstance(w["gate"], str) else "standard")
    shift = w.get("shift", SHIFT_90) if s is None else shift_for_sparsity(s)
    if full_form:
        shift *= math.sqrt(2.0)
    out = []
    for k in range(n):
        seed = 1000 * w["id"] + k
        if g == "standard":
            out.append(standard_layer(w["D"], w["H"], dtype=w["dtype"], seed=seed, shift=shift))
        else:
            Hp = w.get("Hp", w["H"])
            out.append(lopa_layer(w["D"], Hp, w["r"], dtype=w["dtype"], seed=seed, shift=shift))
    return out


def workload_tokens(name: str, n: int | None = None) -> torch.Tensor:
    w = WORKLOADS[name]
    return tokens(w["tokens"] if n is None else n, w["D"], dtype=w["dtype"],
                  seed=1000 * w["id"] + 500)
