"""Operation counts of the gated FFN forward (multiply-adds per token).

TEST INFRASTRUCTURE ONLY (part of the oracle).  Counts follow
"Model casting: compute the gate, then skip most of the FFN" (ai.thesatyajit.com):
  * section "What an FFN actually computes": each of W1, W3, W2 costs H*D
    multiply-adds, so a dense FFN costs 3*H*D;
  * section "The 3x ceiling, and why W1 is always on", Eq. 2: the gate always
    runs, W3 and W2 run only for live units, FLOP-ratio = 3HD / (HD + 2(1-s)HD);
  * section "LoPA Gating: moving the ceiling": the low-rank gate costs r(D+H'),
    the iso-parameter width is H' = D(3H - r)/(r + 2D), and Eq. 4 is the FLOP
    ratio with that gate.
"""
from __future__ import annotations


def dense_macs(D: int, H: int) -> int:
    """3*H*D: the three full matrices."""
    return 3 * H * D


def sparse_macs(D: int, H: int, n_live: float) -> float:
    """Standard gate: H*D for W1 (always on) + n_live*D for W3 rows + n_live*D for W2 columns."""
    return H * D + 2 * n_live * D


def lopa_gate_macs(D: int, Hp: int, r: int) -> int:
    """Low-rank gate U(Vx): r*D for V plus H'*r for U."""
    return r * (D + Hp)


def lopa_macs(D: int, Hp: int, r: int, n_live: float) -> float:
    """Low-rank gate plus the live W3 rows and W2 columns."""
    return lopa_gate_macs(D, Hp, r) + 2 * n_live * D


def iso_width(D: int, H: int, r: int) -> float:
    """H' = D(3H - r)/(r + 2D): the hidden width that keeps the FFN parameter count fixed."""
    return D * (3 * H - r) / (r + 2 * D)


def ratio_standard(s: float) -> float:
    """Eq. 2: 3HD / (HD + 2(1-s)HD) = 3 / (3 - 2s)."""
    return 3.0 / (3.0 - 2.0 * s)


def ratio_lopa(s: float, D: float, H: float, r: float) -> float:
    """Eq. 4: dense 3HD over the low-rank gate plus (1-s) of W3 and W2 at width H' (unrounded)."""
    Hp = iso_width(D, H, r)
    return 3.0 * H * D / (r * (D + Hp) + 2.0 * (1.0 - s) * Hp * D)


def shares_lopa(s: float, D: float, H: float, r: float):
    """Per-matrix cost of the LoPA FFN as a fraction of the dense 3HD: (gate, W3, W2, total)."""
    Hp = iso_width(D, H, r)
    dense = 3.0 * H * D
    gate = r * (D + Hp) / dense
    w3 = (1.0 - s) * Hp * D / dense
    return gate, w3, w3, gate + 2.0 * w3
