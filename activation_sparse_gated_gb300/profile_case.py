"""A small, self-contained forward loop for profiler captures.

    python -m activation_sparse_gated_gb300.profile_case --workload std --calls 8 [--dtype int8]

builds ONE full-size layer of the named workload, runs `--calls` forwards of
`--batch` tokens through the C ABI with a synchronisation after each, and exits
0.  Device memory stays near one layer (110-130 MB for the D=2560 workloads,
350 MB at D=4096); the profiler flushes caches between replays, so DRAM figures
are cold-cache figures.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

CASES = {
    "std": ("std-bf16-D2560-H7168-B1", None),
    "lopa": ("lopa-bf16-D2560-H9787-r400-B1", None),
    "std4096": ("sweep-bf16-D4096-H14336", "standard"),
    "lopa4096": ("sweep-bf16-D4096-H14336", "lopa"),
    "tiny": ("tiny-f32-D384-H1024", None),
}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", choices=sorted(CASES), default="std")
    ap.add_argument("--calls", type=int, default=8)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--dtype", choices=["bf16", "f32", "int8"], default=None,
                    help="handle dtype (default: the workload's); int8 quantises the layer on the device")
    args = ap.parse_args()

    import torch
    import activation_sparse_gated_gb300 as sffn
    from activation_sparse_gated_gb300 import build
    from activation_sparse_gated_gb300 import synthetic as syn

    build.build()
    name, gate = CASES[args.workload]
    lw = syn.workload_layers(name, sets=1, gate=gate)[0]
    ffn = sffn.SparseFFN(lw.D, lw.H, lw.r, "relu", args.dtype or lw.dtype)
    w = {k: (None if t is None else t.cuda()) for k, t in lw.tensors().items()}
    ffn.set_weights(w["W1"] if lw.r == 0 else w["U"], w["V"], w["W3"], w["W2"])
    x = syn.workload_tokens(name, args.calls * args.batch).cuda()
    for c in range(args.calls):
        ffn(x[c * args.batch:(c + 1) * args.batch])
        ffn.synchronize()
    torch.cuda.synchronize()
    print(f"profile_case {args.workload}: {args.calls} calls, live units of the last call: "
          f"{ffn.active_counts(args.batch)}")


if __name__ == "__main__":
    main()
