"""Run a handful of SFI decode steps eagerly (no graph), for profiler captures.

  python -m sparse_long_context_sfi_gb300.profile_step [--workload NAME] [--fast N]

Order of launches on the device: the input generator's kernels, then step 0 (slow):
append, dense attention, evidence, select, compact; then N fast steps: append, sparse
attention. With ncu, `-k regex:attn_kernel -s 0 -c 1` captures the dense attention kernel
and `-k regex:attn_kernel -s 1 -c 1` the first sparse one.
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import numpy as np


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama8b_ctx32k_b4")
    ap.add_argument("--fast", type=int, default=2)
    args = ap.parse_args()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch

    from synth import device as sdev
    from synth.configs import WORKLOADS
    from synth.workload import HostWorkload

    wl = HostWorkload(WORKLOADS[args.workload])
    cfg = wl.cfg
    st = sdev.make_state(wl)
    n = 1 + args.fast
    ins = sdev.DeviceInputs(wl, n, st.k.device)
    out = torch.empty((n, cfg.n_layers, cfg.batch, cfg.n_q_heads, cfg.head_dim),
                      dtype=torch.bfloat16, device=st.k.device)
    torch.cuda.synchronize()
    for t in range(n):
        t0 = time.perf_counter()
        st.step(ins.q[t], ins.k_new[t], ins.v_new[t], np.full(cfg.batch, t == 0), out[t],
                out_fp32=False)
        torch.cuda.synchronize()
        print(f"step {t} ({'slow' if t == 0 else 'fast'}): {1e3 * (time.perf_counter() - t0):.3f} ms")
    err = int(st.err[0])
    print(f"device error word: {err:#x}")
    sys.exit(1 if err else 0)


if __name__ == "__main__":
    main()
