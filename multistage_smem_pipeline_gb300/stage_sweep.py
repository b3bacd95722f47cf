"""Ring-depth (kStage) justification on the current GPU.

    python -m multistage_smem_pipeline_gb300.stage_sweep [--workload c4] [--path pair]
        [--bn 256] [--katoms 1 2] [--wide]

1. Measures the two inputs of the stage-count rule of "第 6 课：Shared Memory
   布局与异步流水" (section 4), S_min = ceil(T_copy / T_compute) + 1, with the
   library's latency probes, per 64-wide K slice of one SM: T_copy = the
   slice's TMA loads (A 128 x 64 and this SM's rows of B x 64 fp16) from issue
   to the full barrier, with every SM loading at once, from a region far
   larger than L2 (HBM) and from one that fits in L2; T_compute = the slice's
   MMAs (4 x tcgen05.mma 128 x bn x 16) on one SM.  A ring stage holds
   `katoms` slices, so in stages S_min becomes ceil(S_min / katoms).  With
   --wide (pair path, units of two n-tiles) a slice carries both tiles' B
   halves (bn rows per SM in all) and feeds both tiles' MMAs, so T_copy is
   probed for A + bn rows of B and T_compute is twice that of one tile.
2. Sweeps kstage from 2 to the deepest ring that fits in shared memory for
   each tile width and slice count on the chosen workload, timing each with
   an L2 flush between launches.
3. Prints one JSON object per measurement and a summary line.

Shared memory per CTA: kstage * (16 KiB + bn * 128 B) + 16 KiB of epilogue
staging; one CTA per SM (persistent), so the page's occupancy collapse
(fewer resident blocks as stages grow) does not arise -- the only cost of a
deeper ring is shared memory the kernel does not otherwise use.
"""
from __future__ import annotations

import argparse
import json
import math

import numpy as np
import torch

from . import binding, synthetic
from .timing import time_launches


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="c4", choices=sorted(synthetic.WORKLOADS))
    ap.add_argument("--path", default="pair", choices=["square", "pair"])
    ap.add_argument("--bn", type=int, nargs="+", default=[256])
    ap.add_argument("--katoms", type=int, nargs="+", default=[1, 2])
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--reps", type=int, default=256)
    ap.add_argument("--wide", action="store_true",
                    help="pair units of two adjacent n-tiles sharing each A slice")
    args = ap.parse_args()
    if args.wide and args.path != "pair":
        ap.error("--wide needs --path pair")

    dev = torch.device("cuda", 0)
    spec = synthetic.WORKLOADS[args.workload]
    M, N, K = spec["M"], spec["N"], spec["K"]
    a_bits, b_bits, _ = synthetic.workload(args.workload)
    a = torch.from_numpy(a_bits.view(np.float16)).to(dev)
    b = torch.from_numpy(b_bits.view(np.float16)).to(dev)
    d = torch.empty((M, N), dtype=torch.float16, device=dev)
    flops = 2.0 * M * N * K
    path = binding.PATH_PAIR if args.path == "pair" else binding.PATH_SQUARE
    summary = {}
    for bn in args.bn:
        # one SM's share of a 64-wide K slice: A 128 x 64, plus B bn x 64
        # (square) or bn/2 x 64 (pair: the other half sits in the peer CTA)
        rows = bn // 2 if path == binding.PATH_PAIR else bn
        if args.wide:
            rows = bn            # both tiles' halves of B
        copy_hbm, comp = binding.probe_latencies(bn=rows, ctas=0, footprint_bytes=4 << 30,
                                                 reps=args.reps // 4)
        copy_l2, _ = binding.probe_latencies(bn=rows, ctas=0, footprint_bytes=32 << 20,
                                             reps=args.reps // 4)
        copy_1sm, _ = binding.probe_latencies(bn=rows, ctas=1, footprint_bytes=4 << 30,
                                              reps=args.reps)
        _, comp = binding.probe_latencies(bn=bn, ctas=1, footprint_bytes=32 << 20,
                                          reps=args.reps)       # 128 x bn x 64 per SM
        if args.wide:
            comp *= 2            # one slice feeds both tiles' MMAs
        s_hbm = binding.minimum_stages(math.ceil(copy_hbm), math.ceil(comp))
        s_l2 = binding.minimum_stages(math.ceil(copy_l2), math.ceil(comp))
        probe = {"kind": "probe", "path": args.path, "bn": bn, "wide": args.wide,
                 "slice_bytes": 16384 + rows * 128,
                 "t_copy_cycles_all_sms_hbm": copy_hbm, "t_copy_cycles_all_sms_l2": copy_l2,
                 "t_copy_cycles_one_sm_hbm": copy_1sm, "t_compute_cycles": comp,
                 "s_min_hbm": s_hbm, "s_min_l2": s_l2}
        print(json.dumps(probe), flush=True)
        for katoms in args.katoms:
            fixed = dict(path=path, bn=bn, katoms=katoms, epi_warps=8 if args.wide else 4,
                         wide=2 if args.wide else (1 if path == binding.PATH_PAIR else 0))
            try:
                deepest = binding.query_config(M, N, K, **fixed)["kstage"]
            except binding.GemmError:
                continue
            best = None
            for ks in range(2, deepest + 1):
                t = time_launches(lambda: binding.gemm_tn_f16_ex(a, b, out=d, kstage=ks, **fixed),
                                  args.steps, args.warmup, dev)
                tf = flops / (t["mean"] * 1e-3) / 1e12
                row = {"kind": "sweep", "workload": args.workload, "path": args.path, "bn": bn,
                       "wide": args.wide,
                       "katoms": katoms, "kstage": ks,
                       "smem_bytes": binding.query_config(M, N, K, kstage=ks, **fixed)["smem_bytes"],
                       "ms_mean": t["mean"], "ms_median": t["median"], "tflops": tf}
                print(json.dumps(row), flush=True)
                if best is None or tf > best[1]:
                    best = (ks, tf)
            summary[f"{bn}/{katoms}"] = {"s_min_hbm": s_hbm, "s_min_l2": s_l2,
                                         "s_min_in_stages": [(s_hbm + katoms - 1) // katoms,
                                                             (s_l2 + katoms - 1) // katoms],
                                         "deepest": deepest, "best_kstage": best[0],
                                         "best_tflops": best[1]}
    status, raw = binding.get_device_error()
    print(json.dumps({"kind": "summary", "workload": args.workload, "per_bn_katoms": summary,
                      "device_status": status}))


if __name__ == "__main__":
    main()
