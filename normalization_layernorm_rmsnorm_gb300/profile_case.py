"""Runs the libnorm calls of chosen workloads a few times and exits: the
program the ncu captures profile (one kernel, a few launches, a few GB).

    python -m normalization_layernorm_rmsnorm_gb300.profile_case \
        --workload bn_f32_256x64x56x56_res_relu --repeat 3

Inputs are the bench's full-size synthetic workloads, and the profile-only
shapes of workloads.PROFILE_ONLY for the paths no bench workload takes.  Most are
well above the
129 MB L2; the LayerNorm fp16 [25216,768] tensors (39 MB each) and the fp16
[128,512,7,7] BatchNorm fit in it, and ncu's default cache control flushes the
caches before each replay pass, so DRAM counters still count cold reads.
"""
from __future__ import annotations

import argparse


def main(argv=None):
    import torch

    import normalization_layernorm_rmsnorm_gb300 as nrm
    from normalization_layernorm_rmsnorm_gb300 import workloads

    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", action="append", required=True)
    ap.add_argument("--phase", choices=("fwd", "bwd", "both"), default="both")
    ap.add_argument("--repeat", type=int, default=3)
    args = ap.parse_args(argv)
    nrm.load()
    dev = torch.device("cuda", 0)
    names = set(args.workload)
    calls = (workloads.build_calls(dev, names) + workloads.build_extra_calls(dev, names)
             + workloads.build_profile_calls(dev, names))
    if not calls:
        ap.error(f"no such workload: {args.workload}")
    for _ in range(args.repeat):
        for c in calls:
            if args.phase in ("both", c.phase):
                c.fn()
    nrm.nrm_sync_status()
    torch.cuda.synchronize()
    print("ran", [f"{c.workload}:{c.phase}" for c in calls], "x", args.repeat)


if __name__ == "__main__":
    main()
