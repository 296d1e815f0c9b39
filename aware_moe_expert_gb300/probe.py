"""Run a few layer calls of one synthetic workload, for profilers.

    python -m aware_moe_expert_gb300.probe --workload mixtral_decode --calls 4 [--T 8]

Builds the workload's seeded inputs (the same generator as bench.py, one copy
of the weights, so the device holds little more than them), calls
moe_layer_forward `--calls` times on the current stream and checks the device
status.  Nothing is timed: under ncu, pick the launch to capture with
`-k regex:<kernel> -s <skip> -c 1`.
"""
from __future__ import annotations

import argparse

import torch

from aware_moe_expert_gb300 import binding as B
from aware_moe_expert_gb300 import workloads as WL
from aware_moe_expert_gb300.inputs import make_layer_inputs


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="mixtral_decode", choices=sorted(WL.ALL))
    ap.add_argument("--T", type=int, default=None, help="override the token count")
    ap.add_argument("--calls", type=int, default=4)
    a = ap.parse_args(argv)
    wl = WL.ALL[a.workload] if a.T is None else WL.ALL[a.workload].with_T(a.T)
    d = make_layer_inputs(wl, "cuda")
    desc = B.desc_for(wl, expert_bias=d["expert_bias"], w_shared_gate_up=d.get("w_shared_gate_up"),
                      w_shared_down=d.get("w_shared_down"))
    layer = B.MoeLayer(desc, "cuda")
    for _ in range(a.calls):
        layer.forward(d["x"], d["router_w"], d["w_gate_up"], d["w_down"], d["k_per_token"])
    torch.cuda.synchronize()
    code = layer.device_status()
    print(f"{wl.name}: {a.calls} layer calls, device status {B.STATUS_NAMES.get(code, code)}, "
          f"{torch.cuda.max_memory_allocated() / 1e9:.2f} GB allocated")
    return 0 if code == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
