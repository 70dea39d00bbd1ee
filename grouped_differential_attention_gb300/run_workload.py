"""Run one named workload a few times through the public API (for profilers).

    python -m grouped_differential_attention_gb300.run_workload prefill \
        gda_3to1_prefill_bf16_B4_L2048_h12+4_d64_dv128 --launches 3
    python -m grouped_differential_attention_gb300.run_workload decode --launches 3
    python -m grouped_differential_attention_gb300.run_workload decode_fp8 --launches 3
    python -m grouped_differential_attention_gb300.run_workload backward --launches 1
    python -m grouped_differential_attention_gb300.run_workload backward_bf16 --launches 3
    python -m grouped_differential_attention_gb300.run_workload prefill2pass --launches 3

Inputs are the seeded synthetic tensors of ``workloads``; prints the mean
device time per launch measured with CUDA events (not meaningful under a
profiler).
"""
from __future__ import annotations

import argparse
import sys

import torch

import grouped_differential_attention_gb300 as gda
from grouped_differential_attention_gb300 import workloads as W


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("kind", choices=["prefill", "prefill2pass", "decode", "decode_fp8", "backward", "backward_bf16"])
    ap.add_argument("workload", nargs="?", default=None)
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--flags", type=int, default=0, help="gda_attn_fwd_ex flags for the prefill kind")
    args = ap.parse_args(argv)
    dev = torch.device("cuda:0")
    if args.kind == "prefill":
        w = W.PREFILL_WORKLOADS[args.workload or W.GDA3_PREFILL_L2048.name]
        inp = [t.to(dev) for t in W.make_prefill_inputs(w)]
        fn = gda.gda_attn_fwd if w.dtype == "bf16" else gda.gda_attn_fwd_f32
        out = torch.empty((w.B, w.L, w.h_s, w.dv), dtype=inp[0].dtype, device=dev)

        def launch():
            fn(*inp, w.lambda_init, causal=w.causal, eps=w.eps, out=out, flags=args.flags)
    elif args.kind == "prefill2pass":
        w = W.PREFILL_WORKLOADS[args.workload or W.GDA3_PREFILL_L2048.name]
        inp = [t.to(dev) for t in W.make_prefill_inputs(w)]
        out = torch.empty((w.B, w.L, w.h_s, w.dv), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(gda.gda_attn_fwd_2pass_workspace_size(w.B, w.L, w.h_s, w.h_n), dtype=torch.uint8,
                         device=dev)

        def launch():
            gda.gda_attn_fwd_2pass(*inp, w.lambda_init, causal=w.causal, eps=w.eps, out=out, workspace=ws)
    elif args.kind == "backward_bf16":
        w = W.PREFILL_WORKLOADS[args.workload or W.GDA3_PREFILL_L2048.name]
        inp = [t.to(dev) for t in W.make_backward_inputs(w)]
        ws = torch.empty(gda.gda_attn_bwd_bf16_workspace_size(w.B, w.L, w.h_s, w.h_n, w.dv), dtype=torch.uint8,
                         device=dev)
        grads = gda.gda_attn_bwd_bf16(*inp[:6], w.lambda_init, inp[6], causal=w.causal, eps=w.eps, workspace=ws)

        def launch():
            gda.gda_attn_bwd_bf16(*inp[:6], w.lambda_init, inp[6], causal=w.causal, eps=w.eps, workspace=ws,
                                  grads=grads)
    elif args.kind == "backward":
        # float32 gradients at a prefill workload's sizes (default: the 3:1 B=4 L=2048 one)
        w = W.PREFILL_WORKLOADS[args.workload or W.GDA3_PREFILL_L2048.name]
        inp = [t.to(dev) for t in W.make_backward_inputs(w, dtype="f32")]
        ws = torch.empty(gda.gda_attn_bwd_workspace_size(w.B, w.L, w.h_s, w.d, w.dv), dtype=torch.uint8,
                         device=dev)
        grads = gda.gda_attn_bwd(*inp[:6], w.lambda_init, inp[6], causal=w.causal, eps=w.eps, workspace=ws)

        def launch():
            gda.gda_attn_bwd(*inp[:6], w.lambda_init, inp[6], causal=w.causal, eps=w.eps, workspace=ws,
                             grads=grads)
    elif args.kind == "decode_fp8":
        w = W.GDA3_DECODE_B64
        inp = [t.to(dev) for t in W.make_decode_inputs_fp8(w)]
        out = torch.empty((w.B, w.h_s, w.dv), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(gda.gda_attn_decode_workspace_size(w.B, w.Lcap, w.h_s, w.h_n, w.dv),
                         dtype=torch.uint8, device=dev)

        def launch():
            gda.gda_attn_decode_fp8(*inp, w.lambda_init, eps=w.eps, out=out, workspace=ws)
    else:
        w = W.GDA3_DECODE_B64
        inp = [t.to(dev) for t in W.make_decode_inputs(w)]
        out = torch.empty((w.B, w.h_s, w.dv), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(gda.gda_attn_decode_workspace_size(w.B, w.Lcap, w.h_s, w.h_n, w.dv),
                         dtype=torch.uint8, device=dev)

        def launch():
            gda.gda_attn_decode(*inp, w.lambda_init, eps=w.eps, out=out, workspace=ws)

    launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.launches):
        launch()
    e1.record()
    torch.cuda.synchronize()
    err = gda.gda_device_error(clear=True)
    print(f"{w.name}: {e0.elapsed_time(e1) / args.launches:.4f} ms per launch, device error word {err}")
    return 0 if err == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
