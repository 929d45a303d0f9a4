"""Run one shape through swiglu_up (or swiglu_down) repeatedly, for timing
and profiling.

    python -m swiglu_mlp_projection_gb300 --M 16 --d 4096 --d_ff 14336 [--dtype bf16]
        [--op up|down] [--path auto|simt|skinny|tc] [--iters 20] [--warmup 3]
        [--copies 1] [--fp8]

--op down times y = h . W_down + residual (bf16; h [M, d_ff], W_down
[d_ff, d], residual [M, d]).  --fp8 quantizes the weights to e4m3 once
(outside the timed calls) and times swiglu_up_fp8 / swiglu_down_fp8 instead
(bf16 activations and outputs).

Inputs are the seeded synthetic operands of swiglu_mlp_projection_gb300.inputs.
Prints the median time per call and the achieved GB/s and TFLOP/s.
"""
import argparse
import json
import statistics


def main():
    import torch
    import swiglu_mlp_projection_gb300 as swg
    from swiglu_mlp_projection_gb300 import inputs, workload

    ap = argparse.ArgumentParser()
    ap.add_argument("--M", type=int, default=16)
    ap.add_argument("--d", type=int, default=4096)
    ap.add_argument("--d_ff", type=int, default=14336)
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f32"])
    ap.add_argument("--path", default="auto", choices=sorted(swg.PATHS))
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--copies", type=int, default=1, help="weight copies rotated per call")
    ap.add_argument("--fp8", action="store_true", help="e4m3 weights (swiglu_up_fp8)")
    ap.add_argument("--op", default="up", choices=["up", "down"])
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    if a.op == "down":
        return run_down(a, dev)
    x, wg, wu = inputs.make_inputs(a.M, a.d, a.d_ff, a.dtype, seed=0)
    x = x.to(dev)
    ws = [(wg.to(dev), wu.to(dev)) for _ in range(a.copies)]
    h = torch.empty(a.M, a.d_ff, dtype=x.dtype, device=dev)
    if a.fp8:
        if a.dtype != "bf16":
            raise SystemExit("--fp8 takes bf16 x and weights")
        qs = [swg.quantize_weights_fp8(g, u) for g, u in ws]
        call = lambda i: swg.swiglu_up_fp8(x, qs[i % a.copies], out=h, path=a.path)
    else:
        call = lambda i: swg.swiglu_up(x, *ws[i % a.copies], out=h, path=a.path)
    ms = time_calls(call, a.warmup, a.iters)
    swg.check_device_status()
    by = (workload.fp8_bytes(a.M, a.d, a.d_ff) if a.fp8
          else workload.algorithmic_bytes(a.M, a.d, a.d_ff, a.dtype))
    fl = workload.flops(a.M, a.d, a.d_ff)
    print(json.dumps({"M": a.M, "d": a.d, "d_ff": a.d_ff, "dtype": "e4m3" if a.fp8 else a.dtype,
                      "path": swg.plan(a.M, a.d, a.d_ff, a.dtype, a.path)["path"],
                      "us": round(ms * 1e3, 2), "GB/s": round(by / ms / 1e6, 1),
                      "TFLOP/s": round(fl / ms / 1e9, 2)}))


def run_down(a, dev):
    import torch
    import swiglu_mlp_projection_gb300 as swg
    from swiglu_mlp_projection_gb300 import inputs, workload
    if a.dtype != "bf16":
        raise SystemExit("the down projection takes bf16")
    h = inputs.make_inputs(a.M, a.d_ff, 8, "bf16", seed=0, x_only=True)[0].to(dev)
    r = inputs.make_inputs(a.M, a.d, 8, "bf16", seed=2, x_only=True)[0].to(dev)
    wds = [inputs.make_inputs(1, a.d_ff, a.d, "bf16", seed=1 + i)[1].to(dev)
           for i in range(a.copies)]
    y = torch.empty(a.M, a.d, dtype=torch.bfloat16, device=dev)
    if a.fp8:
        qs = [swg.quantize_weight_fp8(w) for w in wds]
        call = lambda i: swg.swiglu_down_fp8(h, qs[i % a.copies], residual=r, out=y, path=a.path)
    else:
        call = lambda i: swg.swiglu_down(h, wds[i % a.copies], residual=r, out=y, path=a.path)
    ms = time_calls(call, a.warmup, a.iters)
    swg.check_device_status()
    by = (workload.fp8_down_bytes(a.M, a.d_ff, a.d) if a.fp8
          else workload.down_bytes(a.M, a.d_ff, a.d, "bf16"))
    fl = workload.down_flops(a.M, a.d_ff, a.d)
    print(json.dumps({"op": "down", "M": a.M, "d": a.d, "d_ff": a.d_ff,
                      "dtype": "e4m3" if a.fp8 else "bf16",
                      "path": swg.down_plan(a.M, a.d_ff, a.d, "bf16", a.path)["path"],
                      "us": round(ms * 1e3, 2), "GB/s": round(by / ms / 1e6, 1),
                      "TFLOP/s": round(fl / ms / 1e9, 2)}))


def time_calls(call, warmup, iters):
    """Median milliseconds per call, each call timed with CUDA events."""
    import torch
    for i in range(warmup):
        call(i)
    torch.cuda.synchronize()
    times = []
    for i in range(iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call(i)
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times)


if __name__ == "__main__":
    main()
