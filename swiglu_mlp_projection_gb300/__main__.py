"""Run one shape through swiglu_up repeatedly (for timing and profiling).

    python -m swiglu_mlp_projection_gb300 --M 16 --d 4096 --d_ff 14336 [--dtype bf16]
        [--path auto|simt|skinny|tc] [--iters 20] [--warmup 3] [--copies 1] [--fp8]

--fp8 quantizes the weights to e4m3 once (outside the timed calls) and times
swiglu_up_fp8 instead (bf16 x and h).

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
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
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
    for i in range(a.warmup):
        call(i)
    torch.cuda.synchronize()
    times = []
    for i in range(a.iters):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call(i)
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    swg.check_device_status()
    ms = statistics.median(times)
    by = (workload.fp8_bytes(a.M, a.d, a.d_ff) if a.fp8
          else workload.algorithmic_bytes(a.M, a.d, a.d_ff, a.dtype))
    fl = workload.flops(a.M, a.d, a.d_ff)
    print(json.dumps({"M": a.M, "d": a.d, "d_ff": a.d_ff, "dtype": "e4m3" if a.fp8 else a.dtype,
                      "path": swg.plan(a.M, a.d, a.d_ff, a.dtype, a.path)["path"],
                      "us": round(ms * 1e3, 2), "GB/s": round(by / ms / 1e6, 1),
                      "TFLOP/s": round(fl / ms / 1e9, 2)}))


if __name__ == "__main__":
    main()
