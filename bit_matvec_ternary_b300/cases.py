"""Run one named launch of the hot path a few times (for profiler captures).

    python -m bit_matvec_ternary_b300.cases --case gate_up --n 1 --mode a --reps 3

Cases are the launch groups of one 8B-shaped decoder layer: qkv (q/k/v
grouped, K = 4096), o, gate_up (gate/up grouped), down (K = 12288), quant
(the activation quantiser, K = 12288), chain (the first `--layers`
layers of the 8B stack as one persistent chain launch), stack (the same
layers as the benchmark's CUDA graph of per-group launches; `--mode f`
quantises inside each linear launch), and head (the
151,936 x 4,096 int8 head with its fused argmax).  Each is built from the same seeded
synthetic inputs as the benchmark and launched `reps` times back to back
after `warmup` launches, then the process checks nothing and exits 0.
"""
from __future__ import annotations

import argparse

import numpy as np

from . import synth
from .stack import GROUPS

CASE_GROUPS = {"qkv": 0, "o": 1, "gate_up": 2, "down": 3}


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", default="gate_up",
                    choices=sorted(CASE_GROUPS) + ["quant", "chain", "stack", "head", "blockscale",
                                                   "rmsnorm", "swiglu"])
    ap.add_argument("--n", type=int, default=1)
    ap.add_argument("--mode", default="a", choices=["a", "b", "f"],
                    help="a: bf16, b: int8 from the quantiser, f: int8 quantised in the launch")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--layer", type=int, default=5)
    ap.add_argument("--layers", type=int, default=2)
    args = ap.parse_args()

    import torch
    from . import build as tlbuild
    tlbuild.build()
    from . import tl

    shape = synth.NEUTRINO_8B
    shp = shape.linear_shapes()
    mode = {"a": tl.TL_MODE_BF16, "b": tl.TL_MODE_I8, "f": tl.TL_MODE_I8_FUSED}[args.mode]
    if mode == tl.TL_MODE_I8_FUSED and args.case in ("chain", "quant", "head"):
        raise SystemExit("mode f applies to the per-launch cases and the stack")
    if args.case == "stack":
        from .stack import LinearStack
        st = LinearStack(shape, N=args.n, mode=mode, layers=args.layers)
        st.capture()
        for _ in range(args.warmup + args.reps):
            st.graph.replay()
        torch.cuda.synchronize()
        return
    if args.case == "head":
        V, D = 151_936, 4096
        g = torch.Generator(device="cuda")
        g.manual_seed(1234)
        H = torch.randint(-128, 128, (V, D), dtype=torch.int8, device="cuda", generator=g)
        scale = torch.rand(V, device="cuda", generator=g) * 0.045 + 0.005
        head = tl.Head(H, scale)
        x = synth.activations(args.n, D, seed=55)
        xt = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
        q, s, z = tl.tl_quantize_act(xt)
        for _ in range(args.warmup + args.reps):
            head.argmax(q, s, z)
        torch.cuda.synchronize()
        return
    if args.case == "chain":
        from .stack import LinearStack
        st = LinearStack(shape, N=args.n, mode=mode, layers=args.layers)
        chain = st.chain()
        for _ in range(args.warmup + args.reps):
            chain.run()
        torch.cuda.synchronize()
        if chain.status() != 0:
            raise SystemExit(f"chain status {chain.status()}")
        return
    if args.case == "blockscale":
        # the gate-shaped 12288 x 4096 matrix with one scale per (row, 128-column block)
        M, K = shp["gate"]
        rng = np.random.default_rng(7)
        bw = tl.BlockScaledWeight.from_float(rng.standard_normal((M, K), dtype=np.float32) * 0.02)
        x = synth.activations(args.n, K, seed=3)
        xt = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
        y = torch.empty((args.n, M), dtype=torch.float32, device="cuda")
        for _ in range(args.warmup + args.reps):
            tl.tl_linear_blockscale(bw, xt, out=y)
        torch.cuda.synchronize()
        return
    if args.case in ("rmsnorm", "swiglu"):
        # RMSNorm over the hidden size, SwiGLU over the feed-forward size, each
        # with the per-token quantisation fused
        rng = np.random.default_rng(5)
        D = shp["q"][1] if args.case == "rmsnorm" else shp["gate"][0]

        def bf16(arr):
            return torch.from_numpy(synth.to_bf16_bits(arr.astype(np.float32)).view(np.int16)).view(
                torch.bfloat16).cuda()
        a1 = bf16(rng.standard_normal((args.n, D)))
        a2 = bf16(rng.uniform(0.8, 1.2, D)) if args.case == "rmsnorm" else bf16(rng.standard_normal((args.n, D)))
        for _ in range(args.warmup + args.reps):
            if args.case == "rmsnorm":
                tl.tl_rmsnorm_quant(a1, a2, 1e-6)
            else:
                tl.tl_swiglu_quant(a1, a2)
        torch.cuda.synchronize()
        return
    if args.case == "quant":
        K = shp["down"][1]
        x = synth.activations(args.n, K, seed=1)
        xt = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
        for _ in range(args.warmup + args.reps):
            tl.tl_quantize_act(xt)
        torch.cuda.synchronize()
        return
    grp = GROUPS[CASE_GROUPS[args.case]]
    ws = []
    for p in grp:
        M, K = shp[p]
        seed = synth.matrix_seed(0, args.layer, p)
        W = synth.ternary(M, K, synth.zero_fraction(shape, args.layer, p), seed)
        ws.append(tl.TernaryWeight.from_int8(W, synth.scales(M, seed)))
    K = shp[grp[0]][1]
    x = synth.activations(args.n, K, seed=2)
    xt = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    work = tl.make_workspace([ws], args.n)
    if mode == tl.TL_MODE_I8:
        q, s, z = tl.tl_quantize_act(xt)
        outs = tl.tl_linear_group(ws, q, s, z, mode=mode, workspace=work)
        for _ in range(args.warmup + args.reps):
            tl.tl_linear_group(ws, q, s, z, outs=outs, mode=mode, workspace=work)
    else:
        outs = tl.tl_linear_group(ws, xt, mode=mode, workspace=work)
        for _ in range(args.warmup + args.reps):
            tl.tl_linear_group(ws, xt, outs=outs, mode=mode, workspace=work)
    torch.cuda.synchronize()


if __name__ == "__main__":
    main()
