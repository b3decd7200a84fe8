"""A decoder's stack of ternary projection linears, run through the C ABI.

Per layer the seven projections run in dependency order, as four launches:
[q, k, v] (one grouped launch sharing X) -> o -> [gate, up] (grouped) ->
down (model page "Neutrino-1 8B", "Architecture": seven linears per layer,
36 layers, 252 in all).  The attention and SwiGLU between them are not part
of this path, so each launch reads its own resident input; launches still
follow one another on one stream, and with ``TL_FLAG_PDL`` each one starts
streaming its weights while the previous one drains.  ``capture()`` records
one pass as a CUDA graph.

Mode B adds one activation-quantisation launch in front of every linear
launch (four per layer); the fused mode B (``TL_MODE_I8_FUSED``) quantises
inside the linear's own launch instead.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import synth
from . import tl

GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


def copy_chunks(layers: int):
    """The host-copy chunks of ``LinearStack.capture_e2e`` as lists of
    [first, last) layer ranges: inputs as layer 0, then all the others;
    outputs in runs of about a quarter of the layers, the last layer alone."""
    L = layers
    ins = [(0, 1)] + ([(1, L)] if L > 1 else [])
    every = max(1, (L - 1 + 3) // 4)
    outs = [(lo, min(lo + every, L - 1)) for lo in range(0, L - 1, every)] + [(L - 1, L)]
    return ins, outs


class StackWeights:
    """The packed weights of every layer, resident on the device.

    Matrices are drawn and packed on host threads (seeded per matrix, so the
    result does not depend on the thread count) and copied to the device.
    ``keep_host`` layers also keep their int8 matrices and scales on the host.
    """

    def __init__(self, shape: synth.ModelShape, base_seed: int = 0, layers: int | None = None,
                 keep_host=(), device: str = "cuda", threads: int | None = None):
        self.shape = shape
        self.layers = shape.layers if layers is None else layers
        self.base_seed = base_seed
        self.host = {}
        shp = shape.linear_shapes()
        jobs = [(l, p) for l in range(self.layers) for p in synth.PROJ_ORDER]

        def make(job):
            l, p = job
            M, K = shp[p]
            seed = synth.matrix_seed(base_seed, l, p)
            W = synth.ternary(M, K, synth.zero_fraction(shape, l, p), seed)
            scale = synth.scales(M, seed)
            packed, sc, rs = tl.tl_pack(W, scale)
            return job, packed, sc, rs, (W if l in keep_host else None)

        self.per_layer = [dict() for _ in range(self.layers)]
        n = threads or min(16, os.cpu_count() or 1)
        with ThreadPoolExecutor(n) as ex:
            for (l, p), packed, sc, rs, W in ex.map(make, jobs):
                M, K = shp[p]
                self.per_layer[l][p] = tl.TernaryWeight.from_host(packed, sc, rs, M, K,
                                                                  device=device)
                if W is not None:
                    self.host[(l, p)] = (W, sc)

    def __getitem__(self, layer: int) -> dict:
        return self.per_layer[layer]


class LinearStack:
    def __init__(self, shape: synth.ModelShape, N: int, mode: int = tl.TL_MODE_BF16,
                 out_dtype: int = tl.TL_OUT_F32, base_seed: int = 0, outlier_frac: float = 0.0,
                 unit_rms: bool = False, layers: int | None = None, keep_host=(),
                 device: str = "cuda", symmetric: bool = False,
                 weights: StackWeights | None = None):
        import torch
        self.torch = torch
        self.shape = shape
        self.N, self.mode, self.out_dtype = N, mode, out_dtype
        self.symmetric = symmetric
        if weights is None:
            weights = StackWeights(shape, base_seed, layers, keep_host, device)
        self.stack_weights = weights
        self.layers = weights.layers
        self.device = device
        self.host = weights.host  # (layer, proj) -> (W int8, scale) for kept layers
        shp = shape.linear_shapes()
        self.weights = weights.per_layer   # per layer: dict proj -> TernaryWeight
        # Inputs (one per launch group and layer) live in one flat bf16 buffer
        # and outputs in one flat buffer, so a host round trip is two copies.
        odt = {tl.TL_OUT_F32: torch.float32, tl.TL_OUT_BF16: torch.bfloat16}[out_dtype]
        x_sizes = [N * shp[grp[0]][1] for _ in range(self.layers) for grp in GROUPS]
        y_sizes = [N * shp[p][0] for _ in range(self.layers) for grp in GROUPS for p in grp]
        self.X_flat = torch.empty(sum(x_sizes), dtype=torch.bfloat16, device=device)
        self.Y_flat = torch.empty(sum(y_sizes), dtype=odt, device=device)
        self.X, self.Q, self.S, self.Z, self.Y = [], [], [], [], []
        self.x_span, self.y_span = [], []     # each layer's [lo, hi) in X_flat, Y_flat
        xo = yo = 0
        for l in range(self.layers):
            x_lo, y_lo = xo, yo
            xs, qs, ss, zs, ys = [], [], [], [], []
            for gi, grp in enumerate(GROUPS):
                K = shp[grp[0]][1]
                bits = synth.activations(N, K, seed=base_seed + 100_000 + 10 * l + gi,
                                         outlier_frac=outlier_frac, unit_rms=unit_rms)
                xt = self.X_flat[xo:xo + N * K].view(N, K)
                xo += N * K
                xt.copy_(torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16))
                xs.append(xt)
                if mode == tl.TL_MODE_I8:
                    qs.append(torch.empty((N, K), dtype=torch.int8, device=device))
                    ss.append(torch.empty(N, dtype=torch.float32, device=device))
                    zs.append(torch.empty(N, dtype=torch.int32, device=device))
                outs = []
                for p in grp:
                    M = shp[p][0]
                    outs.append(self.Y_flat[yo:yo + N * M].view(N, M))
                    yo += N * M
                ys.append(outs)
            self.X.append(xs); self.Q.append(qs); self.S.append(ss); self.Z.append(zs)
            self.Y.append(ys)
            self.x_span.append((x_lo, xo))
            self.y_span.append((y_lo, yo))
        groups = [[self.weights[l][p] for p in grp] for l in range(self.layers) for grp in GROUPS]
        self.workspace = tl.make_workspace(groups, N, device=device)
        self.graph = None

    # ------------------------------------------------------------------ run
    @property
    def integer(self) -> bool:
        return self.mode in (tl.TL_MODE_I8, tl.TL_MODE_I8_FUSED)

    @property
    def launches_per_step(self) -> int:
        per_layer = len(GROUPS) * (2 if self.mode == tl.TL_MODE_I8 else 1)
        return per_layer * self.layers

    def run(self, flags: int = tl.TL_FLAG_PDL, stream=None) -> None:
        for l in range(self.layers):
            self.run_layer(l, flags, stream)

    def run_layer(self, l: int, flags: int = tl.TL_FLAG_PDL, stream=None) -> None:
        for gi, grp in enumerate(GROUPS):
            ws = [self.weights[l][p] for p in grp]
            x = self.X[l][gi]
            if self.mode == tl.TL_MODE_I8:
                q, s, z = self.Q[l][gi], self.S[l][gi], self.Z[l][gi]
                tl.tl_quantize_act(x, symmetric=self.symmetric, Q=q, s=s, z=z, stream=stream)
                tl.tl_linear_group(ws, q, s, z, outs=self.Y[l][gi], mode=self.mode,
                                   out_dtype=self.out_dtype, workspace=self.workspace,
                                   flags=flags, stream=stream)
            else:
                if self.mode == tl.TL_MODE_I8_FUSED and self.symmetric:
                    flags |= tl.TL_FLAG_SYMMETRIC
                tl.tl_linear_group(ws, x, outs=self.Y[l][gi], mode=self.mode,
                                   out_dtype=self.out_dtype, workspace=self.workspace,
                                   flags=flags, stream=stream)

    def chain(self, gate=None, wait_limit: int = 0) -> "tl.Chain":
        """The whole pass as one chain: every launch group of every layer, in
        dependency order, run by one persistent launch (mode B quantises each
        group's bf16 input inside the chain)."""
        if self.mode not in (tl.TL_MODE_BF16, tl.TL_MODE_I8):
            raise ValueError("a chain runs mode A or mode B (its quantiser steps are its own)")
        if getattr(self, "_chain", None) is None:
            steps = [([self.weights[l][p] for p in grp], self.X[l][gi], self.Y[l][gi])
                     for l in range(self.layers) for gi, grp in enumerate(GROUPS)]
            self._chain = tl.Chain(steps, self.N, self.mode, self.out_dtype, gate=gate,
                                   wait_limit=wait_limit, device=self.device)
        return self._chain

    def capture(self, flags: int = tl.TL_FLAG_PDL):
        """Record one pass as a CUDA graph (kernels launched by the C ABI)."""
        torch = self.torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run(flags=flags)          # warm: device attributes cached before capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(flags=flags)
        torch.cuda.synchronize()
        self.graph = g
        return g

    def capture_e2e(self, hx, hy, flags: int = tl.TL_FLAG_PDL):
        """Record one pass together with its host copies, as one CUDA graph:
        pinned host inputs ``hx`` (shaped like ``X_flat``) come in on one copy
        stream -- layer 0's first, then all the others -- and the outputs go
        out to pinned ``hy`` (shaped like ``Y_flat``) on a second copy stream
        in chunks of about a quarter of the layers, each as soon as its last
        layer is done, with the last layer alone, so the copies overlap the
        launches.  Each place where the launches wait for a copy or hand one
        an event costs the pass about a microsecond, so the chunks are few:
        measured on the 8B stack at one token, per-layer copies took 1.348 ms
        per pass, these chunks 1.241 ms (1.172 ms without copies; 1.409 ms
        with all inputs copied before the pass and all outputs after it).
        Every replay copies all inputs in and all outputs out."""
        torch = self.torch
        if not (hx.is_pinned() and hy.is_pinned()):
            raise ValueError("the host buffers must be pinned")
        if hx.shape != self.X_flat.shape or hy.shape != self.Y_flat.shape:
            raise ValueError("host buffers must match X_flat and Y_flat")
        L = self.layers
        ins, outs = copy_chunks(L)
        main = torch.cuda.Stream()
        cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
        main.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(main):
            self.run(flags=flags)          # warm: device attributes cached before capture
        torch.cuda.current_stream().wait_stream(main)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        ev_in = [torch.cuda.Event() for _ in ins]
        ev_out = [torch.cuda.Event() for _ in outs]
        with torch.cuda.graph(g, stream=main):
            cin.wait_stream(main)
            cout.wait_stream(main)
            with torch.cuda.stream(cin):
                for i, (l0, l1) in enumerate(ins):
                    lo, hi = self.x_span[l0][0], self.x_span[l1 - 1][1]
                    self.X_flat[lo:hi].copy_(hx[lo:hi], non_blocking=True)
                    ev_in[i].record(cin)
            for l in range(L):
                for i, (l0, _) in enumerate(ins):
                    if l0 == l:
                        main.wait_event(ev_in[i])
                self.run_layer(l, flags, stream=main)
                for i, (l0, l1) in enumerate(outs):
                    if l1 == l + 1:
                        ev_out[i].record(main)
                        with torch.cuda.stream(cout):
                            cout.wait_event(ev_out[i])
                            lo, hi = self.y_span[l0][0], self.y_span[l1 - 1][1]
                            hy[lo:hi].copy_(self.Y_flat[lo:hi], non_blocking=True)
            main.wait_stream(cin)
            main.wait_stream(cout)
        torch.cuda.synchronize()
        self.graph_e2e = g
        return g

    # ------------------------------------------------------------ accounting
    def algorithmic_bytes(self) -> int:
        """Bytes the method must move per pass: packed codes, per-row scales
        (and row sums in mode B), each input once, each output once."""
        shp = self.shape.linear_shapes()
        per_layer = 0
        xb = 2                                         # bf16 inputs, read once
        yb = 4 if self.out_dtype == tl.TL_OUT_F32 else 2
        for grp in GROUPS:
            K = shp[grp[0]][1]
            per_layer += self.N * K * xb
            for p in grp:
                M = shp[p][0]
                per_layer += tl.tl_packed_bytes(M, K) + 4 * M + self.N * M * yb
                if self.integer:
                    per_layer += 4 * M
        if self.mode == tl.TL_MODE_I8:
            per_layer += len(GROUPS) * self.N * 8      # s and z
        return per_layer * self.layers

    def weight_count(self) -> int:
        return self.shape.ternary_weights_per_layer() * self.layers

    def output_bytes(self) -> int:
        return self.Y_flat.numel() * self.Y_flat.element_size()

    def input_bytes(self) -> int:
        return self.X_flat.numel() * self.X_flat.element_size()
