"""The quantized linear layer Y = X W^T + b as sequences of C-ABI calls.

For each recipe the three GEMMs of a linear are issued in the pages' autocast
mode -- both operands are quantized, in the orientation that GEMM consumes,
right before it -- or in pre-quantized mode (the GEMM alone on operands
quantized earlier).  ("How to Optimize Transformer-Based Models for
Low-Precision Training", section "autocast モードの使用と事前量子化の比較"; the
NVFP4 extras -- RHT on Wgrad inputs, SR on gradients, 2D weight blocks, the
extra amax pass -- from section "実モデルにおける結果の解釈".)

Recipes
  bf16         BF16 GEMMs, no quantization (Dgrad / Wgrad read operands MN-major)
  fp8_delayed  per-tensor FP8, scale from the amax history (HYBRID: E4M3 X/W, E5M2 dY)
  fp8_current  per-tensor FP8, scale from the tensor's own amax (extra amax pass)
  mxfp8        1x32 E8M0-scaled E4M3 blocks along the contraction
  nvfp4        1x16 UE4M3-scaled E2M1 blocks; X/dY col copies rotated (RHT),
               dY stochastically rounded, W in 16x16 blocks

Everything here is marshalling: device buffers (torch allocations) and the
order of launches; all arithmetic runs in libte_gb300.so.
"""
from __future__ import annotations

import torch

from . import _lib as L

RECIPES = ("bf16", "fp8_delayed", "fp8_current", "mxfp8", "nvfp4")
PASSES = ("fprop", "dgrad", "wgrad")
LAYER_LINEARS = ("qkv", "attn_out", "mlp_up", "mlp_down")


class DelayedState:
    """DelayedScaling state of a group of tensors: amax history ring, scale, scale_inv, last amax."""

    def __init__(self, n: int, history_len: int, device):
        self.n, self.L = n, history_len
        self.hist = torch.zeros(n * history_len, dtype=torch.float32, device=device)
        self.scale = torch.ones(n, dtype=torch.float32, device=device)
        self.scale_inv = torch.ones(n, dtype=torch.float32, device=device)
        self.amax = torch.zeros(n, dtype=torch.float32, device=device)

    def slot(self, i: int):
        return self.scale[i:i + 1], self.scale_inv[i:i + 1], self.amax[i:i + 1]

    FIELDS = ("hist", "scale", "scale_inv", "amax")

    def state_dict(self) -> dict:
        """Host copy of the recipe state, for a checkpoint (the FP8 metadata a module keeps
        next to its weights: amax history ring, scale, scale_inv, last amax)."""
        out = {k: getattr(self, k).detach().to("cpu", copy=True) for k in self.FIELDS}
        out.update(n=self.n, history_len=self.L)
        return out

    def load_state_dict(self, sd: dict) -> None:
        """Restore a checkpoint taken with ``state_dict`` (same tensor count and history length)."""
        if sd["n"] != self.n or sd["history_len"] != self.L:
            raise ValueError(f"checkpoint holds {sd['n']} tensors x history {sd['history_len']}, "
                             f"state has {self.n} x {self.L}")
        for k in self.FIELDS:
            getattr(self, k).copy_(sd[k])


class QuantLinear:
    """Device buffers of one linear (inputs, outputs, quantized copies) and its GEMM passes."""

    def __init__(self, x: torch.Tensor, w: torch.Tensor, dy: torch.Tensor, bias: torch.Tensor | None,
                 recipes=RECIPES, rht_signs: int = 0, sr_seed: int = 0, fwd_state: DelayedState | None = None,
                 fwd_slots=(0, 1), bwd_state: DelayedState | None = None, bwd_slot: int = 0):
        dev = x.device
        self.x, self.w, self.dy, self.bias = x, w, dy, bias
        M, Kin = x.shape
        Nout = w.shape[0]
        self.M, self.Kin, self.Nout = M, Kin, Nout
        self.name = "linear"
        self.rht_signs, self.sr_seed, self.sr_offset = rht_signs, sr_seed, 0
        bf = torch.bfloat16
        self.y = torch.empty(M, Nout, dtype=bf, device=dev)
        self.dx = torch.empty(M, Kin, dtype=bf, device=dev)
        self.dw = torch.empty(Nout, Kin, dtype=bf, device=dev)
        u8 = dict(dtype=torch.uint8, device=dev)

        def f32():
            return torch.zeros(1, dtype=torch.float32, device=dev)

        # FP8 / MXFP8 copies (shared by the three 8-bit recipes)
        if any(r in recipes for r in ("fp8_delayed", "fp8_current", "mxfp8")):
            self.xr, self.xc = torch.empty(M, Kin, **u8), torch.empty(Kin, M, **u8)
            self.wr, self.wc = torch.empty(Nout, Kin, **u8), torch.empty(Kin, Nout, **u8)
            self.dr, self.dc = torch.empty(M, Nout, **u8), torch.empty(Nout, M, **u8)
        if "fp8_current" in recipes:
            self.cur = {k: (f32(), f32()) for k in ("x", "w", "dy")}    # (amax, scale_inv)
        if "fp8_delayed" in recipes:
            assert fwd_state is not None and bwd_state is not None
            self.dl = {"x": fwd_state.slot(fwd_slots[0]), "w": fwd_state.slot(fwd_slots[1]),
                       "dy": bwd_state.slot(bwd_slot)}
        if "mxfp8" in recipes:
            def sb(r, c):
                return torch.zeros(L.te_scale_bytes(L.E8M0, r, c), **u8)
            self.sxr, self.sxc = sb(M, Kin), sb(Kin, M)
            self.swr, self.swc = sb(Nout, Kin), sb(Kin, Nout)
            self.sdr, self.sdc = sb(M, Nout), sb(Nout, M)
        if "nvfp4" in recipes:
            def nb(r, c):
                return (torch.empty(r, c // 2, **u8), torch.zeros(L.te_scale_bytes(L.UE4M3, r, c), **u8), f32())
            self.nxr, self.nxc = nb(M, Kin), nb(Kin, M)
            self.nwr, self.nwc = nb(Nout, Kin), nb(Kin, Nout)
            self.ndr, self.ndc = nb(M, Nout), nb(Nout, M)
            self.namax = {k: (f32(), f32()) for k in ("x", "w", "dy")}  # (amax, amax after RHT)

    # ---- quantizers (one orientation each, as autocast does per GEMM) -----------------------
    def _q_fp8(self, recipe, name, t, fmt, row=None, col=None):
        if recipe == "fp8_current":
            amax, sinv = self.cur[name]
            L.te_quantize_fp8(t, fmt, None, 1, row, col, amax, sinv)
        else:
            scale, _, amax = self.dl[name]
            L.te_quantize_fp8(t, fmt, scale, 0, row, col, amax, None)

    def _sinv(self, recipe, name):
        return self.cur[name][1] if recipe == "fp8_current" else self.dl[name][1]

    def _q_nv(self, name, t, flags, row=None, col=None, rotated=False):
        amax, amax_rht = self.namax[name]
        # a rotated col copy needs only the rotated amax
        L.te_amax_reduce(t, None if rotated else amax, amax_rht if rotated else None, self.rht_signs)
        rq = row if row is not None else (None, None, None)
        cq = col if col is not None else (None, None, None)
        L.te_quantize_nvfp4(t, flags, self.rht_signs, self.sr_seed, self.sr_offset, amax, amax_rht,
                            rq[0], rq[1], rq[2], cq[0], cq[1], cq[2])

    def quantize(self, recipe: str, pass_: str) -> None:
        """Quantize the two operands of one GEMM (autocast: right before the GEMM)."""
        if recipe == "bf16":
            return
        E4, E5 = L.E4M3, L.E5M2
        if recipe in ("fp8_current", "fp8_delayed"):
            if pass_ == "fprop":
                self._q_fp8(recipe, "x", self.x, E4, row=self.xr)
                self._q_fp8(recipe, "w", self.w, E4, row=self.wr)
            elif pass_ == "dgrad":
                self._q_fp8(recipe, "dy", self.dy, E5, row=self.dr)
                self._q_fp8(recipe, "w", self.w, E4, col=self.wc)
            else:
                self._q_fp8(recipe, "dy", self.dy, E5, col=self.dc)
                self._q_fp8(recipe, "x", self.x, E4, col=self.xc)
        elif recipe == "mxfp8":
            if pass_ == "fprop":
                L.te_quantize_mxfp8(self.x, self.xr, self.sxr)
                L.te_quantize_mxfp8(self.w, self.wr, self.swr)
            elif pass_ == "dgrad":
                L.te_quantize_mxfp8(self.dy, self.dr, self.sdr)
                L.te_quantize_mxfp8(self.w, None, None, self.wc, self.swc)
            else:
                L.te_quantize_mxfp8(self.dy, None, None, self.dc, self.sdc)
                L.te_quantize_mxfp8(self.x, None, None, self.xc, self.sxc)
        elif recipe == "nvfp4":
            RHT, SR, D2 = L.NVFP4_RHT_COL, L.NVFP4_SR, L.NVFP4_2D
            if pass_ == "fprop":
                self._q_nv("x", self.x, 0, row=self.nxr)
                self._q_nv("w", self.w, D2, row=self.nwr)
            elif pass_ == "dgrad":
                self._q_nv("dy", self.dy, SR, row=self.ndr)
                self._q_nv("w", self.w, D2, col=self.nwc)
            else:
                self._q_nv("dy", self.dy, RHT | SR, col=self.ndc, rotated=True)
                self._q_nv("x", self.x, RHT, col=self.nxc, rotated=True)
        else:
            raise ValueError(recipe)

    def gemm(self, recipe: str, pass_: str) -> None:
        """The GEMM of one pass on already-quantized operands."""
        E4, E5 = L.E4M3, L.E5M2
        KM, MN = L.K_MAJOR, L.MN_MAJOR
        if recipe == "bf16":
            if pass_ == "fprop":
                L.te_gemm_bf16(self.x, self.w, self.y, self.bias, KM, KM)
            elif pass_ == "dgrad":
                L.te_gemm_bf16(self.dy, self.w, self.dx, None, KM, MN)
            else:
                L.te_gemm_bf16(self.dy, self.x, self.dw, None, MN, MN)
        elif recipe in ("fp8_current", "fp8_delayed"):
            sx, sw, sd = (self._sinv(recipe, n) for n in ("x", "w", "dy"))
            if pass_ == "fprop":
                L.te_gemm_fp8(self.xr, E4, self.wr, E4, sx, sw, self.y, self.bias)
            elif pass_ == "dgrad":
                L.te_gemm_fp8(self.dr, E5, self.wc, E4, sd, sw, self.dx)
            else:
                L.te_gemm_fp8(self.dc, E5, self.xc, E4, sd, sx, self.dw)
        elif recipe == "mxfp8":
            if pass_ == "fprop":
                L.te_gemm_mxfp8(self.xr, self.sxr, self.wr, self.swr, self.y, self.bias)
            elif pass_ == "dgrad":
                L.te_gemm_mxfp8(self.dr, self.sdr, self.wc, self.swc, self.dx)
            else:
                L.te_gemm_mxfp8(self.dc, self.sdc, self.xc, self.sxc, self.dw)
        elif recipe == "nvfp4":
            if pass_ == "fprop":
                a, b, out, bias = self.nxr, self.nwr, self.y, self.bias
            elif pass_ == "dgrad":
                a, b, out, bias = self.ndr, self.nwc, self.dx, None
            else:
                a, b, out, bias = self.ndc, self.nxc, self.dw, None
            L.te_gemm_nvfp4(a[0], a[1], a[2], b[0], b[1], b[2], out, bias)
        else:
            raise ValueError(recipe)

    def gemm_shape(self, pass_: str):
        if pass_ == "fprop":
            return self.M, self.Nout, self.Kin
        if pass_ == "dgrad":
            return self.M, self.Kin, self.Nout
        return self.Nout, self.Kin, self.M


class Layer:
    """The four linears of one transformer layer with shared DelayedScaling state."""

    def __init__(self, tensors, recipes=RECIPES, history_len: int = 16, rht_signs: int = 0, sr_seed: int = 0,
                 device="cuda", names=None):
        n = len(tensors)
        self.recipes = recipes
        self.fwd = DelayedState(2 * n, history_len, device)
        self.bwd = DelayedState(n, history_len, device)
        self.recipe = L.te_recipe(L.E4M3, L.E5M2, history_len, L.ALGO_MAX, 0, 1)
        self.linears = [QuantLinear(x, w, dy, b, recipes, rht_signs, sr_seed, self.fwd, (2 * i, 2 * i + 1),
                                    self.bwd, i) for i, (x, w, dy, b) in enumerate(tensors)]
        default = LAYER_LINEARS if n == len(LAYER_LINEARS) else tuple(f"linear{i}" for i in range(n))
        for lin, name in zip(self.linears, names or default):
            lin.name = name
        self.step_idx = 0

    def state_dict(self) -> dict:
        """DelayedScaling state of the layer (both directions) and its step counter, on the host."""
        return {"fwd": self.fwd.state_dict(), "bwd": self.bwd.state_dict(), "step": self.step_idx}

    def load_state_dict(self, sd: dict) -> None:
        self.fwd.load_state_dict(sd["fwd"])
        self.bwd.load_state_dict(sd["bwd"])
        self.step_idx = int(sd["step"])

    def scale_update(self) -> None:
        """DelayedScaling bookkeeping after a step: record amaxes, refresh scales (two launches)."""
        L.te_scale_update(self.recipe, 0, self.fwd.hist, self.fwd.amax, self.fwd.scale, self.fwd.scale_inv,
                          self.step_idx)
        L.te_scale_update(self.recipe, 1, self.bwd.hist, self.bwd.amax, self.bwd.scale, self.bwd.scale_inv,
                          self.step_idx)

    def run_linear(self, i: int, recipe: str, autocast: bool = True, on_gemm=None) -> None:
        """The three GEMMs of linear ``i``; ``on_gemm(lin, pass_, phase)`` brackets each GEMM launch."""
        lin = self.linears[i]
        lin.sr_offset = self.step_idx
        for p in PASSES:
            if autocast:
                lin.quantize(recipe, p)
            if on_gemm:
                on_gemm(lin, p, 0)
            lin.gemm(recipe, p)
            if on_gemm:
                on_gemm(lin, p, 1)

    def run(self, recipe: str, autocast: bool = True, on_gemm=None) -> None:
        """One layer's 12 GEMMs, linear by linear, then the DelayedScaling update."""
        for i in range(len(self.linears)):
            self.run_linear(i, recipe, autocast, on_gemm)
        if autocast and recipe == "fp8_delayed":
            self.scale_update()


class HostStreamedLayer:
    """Runs a ``Layer`` whose inputs and outputs live in pinned host memory.

    Per linear, the host-to-device copies of X, W, dY and the bias go on one stream,
    the linear's three GEMMs (with their quantizers) on a second, and the device-to-host
    copies of Y, dX and dW on a third.  Events order each linear's buffers across steps
    (a step's input copies wait until the previous step's GEMMs of that linear are done;
    its GEMMs wait until the previous step's outputs have left), so the transfers of one
    linear overlap the compute of its neighbours.  ``host_in[i] = (x, w, dy, bias)`` and
    ``host_out[i] = (y, dx, dw)`` are pinned CPU tensors shaped like the linear's buffers.
    """

    def __init__(self, layer: Layer, host_in, host_out):
        import torch
        self.layer, self.host_in, self.host_out = layer, host_in, host_out
        self.s_in, self.s_comp, self.s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        n = len(layer.linears)
        self.ev = {k: [torch.cuda.Event() for _ in range(n)] for k in ("in", "comp", "out")}

    def streams(self):
        return self.s_in, self.s_comp, self.s_out

    def step(self, recipe: str, autocast: bool = True) -> None:
        import torch
        ev = self.ev
        for i, (lin, (x, w, dy, b), (y, dx, dw)) in enumerate(zip(self.layer.linears, self.host_in, self.host_out)):
            with torch.cuda.stream(self.s_in):
                self.s_in.wait_event(ev["comp"][i])
                lin.x.copy_(x, non_blocking=True)
                lin.w.copy_(w, non_blocking=True)
                lin.dy.copy_(dy, non_blocking=True)
                if lin.bias is not None and b is not None:
                    lin.bias.copy_(b, non_blocking=True)
                ev["in"][i].record(self.s_in)
            with torch.cuda.stream(self.s_comp):
                self.s_comp.wait_event(ev["in"][i])
                self.s_comp.wait_event(ev["out"][i])
                self.layer.run_linear(i, recipe, autocast)
                ev["comp"][i].record(self.s_comp)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev["comp"][i])
                y.copy_(lin.y, non_blocking=True)
                dx.copy_(lin.dx, non_blocking=True)
                dw.copy_(lin.dw, non_blocking=True)
                ev["out"][i].record(self.s_out)
        if autocast and recipe == "fp8_delayed":
            with torch.cuda.stream(self.s_comp):
                self.layer.scale_update()


class ScheduleStep:
    """A training step's worth of linears under DelayedScaling (the 24-layer schedule).

    Per layer and linear, each tensor is quantized once per step into both copies (the
    DelayedScaling cast records its amax in the same read), then the linear's Fprop, Dgrad
    and Wgrad GEMMs run; after the last layer one batched scale update per direction
    records the amaxes and refreshes every scale ("Introduction to FP8 training using
    Transformer Engine": DelayedScaling with an amax history, HYBRID formats).  Quantized
    copies and outputs are shared by the layers (each layer's are consumed before the next
    layer overwrites them); inputs are per layer.  ``layers[l][i] = (x, w, dy, bias)``.
    """

    def __init__(self, layers, history_len: int = 16, device="cuda", recipe: str = "fp8_delayed"):
        import torch
        assert recipe in ("fp8_delayed", "bf16"), recipe
        self.layers = layers
        self.kind = recipe
        n_lin = sum(len(lin) for lin in layers)
        self.fwd = DelayedState(2 * n_lin, history_len, device)
        self.bwd = DelayedState(n_lin, history_len, device)
        self.recipe = L.te_recipe(L.E4M3, L.E5M2, history_len, L.ALGO_MAX, 0, 1)
        self.history_len = history_len
        u8 = dict(dtype=torch.uint8, device=device)
        bf = torch.bfloat16
        self.bufs = {}
        for lin in layers:
            for x, w, dy, _ in lin:
                key = (x.shape[0], x.shape[1], w.shape[0])
                if key in self.bufs:
                    continue
                M, K, N = key
                self.bufs[key] = dict(y=torch.empty(M, N, dtype=bf, device=device),
                                      dx=torch.empty(M, K, dtype=bf, device=device),
                                      dw=torch.empty(N, K, dtype=bf, device=device))
                if recipe == "fp8_delayed":
                    self.bufs[key].update(xr=torch.empty(M, K, **u8), xc=torch.empty(K, M, **u8),
                                          wr=torch.empty(N, K, **u8), wc=torch.empty(K, N, **u8),
                                          dr=torch.empty(M, N, **u8), dc=torch.empty(N, M, **u8))

    def state_dict(self) -> dict:
        return {"fwd": self.fwd.state_dict(), "bwd": self.bwd.state_dict()}

    def load_state_dict(self, sd: dict) -> None:
        self.fwd.load_state_dict(sd["fwd"])
        self.bwd.load_state_dict(sd["bwd"])

    def run(self, step: int) -> None:
        if self.kind == "bf16":
            return self._run_bf16()
        E4, E5 = L.E4M3, L.E5M2
        k = 0
        fs, fsi, fa = self.fwd.scale, self.fwd.scale_inv, self.fwd.amax
        bs, bsi, ba = self.bwd.scale, self.bwd.scale_inv, self.bwd.amax
        for lin in self.layers:
            for x, w, dy, bias in lin:
                b = self.bufs[(x.shape[0], x.shape[1], w.shape[0])]
                ix, iw = 2 * k, 2 * k + 1
                L.te_quantize_fp8(x, E4, fs[ix:ix + 1], 0, b["xr"], b["xc"], fa[ix:ix + 1])
                L.te_quantize_fp8(w, E4, fs[iw:iw + 1], 0, b["wr"], b["wc"], fa[iw:iw + 1])
                L.te_quantize_fp8(dy, E5, bs[k:k + 1], 0, b["dr"], b["dc"], ba[k:k + 1])
                L.te_gemm_fp8(b["xr"], E4, b["wr"], E4, fsi[ix:ix + 1], fsi[iw:iw + 1], b["y"], bias)
                L.te_gemm_fp8(b["dr"], E5, b["wc"], E4, bsi[k:k + 1], fsi[iw:iw + 1], b["dx"])
                L.te_gemm_fp8(b["dc"], E5, b["xc"], E4, bsi[k:k + 1], fsi[ix:ix + 1], b["dw"])
                k += 1
        L.te_scale_update(self.recipe, 0, self.fwd.hist, fa, fs, fsi, step)
        L.te_scale_update(self.recipe, 1, self.bwd.hist, ba, bs, bsi, step)

    def _run_bf16(self) -> None:
        """The same GEMMs in BF16 on the unquantized tensors (no scaling state)."""
        KM, MN = L.K_MAJOR, L.MN_MAJOR
        for lin in self.layers:
            for x, w, dy, bias in lin:
                b = self.bufs[(x.shape[0], x.shape[1], w.shape[0])]
                L.te_gemm_bf16(x, w, b["y"], bias, KM, KM)
                L.te_gemm_bf16(dy, w, b["dx"], None, KM, MN)
                L.te_gemm_bf16(dy, x, b["dw"], None, MN, MN)

    def gemm_flops(self) -> float:
        return sum(6.0 * x.shape[0] * x.shape[1] * w.shape[0] for lin in self.layers for x, w, _, _ in lin)


class ScheduleGraphs:
    """CUDA-graph replay of a ``ScheduleStep``: one graph per history slot.

    A step's launches differ only in the history slot its scale update writes (step mod
    the history length, with the update interval 1 of the recipe), so one captured graph
    per slot replays any step.  Capture after at least one eager step (first calls set
    kernel attributes)."""

    def __init__(self, sched: ScheduleStep):
        import torch
        self.sched = sched
        self.graphs = []
        stream = torch.cuda.Stream()
        for slot in range(sched.history_len):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                sched.run(slot)
            self.graphs.append(g)

    def run(self, step: int) -> None:
        self.graphs[step % self.sched.history_len].replay()
