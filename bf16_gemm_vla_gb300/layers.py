"""Load-time weight preparation and a static-buffer linear layer.

Load time ("Real-time VLA inference on AMD hardware", "How FlashRT works":
the weights are quantized and packed once, at load, and the choices are
frozen before the graph is recorded):

  FP8:  W fp32 [K x N] --quantize per output channel--> E4M3 bytes + scales
        (optionally produced in FNUZ, as an import from a CDNA3 checkpoint,
        then re-encoded to OCP) --pack--> tile layout.
  BF16: W fp32 --round to bf16 and pack--> tile layout.

A ``Linear`` owns every buffer its forward touches (the quantized
activation, its scale, the quantize workspace and the output), so a
sequence of ``Linear`` calls can be captured into a CUDA graph and replayed
with static pointers and shapes.
"""
from dataclasses import dataclass
from typing import Optional

import torch

from . import frt


@dataclass
class PackedWeight:
    packed: torch.Tensor            # uint8 tile-layout buffer
    K: int
    N: int
    kind: str                       # "e4m3" or "bf16"
    w_scale: Optional[torch.Tensor]  # fp32 [N] (FP8) or None
    bias: Optional[torch.Tensor]    # fp32 [N] or None


def prepare_fp8(w_f32, bias=None, import_fnuz=False):
    """Quantize W per output channel to E4M3 and pack it.  With
    ``import_fnuz`` the bytes are first produced in FNUZ (scale amax/240)
    and re-encoded to OCP in place."""
    K, N = w_f32.shape
    fmt = frt.FNUZ if import_fnuz else frt.OCP
    q, s = frt.frt_quantize_e4m3(w_f32, frt.PER_COL, fmt)
    if import_fnuz:
        frt.frt_fnuz_to_ocp(q.view(-1), out=q.view(-1))
    packed = frt.frt_pack_weights(q, "e4m3")
    # packed weights are load-time data: complete before any GEMM reads them
    torch.cuda.current_stream(packed.device).synchronize()
    return PackedWeight(packed, K, N, "e4m3", s, bias)


@dataclass
class PackedNvfp4:
    packed: torch.Tensor  # uint8 tile-layout buffer of the [K/2 x N] code bytes
    sf: torch.Tensor      # uint8 tiled block scales of the N channels
    g: torch.Tensor       # fp32 [1] tensor scale
    K: int
    N: int
    bias: Optional[torch.Tensor]


def prepare_nvfp4(w_f32, bias=None):
    """Quantize W [K x N] to NVFP4 (blocks of 16 along K, per output channel)
    and pack its codes for the GEMM."""
    K, N = w_f32.shape
    q, sf, g = frt.frt_quantize_nvfp4(w_f32, blocks_along_rows=True)
    packed = frt.frt_pack_weights(q, "e4m3")
    torch.cuda.current_stream(packed.device).synchronize()
    return PackedNvfp4(packed, sf, g, K, N, bias)


def prepare_bf16(w, bias=None):
    """Round W (fp32 or bf16) to bf16 and pack it."""
    K, N = w.shape
    packed = frt.frt_pack_weights(w, "bf16")
    torch.cuda.current_stream(packed.device).synchronize()
    return PackedWeight(packed, K, N, "bf16", None, bias)


class Linear:
    """One linear layer with static buffers, for a fixed number of rows M.

    FP8:  q, s = quantize(x) per tensor (OCP); out = gemm_fp8(q, s, W).
    BF16: out = gemm_bf16(x, W).
    ``act_cols`` output columns get the tanh-GELU.

    FP8 activation scales are dynamic (amax of every input) until
    ``calibrate`` freezes one: then each call only encodes with it (one
    pass over x instead of amax + encode).
    """

    def __init__(self, weight: PackedWeight, M, act_cols=0, out=None, device=None, geglu=False):
        self.w = weight
        self.M = M
        self.act_cols = act_cols
        # merged gate/up (gate channels first) with the GeGLU fused: the
        # output is gelu(gate) * up, N / 2 columns
        self.geglu = geglu
        dev = device if device is not None else weight.packed.device
        n_out = weight.N // 2 if geglu else weight.N
        self.out = out if out is not None else torch.empty((M, n_out), dtype=torch.bfloat16,
                                                            device=dev)
        if weight.kind == "e4m3":
            self.q = torch.empty((M, weight.K), dtype=torch.uint8, device=dev)
            self.a_scale = torch.empty((1,), dtype=torch.float32, device=dev)
            nb = frt.frt_quantize_workspace_bytes(M, weight.K, frt.PER_TENSOR)
            self.ws = torch.zeros((max(nb, 4) // 4,), dtype=torch.float32, device=dev)
            self.static = False
            self.s_out = torch.empty((1,), dtype=torch.float32, device=dev)  # static path's copy
            # header for a previous GEMM that takes this layer's activation
            # scale from its own output (zero-filled once)
            self.sws = frt.next_scale_workspace(dev)
        # the GEMM's own (zero-filled) workspace, or False if it needs none
        gws = frt.gemm_workspace(M, weight.N, weight.K, weight.kind, dev)
        self.gws = False if gws is None else gws

    def calibrate(self, xs, stream=None):
        """Freezes the activation scale at the largest dynamic scale over the
        calibration inputs ``xs`` (each [M x K] bf16): s = max_i amax_i / 448,
        which is the dynamic scale of all of them together since the rounded
        division is monotone.  Later calls encode with it; inputs beyond the
        calibrated range saturate to +-448.  Load-time: synchronises."""
        if self.w.kind != "e4m3":
            raise ValueError("calibrate applies to FP8 layers")
        best = None
        for x in xs:
            frt.frt_quantize_e4m3(x, frt.PER_TENSOR, frt.OCP, q=self.q, scale=self.a_scale,
                                  workspace=self.ws, stream=stream)
            torch.cuda.synchronize(self.a_scale.device)
            s = float(self.a_scale.cpu()[0])
            best = s if best is None or s > best else best
        self.a_scale.fill_(best)
        torch.cuda.synchronize(self.a_scale.device)
        self.static = True
        return best

    def quantize(self, x, stream=None, scale_ready=False):
        """FP8 layers: the activation quantize of x into self.q / self.a_scale
        (nothing for BF16 layers).  scale_ready: the GEMM that produced x has
        written x's scale into self.a_scale already, so this is the encode
        pass alone."""
        if self.w.kind != "e4m3":
            return
        if self.static or scale_ready:
            frt.frt_quantize_e4m3(x, frt.PER_TENSOR, frt.OCP, static_scale=self.a_scale,
                                  q=self.q, scale=self.s_out, stream=stream)
        else:
            frt.frt_quantize_e4m3(x, frt.PER_TENSOR, frt.OCP, q=self.q, scale=self.a_scale,
                                  workspace=self.ws, stream=stream)

    def gemm(self, x, stream=None, next_layer=None):
        """The GEMM alone: FP8 layers read self.q / self.a_scale (x unused),
        BF16 layers read x.  next_layer: an FP8 Linear with a dynamic scale
        whose input is the first next_layer.w.K columns of this layer's
        output; the GEMM then also writes that input's scale into
        next_layer.a_scale (taken in its epilogue), and next_layer's quantize
        is called with scale_ready=True."""
        w = self.w
        if next_layer is not None:
            nl = next_layer
            if nl.w.kind != "e4m3" or nl.static:
                raise ValueError("the next layer's scale is taken for an FP8 layer with a "
                                 "dynamic scale")
            kw = dict(scale_cols=nl.w.K, scale=nl.a_scale, scale_workspace=nl.sws,
                      stream=stream, workspace=self.gws, geglu=self.geglu, bias=w.bias,
                      act_cols=self.act_cols, out=self.out)
            if w.kind == "e4m3":
                return frt.frt_gemm_fp8_next_scale(self.q, self.a_scale, w.packed, w.w_scale, w.N,
                                                   **kw)[0]
            return frt.frt_gemm_bf16_next_scale(x, w.packed, w.N, w_scale=w.w_scale, **kw)[0]
        if w.kind == "e4m3":
            return frt.frt_gemm_fp8(self.q, self.a_scale, w.packed, w.w_scale, w.N, bias=w.bias,
                                    act_cols=self.act_cols, out=self.out, stream=stream,
                                    workspace=self.gws, geglu=self.geglu)
        return frt.frt_gemm_bf16(x, w.packed, w.N, w_scale=w.w_scale, bias=w.bias,
                                 act_cols=self.act_cols, out=self.out, stream=stream,
                                 workspace=self.gws, geglu=self.geglu)

    def __call__(self, x, stream=None):
        self.quantize(x, stream)
        return self.gemm(x, stream)
