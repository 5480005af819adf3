"""The synthetic encoder/decoder stack, captured and replayed as one CUDA graph.

The method records the whole forward once and replays it, so the per-op
launch overhead is paid once at load ("Real-time VLA inference on AMD
hardware", "How FlashRT works"; the recorded region must use static
pointers, no allocation and no host reads, "Deploying DeepSeek-V4-Flash on
AMD MI300X", "HIP Graphs").  The stack here is the linear-layer skeleton of
a pi0.5-style pass:

  encoder: 18 layers at M = 768, hidden 2048, FP8 -- QKV 2048->2560,
           O 2048->2048, merged gate/up 2048->2x16384 (tanh-GELU on the gate
           half), down 16384->2048; every GEMM's input quantized per tensor
           (the first one by the activation quantize; for each later one the
           previous GEMM takes the scale from its own output in its
           epilogue, and the quantize is the encode pass alone; with
           fuse_quantize=False a full quantize, amax included, each);
  decoder: 18 layers at M = 50, hidden 1024, BF16 -- QKV 1024->2560,
           O 2048->1024, gate/up 1024->2x4096, down 4096->1024.

Attention, the GeGLU product, residuals and norms are not part of this
path.  Their places are taken by strided views: O reads the first K columns
of the QKV output, down reads the gate half of the gate/up output, and the
next layer reads the down output.

Weights (N(0, 0.02)) and biases (N(0, 0.1)) are drawn on the device from a
seeded torch generator, one layer after another in the order above.
"""
import torch

from . import frt, layers

ENCODER = (("qkv", 2048, 2560, 0), ("o", 2048, 2048, 0), ("gate_up", 2048, 32768, 16384),
           ("down", 16384, 2048, 0))
DECODER = (("qkv", 1024, 2560, 0), ("o", 2048, 1024, 0), ("gate_up", 1024, 8192, 4096),
           ("down", 4096, 1024, 0))
M_ENC = 768
M_DEC = 50


class SyntheticStack:
    def __init__(self, n_layers=18, seed=1, device="cuda", enc_kind="e4m3", dec_kind="bf16",
                 keep=(0, 17), parts=("enc", "dec"), fuse_quantize=True):
        """parts: the chains to build ("enc", "dec" or both); a chain left out
        is empty and its weights are not drawn (the other chain's draws are
        then not those of the full stack).  fuse_quantize: an FP8 layer fed
        by a GEMM gets its input's scale from that GEMM's epilogue, so its
        quantize is the encode pass alone."""
        self.device = torch.device(device)
        self.fuse_quantize = fuse_quantize
        self.n_layers = n_layers
        g = torch.Generator(device=self.device)
        g.manual_seed(seed)
        self.kept = {}  # (part, layer, name) -> (w fp32 cpu, bias fp32 cpu)
        self.enc = self._build("enc", ENCODER, M_ENC, enc_kind, g, keep) if "enc" in parts else []
        self.dec = self._build("dec", DECODER, M_DEC, dec_kind, g, keep) if "dec" in parts else []
        self.x_enc = torch.zeros((M_ENC, ENCODER[0][1]), dtype=torch.bfloat16, device=self.device)
        self.x_dec = torch.zeros((M_DEC, DECODER[0][1]), dtype=torch.bfloat16, device=self.device)
        self.graph = None

    def _build(self, part, spec, M, kind, g, keep):
        out = []
        for li in range(self.n_layers):
            lay = {}
            for name, K, N, act in spec:
                w = torch.randn((K, N), generator=g, device=self.device, dtype=torch.float32) * 0.02
                b = torch.randn((N,), generator=g, device=self.device, dtype=torch.float32) * 0.1
                if li in keep:
                    self.kept[(part, li, name)] = (w.cpu(), b.cpu())
                pw = layers.prepare_fp8(w, b) if kind == "e4m3" else layers.prepare_bf16(w, b)
                lay[name] = layers.Linear(pw, M, act_cols=act, device=self.device)
                del w
            out.append(lay)
        return out

    def op_list(self):
        """Every launch of one forward in order, as (part, layer, name, op,
        lin, call): op is "quantize" (a full activation quantize), "encode"
        (the quantize of an input whose scale the GEMM before it took),
        "gemm", or "gemm+scale" (the GEMM also takes the next, FP8, layer's
        input scale); lin is the layer's Linear, and call(stream) enqueues
        the launch on the buffers the forward uses."""
        ops = []
        for part, chain in (("enc", self.enc), ("dec", self.dec)):
            flat = [(li, name, lay[name]) for li, lay in enumerate(chain)
                    for name in ("qkv", "o", "gate_up", "down")]
            scaled = False  # this layer's input scale was taken by the previous GEMM
            for i, (li, name, lin) in enumerate(flat):
                x = self.inputs_of(part, li, name)
                nl = flat[i + 1][2] if i + 1 < len(flat) else None
                fuse = (self.fuse_quantize and nl is not None and nl.w.kind == "e4m3"
                        and not nl.static)
                if lin.w.kind == "e4m3":
                    ops.append((part, li, name, "encode" if scaled else "quantize", lin,
                                lambda s=None, lin=lin, x=x, r=scaled:
                                lin.quantize(x, s, scale_ready=r)))
                ops.append((part, li, name, "gemm+scale" if fuse else "gemm", lin,
                            lambda s=None, lin=lin, x=x, nl=(nl if fuse else None):
                            lin.gemm(x, s, next_layer=nl)))
                scaled = fuse
        return ops

    def inputs_of(self, part, li, name):
        """The activation tensor layer (part, li, name) reads, after a forward."""
        chain = self.enc if part == "enc" else self.dec
        lay = chain[li]
        if name == "qkv":
            if li == 0:
                return self.x_enc if part == "enc" else self.x_dec
            return chain[li - 1]["down"].out
        if name == "o":
            return lay["qkv"].out[:, : lay["o"].w.K]
        if name == "gate_up":
            return lay["o"].out
        return lay["gate_up"].out[:, : lay["down"].w.K]

    def forward(self, stream=None):
        """One eager pass (encoder chain, then decoder chain); returns the last
        layer's output of each chain (its input where the chain is empty)."""
        for op in self.op_list():
            op[-1](stream)
        e = self.enc[-1]["down"].out if self.enc else self.x_enc
        d = self.dec[-1]["down"].out if self.dec else self.x_dec
        return e, d

    def launches_per_forward(self):
        """Kernels one forward launches, counted by the library (a full
        quantize takes one grid when its input is dense and fits on chip,
        else two; an encode with a given scale and every GEMM one)."""
        n0 = frt.frt_launch_count()
        self.forward()
        torch.cuda.synchronize(self.device)
        return frt.frt_launch_count() - n0

    def capture(self):
        """Records one forward into a CUDA graph (after one eager warm-up that
        sets every kernel's attributes)."""
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.forward()
        torch.cuda.current_stream(self.device).wait_stream(s)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.forward()
        return self.graph

    def replay(self):
        self.graph.replay()

    def weight_bytes(self):
        return sum(lin.w.packed.numel() for chain in (self.enc, self.dec)
                   for lay in chain for lin in lay.values())
