"""Python binding of libfrt: the same entry points as include/frt.h, taking
torch tensors.  Argument marshalling only -- every step of the path runs in
the library's CUDA kernels; PyTorch provides device memory and the stream.

Outputs that are not passed in are allocated with torch; for CUDA-graph
capture pass every buffer in (the calls then allocate nothing).
"""
import ctypes

import torch

from . import _lib

OCP = "ocp"
FNUZ = "fnuz"
PER_TENSOR = "per_tensor"
PER_COL = "per_col"

_FMT = {OCP: _lib.FRT_E4M3_OCP, FNUZ: _lib.FRT_E4M3_FNUZ}
_MODE = {PER_TENSOR: _lib.FRT_SCALE_PER_TENSOR, PER_COL: _lib.FRT_SCALE_PER_COL}
_XDT = {torch.bfloat16: _lib.FRT_BF16, torch.float32: _lib.FRT_F32}


class FrtError(RuntimeError):
    """A libfrt call returned a status other than FRT_OK."""

    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s" % (fn, _lib.STATUS_NAMES.get(status, status)))


def _check(fn, status):
    if status != _lib.FRT_OK:
        raise FrtError(fn, status)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def lib():
    return _lib.load()


def _rows_view(x, name):
    if x.dim() != 2 or (x.shape[1] > 1 and x.stride(1) != 1) or not x.is_cuda:
        raise ValueError("%s must be a 2-D CUDA tensor with unit column stride" % name)
    return x.shape[0], x.shape[1], x.stride(0)


# ---------------------------------------------------------------- quantize

def frt_launch_count():
    """Kernels this library has launched (or recorded into a capture) so far."""
    return lib().frt_launch_count()


def frt_quantize_workspace_bytes(rows, cols, mode=PER_TENSOR):
    return lib().frt_quantize_workspace_bytes(rows, cols, _MODE[mode])


def frt_quantize_e4m3(x, mode=PER_TENSOR, out_fmt=OCP, static_scale=None, q=None, scale=None,
                      workspace=None, stream=None):
    """E4M3 bytes and dequant scale(s) of a 2-D bf16/fp32 tensor (rows may be
    strided).  Returns (q uint8 [rows x cols], scale fp32 [1] or [cols])."""
    rows, cols, ldx = _rows_view(x, "x")
    L = lib()
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((cols if mode == PER_COL else 1,), dtype=torch.float32, device=x.device)
    if static_scale is None and workspace is None:
        nb = L.frt_quantize_workspace_bytes(rows, cols, _MODE[mode])
        workspace = torch.zeros((max(nb, 4) // 4,), dtype=torch.float32, device=x.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("frt_quantize_e4m3",
           L.frt_quantize_e4m3(x.data_ptr(), _XDT[x.dtype], rows, cols, ldx, _MODE[mode],
                               _FMT[out_fmt], _ptr(static_scale), q.data_ptr(), _ptr(scale),
                               _ptr(workspace), wsb, _stream(stream)))
    return q, scale


def frt_quantize_e4m3_noalloc(x, mode=PER_TENSOR, out_fmt=OCP, static_scale=None, q=None,
                              scale=None, stream=None):
    """frt_quantize_e4m3 for callers that cannot allocate device memory: the
    amax partials use a fixed 1 MiB array inside the library.  Pass q and
    scale in to allocate nothing at all."""
    rows, cols, ldx = _rows_view(x, "x")
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((cols if mode == PER_COL else 1,), dtype=torch.float32, device=x.device)
    _check("frt_quantize_e4m3_noalloc",
           lib().frt_quantize_e4m3_noalloc(x.data_ptr(), _XDT[x.dtype], rows, cols, ldx,
                                           _MODE[mode], _FMT[out_fmt], _ptr(static_scale),
                                           q.data_ptr(), _ptr(scale), _stream(stream)))
    return q, scale


# ---------------------------------------------------------------- FNUZ -> OCP

def frt_fnuz_to_ocp(inp, out=None, stream=None):
    """OCP bytes holding the values of FNUZ bytes (out may be inp)."""
    if inp.dtype != torch.uint8 or not inp.is_contiguous():
        raise ValueError("inp must be a contiguous uint8 tensor")
    if out is None:
        out = torch.empty_like(inp)
    _check("frt_fnuz_to_ocp",
           lib().frt_fnuz_to_ocp(inp.data_ptr(), out.data_ptr(), inp.numel(), _stream(stream)))
    return out


# ---------------------------------------------------------------- pack

def frt_packed_weight_bytes(K, N, packed_dtype="e4m3"):
    dt = _lib.FRT_E4M3_OCP if packed_dtype == "e4m3" else _lib.FRT_BF16
    return lib().frt_packed_weight_bytes(K, N, dt)


def frt_pack_weights(w, packed_dtype="e4m3", packed=None, stream=None):
    """Packs W [K x N] (uint8 OCP E4M3 bytes for 'e4m3'; fp32 or bf16 for
    'bf16') into the kernels' tile layout; returns the uint8 buffer.

    Load-time: a GEMM fetches its weight tiles before waiting for the kernel
    launched just before it, so synchronise (or launch another kernel)
    between packing and the first GEMM that reads the result."""
    K, N, ldw = _rows_view(w, "w")
    if packed_dtype == "e4m3":
        if w.dtype != torch.uint8:
            raise ValueError("e4m3 packing takes OCP E4M3 bytes (uint8)")
        wdt, pdt = _lib.FRT_E4M3_OCP, _lib.FRT_E4M3_OCP
    else:
        wdt, pdt = _XDT[w.dtype], _lib.FRT_BF16
    nbytes = lib().frt_packed_weight_bytes(K, N, pdt)
    if packed is None:
        packed = torch.empty((nbytes,), dtype=torch.uint8, device=w.device)
    _check("frt_pack_weights",
           lib().frt_pack_weights(w.data_ptr(), wdt, K, N, ldw, pdt, packed.data_ptr(),
                                  packed.numel(), _stream(stream)))
    return packed


# ---------------------------------------------------------------- GEMMs

_STATUS = {}


def device_status(device=None):
    """The per-device int32 status word the GEMMs report bounded-wait
    expiry into (zero while healthy)."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device.index)
    if dev not in _STATUS:
        _STATUS[dev] = torch.zeros((1,), dtype=torch.int32, device=dev)
    return _STATUS[dev]


def check_device_status(device=None):
    """Raises FrtError(FRT_ERR_TIMEOUT) if a kernel reported an expired wait
    (synchronises with the device)."""
    st = device_status(device)
    code = int(st.item())
    if code:
        st.zero_()
        raise FrtError("device wait (code 0x%x)" % code, 6)


_GEMM_DTYPE = {"e4m3": _lib.FRT_E4M3_OCP, "bf16": _lib.FRT_BF16}
_GEMM_WS = {}
_GEMM_WS_RETIRED = []


def frt_gemm_workspace_bytes(M, N, K, kind="e4m3"):
    """Bytes of GEMM workspace the plan of this shape uses on the current
    device (0: none).  A workspace must be zero-filled before its first use;
    the GEMM leaves it so."""
    return lib().frt_gemm_workspace_bytes(M, N, K, _GEMM_DTYPE[kind])


def frt_gemm_describe(M, N, K, kind="e4m3", workspace_bytes=None):
    """The launch plan of an M x N x K GEMM on the current device, as a dict
    (kind, bn, kbs, stages, splits, global, tiles, grid, cluster, smem).  workspace_bytes: the usable workspace (None: as much as the plan
    wants, which is what the default shared workspace provides)."""
    if workspace_bytes is None:
        workspace_bytes = (1 << 64) - 1
    buf = ctypes.create_string_buffer(256)
    n = lib().frt_gemm_describe(M, N, K, _GEMM_DTYPE[kind], workspace_bytes, buf, len(buf))
    if n < 0:
        raise FrtError("frt_gemm_describe: unsupported problem", 1)
    plan = {}
    for field in buf.value.decode().split():
        key, val = field.split("=")
        if key == "kind":
            plan[key] = val
        elif "," in val:
            plan[key] = tuple(int(v) for v in val.split(","))
        else:
            plan[key] = int(val)
    return plan


def gemm_workspace(M, N, K, kind="e4m3", device=None):
    """A zero-filled workspace for one layer's GEMM (None if it needs none)."""
    nb = frt_gemm_workspace_bytes(M, N, K, kind)
    if nb == 0:
        return None
    return torch.zeros((nb,), dtype=torch.uint8, device=device)


def _gemm_ws(workspace, M, N, K, kind, device):
    """(pointer, bytes) of the workspace to pass: the caller's; none for
    workspace=False; else a per-device shared one (calls that use it must be
    ordered on one stream), grown on demand."""
    if workspace is False:
        return None, 0
    if workspace is not None:
        return workspace.data_ptr(), workspace.numel() * workspace.element_size()
    nb = frt_gemm_workspace_bytes(M, N, K, kind)
    if nb == 0:
        return None, 0
    ws = _GEMM_WS.get(device)
    if ws is None or ws.numel() < nb:
        if ws is not None:
            _GEMM_WS_RETIRED.append(ws)  # may still be in use by queued work
        ws = torch.zeros((nb,), dtype=torch.uint8, device=device)
        _GEMM_WS[device] = ws
    return ws.data_ptr(), ws.numel()


def _gemm_out(M, N, out, device):
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    if out.dtype != torch.bfloat16:
        raise ValueError("out must be bf16")
    _, _, ldo = _rows_view(out, "out")
    return out, ldo


def _act(act_cols, geglu):
    if geglu:
        return _lib.FRT_ACT_GEGLU, 0
    return (_lib.FRT_ACT_GELU_TANH if act_cols else _lib.FRT_ACT_NONE), act_cols


def frt_gemm_fp8(a_q, a_scale, w_packed, w_scale, N, bias=None, act_cols=0, out=None,
                 stream=None, workspace=None, geglu=False):
    """out = bf16(act(a_scale * w_scale[n] * (A_q . W) + bias[n])), GELU on
    the first act_cols columns.  a_q: [M x K] OCP E4M3 bytes.  workspace: a
    zero-filled uint8 tensor of frt_gemm_workspace_bytes() bytes, False for
    none, or None for the shared per-device one.  geglu: W is a merged
    gate/up weight (gate channels first) and out = gelu(gate) * up, N / 2
    columns."""
    M, K, lda = _rows_view(a_q, "a_q")
    out, ldo = _gemm_out(M, N // 2 if geglu else N, out, a_q.device)
    act, act_cols = _act(act_cols, geglu)
    wp, wb = _gemm_ws(workspace, M, N, K, "e4m3", a_q.device)
    _check("frt_gemm_fp8",
           lib().frt_gemm_fp8(a_q.data_ptr(), lda, _ptr(a_scale), w_packed.data_ptr(),
                              _ptr(w_scale), _ptr(bias), M, N, K, act, act_cols, out.data_ptr(),
                              ldo, wp, wb, device_status(a_q.device).data_ptr(),
                              _stream(stream)))
    return out


def frt_gemm_bf16(a, w_packed, N, w_scale=None, bias=None, act_cols=0, out=None, stream=None,
                  workspace=None, geglu=False):
    """out = bf16(act(w_scale[n] * (A . W) + bias[n])).  a: [M x K] bf16.
    workspace and geglu as for frt_gemm_fp8."""
    M, K, lda = _rows_view(a, "a")
    out, ldo = _gemm_out(M, N // 2 if geglu else N, out, a.device)
    act, act_cols = _act(act_cols, geglu)
    wp, wb = _gemm_ws(workspace, M, N, K, "bf16", a.device)
    _check("frt_gemm_bf16",
           lib().frt_gemm_bf16(a.data_ptr(), lda, w_packed.data_ptr(), _ptr(w_scale), _ptr(bias),
                               M, N, K, act, act_cols, out.data_ptr(), ldo, wp, wb,
                               device_status(a.device).data_ptr(), _stream(stream)))
    return out


def frt_gemm_next_scale_workspace_bytes():
    return lib().frt_gemm_next_scale_workspace_bytes()


def next_scale_workspace(device=None):
    """A zero-filled header for the next layer's scale taken by a GEMM."""
    return torch.zeros((frt_gemm_next_scale_workspace_bytes(),), dtype=torch.uint8, device=device)


def _next_scale(out, scale_cols, scale, scale_workspace):
    if scale_cols is None:
        scale_cols = out.shape[1]
    if scale is None:
        scale = torch.empty((1,), dtype=torch.float32, device=out.device)
    if scale_workspace is None:
        scale_workspace = next_scale_workspace(out.device)
    return (scale_cols, scale, scale_workspace.data_ptr(),
            scale_workspace.numel() * scale_workspace.element_size())


def frt_gemm_fp8_next_scale(a_q, a_scale, w_packed, w_scale, N, bias=None, act_cols=0, out=None,
                            scale_cols=None, scale=None, scale_workspace=None, stream=None,
                            workspace=None, geglu=False):
    """frt_gemm_fp8 that also writes the per-tensor OCP E4M3 scale of its own
    bf16 output out[:, :scale_cols] (amax / 448) for the next FP8 layer,
    whose quantize is then frt_quantize_e4m3(out[:, :scale_cols],
    static_scale=scale).  Returns (out, scale).  scale_workspace: a
    zero-filled header (shared only by calls ordered on one stream;
    allocated when not given)."""
    M, K, lda = _rows_view(a_q, "a_q")
    out, ldo = _gemm_out(M, N // 2 if geglu else N, out, a_q.device)
    cols, scale, sw, swb = _next_scale(out, scale_cols, scale, scale_workspace)
    act, act_cols = _act(act_cols, geglu)
    wp, wb = _gemm_ws(workspace, M, N, K, "e4m3", a_q.device)
    _check("frt_gemm_fp8_next_scale",
           lib().frt_gemm_fp8_next_scale(a_q.data_ptr(), lda, _ptr(a_scale), w_packed.data_ptr(),
                                         _ptr(w_scale), _ptr(bias), M, N, K, act, act_cols,
                                         out.data_ptr(), ldo, cols, scale.data_ptr(), sw, swb,
                                         wp, wb, device_status(a_q.device).data_ptr(),
                                         _stream(stream)))
    return out, scale


def frt_gemm_bf16_next_scale(a, w_packed, N, w_scale=None, bias=None, act_cols=0, out=None,
                             scale_cols=None, scale=None, scale_workspace=None, stream=None,
                             workspace=None, geglu=False):
    """frt_gemm_bf16 that also writes the next FP8 layer's scale (as
    frt_gemm_fp8_next_scale).  Returns (out, scale)."""
    M, K, lda = _rows_view(a, "a")
    out, ldo = _gemm_out(M, N // 2 if geglu else N, out, a.device)
    cols, scale, sw, swb = _next_scale(out, scale_cols, scale, scale_workspace)
    act, act_cols = _act(act_cols, geglu)
    wp, wb = _gemm_ws(workspace, M, N, K, "bf16", a.device)
    _check("frt_gemm_bf16_next_scale",
           lib().frt_gemm_bf16_next_scale(a.data_ptr(), lda, w_packed.data_ptr(), _ptr(w_scale),
                                          _ptr(bias), M, N, K, act, act_cols, out.data_ptr(), ldo,
                                          cols, scale.data_ptr(), sw, swb, wp, wb,
                                          device_status(a.device).data_ptr(), _stream(stream)))
    return out, scale


# ---------------------------------------------------------------- NVFP4

def frt_nvfp4_scale_bytes(vectors, K):
    return lib().frt_nvfp4_scale_bytes(vectors, K)


def nvfp4_workspace(device=None):
    """A zero-filled 16-byte workspace for frt_quantize_nvfp4's amax."""
    return torch.zeros((lib().frt_quantize_nvfp4_workspace_bytes(),), dtype=torch.uint8,
                       device=device)


def frt_quantize_nvfp4(x, blocks_along_rows=False, static_scale=None, q=None, sf=None,
                       scale=None, workspace=None, stream=None):
    """NVFP4 codes (two per byte along K), tiled block scales and the tensor
    scale g of a 2-D bf16/fp32 tensor.  blocks_along_rows=False: x is
    [M x K] and q [M x K/2]; True: x is a weight [K x N] and q [K/2 x N].
    Returns (q uint8, sf uint8, scale fp32 [1])."""
    rows, cols, ldx = _rows_view(x, "x")
    V, K = (cols, rows) if blocks_along_rows else (rows, cols)
    qshape = (rows // 2, cols) if blocks_along_rows else (rows, cols // 2)
    if q is None:
        q = torch.empty(qshape, dtype=torch.uint8, device=x.device)
    nsf = lib().frt_nvfp4_scale_bytes(V, K)
    if sf is None:
        sf = torch.empty((max(nsf, 1),), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty((1,), dtype=torch.float32, device=x.device)
    if static_scale is None and workspace is None:
        workspace = nvfp4_workspace(x.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("frt_quantize_nvfp4",
           lib().frt_quantize_nvfp4(x.data_ptr(), _XDT[x.dtype], rows, cols, ldx,
                                    1 if blocks_along_rows else 0, _ptr(static_scale),
                                    q.data_ptr(), sf.data_ptr(), sf.numel(), _ptr(scale),
                                    _ptr(workspace), wsb, _stream(stream)))
    return q, sf, scale


def frt_gemm_nvfp4(a_q, a_sf, a_scale, w_packed, w_sf, w_scale, N, bias=None, act_cols=0,
                   out=None, stream=None):
    """out = bf16(act(g_a g_w sum_k a[m,k] w[k,n] + bias[n])) on NVFP4
    operands: a_q [M x K/2] codes with tiled scales a_sf and tensor scale
    a_scale; the weight packed by frt_pack_weights from its [K/2 x N] codes,
    its tiled scales w_sf and tensor scale w_scale."""
    M, Kh, lda = _rows_view(a_q, "a_q")
    K = 2 * Kh
    out, ldo = _gemm_out(M, N, out, a_q.device)
    act, act_cols = _act(act_cols, False)
    _check("frt_gemm_nvfp4",
           lib().frt_gemm_nvfp4(a_q.data_ptr(), lda, a_sf.data_ptr(), _ptr(a_scale),
                                w_packed.data_ptr(), w_sf.data_ptr(), _ptr(w_scale), _ptr(bias),
                                M, N, K, act, act_cols, out.data_ptr(), ldo,
                                device_status(a_q.device).data_ptr(), _stream(stream)))
    return out


def frt_gate_residual_ada_norm_bf16(residual, output, gate, style, eps=1e-6, normalized=None,
                                    next_gate=None, stream=None):
    """The decoder block boundary: residual <- bf16(residual + output * gate)
    (in place), normalized = bf16(rms_norm(residual) * (1 + scale) + shift)
    and next_gate from style = [scale | shift | next gate] ([M x 3H]).  All
    bf16, contiguous.  Returns (normalized, next_gate)."""
    M, H = residual.shape
    for t, shape, name in ((output, (M, H), "output"), (gate, (M, H), "gate"),
                           (style, (M, 3 * H), "style")):
        if tuple(t.shape) != shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous bf16 tensor of shape %s" % (name, shape))
    if residual.dtype != torch.bfloat16 or not residual.is_contiguous():
        raise ValueError("residual must be a contiguous bf16 tensor")
    if normalized is None:
        normalized = torch.empty((M, H), dtype=torch.bfloat16, device=residual.device)
    if next_gate is None:
        next_gate = torch.empty((M, H), dtype=torch.bfloat16, device=residual.device)
    _check("frt_gate_residual_ada_norm_bf16",
           lib().frt_gate_residual_ada_norm_bf16(residual.data_ptr(), output.data_ptr(),
                                                 gate.data_ptr(), style.data_ptr(), M, H, eps,
                                                 normalized.data_ptr(), next_gate.data_ptr(),
                                                 _stream(stream)))
    return normalized, next_gate
