"""BitLinear forward of BitNet b1.58 for B300 (sm_103a).

Thin Python binding over the C ABI in include/bitlinear.h: it checks tensor
placement and dtypes, passes raw device pointers and the current CUDA stream,
and raises BitLinearError on any non-OK status. Every step of the computation
runs in the library's CUDA kernels; there is no CPU or PyTorch fallback.

    packed, s_w = pack(W)                    # W [N, K] fp32 on the GPU
    Y = forward(X, packed, s_w)              # X [M, K] fp32 or bf16
    Y = ffn(X, up, s_up, down, s_down)       # up->ReLU^2->requant->down
    Y = forward_rmsnorm(X, packed, s_w, g)   # RMSNorm fused into the quantization
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import (BL_DTYPE_BF16, BL_DTYPE_F32, BL_DTYPE_I8, BL_MAX_BATCH, BL_OP_FFN, BL_OP_FFN_GATED,  # noqa: F401
                   BL_OP_FORWARD,
                   BL_OP_FORWARD_BATCH, BL_OP_PACK, BitLinearError, ForwardDesc, check)

EPS = 1e-5
EPS_NORM = 1e-5

__all__ = ["pack", "quant_act", "quant_act_tc", "forward", "forward_batch", "forward_q8", "forward_tc",
           "forward_noalloc", "ffn", "ffn_gated", "rmsnorm_quant", "forward_rmsnorm", "ffn_subln", "unpack",
           "workspace_bytes", "workspace_status", "Workspace", "BitLinearError", "EPS", "EPS_NORM",
           "library_path"]


def library_path() -> str:
    return _lib.LIB_PATH


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else int(t.data_ptr())


def _need_cuda(t: torch.Tensor, name: str, dtypes) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _x_dtype(X: torch.Tensor) -> int:
    if X.dtype == torch.float32:
        return BL_DTYPE_F32
    if X.dtype == torch.bfloat16:
        return BL_DTYPE_BF16
    raise ValueError(f"X must be float32 or bfloat16, got {X.dtype}")


def workspace_bytes(op: int, M: int, N: int, K: int) -> int:
    return int(_lib.lib().bitlinear_workspace_bytes(op, M, N, K))


class Workspace:
    """Caller-owned scratch for the library (zero-initialized once; grows on demand).
    Calls that share one Workspace must run in order on one stream."""

    def __init__(self, nbytes: int = 0, device=None):
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.buf = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=self.device)

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self.buf = torch.zeros(int(nbytes), dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws: dict[int, Workspace] = {}


def _workspace(ws: Workspace | None, nbytes: int) -> torch.Tensor:
    if ws is None:
        dev = torch.cuda.current_device()
        ws = _default_ws.setdefault(dev, Workspace(0, torch.device("cuda", dev)))
    return ws.get(nbytes)


def pack(W: torch.Tensor, eps: float = EPS, workspace: Workspace | None = None, stream=None):
    """Absmean ternary quantization + 2-bit packing. Returns (packed uint8 [N, K/4], s_w fp32 [1])."""
    _need_cuda(W, "W", (torch.float32,))
    N, K = W.shape
    packed = torch.empty((N, K // 4), dtype=torch.uint8, device=W.device)
    s_w = torch.empty(4, dtype=torch.float32, device=W.device)[:1]
    nb = workspace_bytes(BL_OP_PACK, 0, N, K)
    ws = _workspace(workspace, nb)
    check(_lib.lib().bitlinear_pack(_ptr(W), N, K, eps, _ptr(packed), _ptr(s_w), _ptr(ws), ws.numel(),
                                    _stream(stream)), "bitlinear_pack")
    return packed, s_w


def quant_act(X: torch.Tensor, eps: float = EPS, stream=None):
    """Per-token absmax int8 quantization. Returns (q int8 [M, K], m fp32 [M])."""
    _need_cuda(X, "X", (torch.float32, torch.bfloat16))
    M, K = X.shape
    q = torch.empty((M, K), dtype=torch.int8, device=X.device)
    m = torch.empty(max(M, 4), dtype=torch.float32, device=X.device)[:M]
    check(_lib.lib().bitlinear_quant_act(_ptr(X), _x_dtype(X), M, K, eps, _ptr(q), _ptr(m), _stream(stream)),
          "bitlinear_quant_act")
    return q, m


def forward(X: torch.Tensor, packed: torch.Tensor, s_w: torch.Tensor, eps: float = EPS, return_acc: bool = False,
            out: torch.Tensor | None = None, workspace: Workspace | None = None, stream=None):
    """Y = BitLinear(X) with packed ternary weights [N, K/4] and scale s_w [1]."""
    _need_cuda(X, "X", (torch.float32, torch.bfloat16))
    _need_cuda(packed, "packed", (torch.uint8,))
    _need_cuda(s_w, "s_w", (torch.float32,))
    M, K = X.shape
    N = packed.shape[0]
    if packed.shape[1] * 4 != K:
        raise ValueError(f"packed has {packed.shape[1]} bytes per row, expected K/4 = {K // 4}")
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=X.device)
    acc = torch.empty((M, N), dtype=torch.int32, device=X.device) if return_acc else None
    nb = workspace_bytes(BL_OP_FORWARD, M, N, K)
    ws = _workspace(workspace, nb)
    check(_lib.lib().bitlinear_forward(_ptr(X), _x_dtype(X), M, K, _ptr(packed), _ptr(s_w), N, eps, _ptr(Y),
                                       _ptr(acc), _ptr(ws), ws.numel(), _stream(stream)), "bitlinear_forward")
    return (Y, acc) if return_acc else Y


def forward_batch(problems, eps: float = EPS, workspace: Workspace | None = None, stream=None, descs=None):
    """Independent BitLinear forwards in one call. `problems` is a sequence of
    (X, packed, s_w, Y), (X, packed, s_w, Y, acc) or (q, packed, s_w, Y, acc, m)
    with device tensors: X fp32/bf16, or q int8 already quantized with its
    per-token scales m (acc may be None). The outputs Y (and acc) are written in
    place. Returns the ctypes descriptor array, which can be passed back as
    `descs` to skip rebuilding it."""
    if descs is None:
        if len(problems) > BL_MAX_BATCH:
            raise ValueError(f"at most {BL_MAX_BATCH} problems per call")
        descs = (ForwardDesc * len(problems))()
        for d, prob in zip(descs, problems):
            X, packed, s_w, Y = prob[:4]
            acc = prob[4] if len(prob) > 4 else None
            m = prob[5] if len(prob) > 5 else None
            _need_cuda(X, "X", (torch.float32, torch.bfloat16, torch.int8))
            _need_cuda(packed, "packed", (torch.uint8,))
            _need_cuda(Y, "Y", (torch.float32,))
            M, K = X.shape
            N = packed.shape[0]
            if packed.shape[1] * 4 != K or tuple(Y.shape) != (M, N):
                raise ValueError("forward_batch: shapes of X, packed and Y do not match")
            if X.dtype == torch.int8:
                if m is None:
                    raise ValueError("forward_batch: an int8 input needs its per-token scales m")
                _need_cuda(m, "m", (torch.float32,))
                d.x_dtype, d.m = BL_DTYPE_I8, _ptr(m)
            else:
                d.x_dtype, d.m = _x_dtype(X), None
            d.X, d.M, d.K, d.N = _ptr(X), M, K, N
            d.packed, d.s_w, d.Y, d.acc = _ptr(packed), _ptr(s_w), _ptr(Y), _ptr(acc)
    tokens = sum(int(d.M) for d in descs if d.x_dtype != BL_DTYPE_I8)
    kmax = max((int(d.K) for d in descs), default=64)
    nb = workspace_bytes(BL_OP_FORWARD_BATCH, tokens, 0, kmax)
    ws = _workspace(workspace, nb)
    check(_lib.lib().bitlinear_forward_batch(descs, len(descs), eps, _ptr(ws), ws.numel(), _stream(stream)),
          "bitlinear_forward_batch")
    return descs


def forward_q8(q: torch.Tensor, m: torch.Tensor, packed: torch.Tensor, s_w: torch.Tensor, return_acc: bool = False,
               out: torch.Tensor | None = None, workspace: Workspace | None = None, stream=None):
    """BitLinear on an already-quantized input (q int8 [M, K], m fp32 [M] from quant_act)."""
    _need_cuda(q, "q", (torch.int8,))
    _need_cuda(m, "m", (torch.float32,))
    _need_cuda(packed, "packed", (torch.uint8,))
    _need_cuda(s_w, "s_w", (torch.float32,))
    M, K = q.shape
    N = packed.shape[0]
    if packed.shape[1] * 4 != K:
        raise ValueError(f"packed has {packed.shape[1]} bytes per row, expected K/4 = {K // 4}")
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=q.device)
    acc = torch.empty((M, N), dtype=torch.int32, device=q.device) if return_acc else None
    nb = workspace_bytes(BL_OP_FORWARD, M, N, K)
    ws = _workspace(workspace, nb)
    check(_lib.lib().bitlinear_forward_q8(_ptr(q), _ptr(m), M, K, _ptr(packed), _ptr(s_w), N, _ptr(Y), _ptr(acc),
                                          _ptr(ws), ws.numel(), _stream(stream)), "bitlinear_forward_q8")
    return (Y, acc) if return_acc else Y


def quant_act_tc(X: torch.Tensor, eps: float = EPS, stream=None):
    """Per-token absmax quantization into the tensor-core operand form.
    Returns (act fp16 [M, K], m fp32 [M]) for forward_tc."""
    _need_cuda(X, "X", (torch.float32, torch.bfloat16))
    M, K = X.shape
    act = torch.empty((M, K), dtype=torch.float16, device=X.device)
    m = torch.empty(max(M, 4), dtype=torch.float32, device=X.device)[:M]
    check(_lib.lib().bitlinear_quant_act_tc(_ptr(X), _x_dtype(X), M, K, eps, _ptr(act), _ptr(m), _stream(stream)),
          "bitlinear_quant_act_tc")
    return act, m


def forward_tc(act: torch.Tensor, m: torch.Tensor, packed: torch.Tensor, s_w: torch.Tensor,
               return_acc: bool = False, out: torch.Tensor | None = None, workspace: Workspace | None = None,
               stream=None):
    """BitLinear on an input from quant_act_tc: the tensor-core contraction only."""
    _need_cuda(act, "act", (torch.float16,))
    _need_cuda(m, "m", (torch.float32,))
    _need_cuda(packed, "packed", (torch.uint8,))
    _need_cuda(s_w, "s_w", (torch.float32,))
    M, K = act.shape
    N = packed.shape[0]
    if packed.shape[1] * 4 != K:
        raise ValueError(f"packed has {packed.shape[1]} bytes per row, expected K/4 = {K // 4}")
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=act.device)
    acc = torch.empty((M, N), dtype=torch.int32, device=act.device) if return_acc else None
    # room for [M][N] int32 partial sums lets few tokens cut K across more SMs
    ws = _workspace(workspace, 256 + (4 * M * N if M <= 128 else 0))
    check(_lib.lib().bitlinear_forward_tc(_ptr(act), _ptr(m), M, K, _ptr(packed), _ptr(s_w), N, _ptr(Y), _ptr(acc),
                                          _ptr(ws), ws.numel(), _stream(stream)), "bitlinear_forward_tc")
    return (Y, acc) if return_acc else Y


def forward_noalloc(X: torch.Tensor, packed: torch.Tensor, s_w: torch.Tensor, eps: float = EPS,
                    return_acc: bool = False, out: torch.Tensor | None = None, stream=None):
    """forward() for callers that cannot provide device scratch: the library
    uses its own fixed 8 MiB device array instead of a workspace. The first
    call on a device does a one-time address lookup (make it before any stream
    capture); calls that overlap on the GPU race on the shared array."""
    _need_cuda(X, "X", (torch.float32, torch.bfloat16))
    _need_cuda(packed, "packed", (torch.uint8,))
    _need_cuda(s_w, "s_w", (torch.float32,))
    M, K = X.shape
    N = packed.shape[0]
    if packed.shape[1] * 4 != K:
        raise ValueError(f"packed has {packed.shape[1]} bytes per row, expected K/4 = {K // 4}")
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=X.device)
    acc = torch.empty((M, N), dtype=torch.int32, device=X.device) if return_acc else None
    check(_lib.lib().bitlinear_forward_noalloc(_ptr(X), _x_dtype(X), M, K, _ptr(packed), _ptr(s_w), N, eps,
                                               _ptr(Y), _ptr(acc), _stream(stream)), "bitlinear_forward_noalloc")
    return (Y, acc) if return_acc else Y


def ffn(X: torch.Tensor, up: torch.Tensor, s_up: torch.Tensor, down: torch.Tensor, s_down: torch.Tensor,
        eps: float = EPS, out: torch.Tensor | None = None, workspace: Workspace | None = None, stream=None):
    """Ungated FFN: down(ReLU^2(up(X))), each projection a BitLinear."""
    _need_cuda(X, "X", (torch.float32, torch.bfloat16))
    for t, n in ((up, "up"), (down, "down")):
        _need_cuda(t, n, (torch.uint8,))
    M, D = X.shape
    F = up.shape[0]
    if up.shape[1] * 4 != D or down.shape[0] != D or down.shape[1] * 4 != F:
        raise ValueError("FFN weight shapes do not match X")
    Y = out if out is not None else torch.empty((M, D), dtype=torch.float32, device=X.device)
    nb = workspace_bytes(BL_OP_FFN, M, F, D)
    ws = _workspace(workspace, nb)
    check(_lib.lib().bitlinear_ffn(_ptr(X), _x_dtype(X), M, D, _ptr(up), _ptr(s_up), _ptr(down), _ptr(s_down), F,
                                   eps, _ptr(Y), _ptr(ws), ws.numel(), _stream(stream)), "bitlinear_ffn")
    return Y


def ffn_gated(X: torch.Tensor, up: torch.Tensor, s_up: torch.Tensor, gate: torch.Tensor, s_gate: torch.Tensor,
              down: torch.Tensor, s_down: torch.Tensor, eps: float = EPS, out: torch.Tensor | None = None,
              workspace: Workspace | None = None, stream=None):
    """Gated FFN: down(ReLU^2(gate(X)) * up(X)), each projection a BitLinear."""
    _need_cuda(X, "X", (torch.float32, torch.bfloat16))
    for t, n in ((up, "up"), (gate, "gate"), (down, "down")):
        _need_cuda(t, n, (torch.uint8,))
    M, D = X.shape
    F = up.shape[0]
    if (up.shape[1] * 4 != D or tuple(gate.shape) != tuple(up.shape) or down.shape[0] != D
            or down.shape[1] * 4 != F):
        raise ValueError("gated FFN weight shapes do not match X")
    Y = out if out is not None else torch.empty((M, D), dtype=torch.float32, device=X.device)
    nb = workspace_bytes(BL_OP_FFN_GATED, M, F, D)
    ws = _workspace(workspace, nb)
    check(_lib.lib().bitlinear_ffn_gated(_ptr(X), _x_dtype(X), M, D, _ptr(up), _ptr(s_up), _ptr(gate), _ptr(s_gate),
                                         _ptr(down), _ptr(s_down), F, eps, _ptr(Y), _ptr(ws), ws.numel(),
                                         _stream(stream)), "bitlinear_ffn_gated")
    return Y


def _need_gain(g: torch.Tensor | None, K: int, name: str) -> None:
    if g is None:
        return
    _need_cuda(g, name, (torch.float32,))
    if g.dim() != 1 or g.shape[0] != K:
        raise ValueError(f"{name} must be a [{K}] gain vector, got {tuple(g.shape)}")


def rmsnorm_quant(X: torch.Tensor, g: torch.Tensor | None = None, eps_norm: float = EPS_NORM, eps: float = EPS,
                  stream=None):
    """RMSNorm (gain g [K], None = 1) fused into the per-token absmax quant.
    Returns (q int8 [M, K], m fp32 [M]) with the norm factor folded into m."""
    _need_cuda(X, "X", (torch.float32, torch.bfloat16))
    M, K = X.shape
    _need_gain(g, K, "g")
    q = torch.empty((M, K), dtype=torch.int8, device=X.device)
    m = torch.empty(max(M, 4), dtype=torch.float32, device=X.device)[:M]
    check(_lib.lib().bitlinear_rmsnorm_quant(_ptr(X), _x_dtype(X), M, K, _ptr(g), eps_norm, eps, _ptr(q), _ptr(m),
                                             _stream(stream)), "bitlinear_rmsnorm_quant")
    return q, m


def forward_rmsnorm(X: torch.Tensor, packed: torch.Tensor, s_w: torch.Tensor, g: torch.Tensor | None = None,
                    eps_norm: float = EPS_NORM, eps: float = EPS, return_acc: bool = False,
                    out: torch.Tensor | None = None, workspace: Workspace | None = None, stream=None):
    """Y = BitLinear(RMSNorm_g(X)), the norm fused into the activation quantization."""
    _need_cuda(X, "X", (torch.float32, torch.bfloat16))
    _need_cuda(packed, "packed", (torch.uint8,))
    _need_cuda(s_w, "s_w", (torch.float32,))
    M, K = X.shape
    _need_gain(g, K, "g")
    N = packed.shape[0]
    if packed.shape[1] * 4 != K:
        raise ValueError(f"packed has {packed.shape[1]} bytes per row, expected K/4 = {K // 4}")
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=X.device)
    acc = torch.empty((M, N), dtype=torch.int32, device=X.device) if return_acc else None
    ws = _workspace(workspace, workspace_bytes(BL_OP_FORWARD, M, N, K))
    check(_lib.lib().bitlinear_forward_rmsnorm(_ptr(X), _x_dtype(X), M, K, _ptr(g), eps_norm, _ptr(packed),
                                               _ptr(s_w), N, eps, _ptr(Y), _ptr(acc), _ptr(ws), ws.numel(),
                                               _stream(stream)), "bitlinear_forward_rmsnorm")
    return (Y, acc) if return_acc else Y


def ffn_subln(X: torch.Tensor, up: torch.Tensor, s_up: torch.Tensor, down: torch.Tensor, s_down: torch.Tensor,
              g_in: torch.Tensor | None = None, g_sub: torch.Tensor | None = None, gate: torch.Tensor | None = None,
              s_gate: torch.Tensor | None = None, eps_norm: float = EPS_NORM, eps: float = EPS,
              out: torch.Tensor | None = None, workspace: Workspace | None = None, stream=None):
    """FFN block with SubLN: RMSNorm(g_in) on X, up (and gate), ReLU^2 (times up
    when gated), RMSNorm(g_sub) on h, down."""
    _need_cuda(X, "X", (torch.float32, torch.bfloat16))
    gated = gate is not None
    if gated != (s_gate is not None):
        raise ValueError("gate and s_gate go together")
    for t, n in ((up, "up"), (down, "down")) + (((gate, "gate"),) if gated else ()):
        _need_cuda(t, n, (torch.uint8,))
    M, D = X.shape
    F = up.shape[0]
    if (up.shape[1] * 4 != D or down.shape[0] != D or down.shape[1] * 4 != F
            or (gated and tuple(gate.shape) != tuple(up.shape))):
        raise ValueError("FFN weight shapes do not match X")
    _need_gain(g_in, D, "g_in")
    _need_gain(g_sub, F, "g_sub")
    Y = out if out is not None else torch.empty((M, D), dtype=torch.float32, device=X.device)
    ws = _workspace(workspace, workspace_bytes(BL_OP_FFN_GATED if gated else BL_OP_FFN, M, F, D))
    check(_lib.lib().bitlinear_ffn_subln(_ptr(X), _x_dtype(X), M, D, _ptr(g_in), _ptr(up), _ptr(s_up), _ptr(gate),
                                         _ptr(s_gate), _ptr(g_sub), _ptr(down), _ptr(s_down), F, eps_norm, eps,
                                         _ptr(Y), _ptr(ws), ws.numel(), _stream(stream)), "bitlinear_ffn_subln")
    return Y


def unpack(packed: torch.Tensor, K: int, stream=None) -> torch.Tensor:
    """Decode packed codes to int8 ternary values [N, K]."""
    _need_cuda(packed, "packed", (torch.uint8,))
    N = packed.shape[0]
    t = torch.empty((N, K), dtype=torch.int8, device=packed.device)
    check(_lib.lib().bitlinear_unpack(_ptr(packed), N, K, _ptr(t), _stream(stream)), "bitlinear_unpack")
    return t


def workspace_status(ws: Workspace | torch.Tensor | None = None, stream=None) -> int:
    """Reads and clears the sticky device status of a workspace (0 = OK)."""
    if ws is None:
        ws = _default_ws.get(torch.cuda.current_device())
        if ws is None:
            return 0
    buf = ws.buf if isinstance(ws, Workspace) else ws
    return int(_lib.lib().bitlinear_workspace_status(_ptr(buf), _stream(stream)))
