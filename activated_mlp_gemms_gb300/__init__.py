"""Fused transformer MLP block on one GB300 (sm_103a): Python binding of libmlp.so.

Argument marshalling only: every step of the forward and backward passes
runs in the library's CUDA kernels.  PyTorch supplies device memory and
streams.  The functions carry the names of the C ABI (include/mlp.h):

    mlp_workspace_size, mlp_fwd, mlp_fwd_infer, mlp_bwd, mlp_bwd_recompute,
    mlp_status_string, mlp_device_status, mlp_version

and mlp_func (module `autograd`) is the same forward and backward as one
differentiable PyTorch function.

Tensors are CUDA, contiguous, bf16 (fp32 for accumulated weight gradients),
with x [M,H], Wg/Wu [I,H], Wd [H,I].  A missing library raises at the first
call: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "ACTS", "MlpError", "Problem", "lib", "mlp_workspace_size", "mlp_fwd", "mlp_fwd_infer",
    "mlp_bwd", "mlp_bwd_recompute", "mlp_status_string", "mlp_device_status", "mlp_version",
    "MODE_FWD", "MODE_INFER", "MODE_BWD", "MODE_BWD_RECOMPUTE", "mlp_trace_enable",
    "mlp_trace_read", "mlp_kernel_name", "mlp_set_tile_policy", "mlp_fwd_infer_noalloc",
    "Block", "block", "mlp_block_fwd", "mlp_block_bwd", "mlp_fp8_quantize", "mlp_fp8_fwd",
    "MODE_FP8_FWD", "mlp_fp8_bwd", "MODE_FP8_BWD",
    "NOALLOC_SCRATCH_BYTES", "mlp_set_wait_timeout_ms", "mlp_debug_set_flags", "DEBUG_NO_WORK", "DEBUG_DECODE_FMA",
    "DEBUG_DECODE_MMA",
    "mlp_noalloc_status", "mlp_fp8_refresh_scales", "Plan", "mlp_plan", "mlp_debug_hold_sms",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmlp.so")

ACTS = {"swiglu": 0, "relu_sq": 1, "gelu_tanh_approx": 2, "relu": 3, "reglu": 4, "geglu": 5,
        "glu": 6}
GATED_ACTS = ("swiglu", "reglu", "geglu", "glu")
MODE_FWD, MODE_INFER, MODE_BWD, MODE_BWD_RECOMPUTE, MODE_FP8_FWD, MODE_FP8_BWD = 0, 1, 2, 3, 4, 5
NOALLOC_SCRATCH_BYTES = 16 << 20  # MLP_NOALLOC_SCRATCH_BYTES
DEBUG_NO_WORK = 1  # MLP_DEBUG_NO_WORK
DEBUG_DECODE_FMA = 2  # MLP_DEBUG_DECODE_FMA
DEBUG_DECODE_MMA = 4  # MLP_DEBUG_DECODE_MMA


class MlpError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {mlp_status_string(code)} ({code})")


class Problem(ctypes.Structure):
    """mlp_problem_t"""
    _fields_ = [("M", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("act", ctypes.c_int), ("gate_mult", ctypes.c_float),
                ("down_mult", ctypes.c_float)]


class Block(ctypes.Structure):
    """mlp_block_t: y = resid_lambda * x + post_lambda * MLP(x / sqrt(mean x^2 + eps))"""
    _fields_ = [("resid_lambda", ctypes.c_float), ("post_lambda", ctypes.c_float),
                ("eps", ctypes.c_float)]


class Plan(ctypes.Structure):
    """mlp_plan_t: what one call launches (see mlp_plan)."""
    _fields_ = [("decode", ctypes.c_int), ("fused_forward", ctypes.c_int),
                ("cta_group", ctypes.c_int), ("out_split", ctypes.c_int),
                ("wgrad_cta_group", ctypes.c_int), ("wgrad_split", ctypes.c_int)]

    def as_dict(self):
        return {k: int(getattr(self, k)) for k, _ in self._fields_}


_LIB = None
_VP = ctypes.c_void_p


def lib():
    """Load libmlp.so (built in-tree by __graft_entry__.build())."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libmlp.so is not built ({LIB_PATH} missing); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(Problem)
    L.mlp_workspace_size.argtypes = [P, ctypes.c_int]
    L.mlp_workspace_size.restype = ctypes.c_size_t
    L.mlp_fwd.argtypes = [P] + [_VP] * 7 + [_VP, ctypes.c_size_t, _VP]
    L.mlp_fwd.restype = ctypes.c_int
    L.mlp_fwd_infer.argtypes = [P] + [_VP] * 5 + [_VP, ctypes.c_size_t, _VP]
    L.mlp_fwd_infer.restype = ctypes.c_int
    L.mlp_bwd.argtypes = [P] + [_VP] * 11 + [ctypes.c_int, _VP, ctypes.c_size_t, _VP]
    L.mlp_bwd.restype = ctypes.c_int
    L.mlp_bwd_recompute.argtypes = [P] + [_VP] * 9 + [ctypes.c_int, _VP, ctypes.c_size_t, _VP]
    L.mlp_bwd_recompute.restype = ctypes.c_int
    L.mlp_fp8_quantize.argtypes = [_VP, ctypes.c_longlong, _VP, _VP, _VP, _VP]
    L.mlp_fp8_quantize.restype = ctypes.c_int
    L.mlp_fp8_fwd.argtypes = [P] + [_VP] * 8 + [_VP, ctypes.c_size_t, _VP]
    L.mlp_fp8_fwd.restype = ctypes.c_int
    L.mlp_fp8_bwd.argtypes = [P] + [_VP] * 11 + [_VP, ctypes.c_size_t, _VP]
    L.mlp_fp8_bwd.restype = ctypes.c_int
    B = ctypes.POINTER(Block)
    L.mlp_block_fwd.argtypes = [P, B] + [_VP] * 8 + [_VP, ctypes.c_size_t, _VP]
    L.mlp_block_fwd.restype = ctypes.c_int
    L.mlp_block_bwd.argtypes = [P, B] + [_VP] * 12 + [ctypes.c_int, _VP, ctypes.c_size_t, _VP]
    L.mlp_block_bwd.restype = ctypes.c_int
    L.mlp_status_string.argtypes = [ctypes.c_int]
    L.mlp_status_string.restype = ctypes.c_char_p
    L.mlp_device_status.argtypes = [_VP, _VP]
    L.mlp_device_status.restype = ctypes.c_int
    L.mlp_version.argtypes = []
    L.mlp_version.restype = ctypes.c_char_p
    L.mlp_fwd_infer_noalloc.argtypes = [P] + [_VP] * 5 + [_VP]
    L.mlp_fwd_infer_noalloc.restype = ctypes.c_int
    L.mlp_noalloc_status.argtypes = [_VP]
    L.mlp_noalloc_status.restype = ctypes.c_int
    L.mlp_fp8_refresh_scales.argtypes = [_VP, _VP, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                         ctypes.c_float, _VP]
    L.mlp_fp8_refresh_scales.restype = ctypes.c_int
    L.mlp_plan.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Plan)]
    L.mlp_plan.restype = ctypes.c_int
    L.mlp_debug_hold_sms.argtypes = [ctypes.c_int, ctypes.c_uint, _VP]
    L.mlp_debug_hold_sms.restype = ctypes.c_int
    L.mlp_set_wait_timeout_ms.argtypes = [ctypes.c_uint]
    L.mlp_set_wait_timeout_ms.restype = ctypes.c_int
    L.mlp_debug_set_flags.argtypes = [ctypes.c_int]
    L.mlp_debug_set_flags.restype = ctypes.c_int
    L.mlp_set_tile_policy.argtypes = [ctypes.c_int]
    L.mlp_set_tile_policy.restype = ctypes.c_int
    L.mlp_trace_enable.argtypes = [ctypes.c_int]
    L.mlp_trace_enable.restype = ctypes.c_int
    L.mlp_trace_read.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_float),
                                 ctypes.c_int]
    L.mlp_trace_read.restype = ctypes.c_int
    L.mlp_kernel_name.argtypes = [ctypes.c_int]
    L.mlp_kernel_name.restype = ctypes.c_char_p
    _LIB = L
    return L


def problem(M, H, I, act="swiglu", gate_mult=1.0, down_mult=1.0) -> Problem:
    if act not in ACTS:
        raise ValueError(f"unknown activation {act!r}; one of {list(ACTS)}")
    return Problem(int(M), int(H), int(I), ACTS[act], float(gate_mult), float(down_mult))


def block(resid_lambda=1.0, post_lambda=1.0, eps=2.0 ** -7) -> Block:
    return Block(float(resid_lambda), float(post_lambda), float(eps))


def _ptr(t, dtype=torch.bfloat16, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc, where):
    if rc != 0:
        raise MlpError(rc, where)


def mlp_status_string(code: int) -> str:
    return lib().mlp_status_string(int(code)).decode()


def mlp_version() -> str:
    return lib().mlp_version().decode()


def mlp_workspace_size(prob: Problem, mode: int) -> int:
    return int(lib().mlp_workspace_size(ctypes.byref(prob), int(mode)))


def alloc_workspace(prob: Problem, mode: int, device=None) -> torch.Tensor:
    n = mlp_workspace_size(prob, mode)
    if n == 0:
        raise MlpError(-1, "mlp_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _ws(ws, prob, mode, device):
    if ws is None:
        ws = alloc_workspace(prob, mode, device)
    if not (ws.is_cuda and ws.dtype == torch.uint8 and ws.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA uint8 tensor")
    return ws


def mlp_fwd(prob: Problem, x, Wg, Wu, Wd, out, G_save=None, U_save=None, ws=None, stream=None):
    """Training forward: out = down_mult * Wd (gate_mult * act(x Wg^T) * (x Wu^T)); optionally
    stores the preacts G = x Wg^T, U = x Wu^T (bf16 [M,I]).  Returns the workspace used."""
    ws = _ws(ws, prob, MODE_FWD, x.device)
    rc = lib().mlp_fwd(ctypes.byref(prob), _ptr(x, name="x"), _ptr(Wg, name="Wg"),
                       _ptr(Wu, name="Wu"), _ptr(Wd, name="Wd"), _ptr(out, name="out"),
                       _ptr(G_save, name="G_save"), _ptr(U_save, name="U_save"),
                       ws.data_ptr(), ws.numel(), _stream(stream))
    _check(rc, "mlp_fwd")
    return ws


def mlp_fwd_infer(prob: Problem, x, Wg, Wu, Wd, out, ws=None, stream=None):
    """No-grad forward; stores no intermediates outside the workspace."""
    ws = _ws(ws, prob, MODE_INFER, x.device)
    rc = lib().mlp_fwd_infer(ctypes.byref(prob), _ptr(x, name="x"), _ptr(Wg, name="Wg"),
                             _ptr(Wu, name="Wu"), _ptr(Wd, name="Wd"), _ptr(out, name="out"),
                             ws.data_ptr(), ws.numel(), _stream(stream))
    _check(rc, "mlp_fwd_infer")
    return ws


def _wdt(fuse):
    return torch.float32 if fuse else torch.bfloat16


def mlp_bwd(prob: Problem, dout, x, Wg, Wu, Wd, G, U, dx=None, dWg=None, dWu=None, dWd=None,
            fuse_grad_accum=False, ws=None, stream=None):
    """Backward from saved preacts G, U (overwritten with dG, dU).  Outputs that are None
    are skipped; weight gradients are bf16 (overwritten) or fp32 (+= in place) when
    fuse_grad_accum."""
    ws = _ws(ws, prob, MODE_BWD, x.device)
    wd = _wdt(fuse_grad_accum)
    rc = lib().mlp_bwd(ctypes.byref(prob), _ptr(dout, name="dout"), _ptr(x, name="x"),
                       _ptr(Wg, name="Wg"), _ptr(Wu, name="Wu"), _ptr(Wd, name="Wd"),
                       _ptr(G, name="G"), _ptr(U, name="U"), _ptr(dx, name="dx"),
                       _ptr(dWg, wd, "dWg"), _ptr(dWu, wd, "dWu"), _ptr(dWd, wd, "dWd"),
                       int(bool(fuse_grad_accum)), ws.data_ptr(), ws.numel(), _stream(stream))
    _check(rc, "mlp_bwd")
    return ws


def mlp_bwd_recompute(prob: Problem, dout, x, Wg, Wu, Wd, dx=None, dWg=None, dWu=None, dWd=None,
                      fuse_grad_accum=False, ws=None, stream=None):
    """Backward that recomputes the preacts from x (save-only-x training)."""
    ws = _ws(ws, prob, MODE_BWD_RECOMPUTE, x.device)
    wd = _wdt(fuse_grad_accum)
    rc = lib().mlp_bwd_recompute(ctypes.byref(prob), _ptr(dout, name="dout"), _ptr(x, name="x"),
                                 _ptr(Wg, name="Wg"), _ptr(Wu, name="Wu"), _ptr(Wd, name="Wd"),
                                 _ptr(dx, name="dx"), _ptr(dWg, wd, "dWg"), _ptr(dWu, wd, "dWu"),
                                 _ptr(dWd, wd, "dWd"), int(bool(fuse_grad_accum)),
                                 ws.data_ptr(), ws.numel(), _stream(stream))
    _check(rc, "mlp_bwd_recompute")
    return ws


def mlp_block_fwd(prob: Problem, blk: Block, x, Wg, Wu, Wd, y, G_save=None, U_save=None,
                  rstd=None, ws=None, stream=None):
    """The MLP block: y = resid_lambda x + post_lambda MLP(RMSNorm(x)).  Returns
    (rstd, ws): the fp32 per-token 1/r the backward takes, and the workspace."""
    ws = _ws(ws, prob, MODE_FWD, x.device)
    if rstd is None:
        rstd = torch.empty(prob.M, dtype=torch.float32, device=x.device)
    rc = lib().mlp_block_fwd(ctypes.byref(prob), ctypes.byref(blk), _ptr(x, name="x"),
                             _ptr(Wg, name="Wg"), _ptr(Wu, name="Wu"), _ptr(Wd, name="Wd"),
                             _ptr(y, name="y"), _ptr(G_save, name="G_save"),
                             _ptr(U_save, name="U_save"), _ptr(rstd, torch.float32, "rstd"),
                             ws.data_ptr(), ws.numel(), _stream(stream))
    _check(rc, "mlp_block_fwd")
    return rstd, ws


def mlp_block_bwd(prob: Problem, blk: Block, dy, x, Wg, Wu, Wd, G, U, rstd, dx=None, dWg=None,
                  dWu=None, dWd=None, fuse_grad_accum=False, ws=None, stream=None):
    """Backward of mlp_block_fwd from its saved G, U (overwritten) and rstd."""
    ws = _ws(ws, prob, MODE_BWD, x.device)
    wd = _wdt(fuse_grad_accum)
    rc = lib().mlp_block_bwd(ctypes.byref(prob), ctypes.byref(blk), _ptr(dy, name="dy"),
                             _ptr(x, name="x"), _ptr(Wg, name="Wg"), _ptr(Wu, name="Wu"),
                             _ptr(Wd, name="Wd"), _ptr(G, name="G"), _ptr(U, name="U"),
                             _ptr(rstd, torch.float32, "rstd"), _ptr(dx, name="dx"),
                             _ptr(dWg, wd, "dWg"), _ptr(dWu, wd, "dWu"), _ptr(dWd, wd, "dWd"),
                             int(bool(fuse_grad_accum)), ws.data_ptr(), ws.numel(),
                             _stream(stream))
    _check(rc, "mlp_block_bwd")
    return ws


def _u8(t, name):
    if t is None:
        return None
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()
            and t.dtype in (torch.uint8, torch.float8_e4m3fn, torch.float8_e5m2)):
        raise ValueError(f"{name} must be a contiguous CUDA uint8 / float8 tensor")
    return t.data_ptr()


def mlp_fp8_quantize(src, scale, dst, amax=None, stream=None):
    """dst (e4m3 codes) = e4m3(src * (1 / scale[0])); max|src| atomically into amax[0]."""
    rc = lib().mlp_fp8_quantize(_ptr(src, name="src"), src.numel(),
                                _ptr(scale, torch.float32, "scale"), _u8(dst, "dst"),
                                _ptr(amax, torch.float32, "amax"), _stream(stream))
    _check(rc, "mlp_fp8_quantize")


def mlp_fp8_fwd(prob: Problem, x8, W1_8, W2_8, scales, out, a8_save=None, amax_a=None, ws=None,
                stream=None, pre_save=None):
    """e4m3 forward of the ReLU^2 MLP; scales = fp32 device tensor {sx, s1, s2, s_post, ...};
    pre_save (bf16 [M, I]) receives the preact for mlp_fp8_bwd."""
    ws = _ws(ws, prob, MODE_FP8_FWD, out.device)
    rc = lib().mlp_fp8_fwd(ctypes.byref(prob), _u8(x8, "x8"), _u8(W1_8, "W1_8"), _u8(W2_8, "W2_8"),
                           _ptr(scales, torch.float32, "scales"), _ptr(out, name="out"),
                           _u8(a8_save, "a8_save"), _ptr(pre_save, name="pre_save"),
                           _ptr(amax_a, torch.float32, "amax_a"),
                           ws.data_ptr(), ws.numel(), _stream(stream))
    _check(rc, "mlp_fp8_fwd")
    return ws


def mlp_fp8_bwd(prob: Problem, dout, x8, W1_8, W2_8, pre, a8, scales, dx=None, dW1=None, dW2=None,
                amax_dpre=None, ws=None, stream=None):
    """8-bit backward of the ReLU^2 MLP (e5m2 gradients); scales = fp32 [6] device tensor
    {sx, s1, s2, s_post, sg, s_dpre}; dx [M,H], dW1 [I,H], dW2 [H,I] bf16 outputs."""
    ws = _ws(ws, prob, MODE_FP8_BWD, dout.device)
    if scales is not None and scales.numel() < 6:
        raise ValueError("scales must hold {sx, s1, s2, s_post, sg, s_dpre}")
    rc = lib().mlp_fp8_bwd(ctypes.byref(prob), _ptr(dout, name="dout"), _u8(x8, "x8"),
                           _u8(W1_8, "W1_8"), _u8(W2_8, "W2_8"), _ptr(pre, name="pre"),
                           _u8(a8, "a8"), _ptr(scales, torch.float32, "scales"),
                           _ptr(dx, name="dx"), _ptr(dW1, name="dW1"), _ptr(dW2, name="dW2"),
                           _ptr(amax_dpre, torch.float32, "amax_dpre"),
                           ws.data_ptr(), ws.numel(), _stream(stream))
    _check(rc, "mlp_fp8_bwd")
    return ws


def mlp_fp8_refresh_scales(amax, scale, gain, floor, stream=None) -> None:
    """The delayed-scale refresh on the device: amax fp32 [n] or [n, width],
    scale fp32 [n]; scale = max(a * gain, floor) where the slot's amax a is
    finite and > 0, and the amax is cleared (gpt.py _refresh_delayed_scale)."""
    n = scale.numel()
    width = amax.numel() // n if n else 1
    if n and amax.numel() != n * width:
        raise ValueError("amax must hold n * width values")
    rc = lib().mlp_fp8_refresh_scales(_ptr(amax, torch.float32, "amax"),
                                      _ptr(scale, torch.float32, "scale"), int(n), int(width),
                                      float(gain), float(floor), _stream(stream))
    _check(rc, "mlp_fp8_refresh_scales")


def mlp_plan(prob: Problem, mode: int, fuse_grad_accum: bool = False) -> dict:
    """What one call in `mode` launches on the current device (mlp_plan_t as a dict)."""
    plan = Plan()
    rc = lib().mlp_plan(ctypes.byref(prob), int(mode), int(bool(fuse_grad_accum)),
                        ctypes.byref(plan))
    _check(rc, "mlp_plan")
    return plan.as_dict()


def mlp_debug_hold_sms(ctas: int, us: int, stream=None) -> None:
    """Testing hook: keep `ctas` SMs busy for `us` microseconds on `stream`."""
    _check(lib().mlp_debug_hold_sms(int(ctas), int(us), _stream(stream)), "mlp_debug_hold_sms")


def mlp_device_status(ws, stream=None) -> int:
    """Synchronises the stream and returns the device status word (0 = OK)."""
    return int(lib().mlp_device_status(ws.data_ptr(), _stream(stream)))


def mlp_trace_enable(on: bool = True) -> None:
    """Bracket every kernel launch of later calls with CUDA events (timing)."""
    _check(lib().mlp_trace_enable(1 if on else 0), "mlp_trace_enable")


def mlp_kernel_name(tag: int) -> str:
    return lib().mlp_kernel_name(int(tag)).decode()


def mlp_trace_read(capacity: int = 4096):
    """Returns [(kernel name, ms), ...] for the launches recorded since the
    last read, in launch order, and frees the records."""
    tags = (ctypes.c_int * capacity)()
    ms = (ctypes.c_float * capacity)()
    n = lib().mlp_trace_read(tags, ms, capacity)
    if n < 0:
        raise MlpError(n, "mlp_trace_read")
    return [(mlp_kernel_name(tags[i]), float(ms[i])) for i in range(n)]


def mlp_set_tile_policy(policy: int) -> None:
    """0 = automatic, 1 = single-CTA 128x256 tiles, 2 = CTA-pair 256x256 tiles,
    3 = automatic tiles with the gated forward's two GEMMs as separate launches."""
    _check(lib().mlp_set_tile_policy(int(policy)), "mlp_set_tile_policy")


def mlp_fwd_infer_noalloc(prob: Problem, x, Wg, Wu, Wd, out, stream=None) -> None:
    """Inference forward for callers that may not allocate device memory: the
    scratch is a fixed array inside the library (NOALLOC_SCRATCH_BYTES), shared
    by all calls, so calls must be ordered (e.g. one stream).  The first call
    on a device looks up the array's address; make it before any stream
    capture.  Raises MlpError(MLP_ERR_WORKSPACE_TOO_SMALL) for problems whose
    inference workspace exceeds the array."""
    rc = lib().mlp_fwd_infer_noalloc(ctypes.byref(prob), _ptr(x, name="x"), _ptr(Wg, name="Wg"),
                                     _ptr(Wu, name="Wu"), _ptr(Wd, name="Wd"),
                                     _ptr(out, name="out"), _stream(stream))
    _check(rc, "mlp_fwd_infer_noalloc")


def mlp_noalloc_status(stream=None) -> int:
    """Synchronises the stream and returns the status word of
    mlp_fwd_infer_noalloc's scratch on the current device (0 = OK)."""
    return int(lib().mlp_noalloc_status(_stream(stream)))


def mlp_set_wait_timeout_ms(ms: int) -> None:
    """Bound of the kernels' device-side waits for later calls (0 = default)."""
    _check(lib().mlp_set_wait_timeout_ms(int(ms)), "mlp_set_wait_timeout_ms")


def mlp_debug_set_flags(flags: int) -> None:
    """Testing hooks: DEBUG_NO_WORK makes later calls time out on purpose;
    DEBUG_DECODE_FMA / DEBUG_DECODE_MMA force the decode-sized forward onto
    the CUDA-core or the warp-MMA weight stream."""
    _check(lib().mlp_debug_set_flags(int(flags)), "mlp_debug_set_flags")


from .autograd import mlp_block_func, mlp_func  # noqa: E402  (differentiable forms)

__all__ += ["mlp_func", "mlp_block_func"]
