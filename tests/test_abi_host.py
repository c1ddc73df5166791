"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol include/mlp.h declares, and rejects bad arguments before
enqueueing anything (fake, never-dereferenced pointers are used)."""
import ctypes
import os
import re

import pytest

import activated_mlp_gemms_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mlp.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(m.LIB_PATH):
        from activated_mlp_gemms_gb300 import _build
        _build.build()
    return m.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_]+\s*\*?\s*(mlp_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    assert names == sorted(["mlp_workspace_size", "mlp_fwd", "mlp_fwd_infer", "mlp_bwd",
                            "mlp_bwd_recompute", "mlp_status_string", "mlp_device_status",
                            "mlp_version", "mlp_trace_enable", "mlp_trace_read",
                            "mlp_kernel_name", "mlp_set_tile_policy",
                            "mlp_fwd_infer_noalloc", "mlp_set_wait_timeout_ms",
                            "mlp_debug_set_flags", "mlp_block_fwd", "mlp_block_bwd",
                            "mlp_fp8_quantize", "mlp_fp8_fwd", "mlp_fp8_bwd",
                            "mlp_fp8_refresh_scales", "mlp_plan", "mlp_debug_hold_sms",
                            "mlp_noalloc_status"])


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n
    assert m.mlp_version() == "0.1.0"


def test_status_strings(L):
    assert m.mlp_status_string(0) == "MLP_OK"
    assert m.mlp_status_string(-4) == "MLP_ERR_WORKSPACE_TOO_SMALL"
    assert m.mlp_status_string(-6) == "MLP_ERR_TIMEOUT"
    assert m.mlp_status_string(12345) == "MLP_ERR_UNKNOWN"


def test_workspace_sizes(L):
    p = m.problem(2048, 4096, 11008)
    inter = 2048 * 11008 * 2
    assert m.mlp_workspace_size(p, m.MODE_FWD) == 1024 + inter
    assert m.mlp_workspace_size(p, m.MODE_INFER) == 1024 + inter
    assert m.mlp_workspace_size(p, m.MODE_BWD) == 1024 + inter
    assert m.mlp_workspace_size(p, m.MODE_BWD_RECOMPUTE) == 1024 + 3 * inter
    q = m.problem(49152, 768, 3072, "relu_sq")
    assert m.mlp_workspace_size(q, m.MODE_BWD_RECOMPUTE) == 1024 + 2 * 49152 * 3072 * 2
    # decode-sized M: the down projection splits K and needs an fp32 [M,H] region
    d = m.problem(16, 4096, 14336)
    r256 = lambda n: (n + 255) // 256 * 256  # noqa: E731
    assert m.mlp_workspace_size(d, m.MODE_INFER) == 1024 + r256(16 * 14336 * 2) + 16 * 4096 * 4
    assert m.mlp_workspace_size(d, m.MODE_BWD) == 1024 + r256(16 * 14336 * 2) + 16 * 4096 * 4
    # a partial wave of down-projection tiles (512 tokens: 32 tiles of 256 x 256
    # on 76 CTA pairs): the forward splits K and needs the fp32 region, the
    # backward's dx does not
    e = m.problem(512, 4096, 14336)
    assert m.mlp_workspace_size(e, m.MODE_INFER) == 1024 + 512 * 14336 * 2 + 512 * 4096 * 4
    assert m.mlp_workspace_size(e, m.MODE_FWD) == 1024 + 512 * 14336 * 2 + 512 * 4096 * 4
    assert m.mlp_workspace_size(e, m.MODE_BWD) == 1024 + 512 * 14336 * 2
    # more than half the pairs (1024 tokens: 64 tiles) is left whole
    f = m.problem(1024, 4096, 14336)
    assert m.mlp_workspace_size(f, m.MODE_INFER) == 1024 + 1024 * 14336 * 2
    assert m.mlp_workspace_size(m.problem(64, 128, 352), m.MODE_INFER) == 1024 + 64 * 352 * 2
    assert m.mlp_workspace_size(m.problem(0, 8, 8), 0) == 0
    assert m.mlp_workspace_size(m.problem(8, 12, 8), 0) == 0  # H % 8 != 0
    assert m.mlp_workspace_size(p, 7) == 0


FAKE = 0x10000  # aligned, never dereferenced: validation fails before any launch


def _fwd(L, prob, x=FAKE, Wg=FAKE, Wu=FAKE, Wd=FAKE, out=FAKE, ws=FAKE, ws_bytes=1 << 40):
    return L.mlp_fwd_infer(ctypes.byref(prob), x, Wg, Wu, Wd, out, ws, ws_bytes, None)


def test_validation_errors(L):
    assert _fwd(L, m.problem(0, 128, 352)) == -1            # M <= 0
    assert _fwd(L, m.problem(64, 130, 352)) == -2           # H % 8
    assert _fwd(L, m.problem(64, 128, 350)) == -2           # I % 8
    assert _fwd(L, m.problem(64, 128, 352), x=None) == -1   # null input
    assert _fwd(L, m.problem(64, 128, 352), Wg=FAKE + 2) == -2  # misaligned
    assert _fwd(L, m.problem(64, 128, 352), Wu=None) == -1  # gated needs Wu
    assert _fwd(L, m.problem(64, 128, 352, "relu_sq")) == -1  # non-gated takes no Wu
    assert _fwd(L, m.problem(64, 128, 352), ws_bytes=100) == -4
    assert _fwd(L, m.problem(64, 128, 352), ws=FAKE + 16) == -2  # workspace 256-aligned
    bad = m.problem(64, 128, 352)
    bad.act = 9
    assert _fwd(L, bad) == -1
    nanp = m.problem(64, 128, 352, gate_mult=float("nan"))
    assert _fwd(L, nanp) == -1
    assert L.mlp_fwd_infer(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == -1


def test_backward_validation(L):
    p = m.problem(64, 128, 352)
    args = [FAKE] * 5  # dout, x, Wg, Wu, Wd
    # saved mode needs G and U
    assert L.mlp_bwd(ctypes.byref(p), *args, None, FAKE, FAKE, None, None, None, 0, FAKE,
                     1 << 40, None) == -1
    # fuse flag must be 0/1
    assert L.mlp_bwd(ctypes.byref(p), *args, FAKE, FAKE, FAKE, None, None, None, 3, FAKE,
                     1 << 40, None) == -1
    # recompute-mode workspace is larger
    need = m.mlp_workspace_size(p, m.MODE_BWD_RECOMPUTE)
    assert L.mlp_bwd_recompute(ctypes.byref(p), *args, FAKE, None, None, None, 0, FAKE,
                               need - 1, None) == -4
    # non-gated: dWu must be NULL
    q = m.problem(64, 128, 352, "relu_sq")
    assert L.mlp_bwd_recompute(ctypes.byref(q), FAKE, FAKE, FAKE, None, FAKE, None, None, FAKE,
                               None, 0, FAKE, 1 << 40, None) == -1


def test_block_validation(L):
    p = m.problem(64, 128, 352, "relu_sq")
    b = m.block(1.1 ** 0.5, 0.8, 2.0 ** -7)
    ws = 1 << 40
    fwd = lambda prob, blk, rstd=FAKE: L.mlp_block_fwd(  # noqa: E731
        ctypes.byref(prob), blk, FAKE, FAKE, None, FAKE, FAKE, None, None, rstd, FAKE, ws, None)
    assert fwd(p, None) == -1                       # no block
    assert fwd(p, ctypes.byref(b), rstd=None) == -1  # rstd required
    assert fwd(p, ctypes.byref(b), rstd=FAKE + 4) == -2  # rstd 16-byte aligned
    assert fwd(p, ctypes.byref(m.block(eps=-1.0))) == -1
    assert fwd(p, ctypes.byref(m.block(post_lambda=float("inf")))) == -1
    bwd = lambda dx: L.mlp_block_bwd(  # noqa: E731
        ctypes.byref(p), ctypes.byref(b), FAKE + 256, FAKE, FAKE, None, FAKE, FAKE, None, FAKE,
        dx, None, None, None, 0, FAKE, ws, None)
    assert bwd(FAKE) == -1        # dx aliases x
    assert bwd(FAKE + 256) == -1  # dx aliases dy


def test_fp8_validation_and_workspace(L):
    p = m.problem(2048, 768, 3072, "relu_sq")
    assert m.mlp_workspace_size(p, m.MODE_FP8_FWD) == 1024 + 2048 * 3072
    ws = 1 << 40
    f = lambda prob, scales=FAKE: L.mlp_fp8_fwd(  # noqa: E731
        ctypes.byref(prob), FAKE, FAKE, FAKE, scales, FAKE, None, None, None, FAKE, ws, None)
    assert f(m.problem(64, 128, 352)) == -3            # SwiGLU: unsupported
    assert f(m.problem(64, 136, 352, "relu_sq")) == -2  # H % 16
    assert f(p, scales=None) == -1
    assert L.mlp_fp8_quantize(FAKE, 12, FAKE, FAKE, None, None) == -1   # n % 8
    assert L.mlp_fp8_quantize(FAKE, 0, FAKE, FAKE, None, None) == 0     # nothing to do
    assert L.mlp_fp8_quantize(FAKE, 16, None, FAKE, None, None) == -1   # no scale


def test_fp8_backward_validation_and_workspace(L):
    p = m.problem(1000, 768, 3072, "relu_sq")
    r = lambda n: (n + 255) // 256 * 256  # noqa: E731
    need = 1024 + r(1000 * 768) + r(1000 * 3072)
    assert m.mlp_workspace_size(p, m.MODE_FP8_BWD) == need
    ws = 1 << 40

    def b(prob=p, dout=FAKE, x8=FAKE, W1=FAKE, W2=FAKE, pre=FAKE, a8=FAKE, scales=FAKE, dx=FAKE,
          dW1=FAKE, dW2=FAKE, ws_bytes=ws):
        return L.mlp_fp8_bwd(ctypes.byref(prob), dout, x8, W1, W2, pre, a8, scales, dx, dW1, dW2,
                             None, FAKE, ws_bytes, None)
    assert b(prob=m.problem(64, 128, 352)) == -3             # SwiGLU: unsupported
    assert b(prob=m.problem(64, 136, 352, "relu_sq")) == -2  # H % 16
    assert b(scales=None) == -1
    assert b(dout=None) == -1
    assert b(dout=FAKE + 8) == -2                 # 16-byte alignment
    assert b(W1=None) == -1                       # dx needs W1_8
    assert b(x8=None) == -1                       # dW1 needs x8
    assert b(a8=None) == -1                       # dW2 needs a8
    # without the saved preact the derivative recomputes it: x8 and W1_8 are then needed
    assert b(pre=None, x8=None, dW1=None) == -1
    assert b(pre=None, W1=None, dx=None) == -1
    assert b(W2=None) == -1                       # ... and W2_8
    assert b(ws_bytes=need - 1) == -4
    # nothing requested: returns before any CUDA call; absent operands of
    # unrequested outputs are fine
    assert b(dx=None, dW1=None, dW2=None, x8=None, W1=None, W2=None, pre=None, a8=None) == 0


def test_kernel_names_and_empty_trace(L):
    assert m.mlp_kernel_name(2) == "dgated"
    assert m.mlp_kernel_name(6) == "convert"
    assert m.mlp_kernel_name(7) == "dact_recompute"
    assert m.mlp_kernel_name(8) == "rstd"
    assert m.mlp_kernel_name(9) == "rmsnorm_bwd"
    assert m.mlp_kernel_name(10) == "quant_f8"
    assert m.mlp_kernel_name(11) == "fwd_fused"
    assert m.mlp_kernel_name(99) == "unknown"
    # every tag the header declares has a name of its own
    hdr = open(os.path.join(ROOT, "include", "mlp.h")).read()
    tags = [int(v) for v in re.findall(r"MLP_KERNEL_\w+ = (\d+)", hdr)]
    assert tags == list(range(len(tags)))
    names = [m.mlp_kernel_name(t) for t in tags]
    assert "unknown" not in names and len(set(names)) == len(names)
    assert m.mlp_trace_read() == []  # nothing recorded: no CUDA call is made


def test_tile_policy_values(L):
    assert L.mlp_set_tile_policy(4) == -1
    assert L.mlp_set_tile_policy(-1) == -1
    for v in (1, 2, 3, 0):
        assert L.mlp_set_tile_policy(v) == 0


def test_debug_hooks_validate(L):
    assert L.mlp_debug_set_flags(8) == -1
    assert L.mlp_debug_set_flags(-1) == -1
    assert L.mlp_debug_set_flags(2) == 0  # MLP_DEBUG_DECODE_FMA
    assert L.mlp_debug_set_flags(4) == 0  # MLP_DEBUG_DECODE_MMA
    assert L.mlp_debug_set_flags(0) == 0
    assert L.mlp_set_wait_timeout_ms(0) == 0


def test_refresh_scales_validates(L):
    # rejected before any launch (fake, never-dereferenced pointers)
    r = L.mlp_fp8_refresh_scales
    assert r(FAKE, FAKE, -1, 1, 1.0, 0.0, None) == -1
    assert r(FAKE, FAKE, 1, 0, 1.0, 0.0, None) == -1
    assert r(None, FAKE, 1, 1, 1.0, 0.0, None) == -1
    assert r(FAKE, None, 1, 1, 1.0, 0.0, None) == -1
    assert r(FAKE, FAKE, 1, 1, float("inf"), 0.0, None) == -1
    assert r(FAKE, FAKE, 1, 1, 1.0, float("nan"), None) == -1
    assert r(FAKE + 2, FAKE, 1, 1, 1.0, 0.0, None) == -2
    assert r(FAKE, FAKE, 0, 1, 1.0, 0.0, None) == 0  # nothing to do: nothing enqueued
    assert m.mlp_kernel_name(12) == "refresh_scales"


def test_plan_and_hold_validate(L):
    plan = m.Plan()
    p = m.problem(2048, 4096, 11008)
    assert L.mlp_plan(ctypes.byref(p), m.MODE_FWD, 0, None) == -1
    assert L.mlp_plan(ctypes.byref(p), 9, 0, ctypes.byref(plan)) == -1
    assert L.mlp_plan(ctypes.byref(p), m.MODE_BWD, 2, ctypes.byref(plan)) == -1
    assert L.mlp_plan(ctypes.byref(m.problem(0, 8, 8)), 0, 0, ctypes.byref(plan)) == -1
    assert L.mlp_debug_hold_sms(0, 10, None) == -1
    assert L.mlp_debug_hold_sms(70000, 10, None) == -1
