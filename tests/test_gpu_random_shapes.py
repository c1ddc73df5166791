"""Seeded random shapes through the whole path against the fp64 oracle: the
training forward and the backward (saved or recomputed preacts, bf16 or
fp32-accumulated weight gradients), every activation.

The launch plan makes size-dependent choices: the weight-streaming forward
for 1-8 tokens (CUDA-core or warp-MMA stream), split-K for [M,H] outputs
with few tiles, the one-launch gated forward, single-CTA or CTA-pair tiles.
Hand-picked test shapes sit where their authors expected the boundaries;
these are drawn at random (with a fixed seed) from ranges that straddle
them, with ragged tails in every dimension and dimensions below one tile or
one k-block.  Each case records the choices mlp_plan reports, and the last
test checks that the draw reached every one of them."""
import numpy as np
import pytest

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import make_inputs
from mlp_gpu_helpers import compare_full, dev_tensors, dw_floor, oracle_full, run_gpu

pytestmark = pytest.mark.gpu

ACTS = list(m.ACTS)
MULTS = [(1.0, 1.0), (1.125, 2.0), (0.75, 1.5)]


def _draw(n=48, seed=20261203, max_mhi=2.2e9):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        r = rng.random()
        if r < 0.35:
            M = int(rng.integers(1, 17))            # weight-streaming forward
        elif r < 0.6:
            M = int(rng.integers(17, 300))          # split-K at decode sizes
        else:
            M = int(rng.integers(300, 1100))        # CTA pairs, the prefill split
        H = 8 * int(rng.choice([rng.integers(1, 40), rng.integers(40, 513)]))
        I = 8 * int(rng.choice([rng.integers(1, 40), rng.integers(40, 513)]))
        if M * H * I > max_mhi:
            continue
        act = ACTS[int(rng.integers(len(ACTS)))]
        gm, dm = MULTS[int(rng.integers(len(MULTS)))]
        mode = "saved" if rng.random() < 0.5 else "recompute"
        fuse = bool(rng.random() < 0.4)
        out.append((M, H, I, act, gm, dm, mode, fuse))
    return out


CASES = _draw()
SEEN = set()


def _choices(M, H, I, act, gm, dm, mode):
    prob = m.problem(M, H, I, act, gm, dm)
    fwd = m.mlp_plan(prob, m.MODE_FWD)
    bwd = m.mlp_plan(prob, m.MODE_BWD if mode == "saved" else m.MODE_BWD_RECOMPUTE)
    got = {("decode", fwd["decode"]), ("cta_group", fwd["cta_group"])}
    if fwd["decode"] == 0:
        got.add(("forward_split", fwd["out_split"] > 1))
        if act in m.GATED_ACTS:
            got.add(("fused_forward", fwd["fused_forward"]))
    got.add(("dx_split", bwd["out_split"] > 1))
    return got


@pytest.mark.parametrize("M,H,I,act,gm,dm,mode,fuse", CASES,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}-{c[3]}-{c[6]}-{'f32' if c[7] else 'bf16'}"
                              for c in CASES])
def test_random_shape_parity(M, H, I, act, gm, dm, mode, fuse):
    SEEN.update(_choices(M, H, I, act, gm, dm, mode))
    t = make_inputs(M, H, I, act, seed=M * 7919 + H * 31 + I, dW_prev=fuse)
    tc = {k: v for k, v in t.items() if not k.endswith("_prev")}
    prev = {k: v for k, v in t.items() if k.endswith("_prev")} if fuse else None
    got, bad, _ = run_gpu(dev_tensors(tc), M, H, I, act, gm, dm, mode=mode, fuse=fuse, dW_prev=prev)
    assert not bad, f"guard band overwritten: {bad}"
    ref = oracle_full(tc, act, gm, dm, dW_prev=prev)
    compare_full(got, ref, fuse, floor=dw_floor(tc, act, gm, dm, mode, ref, prev) if fuse else None)


def test_the_draw_covers_every_launch_choice():
    """Runs after the cases above (file order): every size-dependent choice
    of the plan was taken by at least one drawn shape."""
    if len(SEEN) == 0:
        pytest.skip("the random cases did not run")
    want = {("decode", 0), ("decode", 1), ("decode", 2), ("cta_group", 1), ("cta_group", 2),
            ("forward_split", True), ("forward_split", False), ("fused_forward", 1),
            ("dx_split", True), ("dx_split", False)}
    assert want <= SEEN, sorted(want - SEEN)
