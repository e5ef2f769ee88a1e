"""GPU parity of the backward (fa_bwd) against the fp64 backward oracle.

Tolerance, derived from the arithmetic (the pages give none for gradients):
bf16 inputs, P and dS rounded to bf16 (relative 2^-9) before the gradient
GEMMs, fp32 accumulation, bf16 outputs.  Per gradient G:
  max |G_gpu - G_ref| <= 2e-2 * max |G_ref| + 1e-4
  mean |G_gpu - G_ref| <= 1e-2 * mean |G_ref| + 1e-5
The absolute terms cover gradients that are exactly zero (one visible key:
dS = P (dP - D) vanishes, up to the rounding of O inside D).
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from oracle import backward  # noqa: E402
from exact_attention_28_gb300 import inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_28_gb300 import build, ops as _ops
    build.build()
    _ops.load_library()
    return _ops


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def check(name, got, ref):
    got = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    top = np.max(np.abs(ref))
    assert np.all(np.isfinite(got)), name
    assert err.max() <= 2e-2 * top + 1e-4, f"{name}: max err {err.max():.3e} vs max |ref| {top:.3e}"
    assert err.mean() <= 1e-2 * np.mean(np.abs(ref)) + 1e-5, f"{name}: mean err {err.mean():.3e}"


def run_case(ops, B, H, Nq, Nk, d, causal, seed=0, scale=None):
    q, k, v = inputs.custom_inputs(1234 + seed, B, H, Nq, Nk, d)
    do = inputs.normal_bf16(99 + seed, (B, H, Nq, d))
    scale = float(np.float32(1 / math.sqrt(d))) if scale is None else scale
    Q, K, V, dO = to_dev(q), to_dev(k), to_dev(v), to_dev(do)
    O, L = ops.fa_fwd(Q, K, V, scale=scale, causal=causal)
    dQ, dK, dV = ops.fa_bwd(Q, K, V, O, L, dO, scale=scale, causal=causal)
    ops.check_device_status()
    f = oracle.bf16_bits_to_f64
    rQ, rK, rV = backward.backward_heads(f(q), f(k), f(v), f(do), float(np.float32(scale)), causal)
    check("dQ", dQ, rQ)
    check("dK", dK, rK)
    check("dV", dV, rV)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(256, 256), (384, 640), (640, 384), (300, 200), (129, 257), (1, 130), (128, 1)])
def test_backward_against_oracle(ops, d, causal, Nq, Nk):
    run_case(ops, 1, 2, Nq, Nk, d, causal, seed=Nq + Nk)


def test_backward_many_heads(ops):
    run_case(ops, 2, 8, 512, 512, 128, True, seed=7)


@pytest.mark.parametrize("scale", [0.5, -0.2])
def test_backward_other_scales(ops, scale):
    run_case(ops, 1, 2, 200, 300, 64, False, seed=11, scale=scale)


def test_backward_zero_upstream_gradient_gives_zero(ops):
    q, k, v = inputs.custom_inputs(5, 1, 2, 256, 256, 128)
    Q, K, V = to_dev(q), to_dev(k), to_dev(v)
    O, L = ops.fa_fwd(Q, K, V, causal=True)
    dQ, dK, dV = ops.fa_bwd(Q, K, V, O, L, torch.zeros_like(Q), causal=True)
    ops.check_device_status()
    for g in (dQ, dK, dV):
        assert torch.count_nonzero(g).item() == 0


def test_autograd_wrapper_matches_the_oracle(ops):
    # flash_attention(...).backward(dO) runs fa_fwd then fa_bwd; compare with the oracle
    B, H, Nq, Nk, d = 1, 2, 200, 300, 64
    q, k, v = inputs.custom_inputs(777, B, H, Nq, Nk, d)
    do = inputs.normal_bf16(778, (B, H, Nq, d))
    Q, K, V = (to_dev(a).requires_grad_(True) for a in (q, k, v))
    O = ops.flash_attention(Q, K, V, causal=True)
    O.backward(to_dev(do))
    ops.check_device_status()
    f = oracle.bf16_bits_to_f64
    scale = 1 / math.sqrt(d)
    O_ref, _ = oracle.attention(q, k, v, scale, True)
    assert np.abs(O.detach().float().cpu().numpy() - O_ref).max() <= 2e-2
    rQ, rK, rV = backward.backward_heads(f(q), f(k), f(v), f(do), scale, True)
    check("dQ", Q.grad, rQ)
    check("dK", K.grad, rK)
    check("dV", V.grad, rV)


def elementwise_bounds(q, k, v, do, scale, causal):
    """Per-element error bounds of dQ, dK, dV from the arithmetic, in fp64.

    The kernels round P and dS = P (dP - D) to bf16 (relative error <= 2^-9)
    before the gradient GEMMs, accumulate in fp32 and round the result to
    bf16 (<= 2^-9 of the element).  So element (i, c) of dQ = scale dS K is
    off by at most 2^-9 |dQ_ic| + 2^-9 scale sum_j |dS_ij| |K_jc| plus fp32
    accumulation error, and dK, dV likewise with dS^T Q and P^T dO.  D =
    rowsum(dO * O) is formed from the forward's bf16 O (relative error about
    2^-9 per element), so dS_ij also carries -P_ij dD_i with |dD_i| <= 2^-9
    sum_c |dO_ic| |O_ic|: on rows whose exact dS vanishes (a query that sees
    one key) this is the whole gradient.  The bounds below take twice those
    factors (2^-8), which also covers the recomputation of P from the stored
    LSE in fp32.
    """
    f = oracle.bf16_bits_to_f64
    Q, K, V, dO = f(q), f(k), f(v), f(do)
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    vis = np.ones((Nq, Nk), dtype=bool) if not causal else (np.arange(Nk)[None, :] <= np.arange(Nq)[:, None])
    bounds = [np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)]
    for b in range(B):
        for h in range(H):
            S = np.where(vis, scale * (Q[b, h] @ K[b, h].T), -np.inf)
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            O = P @ V[b, h]
            dS = P * (dO[b, h] @ V[b, h].T - (dO[b, h] * O).sum(axis=1, keepdims=True))
            dD = 2.0 ** -8 * (np.abs(dO[b, h]) * np.abs(O)).sum(axis=1)     # error of D from the bf16 O
            bounds[0][b, h] = 2.0 ** -8 * abs(scale) * (np.abs(dS) @ np.abs(K[b, h])) + \
                abs(scale) * dD[:, None] * (P @ np.abs(K[b, h]))
            bounds[1][b, h] = 2.0 ** -8 * abs(scale) * (np.abs(dS).T @ np.abs(Q[b, h])) + \
                abs(scale) * (P.T @ (dD[:, None] * np.abs(Q[b, h])))
            bounds[2][b, h] = 2.0 ** -8 * (P.T @ np.abs(dO[b, h]))
    return bounds


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(128, 128), (200, 300), (257, 129)])
def test_backward_every_element_within_its_bound(ops, d, causal, Nq, Nk):
    # element-wise: |G_gpu - G_ref| <= 2^-8 |G_ref| + (bf16 rounding of the
    # summed terms, see elementwise_bounds) + 1e-6, on every entry
    q, k, v = inputs.custom_inputs(4321 + Nq, 1, 2, Nq, Nk, d)
    do = inputs.normal_bf16(77 + Nk, (1, 2, Nq, d))
    scale = float(np.float32(1 / math.sqrt(d)))
    Q, K, V, dO = to_dev(q), to_dev(k), to_dev(v), to_dev(do)
    O, L = ops.fa_fwd(Q, K, V, scale=scale, causal=causal)
    grads = ops.fa_bwd(Q, K, V, O, L, dO, scale=scale, causal=causal)
    ops.check_device_status()
    f = oracle.bf16_bits_to_f64
    refs = backward.backward_heads(f(q), f(k), f(v), f(do), scale, causal)
    for name, g, r, extra in zip(("dQ", "dK", "dV"), grads, refs, elementwise_bounds(q, k, v, do, scale, causal)):
        err = np.abs(g.float().cpu().numpy().astype(np.float64) - r)
        bound = 2.0 ** -8 * np.abs(r) + extra + 1e-6
        worst = np.unravel_index(np.argmax(err / bound), err.shape)
        assert np.all(err <= bound), (f"{name}: element {worst} error {err[worst]:.3e} > bound {bound[worst]:.3e} "
                                      f"(ref {r[worst]:.3e})")
