"""Pins of the oracle's trainer backward (QUADS §3.2 Eq. 13, straight-through
estimator: the fake-quantizer is the identity in the backward, so the
gradients are the plain derivatives of the layer's forward).  The chain of
combine_grad, a dgrad product, swiglu_grad, segment_wgrad and the routed-row
gather-sum must equal central finite differences of the binary64 forward
combine(swiglu(scatter(x) W13^T) Wd^T) with the loss <out, dout> -- a wrong
sign, a swapped gate/up, a transposed operand or a row taken from the wrong
segment fails it."""
import numpy as np

import oracle


def _layer(T=6, H=32, I=16, E=3, topk=2, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 2] -= 100.0  # expert 2 gets no tokens: an empty segment
    w13 = rng.standard_normal((E, 2 * I, H)) * 0.3
    wd = rng.standard_normal((E, H, I)) * 0.3
    dout = rng.standard_normal((T, H))
    ids, rw = oracle.route_topk(logits, topk)
    counts, offs, dst = oracle.route_layout(ids, E)
    return x, w13, wd, dout, ids, rw.astype(np.float64), counts, offs, dst


def _forward(x, w13, wd, ids, rw, offs, dst):
    E, N13, H = w13.shape
    I = N13 // 2
    R = int(offs[-1])
    xr = np.zeros((R, H))
    T, topk = dst.shape
    for t in range(T):
        xr[dst[t]] = x[t]
    gu = np.zeros((R, 2 * I))
    for e in range(E):
        gu[offs[e]:offs[e + 1]] = xr[offs[e]:offs[e + 1]] @ w13[e].T
    h = oracle.swiglu(gu, I)
    y = np.zeros((R, H))
    for e in range(E):
        y[offs[e]:offs[e + 1]] = h[offs[e]:offs[e + 1]] @ wd[e].T
    return xr, gu, h, y, oracle.combine(y, dst.astype(np.int32), rw)


def _backward(x, w13, wd, dout, ids, rw, offs, dst):
    E = w13.shape[0]
    xr, gu, h, y, out = _forward(x, w13, wd, ids, rw, offs, dst)
    R = xr.shape[0]
    dy, dw = oracle.combine_grad(dout, y, dst, rw, R)
    dh = np.zeros_like(h)
    for e in range(E):
        dh[offs[e]:offs[e + 1]] = dy[offs[e]:offs[e + 1]] @ wd[e]
    dwd = oracle.segment_wgrad(dy, h, offs)
    dgu = oracle.swiglu_grad(gu, dh)
    dxr = np.zeros_like(xr)
    for e in range(E):
        dxr[offs[e]:offs[e + 1]] = dgu[offs[e]:offs[e + 1]] @ w13[e]
    dw13 = oracle.segment_wgrad(dgu, xr, offs)
    dx = oracle.combine(dxr, dst.astype(np.int32), np.ones(dst.shape))
    return dx, dw13, dwd, dw


def _fd(f, a, idx, eps=1e-6):
    a0 = a[idx]
    a[idx] = a0 + eps
    lp = f()
    a[idx] = a0 - eps
    lm = f()
    a[idx] = a0
    return (lp - lm) / (2 * eps)


def test_backward_matches_finite_differences():
    x, w13, wd, dout, ids, rw, counts, offs, dst = _layer()
    assert counts[2] == 0
    dx, dw13, dwd, dw = _backward(x, w13, wd, dout, ids, rw, offs, dst)
    loss = lambda: float(np.sum(_forward(x, w13, wd, ids, rw, offs, dst)[-1] * dout))
    rng = np.random.default_rng(1)
    for arr, grad in ((x, dx), (w13, dw13), (wd, dwd)):
        for _ in range(25):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            num = _fd(loss, arr, idx)
            assert abs(num - grad[idx]) <= 1e-6 * max(1.0, abs(num)), (idx, num, grad[idx])
    assert not dw13[2].any() and not dwd[2].any()  # the empty expert
    # the combine weights' gradient: d loss / d w[t,s] with the routing held fixed
    for t, s in [(0, 0), (3, 1), (5, 0)]:
        num = _fd(loss, rw, (t, s))
        assert abs(num - dw[t, s]) <= 1e-6 * max(1.0, abs(num))


def test_swiglu_grad_closed_form_points():
    # at g = 0: s = 1/2, so dg = dh * u / 2 and du = 0
    gu = np.array([[0.0, 3.0]])
    dh = np.array([[2.0]])
    assert np.allclose(oracle.swiglu_grad(gu, dh), [[3.0, 0.0]], rtol=0, atol=1e-15)
    # large g: silu(g) -> g, silu'(g) -> 1
    gu = np.array([[40.0, 0.5]])
    assert np.allclose(oracle.swiglu_grad(gu, dh), [[1.0, 80.0]], rtol=1e-12)
