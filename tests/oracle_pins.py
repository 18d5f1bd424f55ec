"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each pin is a function of an `oracle.Oracle` instance and raises
AssertionError when the oracle disagrees with:
  - closed forms of special cases (constant rows, eps = 0 worked example);
  - invariants that hold for every input (zero-mean / variance of LayerNorm
    output, mean square of RMSNorm output, the gradient identities);
  - central finite differences of the oracle's own forward (which pin the
    backward to the derivative of the forward);
  - an independent library routine: torch CPU float64 layer_norm /
    rms_norm and autograd;
  - symmetries (column permutation, LayerNorm shift invariance, scaling);
  - exact bf16 widening (torch's own bf16 -> float64 conversion);
  - the E4M3 format's closed-form code values and torch's float8_e4m3fn
    conversion (an independent library) for the FP8 output, and the
    defining properties of the two scalings (row maximum maps to 448; MX
    block maximum lands in [256, 512) after a power-of-two scale).
The definitions these facts follow are the LayerNorm/RMSNorm and
backward-pass paragraphs of "PyTorch atinge desempenho SOTA em normalizacao
com torch.compile" (matsubara.tec.br); eps inside the square root, the
population variance and y = xhat * gamma (+ beta) are the readings used
throughout.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

RMS, LAYER = 0, 1


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    err = np.abs(a - b)
    bound = atol + rtol * np.abs(b)
    if not np.all(err <= bound):
        k = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: max violation at {k}: got {a.flat[k]!r}, "
                             f"want {b.flat[k]!r}")


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- closed forms
def pin_rms_constant_row(orc):
    """RMSNorm of x = c * 1: mean square c^2, so y = gamma * c / sqrt(c^2 + eps),
    which tends to gamma * sign(c) as eps -> 0; c = 0 gives y = 0."""
    N = 16
    gamma = _rng(1).uniform(0.5, 1.5, N)
    # eps = 0 and c = 3: sqrt(9) = 3 exactly, y = gamma exactly.
    y, r, _ = orc.fwd_f64(np.full((1, N), 3.0), gamma, None, 0.0, RMS)
    _close(y[0], gamma, 0, what="rms const eps=0")
    _close(r, [1.0 / 3.0], 1e-15, what="rms const rstd")
    y, _, _ = orc.fwd_f64(np.full((1, N), -2.5), gamma, None, 0.0, RMS)
    _close(y[0], -gamma, 1e-15, what="rms const negative")
    # eps = c^2: r = 1 / sqrt(2 c^2), y = gamma / sqrt(2) * sign(c).
    y, r, _ = orc.fwd_f64(np.full((1, N), 2.0), gamma, None, 4.0, RMS)
    _close(y[0], gamma / np.sqrt(2.0), 1e-15, what="rms const eps=c^2")
    _close(r, [1.0 / np.sqrt(8.0)], 1e-15, what="rms const eps=c^2 rstd")
    # tiny eps: y -> gamma * sign(c)
    y, _, _ = orc.fwd_f64(np.full((1, N), 0.75), gamma, None, 1e-12, RMS)
    _close(y[0], gamma, 1e-11, what="rms const eps->0")
    y, _, _ = orc.fwd_f64(np.zeros((1, N)), gamma, None, 1e-6, RMS)
    assert np.all(y == 0.0), "rms zero row"


def pin_layer_constant_row(orc):
    """LayerNorm of a constant row: variance 0, xhat = 0, y = beta,
    rstd = 1/sqrt(eps), and dx = rstd * (g - mean(g)) with g = dy * gamma."""
    N = 12
    rng = _rng(2)
    gamma = rng.uniform(0.5, 1.5, N)
    beta = rng.normal(0, 0.1, N)
    eps = 1e-5
    x = np.full((1, N), 0.625)  # exactly representable, so the mean is exact
    y, r, mu = orc.fwd_f64(x, gamma, beta, eps, LAYER)
    _close(y[0], beta, 0, 1e-15, what="ln const y")
    _close(mu, [0.625], 0, what="ln const mean")
    _close(r, [1.0 / np.sqrt(eps)], 1e-15, what="ln const rstd")
    dy = rng.normal(0, 1, (1, N))
    dx, dg, db = orc.bwd_f64(dy, x, gamma, eps, LAYER)
    g = dy[0] * gamma
    _close(dx[0], (g - g.mean()) / np.sqrt(eps), 1e-12, 1e-12, what="ln const dx")
    _close(dg, np.zeros(N), 0, 1e-15, what="ln const dgamma")
    _close(db, dy[0], 0, 0, what="ln const dbeta")


def pin_zscore_worked_example(orc):
    """x = [1, 2, 3, 4], eps = 0, gamma = 1, beta = 0: LayerNorm output is the
    population z-score (x - 2.5) / sqrt(1.25); RMSNorm of [3, 4] with eps = 0
    is [3, 4] / sqrt(12.5)."""
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    y, r, mu = orc.fwd_f64(x, np.ones(4), np.zeros(4), 0.0, LAYER)
    _close(y[0], (x[0] - 2.5) / np.sqrt(1.25), 1e-15, what="zscore")
    _close(mu, [2.5], 0, what="zscore mean")
    y, _, _ = orc.fwd_f64(np.array([[3.0, 4.0]]), np.ones(2), None, 0.0, RMS)
    _close(y[0], np.array([3.0, 4.0]) / np.sqrt(12.5), 1e-15, what="rms 3-4")


# ------------------------------------------------------------------ invariants
def pin_layer_output_moments(orc):
    """gamma = 1, beta = 0: each output row has mean 0 and population variance
    v / (v + eps), v the population variance of the input row (numpy.var)."""
    rng = _rng(3)
    for N, eps in ((7, 1e-5), (64, 1e-2), (1000, 1e-5), (33, 0.5)):
        x = rng.normal(0.3, 1.7, (5, N))
        y, _, mu = orc.fwd_f64(x, np.ones(N), np.zeros(N), eps, LAYER)
        v = x.var(axis=1)
        _close(y.mean(axis=1), np.zeros(5), 0, 1e-13, what="ln out mean")
        _close(y.var(axis=1), v / (v + eps), 1e-12, what="ln out var")
        _close(mu, x.mean(axis=1), 1e-13, 1e-15, what="ln mean")


def pin_rms_output_moment(orc):
    """gamma = 1: the mean of y^2 over a row is m / (m + eps), m = mean(x^2)."""
    rng = _rng(4)
    for N, eps in ((5, 1e-6), (128, 1e-2), (999, 1e-6), (16, 2.0)):
        x = rng.normal(-0.2, 0.9, (4, N))
        y, r, mu = orc.fwd_f64(x, np.ones(N), None, eps, RMS)
        m = (x * x).mean(axis=1)
        _close((y * y).mean(axis=1), m / (m + eps), 1e-12, what="rms out moment")
        assert np.all(mu == 0.0), "rms mean output must be 0"


def pin_gradient_identities(orc):
    """For every row: LayerNorm  sum_j dx_j = 0 and
    sum_j xhat_j dx_j = r N c eps / (v + eps); RMSNorm  sum_j x_j dx_j =
    N c eps / (m + eps); with c = mean_j(dy_j gamma_j xhat_j).  xhat, v, m
    and r are computed here from numpy's mean/var."""
    rng = _rng(5)
    for N, eps in ((9, 1e-5), (256, 1e-3), (77, 0.25)):
        x = rng.normal(0.5, 1.3, (6, N))
        dy = rng.normal(0, 1, (6, N))
        gamma = rng.uniform(0.5, 1.5, N)
        # LayerNorm
        dx, _, _ = orc.bwd_f64(dy, x, gamma, eps, LAYER)
        v = x.var(axis=1, keepdims=True)
        r = 1.0 / np.sqrt(v + eps)
        xhat = (x - x.mean(axis=1, keepdims=True)) * r
        c = (dy * gamma * xhat).mean(axis=1)
        scale = np.abs(dx).sum(axis=1)
        _close(dx.sum(axis=1), np.zeros(6), 0, 1e-13 * scale.max(), what="ln sum dx")
        _close((xhat * dx).sum(axis=1), r[:, 0] * N * c * eps / (v[:, 0] + eps),
               1e-9, 1e-13 * scale.max(), what="ln xhat.dx")
        # RMSNorm
        dx, _, _ = orc.bwd_f64(dy, x, gamma, eps, RMS)
        m = (x * x).mean(axis=1, keepdims=True)
        xhat = x / np.sqrt(m + eps)
        c = (dy * gamma * xhat).mean(axis=1)
        _close((x * dx).sum(axis=1), N * c * eps / (m[:, 0] + eps), 1e-9,
               1e-13 * np.abs(x * dx).sum(axis=1).max(), what="rms x.dx")


def pin_column_sums(orc):
    """dgamma / dbeta accumulate over rows: the result for a block of rows is
    the sum of the results for each single row (checked row by row), and dbeta
    is exactly the column sum of dy in LayerNorm mode, zero in RMSNorm."""
    rng = _rng(6)
    M, N = 5, 24
    x = rng.normal(0, 1, (M, N))
    dy = rng.normal(0, 1, (M, N))
    gamma = rng.uniform(0.5, 1.5, N)
    for mode in (RMS, LAYER):
        _, dg, db = orc.bwd_f64(dy, x, gamma, 1e-5, mode)
        acc = np.zeros(N)
        for i in range(M):
            _, dgi, _ = orc.bwd_f64(dy[i:i + 1], x[i:i + 1], gamma, 1e-5, mode)
            acc += dgi
        _close(dg, acc, 1e-13, 1e-15, what="dgamma additivity")
        if mode == LAYER:
            _close(db, dy.sum(axis=0), 1e-15, 1e-15, what="dbeta = colsum dy")
        else:
            assert np.all(db == 0.0), "rms dbeta must be zero"


# ---------------------------------------------------------- finite differences
def _loss(orc, x, gamma, beta, dy, eps, mode):
    y, _, _ = orc.fwd_f64(x, gamma, beta, eps, mode)
    return float(np.sum(dy * y))


def pin_finite_differences(orc):
    """Central differences (h = 1e-6) of L = sum(dy * y) with respect to x,
    gamma and beta agree with the analytic dx, dgamma and dbeta."""
    rng = _rng(7)
    h = 1e-6
    cases = [(1, 1), (2, 2), (3, 3), (2, 8), (3, 17)]
    for mode in (RMS, LAYER):
        for M, N in cases:
            for eps in (1e-5, 0.3):
                x = rng.normal(0.2, 1.0, (M, N))
                dy = rng.normal(0, 1, (M, N))
                gamma = rng.uniform(0.5, 1.5, N)
                beta = rng.normal(0, 0.1, N) if mode == LAYER else None
                dx, dg, db = orc.bwd_f64(dy, x, gamma, eps, mode)
                fd = np.zeros_like(x)
                for i in range(M):
                    for j in range(N):
                        xp = x.copy(); xp[i, j] += h
                        xm = x.copy(); xm[i, j] -= h
                        fd[i, j] = (_loss(orc, xp, gamma, beta, dy, eps, mode)
                                    - _loss(orc, xm, gamma, beta, dy, eps, mode)) / (2 * h)
                tol = 1e-6 * max(1.0, np.abs(dx).max())
                _close(dx, fd, 1e-6, tol, what=f"fd dx mode={mode} {M}x{N}")
                fdg = np.zeros(N)
                fdb = np.zeros(N)
                for j in range(N):
                    gp = gamma.copy(); gp[j] += h
                    gm = gamma.copy(); gm[j] -= h
                    fdg[j] = (_loss(orc, x, gp, beta, dy, eps, mode)
                              - _loss(orc, x, gm, beta, dy, eps, mode)) / (2 * h)
                    if mode == LAYER:
                        bp = beta.copy(); bp[j] += h
                        bm = beta.copy(); bm[j] -= h
                        fdb[j] = (_loss(orc, x, gamma, bp, dy, eps, mode)
                                  - _loss(orc, x, gamma, bm, dy, eps, mode)) / (2 * h)
                tol = 1e-6 * max(1.0, np.abs(dg).max())
                _close(dg, fdg, 1e-6, tol, what=f"fd dgamma mode={mode} {M}x{N}")
                if mode == LAYER:
                    _close(db, fdb, 1e-6, 1e-6 * max(1.0, np.abs(db).max()),
                           what=f"fd dbeta {M}x{N}")
    # near-constant row where eps dominates the variance
    x = np.array([[1.0, 1.0 + 1e-4, 1.0 - 1e-4, 1.0, 1.0 + 2e-4]])
    dy = rng.normal(0, 1, x.shape)
    gamma = rng.uniform(0.5, 1.5, 5)
    beta = rng.normal(0, 0.1, 5)
    for mode in (RMS, LAYER):
        dx, _, _ = orc.bwd_f64(dy, x, gamma, 1e-3, mode)
        fd = np.zeros_like(x)
        for j in range(5):
            xp = x.copy(); xp[0, j] += h
            xm = x.copy(); xm[0, j] -= h
            fd[0, j] = (_loss(orc, xp, gamma, beta, dy, 1e-3, mode)
                        - _loss(orc, xm, gamma, beta, dy, 1e-3, mode)) / (2 * h)
        _close(dx, fd, 1e-6, 1e-6 * max(1.0, np.abs(dx).max()),
               what=f"fd near-const mode={mode}")


# ------------------------------------------------------------- library routine
def pin_torch_float64(orc):
    """torch CPU float64 layer_norm / rms_norm and autograd give the same y,
    dx, dgamma and dbeta (an implementation independent of this oracle)."""
    rng = _rng(8)
    for M, N in ((3, 1), (4, 8), (7, 100), (16, 1024), (2, 4104)):
        for eps in (1e-6, 1e-5, 0.1):
            x = rng.normal(0.1, 1.5, (M, N))
            dy = rng.normal(0, 1, (M, N))
            gamma = rng.uniform(0.5, 1.5, N)
            beta = rng.normal(0, 0.1, N)
            for mode in (RMS, LAYER):
                xt = torch.tensor(x, requires_grad=True)
                gt = torch.tensor(gamma, requires_grad=True)
                bt = torch.tensor(beta, requires_grad=True)
                if mode == LAYER:
                    yt = F.layer_norm(xt, (N,), gt, bt, eps)
                else:
                    yt = F.rms_norm(xt, (N,), gt, eps)
                gx, gg = torch.autograd.grad(yt, (xt, gt), torch.tensor(dy),
                                             retain_graph=True)
                y, _, _ = orc.fwd_f64(x, gamma, beta if mode == LAYER else None, eps, mode)
                dx, dg, db = orc.bwd_f64(dy, x, gamma, eps, mode)
                ys = np.abs(y).max()
                _close(y, yt.detach().numpy(), 1e-12, 1e-14 * ys, what=f"torch y {mode}")
                _close(dx, gx.numpy(), 1e-10, 1e-12 * max(1, np.abs(dx).max()),
                       what=f"torch dx {mode} {M}x{N}")
                _close(dg, gg.numpy(), 1e-10, 1e-12 * max(1, np.abs(dg).max()),
                       what=f"torch dgamma {mode}")
                if mode == LAYER:
                    (gb,) = torch.autograd.grad(yt, (bt,), torch.tensor(dy))
                    _close(db, gb.numpy(), 1e-12, 1e-13, what="torch dbeta")


# ------------------------------------------------------------------ symmetries
def pin_symmetries(orc):
    """Permuting columns (with gamma, beta) permutes every output; LayerNorm
    is invariant to adding a constant to a row; scaling x by alpha equals the
    normalisation with eps / alpha^2."""
    rng = _rng(9)
    M, N = 4, 37
    x = rng.normal(0, 1, (M, N))
    dy = rng.normal(0, 1, (M, N))
    gamma = rng.uniform(0.5, 1.5, N)
    beta = rng.normal(0, 0.1, N)
    perm = rng.permutation(N)
    for mode in (RMS, LAYER):
        b = beta if mode == LAYER else None
        y, r, mu = orc.fwd_f64(x, gamma, b, 1e-5, mode)
        yp, rp, _ = orc.fwd_f64(x[:, perm], gamma[perm], None if b is None else b[perm],
                                1e-5, mode)
        _close(yp, y[:, perm], 1e-13, 1e-15, what="perm y")
        _close(rp, r, 1e-13, what="perm rstd")
        dx, dg, db = orc.bwd_f64(dy, x, gamma, 1e-5, mode)
        dxp, dgp, dbp = orc.bwd_f64(dy[:, perm], x[:, perm], gamma[perm], 1e-5, mode)
        _close(dxp, dx[:, perm], 1e-11, 1e-13, what="perm dx")
        _close(dgp, dg[perm], 1e-11, 1e-13, what="perm dgamma")
        alpha = 4.0
        ya, ra, _ = orc.fwd_f64(alpha * x, gamma, b, 1e-5, mode)
        ys, rs, _ = orc.fwd_f64(x, gamma, b, 1e-5 / alpha ** 2, mode)
        _close(ya, ys, 1e-13, 1e-15, what="scale y")
        _close(ra * alpha, rs, 1e-13, what="scale rstd")
    y0, _, mu0 = orc.fwd_f64(x, gamma, beta, 1e-5, LAYER)
    y1, _, mu1 = orc.fwd_f64(x + 3.0, gamma, beta, 1e-5, LAYER)
    _close(y1, y0, 1e-10, 1e-12, what="ln shift")
    _close(mu1, mu0 + 3.0, 1e-13, what="ln shift mean")


# ---------------------------------------------------------- bf16 entry points
def pin_bf16_entry_points(orc):
    """The bf16 entry points equal the f64 ones on the exactly widened values
    (widening checked against torch's bf16 -> float64 conversion); row lists
    select rows; param grads equal the f64 column sums."""
    g = torch.Generator().manual_seed(11)
    M, N = 9, 40
    x = (torch.randn(M, N, generator=g) * 3).to(torch.bfloat16)
    dy = torch.randn(M, N, generator=g).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(N, generator=g)).to(torch.bfloat16)
    beta = (0.1 * torch.randn(N, generator=g)).to(torch.bfloat16)

    def bits(t):
        return t.view(torch.int16).numpy().view(np.uint16)

    xf, dyf = x.double().numpy(), dy.double().numpy()
    gf, bf = gamma.double().numpy(), beta.double().numpy()
    rows = np.array([8, 0, 3, 3])
    for mode in (RMS, LAYER):
        b_bits = bits(beta) if mode == LAYER else None
        b_f = bf if mode == LAYER else None
        y, r, mu = orc.fwd_bf16(bits(x), bits(gamma), b_bits, 1e-5, mode)
        y2, r2, mu2 = orc.fwd_f64(xf, gf, b_f, 1e-5, mode)
        assert np.array_equal(y, y2) and np.array_equal(r, r2) and np.array_equal(mu, mu2), \
            "bf16 fwd != f64 fwd on widened inputs"
        ys, rs, _ = orc.fwd_bf16(bits(x), bits(gamma), b_bits, 1e-5, mode, rows=rows)
        assert np.array_equal(ys, y[rows]) and np.array_equal(rs, r[rows]), "row selection"
        dx, dg, db = orc.bwd_f64(dyf, xf, gf, 1e-5, mode)
        dxs = orc.bwd_dx_bf16(bits(dy), bits(x), bits(gamma), 1e-5, mode, rows=rows)
        assert np.array_equal(dxs, dx[rows]), "bf16 dx rows"
        pg, pb, pga, pba = orc.param_grads_bf16(bits(dy), bits(x), bits(gamma), 1e-5, mode)
        assert np.array_equal(pg, dg) and np.array_equal(pb, db), "param grads"
        assert np.all(pga >= np.abs(pg)) and np.all(pba >= np.abs(pb)), "abs sums"


# ------------------------------------------------- fused residual add + norm
def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def pin_residual_add_rounding(orc):
    """h = bf16(x + r) with the sum in binary32 and round-to-nearest-even:
    equal, bit for bit, to torch's own float32 add and bf16 conversion, on
    values that exercise carries, cancellation, ties, overflow to inf and
    operands many binades apart."""
    g = torch.Generator().manual_seed(12)
    x = torch.randn(64, 96, generator=g) * torch.exp2(torch.randint(-20, 20, (64, 96), generator=g).float())
    r = torch.randn(64, 96, generator=g) * torch.exp2(torch.randint(-20, 20, (64, 96), generator=g).float())
    r[:8] = -x[:8]                      # exact cancellation
    r[8:16] = x[8:16] * 2.0 ** -8       # sums that land on bf16 ties
    x[16, :4] = 3.0e38
    r[16, :4] = 3.0e38                  # overflow to inf
    xb, rb = x.to(torch.bfloat16), r.to(torch.bfloat16)
    want = (xb.float() + rb.float()).to(torch.bfloat16)
    got = orc.residual_add_bf16(_bits(xb), _bits(rb))
    assert np.array_equal(got, _bits(want)), "residual add bits differ from float32 add + RNE"


def pin_add_norm_composition(orc):
    """The fused forward is the norm of h; the fused backward is the norm's
    dx at h plus the residual gradient dh, added (not subtracted, not scaled)."""
    g = torch.Generator().manual_seed(13)
    M, N = 6, 40
    x = torch.randn(M, N, generator=g).to(torch.bfloat16)
    r = torch.randn(M, N, generator=g).to(torch.bfloat16)
    dy = torch.randn(M, N, generator=g).to(torch.bfloat16)
    dh = torch.randn(M, N, generator=g).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(N, generator=g)).to(torch.bfloat16)
    beta = (0.1 * torch.randn(N, generator=g)).to(torch.bfloat16)
    for mode in (RMS, LAYER):
        bb = _bits(beta) if mode == LAYER else None
        h, y, rs, mu = orc.add_fwd_bf16(_bits(x), _bits(r), _bits(gamma), bb, 1e-5, mode)
        y2, rs2, mu2 = orc.fwd_bf16(h, _bits(gamma), bb, 1e-5, mode)
        assert np.array_equal(y, y2) and np.array_equal(rs, rs2)
        dx = orc.add_bwd_dx_bf16(_bits(dy), h, _bits(dh), _bits(gamma), 1e-5, mode)
        dx0 = orc.bwd_dx_bf16(_bits(dy), h, _bits(gamma), 1e-5, mode)
        assert np.array_equal(dx, dx0 + dh.double().numpy()), "dx must be norm dx + dh"
        rows = np.array([5, 0, 2])
        dxs = orc.add_bwd_dx_bf16(_bits(dy), h, _bits(dh), _bits(gamma), 1e-5, mode, rows=rows)
        assert np.array_equal(dxs, dx[rows]), "row selection of the fused backward"


FP8_ROW, FP8_MX = 0, 1


def _e4m3_spacing(v):
    """Distance between adjacent E4M3 values around |v| (< 448): 2^(e-3) in
    binade e, 2^-9 in the subnormal range."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.exp2(np.maximum(e, -6.0) - 3.0)


def _check_nearest(codes, v, orc, what):
    """decode(codes) is a nearest E4M3 value of v (saturating at 448), with
    the sign of v."""
    d = orc.e4m3_decode(codes)
    v = np.asarray(v, np.float64)
    sat = np.abs(v) >= 448.0
    assert np.all(np.abs(d[sat]) == 448.0), f"{what}: saturation"
    ok = np.abs(d - v) <= 0.5 * _e4m3_spacing(v)
    assert np.all(ok | sat), f"{what}: {int((~(ok | sat)).sum())} codes are not nearest"
    wrong_sign = (v != 0) & (d != 0) & ((d < 0) != (v < 0))
    assert not wrong_sign.any(), f"{what}: sign"


def pin_e4m3_codes(orc):
    """E4M3 codes: every value equals the format's closed form and torch's
    float8_e4m3fn decoding; encoding inverts decoding, breaks ties to the
    even mantissa, saturates at +-448 and agrees with torch's float32 ->
    float8_e4m3fn conversion on in-range values."""
    codes = np.arange(256, dtype=np.uint8)
    d = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(d), nan) and nan.sum() == 2, "NaN codes"
    assert np.array_equal(d[~nan], ref[~nan]), "E4M3 decoding differs from torch"
    assert d[0x7E] == 448.0 and d[0x01] == 2.0 ** -9 and d[0x08] == 2.0 ** -6
    assert d[0x38] == 1.0 and d[0x80] == 0.0 and np.signbit(d[0x80])
    fin = codes[~nan]
    assert np.array_equal(orc.e4m3_encode(d[~nan]), fin), "encode(decode(c)) != c"
    pos = np.arange(0x00, 0x7E, dtype=np.int64)          # adjacent pairs (c, c+1)
    lo, hi = d[pos], d[pos + 1]
    mid = 0.5 * (lo + hi)
    even = np.where(pos % 2 == 0, pos, pos + 1)
    assert np.array_equal(orc.e4m3_encode(mid), even.astype(np.uint8)), "ties to even"
    assert np.array_equal(orc.e4m3_encode(-mid), (even | 0x80).astype(np.uint8)), "negative ties"
    below = mid - (hi - lo) * 2.0 ** -20
    above = mid + (hi - lo) * 2.0 ** -20
    assert np.array_equal(orc.e4m3_encode(below), pos.astype(np.uint8)), "below midpoint"
    assert np.array_equal(orc.e4m3_encode(above), (pos + 1).astype(np.uint8)), "above midpoint"
    big = np.array([448.0 * (1 + 2.0 ** -20), 464.0, 480.0, 1e30, np.inf])
    assert np.all(orc.e4m3_encode(big) == 0x7E) and np.all(orc.e4m3_encode(-big) == 0xFE)
    assert orc.e4m3_encode(np.array([np.nan]))[0] == 0x7F
    g = torch.Generator().manual_seed(21)
    mag = torch.exp2(torch.empty(20000, dtype=torch.float64).uniform_(-12.0, 8.77, generator=g))
    sgn = torch.where(torch.rand(20000, generator=g) < 0.5, -1.0, 1.0).double()
    v32 = (mag * sgn).float()
    want = v32.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode(v32.double().numpy())
    assert np.array_equal(got, want), "E4M3 encoding differs from torch's conversion"


def _fp8_inputs(seed, M, N, block_scales=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, N, generator=g)
    x[1] *= 50.0
    x[2, 3] = 80.0                                       # outlier
    gamma = 1 + 0.1 * torch.randn(N, generator=g)
    if block_scales:
        # very different block magnitudes, one block below 2^-119 (E8M0 clamp)
        nb = N // 32
        mult = torch.exp2(torch.tensor([(-8.0 + 5.0 * b) for b in range(nb)]))
        mult[-1] = 2.0 ** -128
        gamma = gamma * mult.repeat_interleave(32)
    beta = 0.1 * torch.randn(N, generator=g)
    if block_scales:
        beta = beta * mult.repeat_interleave(32)
    x = x.to(torch.bfloat16)
    x[3] = 0                                             # zero row
    return x, gamma.to(torch.bfloat16), beta.to(torch.bfloat16)


def pin_fp8_row_scaling(orc):
    """Per-row scaling: amax is the row's max |y| of the (already pinned)
    forward, scale = amax / 448, the row maximum gets code +-448, every code
    is a nearest E4M3 value of y / scale; a zero row has scale 1 and codes 0."""
    M, N = 5, 64
    x, gamma, beta = _fp8_inputs(31, M, N)
    for mode in (RMS, LAYER):
        bb = _bits(beta) if mode == LAYER else None
        # RMS: row 3 is zero -> y = 0; LayerNorm: y = beta there (nonzero)
        o = orc.fwd_fp8_bf16(_bits(x), None, _bits(gamma), bb, 1e-5, mode, FP8_ROW)
        y, _, _ = orc.fwd_bf16(_bits(x), _bits(gamma), bb, 1e-5, mode)
        assert np.array_equal(o["y"], y)
        amax = np.abs(y).max(axis=1)
        assert np.array_equal(o["amax"], amax)
        nz = amax > 0
        assert mode == LAYER or not nz[3], "zero row"
        _close(o["scale"][nz], amax[nz] / 448.0, 1e-15, what="row scale")
        assert np.all(o["scale"][~nz] == 1.0) and np.all(o["q"][~nz] & 0x7F == 0)
        dq = orc.e4m3_decode(o["q"])
        assert np.all(np.abs(dq[nz]).max(axis=1) == 448.0), "row max must map to 448"
        v = (y[nz] / amax[nz][:, None]) * 448.0
        _check_nearest(o["q"][nz], v, orc, f"row codes mode {mode}")


def pin_fp8_mx_scaling(orc):
    """MX scaling: each 32-column block gets X = 2^e with the block maximum
    in [256, 512) after scaling (e clamped at -127 for tiny blocks, E8M0
    byte e + 127), and every code is a nearest E4M3 value of y / X,
    saturating at 448."""
    M, N = 5, 256
    x, gamma, beta = _fp8_inputs(32, M, N, block_scales=True)
    nb = N // 32
    for mode in (RMS, LAYER):
        bb = _bits(beta) if mode == LAYER else None
        o = orc.fwd_fp8_bf16(_bits(x), None, _bits(gamma), bb, 1e-5, mode, FP8_MX)
        y, _, _ = orc.fwd_bf16(_bits(x), _bits(gamma), bb, 1e-5, mode)
        yb = y.reshape(M, nb, 32)
        amax = np.abs(yb).max(axis=2)
        assert np.array_equal(o["amax"], amax)
        X = o["scale"]
        e = np.log2(X)
        assert np.array_equal(e, np.round(e)), "MX scale must be a power of two"
        assert np.array_equal(o["ebyte"].astype(np.int64), e.astype(np.int64) + 127)
        live = amax > 0
        s = amax[live] / X[live]
        clamped = e[live] == -127
        assert np.all(s < 512.0) and np.all((s >= 256.0) | clamped), "block max not in [256, 512)"
        assert np.any(clamped), "the tiny block must hit the E8M0 clamp"
        assert np.all(e[~live] == -127)
        assert len(np.unique(e[0])) > 3, "scales must be per block"
        v = (yb / X[:, :, None]).reshape(M, N)
        _check_nearest(o["q"], v, orc, f"MX codes mode {mode}")


def pin_fp8_residual_composition(orc):
    """FP8 output of the fused residual form is the FP8 output of h."""
    g = torch.Generator().manual_seed(33)
    M, N = 4, 96
    x = torch.randn(M, N, generator=g).to(torch.bfloat16)
    r = torch.randn(M, N, generator=g).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(N, generator=g)).to(torch.bfloat16)
    h = orc.residual_add_bf16(_bits(x), _bits(r))
    for mode in (RMS, LAYER):
        for sc in (FP8_ROW, FP8_MX):
            a = orc.fwd_fp8_bf16(_bits(x), _bits(r), _bits(gamma), None, 1e-5, mode, sc)
            b = orc.fwd_fp8_bf16(h, None, _bits(gamma), None, 1e-5, mode, sc)
            for k in a:
                assert np.array_equal(a[k], b[k]), k
            rows = np.array([3, 1])
            c = orc.fwd_fp8_bf16(_bits(x), _bits(r), _bits(gamma), None, 1e-5, mode, sc,
                                 rows=rows)
            assert np.array_equal(c["q"], a["q"][rows]) and np.array_equal(c["scale"], a["scale"][rows])


# ------------------------------------------------ norm feeding a GEMM
def _gemm_case(seed, M, K, Nout, offset=0.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(M, K, generator=g) + offset).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(K, generator=g)).to(torch.bfloat16)
    beta = (0.1 * torch.randn(K, generator=g)).to(torch.bfloat16)
    w = (torch.randn(Nout, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    return x, gamma, beta, w


def pin_norm_gemm_selection(orc):
    """W whose row o holds one power of two s_o at column p(o) picks out
    column p(o) of the normalised rows: out[:, o] = s_o * y[:, p(o)] exactly.
    Pins the operand order (W is [Nout, K], one row per output feature) with
    a non-square W and a permutation that is not its own inverse."""
    K, Nout = 16, 24
    x, gamma, beta, _ = _gemm_case(21, 5, K, Nout)
    p = np.array([(3 * o + 1) % K for o in range(Nout)])
    s = 2.0 ** np.array([(o % 5) - 2 for o in range(Nout)])
    w = torch.zeros(Nout, K, dtype=torch.float64)
    w[np.arange(Nout), p] = torch.tensor(s)
    wb = _bits(w.to(torch.bfloat16))
    for mode in (RMS, LAYER):
        bb = _bits(beta) if mode == LAYER else None
        y, rs, mu = orc.fwd_bf16(_bits(x), _bits(gamma), bb, 1e-5, mode)
        out, rs2, mu2 = orc.norm_gemm_bf16(_bits(x), _bits(gamma), bb, wb, 1e-5, mode)
        assert out.shape == (5, Nout)
        assert np.array_equal(out, y[:, p] * s), f"selection W, mode {mode}"
        assert np.array_equal(rs, rs2) and np.array_equal(mu, mu2), "saved stats"
        rows = np.array([4, 0, 2])
        o2, _, _ = orc.norm_gemm_bf16(_bits(x), _bits(gamma), bb, wb, 1e-5, mode, rows=rows)
        assert np.array_equal(o2, out[rows]), "row selection"


def pin_norm_gemm_torch(orc):
    """torch CPU float64 layer_norm / rms_norm followed by F.linear (a library
    implementation independent of the oracle) gives the same output."""
    for M, K, Nout, off in ((3, 8, 5, 0.0), (7, 64, 40, 0.0), (9, 200, 33, 2.0),
                            (4, 1024, 96, 0.5)):
        x, gamma, beta, w = _gemm_case(22 + K, M, K, Nout, off)
        xt, gt, bt, wt = (t.double() for t in (x, gamma, beta, w))
        for mode in (RMS, LAYER):
            if mode == LAYER:
                yt = F.layer_norm(xt, (K,), gt, bt, 1e-5)
            else:
                yt = F.rms_norm(xt, (K,), gt, 1e-5)
            want = F.linear(yt, wt).numpy()
            scale = (yt.abs() @ wt.abs().T).numpy()
            bb = _bits(beta) if mode == LAYER else None
            out, _, _ = orc.norm_gemm_bf16(_bits(x), _bits(gamma), bb, _bits(w), 1e-5, mode)
            _close(out, want, 0, 1e-13 * scale.max(), what=f"torch norm+linear {mode} {K}")


def pin_norm_gemm_factorisation(orc):
    """The lazy pre-norm identity that lets a GEMM normalise after the
    contraction: with W' = W * gamma (per column), u = W' 1 and v = W beta,
    out = rstd * (x W'^T - mean * u) + v, each term formed separately in
    float64 from the raw x (row statistics taken with numpy)."""
    for off in (0.0, 3.0):
        x, gamma, beta, w = _gemm_case(31, 6, 48, 20, off)
        X, G, B, W = (t.double().numpy() for t in (x, gamma, beta, w))
        Wg = W * G[None, :]
        u = Wg.sum(axis=1)
        v = W @ B
        for mode in (RMS, LAYER):
            mu = X.mean(axis=1) if mode == LAYER else np.zeros(X.shape[0])
            var = ((X - mu[:, None]) ** 2).mean(axis=1) if mode == LAYER else (X ** 2).mean(axis=1)
            r = 1.0 / np.sqrt(var + 1e-5)
            want = r[:, None] * (X @ Wg.T - mu[:, None] * u[None, :])
            if mode == LAYER:
                want = want + v[None, :]
            bb = _bits(beta) if mode == LAYER else None
            out, rs, mean = orc.norm_gemm_bf16(_bits(x), _bits(gamma), bb, _bits(w), 1e-5, mode)
            scale = np.abs(r)[:, None] * (np.abs(X) @ np.abs(Wg).T) + np.abs(v)[None, :]
            _close(out, want, 0, 1e-12 * scale.max(), what=f"factorisation {mode} off={off}")
            _close(rs, r, 1e-13, what="rstd")


def pin_norm_gemm_layer_constant_weights(orc):
    """LayerNorm with gamma = 1: a constant weight row c sums the normalised
    row, sum_j xhat_j = 0, so out = c * sum_j beta_j (and 0 with beta = 0)."""
    K, Nout = 40, 6
    x, _, beta, _ = _gemm_case(41, 7, K, Nout, 1.5)
    ones = _bits(torch.ones(K, dtype=torch.bfloat16))
    c = torch.tensor([1.0, -2.0, 0.5, 3.0, 0.25, -1.0], dtype=torch.float64)
    wb = _bits(c[:, None].expand(Nout, K).to(torch.bfloat16).contiguous())
    out, _, _ = orc.norm_gemm_bf16(_bits(x), ones, None, wb, 1e-5, LAYER)
    _close(out, np.zeros_like(out), 0, 1e-12 * K, what="sum of xhat")
    out, _, _ = orc.norm_gemm_bf16(_bits(x), ones, _bits(beta), wb, 1e-5, LAYER)
    want = np.broadcast_to(c.numpy()[None, :] * beta.double().sum().item(), out.shape)
    _close(out, want, 0, 1e-12 * K, what="c * sum beta")


ALL_PINS = [
    pin_rms_constant_row,
    pin_layer_constant_row,
    pin_zscore_worked_example,
    pin_layer_output_moments,
    pin_rms_output_moment,
    pin_gradient_identities,
    pin_column_sums,
    pin_finite_differences,
    pin_torch_float64,
    pin_symmetries,
    pin_bf16_entry_points,
    pin_residual_add_rounding,
    pin_add_norm_composition,
    pin_e4m3_codes,
    pin_fp8_row_scaling,
    pin_fp8_mx_scaling,
    pin_fp8_residual_composition,
    pin_norm_gemm_selection,
    pin_norm_gemm_torch,
    pin_norm_gemm_factorisation,
    pin_norm_gemm_layer_constant_weights,
]
