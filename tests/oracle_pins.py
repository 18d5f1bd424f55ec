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
  - exact bf16 widening (torch's own bf16 -> float64 conversion).
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
]
