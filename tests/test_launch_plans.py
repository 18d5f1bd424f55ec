"""CPU checks of every launch plan the library would use on a GB300
(152 SMs, 227 KB opt-in shared memory): all accesses in bounds, alignment
rules met, every tile and column owned exactly once."""
import pytest

import memory_bound_normalization_rmsnorm_gb300 as gb
from memory_bound_normalization_rmsnorm_gb300.workloads import WORKLOADS

import launch_check

SMS = 152
OPTIN = 232448

SMALL_N = [8, 16, 24, 40, 64, 72, 104, 128, 200, 256, 264, 512, 520, 768, 776, 1000,
           1024, 1032, 2048, 2056, 3072, 4096, 4104, 5120, 8192, 8200, 12296, 16384,
           16392, 32768, 40000, 65536, 131072, 131080, 262144]
SMALL_M = [1, 2, 3, 17, 65, 257, 1000]


def _cases():
    for w in WORKLOADS.values():
        yield w.M, w.N, w.mode
    for n in SMALL_N:
        for m in SMALL_M:
            for mode in (0, 1):
                yield m, n, mode


@pytest.mark.parametrize("backward", [False, True])
def test_all_plans_in_bounds(backward):
    n = 0
    for M, N, mode in _cases():
        p = gb.norm_plan(M, N, mode, backward, SMS, OPTIN)
        launch_check.check_plan(p, M, N, mode, backward, OPTIN)
        if backward:
            launch_check.check_reduce(p["partials"], N, 2 if mode == 1 else 1)
        n += 1
    assert n > 400


@pytest.mark.parametrize("backward", [False, True])
def test_fused_residual_plans_in_bounds(backward):
    n = 0
    for M, N, mode in _cases():
        p = gb.norm_plan(M, N, mode, backward, SMS, OPTIN, residual=True)
        launch_check.check_plan(p, M, N, mode, backward, OPTIN, residual=True)
        n += 1
    assert n > 200


@pytest.mark.parametrize("residual", [False, True])
def test_fp8_plans_in_bounds(residual):
    """Every E4M3-output plan is in bounds, and satisfies the MX block rule
    when N is a multiple of 32 (register-resident and long-row plans)."""
    n = 0
    for M, N, mode in _cases():
        try:
            p = gb.norm_plan(M, N, mode, False, SMS, OPTIN, residual=residual)
        except gb.NormError as e:
            assert residual and e.status == 6
            continue
        p8 = gb.norm_plan(M, N, mode, False, SMS, OPTIN, residual=residual, fp8=True)
        launch_check.check_plan(p8, M, N, mode, False, OPTIN, residual=residual)
        if p8["cluster"] == 1:
            launch_check.check_fp8_plan(p8, M, N, "row")
        if N % 32 == 0:
            launch_check.check_fp8_plan(p8, M, N, "mx")
        n += 1
    assert n > 400


def test_plan_rejects_unsupported():
    with pytest.raises(gb.NormError):
        gb.norm_plan(4, 12, 0, False, SMS, OPTIN)  # N % 8 != 0
    with pytest.raises(gb.NormError):
        gb.norm_plan(0, 16, 0, False, SMS, OPTIN)  # M < 1
    with pytest.raises(gb.NormError):
        gb.norm_plan(4, (1 << 24) + 8, 0, False, SMS, OPTIN)  # N > NORM_MAX_N
    for which in (dict(residual=True), dict(fp8=True)):  # fused variants stop earlier
        with pytest.raises(gb.NormError):
            gb.norm_plan(4, 262152, 0, False, SMS, OPTIN, **which)
    with pytest.raises(gb.NormError):
        gb.norm_plan(4, 262152, 0, True, SMS, OPTIN, residual=True)


def test_regimes_by_row_length():
    """Warp (or sub-warp) per row for short rows, several warps per row for
    medium rows, a thread-block cluster per row for long rows."""
    p = gb.norm_plan(262144, 256, 0, False, SMS, OPTIN)
    assert p["threads_per_row"] == 32 and p["cluster"] == 1
    p = gb.norm_plan(1000, 64, 0, False, SMS, OPTIN)
    assert p["threads_per_row"] == 8
    p = gb.norm_plan(32768, 4096, 1, False, SMS, OPTIN)
    assert p["threads_per_row"] > 32 and p["cluster"] == 1
    p = gb.norm_plan(4096, 131072, 0, False, SMS, OPTIN)
    assert p["cluster"] > 1
    p = gb.norm_plan(4096, 131072, 0, True, SMS, OPTIN)
    assert p["cluster"] > 1


def test_random_shapes_every_plan_kind():
    """Seeded random (M, N) for every pass and variant: each plan the library
    would launch on a GB300 is in bounds (plain, fused residual, E4M3)."""
    import numpy as np

    rng = np.random.default_rng(7)
    n = 0
    for _ in range(150):
        N = int(rng.integers(1, 262144 // 8 + 1)) * 8
        M = int(rng.choice([1, 3, 17, 1000, 4099, 65537]))
        mode = int(rng.integers(0, 2))
        for backward in (False, True):
            for residual in (False, True):
                p = gb.norm_plan(M, N, mode, backward, SMS, OPTIN, residual=residual)
                launch_check.check_plan(p, M, N, mode, backward, OPTIN, residual=residual)
                if backward:
                    launch_check.check_reduce(p["partials"], N, 2 if mode == 1 else 1)
                n += 1
            if not backward:
                p8 = gb.norm_plan(M, N, mode, False, SMS, OPTIN, fp8=True)
                launch_check.check_plan(p8, M, N, mode, False, OPTIN)
                launch_check.check_fp8_plan(p8, M, N, "row")
                if N % 32 == 0:
                    launch_check.check_fp8_plan(p8, M, N, "mx")
    assert n == 600


SPLIT_SHAPES = [(6, 524288), (33, 1048576), (4096, 524288), (1, 262152), (4097, 300008),
                (5, 1 << 24), (2, 262144 + 4096 * 3 + 8)]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("backward", [False, True])
@pytest.mark.parametrize("other", [False, True])
def test_split_plans_in_bounds(mode, backward, other, monkeypatch):
    """Rows wider than one cluster holds take the two-pass path: both passes
    of the forward and of the backward stay in bounds, and the dx pass's
    dgamma / dbeta slots are distinct and read back exactly.  (stream=0
    keeps the RMSNorm backward at 524288 columns, which streams by default,
    on the two-pass path.)"""
    monkeypatch.setenv("GBNORM_PLAN", "stream=0")
    phase = (2 if backward else 0) + (1 if other else 0)
    for M, N in SPLIT_SHAPES:
        p = gb.norm_plan(M, N, mode, backward, SMS, OPTIN, other_pass=other)
        assert p["split_segments"] == -(-N // 4096)
        launch_check.check_split_plan(p, M, N, mode, phase, OPTIN)


@pytest.mark.parametrize("backward", [False, True])
def test_split_forced_small_rows(backward, monkeypatch):
    """The plan override split=1 (with W=1024 segments) puts short rows on
    the two-pass path, which the GPU parity tests use for ragged and
    many-segment cases at sizes the oracle checks in full."""
    monkeypatch.setenv("GBNORM_PLAN", "split=1,W=1024")
    for mode in (0, 1):
        for M, N in ((37, 1024), (130, 3000), (70, 4104), (9, 8200), (1, 8), (3, 1016)):
            for other in (False, True):
                p = gb.norm_plan(M, N, mode, backward, SMS, OPTIN, other_pass=other)
                assert p["split_segments"] == -(-N // 1024)
                launch_check.check_split_plan(p, M, N, mode,
                                              (2 if backward else 0) + (1 if other else 0), OPTIN)


def test_split_random_shapes(monkeypatch):
    import numpy as np

    monkeypatch.setenv("GBNORM_PLAN", "stream=0")

    rng = np.random.default_rng(7)
    for _ in range(60):
        N = int(rng.integers(262152 // 8, (1 << 24) // 8 + 1)) * 8
        M = int(rng.integers(1, 5000))
        mode = int(rng.integers(0, 2))
        for phase in range(4):
            p = gb.norm_plan(M, N, mode, phase >= 2, SMS, OPTIN, other_pass=bool(phase & 1))
            launch_check.check_split_plan(p, M, N, mode, phase, OPTIN)


def test_one_pass_up_to_its_limit():
    for bwd in (False, True):
        assert gb.norm_plan(4096, 262144, 0, bwd, SMS, OPTIN)["split_segments"] == 0
        assert gb.norm_plan(4096, 262152, 0, bwd, SMS, OPTIN)["split_segments"] > 0


STREAM_SHAPES = [(1, 32768), (5, 32768), (4096, 32768), (3, 65536), (4099, 65536),
                 (2, 131072), (4096, 131072), (45, 131072), (7, 262144), (2048, 262144),
                 (3, 524288), (1024, 524288), (11, 98304)]


@pytest.mark.parametrize("mode", [0, 1])
def test_stream_plans_in_bounds(mode, monkeypatch):
    """The streaming backward (forced at every width it takes, and where it
    is the default): pieces, copies, shared and tensor memory, partials."""
    for M, N in STREAM_SHAPES:
        monkeypatch.setenv("GBNORM_PLAN", "stream=1")
        p = gb.norm_plan(M, N, mode, True, SMS, OPTIN)
        launch_check.check_plan(p, M, N, mode, True, OPTIN)
        launch_check.check_reduce(p["partials"], N, 2 if mode == 1 else 1)
        assert p["piece_cols"] == 16384
        monkeypatch.setenv("GBNORM_PLAN", "stream=1,W=8192")  # the fused variant's pieces
        p8 = gb.norm_plan(M, N, mode, True, SMS, OPTIN)
        assert p8["piece_cols"] == 8192
        launch_check.check_plan(p8, M, N, mode, True, OPTIN)
        monkeypatch.setenv("GBNORM_PLAN", "stream=1")
        if N <= 262144:  # the fused residual variant (dh in the dx pass's pieces)
            p = gb.norm_plan(M, N, mode, True, SMS, OPTIN, residual=True)
            assert p["streamed"] == 1
            launch_check.check_plan(p, M, N, mode, True, OPTIN, residual=True)
        monkeypatch.delenv("GBNORM_PLAN")
        p = gb.norm_plan(M, N, mode, True, SMS, OPTIN)
        if p["streamed"]:
            launch_check.check_plan(p, M, N, mode, True, OPTIN)


def test_stream_default_widths():
    """Where the backward streams by default (the widths it measured faster
    at) and where it keeps the resident long-row kernel or the two-pass
    path."""
    want = {(0, 32768): 1, (0, 65536): 1, (0, 131072): 1, (0, 262144): 1, (0, 524288): 1,
            (1, 32768): 1, (1, 65536): 1, (1, 131072): 1, (1, 262144): 1, (1, 524288): 1,
            (0, 98304): 0, (0, 16384): 0, (1, 1048576): 0}
    for (mode, N), s in want.items():
        p = gb.norm_plan(4096, N, mode, True, SMS, OPTIN)
        assert p["streamed"] == s, (mode, N)
        if N > 262144 and not s:
            assert p["split_segments"] > 0
        # the forward streams only RMSNorm rows beyond 262144 columns
        # (slices of 65536, else 32768, in clusters of up to 16); the fused
        # residual backward streams where the plain one does (its entry
        # points stop at 262144 columns)
        pf = gb.norm_plan(4096, N, mode, False, SMS, OPTIN)
        fwd_streams = mode == 0 and N > 262144 and N // 65536 <= 16
        if fwd_streams:
            assert pf["cols_per_cta"] == 65536 and pf["piece_cols"] == 16384
        assert pf["streamed"] == int(fwd_streams), (mode, N, pf)
        if fwd_streams:
            launch_check.check_plan(pf, 4096, N, mode, False, OPTIN)
        if N <= 262144:
            pr = gb.norm_plan(4096, N, mode, True, SMS, OPTIN, residual=True)
            assert pr["streamed"] == s
            if s:
                launch_check.check_plan(pr, 4096, N, mode, True, OPTIN, residual=True)


def test_wait_hint_only_where_tuned(monkeypatch):
    """The register-resident LayerNorm 4096 forward waits with a suspend
    hint; no other default plan does, and the override hint= applies only to
    the plans that have a hinted variant (exact, single CTA, plain, 2 or 4
    chunks per thread)."""
    assert gb.norm_plan(32768, 4096, 1, False, SMS, OPTIN)["wait_hint_ns"] == 2000
    for mode, N in ((1, 2048), (0, 4096), (0, 1024), (1, 8192), (0, 131072)):
        assert gb.norm_plan(32768, N, mode, False, SMS, OPTIN)["wait_hint_ns"] == 0
    assert gb.norm_plan(32768, 4096, 1, True, SMS, OPTIN)["wait_hint_ns"] == 0
    monkeypatch.setenv("GBNORM_PLAN", "hint=1500")
    p = gb.norm_plan(32768, 2048, 0, False, SMS, OPTIN)
    assert p["wait_hint_ns"] == (1500 if p["chunks_per_thread"] in (2, 4) and p["exact"] else 0)
    assert gb.norm_plan(4096, 131072, 0, False, SMS, OPTIN)["wait_hint_ns"] == 0  # long rows


@pytest.mark.parametrize("mode", [0, 1])
def test_stream_forward_plans_in_bounds(mode, monkeypatch):
    """The streaming forward, forced (stream=1) at every width it takes and
    with 8-piece slices (K=16, RMSNorm), and where it is the default."""
    shapes = [(1, 32768), (7, 65536), (300, 131072), (5, 262144), (3, 524288), (4099, 524288)]
    for M, N in shapes:
        monkeypatch.setenv("GBNORM_PLAN", "stream=1")
        p = gb.norm_plan(M, N, mode, False, SMS, OPTIN)
        assert p["streamed"] == 1 and p["cols_per_cta"] == 32768
        assert p["piece_cols"] == (16384 if mode == 0 else 8192)
        launch_check.check_plan(p, M, N, mode, False, OPTIN)
        if mode == 0 and N >= 65536:
            monkeypatch.setenv("GBNORM_PLAN", "stream=1,K=16")
            p = gb.norm_plan(M, N, mode, False, SMS, OPTIN)
            assert p["streamed"] == 1 and p["cols_per_cta"] == 65536
            launch_check.check_plan(p, M, N, mode, False, OPTIN)
    monkeypatch.delenv("GBNORM_PLAN")
    for M, N in ((2048, 524288), (1024, 1048576)):
        p = gb.norm_plan(M, N, mode, False, SMS, OPTIN)
        if p["streamed"]:
            launch_check.check_plan(p, M, N, mode, False, OPTIN)
