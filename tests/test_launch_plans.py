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
        gb.norm_plan(4, 262152, 0, False, SMS, OPTIN)  # N > NORM_MAX_N


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
