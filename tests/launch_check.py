"""Host-side check of the kernels' index arithmetic for a launch plan.

Restates, for every CTA of a launch, the addresses the forward / backward /
reduce kernels form (tiles, rows, 16-byte chunks, bulk-copy sizes, shared
memory slots, partial rows) and asserts that each stays inside its buffer
and meets the alignment rules of the copies.  Run on the CPU before a plan
reaches the GPU; uses only the plan the library reports (norm_plan).
"""
from __future__ import annotations

MAX_THREADS = 512
XCH_BUFFERS = 4
TX_LIMIT = 1 << 20


def _align16(v):
    return (v + 15) & ~15


def smem_layout(RT, NS, S, G, tpr, ntensors, stats, C, par_bytes=0):
    """Same region order as the kernels' shared-memory layout."""
    tensor = RT * NS * 2
    stage = tensor * ntensors
    off = stage * S
    L = {"tensor": tensor, "stage": stage, "params": off}
    off = _align16(off + par_bytes)
    L["stats"] = off
    if stats:
        off = _align16(off + S * RT * 2 * 4)
    L["red"] = off
    if tpr > 32:
        off = _align16(off + 2 * G * (tpr // 32) * 4 * 4)
    L["xch"] = off
    if C > 1:
        off = _align16(off + XCH_BUFFERS * RT * C * 4 * 4 + 8 * XCH_BUFFERS)
    L["bar"] = off
    off = _align16(off + S * 8)
    L["flag"] = off
    off = _align16(off + 4 + 4 * S)
    L["total"] = off
    return L


STREAM_THREADS = 512
STREAM_SLICE = 32768  # backward slice; the forward's is this or twice it


def stream_layout(S, C, ntensors, piece):
    """Shared memory of the streaming kernels, in their order: stages of
    `piece` columns of x (forward), x and dy (backward) or x, dy and dh
    (fused residual backward)."""
    tensor = piece * 2
    stage = ntensors * tensor
    off = stage * S
    L = {"tensor": tensor, "stage": stage, "red": off}
    # per-warp row partials [buffer][warp][2 or 4] floats, then one counter per buffer
    per_warp = 4 if ntensors == 1 else 2
    L["per_warp"] = per_warp
    off = _align16(off + XCH_BUFFERS * (STREAM_THREADS // 32) * per_warp * 4 + 4 * XCH_BUFFERS)
    L["xch"] = off
    off = _align16(off + XCH_BUFFERS * C * 4 * 4 + 8 * XCH_BUFFERS)  # also for C = 1
    L["bar"] = off
    off = _align16(off + S * 8)
    L["flag"] = off
    off = _align16(off + 4 + 4 * S + 4)  # abort flag, S warp counters, TMEM slot
    L["total"] = off
    return L


def stream_piece_at(q, np_, nr):
    """(pass, row index j, piece p) of piece q of a cluster's sequence: pass 1
    of row 0, then pass 1 of row j and pass 2 of row j - 1, then pass 2 of
    the last row."""
    if q < np_:
        return 0, 0, q
    q2 = q - np_
    b, w = divmod(q2, 2 * np_)
    if b < nr - 1:
        return (0, b + 1, w) if w < np_ else (1, b, w - np_)
    return 1, nr - 1, w


def check_stream_plan(p, M, N, mode, smem_optin=232448, residual=False, backward=True):
    """The streaming kernels' accesses for plan `p`: every (row, pass,
    piece) issued once per cluster in pipeline order, each bulk copy inside
    its tensor and 16-byte aligned, the shared-memory regions in bounds, the
    backward's tensor-memory columns within 512 and its partial rows inside
    the workspace."""
    C, NS, S, grid, P = p["cluster"], p["cols_per_cta"], p["stages"], p["grid"], p["partials"]
    assert p["streamed"] == 1 and p["threads"] == STREAM_THREADS and p["exact"] == 1
    piece = p["piece_cols"]
    kp = piece // (STREAM_THREADS * 8)  # chunks per thread per piece
    assert kp in (2, 4) and piece == STREAM_THREADS * kp * 8
    np_ = NS // piece
    assert NS % piece == 0 and N == C * NS and 1 <= C <= 16
    assert NS == STREAM_SLICE or (not backward and NS == 2 * STREAM_SLICE)
    assert p["chunks_per_thread"] * STREAM_THREADS * 8 == NS
    assert p["tiles"] == M and grid % C == 0 and grid // C == P and 1 <= P <= M
    nt = (3 if residual else 2) if backward else 1
    L = stream_layout(S, C, nt, piece)
    assert p["smem_bytes"] == L["total"] <= smem_optin - 1024 and S >= 2
    # pass 1 pieces land x (and dy), pass 2 pieces also dh: inside the stage
    assert nt * L["tensor"] == L["stage"]
    assert L["stage"] < TX_LIMIT and L["bar"] % 8 == 0 and L["flag"] % 4 == 0
    # per-warp partials (buffer < 4, warp < 16, 2 or 4 floats), the 4
    # counters, then the exchange slots [buffer][rank] and their 4 mbarriers
    warps, pw = STREAM_THREADS // 32, L["per_warp"]
    hi = ((XCH_BUFFERS - 1) * warps + (warps - 1)) * pw + pw
    assert L["red"] + hi * 4 <= L["red"] + XCH_BUFFERS * warps * pw * 4
    assert L["red"] + XCH_BUFFERS * warps * pw * 4 + 4 * XCH_BUFFERS <= L["xch"]
    bars = L["xch"] + XCH_BUFFERS * C * 16
    assert bars % 8 == 0 and bars + 8 * XCH_BUFFERS <= L["bar"]
    # thread t, chunk k of a piece: smem byte t*16 + k*threads*16 (+16) in the
    # tensor; global column piece*W + (k*threads + t)*8 (+8) in the slice
    assert (STREAM_THREADS - 1) * 16 + (kp - 1) * STREAM_THREADS * 16 + 16 <= L["tensor"]
    assert (np_ - 1) * piece + ((kp - 1) * STREAM_THREADS + STREAM_THREADS - 1) * 8 + 8 <= NS
    nacc = 2 if mode == 1 else 1
    groups = STREAM_THREADS // 32 // 4
    if backward:
        assert groups * np_ * kp * 8 * nacc <= 512, "accumulators exceed TMEM"
    seen = 0
    for cid in range(P):
        nr = -(-(M - cid) // P)
        order = []
        for q in range(2 * np_ * nr):
            ps, j, pc = stream_piece_at(q, np_, nr)
            assert 0 <= j < nr and 0 <= pc < np_
            row = cid + j * P
            assert row < M
            for crank in range(C):
                off = row * N + crank * NS + pc * piece
                assert (off * 2) % 16 == 0 and off + piece <= M * N
            order.append((ps, j, pc))
        assert len(set(order)) == len(order) == 2 * np_ * nr
        # consumed in this order by the kernel's loop: pass 1 of row j, then
        # pass 2 of row j - 1, each piece in increasing order
        want = []
        for j in range(nr + 1):
            if j < nr:
                want += [(0, j, pc) for pc in range(np_)]
            if j >= 1:
                want += [(1, j - 1, pc) for pc in range(np_)]
        assert order == want
        seen += nr
        if backward:
            last = ((nacc - 1) * P + cid) * N + (C - 1) * NS + NS
            assert last <= nacc * P * N, "partial row write out of the workspace"
    assert seen == M
    return True


def check_plan(p, M, N, mode, backward, smem_optin=232448, residual=False):
    """Raise AssertionError if any access of the launch described by `p`
    (a norm_plan dict) would leave its buffer or break an alignment rule."""
    if p.get("streamed"):
        assert not (residual and not backward)
        return check_stream_plan(p, M, N, mode, smem_optin, residual, backward)
    C, NS, tpr, K = p["cluster"], p["cols_per_cta"], p["threads_per_row"], p["chunks_per_thread"]
    G, rpg, RT, S = p["groups"], p["rows_per_group"], p["rows_per_tile"], p["stages"]
    threads, smem, ntiles, grid, P = p["threads"], p["smem_bytes"], p["tiles"], p["grid"], p["partials"]
    nc = N // 8
    nsc = NS // 8
    assert N % 8 == 0 and NS % 8 == 0
    assert threads == G * tpr <= MAX_THREADS and threads % 32 == 0
    assert tpr >= 32 and tpr % 32 == 0 or (tpr < 32 and 32 % tpr == 0)
    if tpr > 32:
        assert 1 + (G - 1) <= 15, "named barrier id out of range"
    assert RT == G * rpg and S >= 2
    assert C >= 1 and grid % C == 0 and grid // C == P and P >= 1
    assert C == 1 or rpg == 1
    assert not residual or C == 1 or p["long_rows"]  # no register-path cluster variants
    assert ntiles == -(-M // RT) and P <= ntiles
    assert K * tpr >= nsc, "a chunk has no owner"
    if p["exact"]:
        assert tpr % 32 == 0 and K * tpr == nsc and nc % C == 0, "EXACT plan is not exact"
    # the long-row fused residual backward keeps dh out of the stage
    ntensors = (2 if backward else 1) + (1 if residual and not (backward and p["long_rows"]) else 0)
    par = p["param_smem_bytes"]
    nvec = 2 if mode == 1 else 1
    assert par == 0 or (not backward and p["exact"] and K in (5, 6, 8) and C == 1
                        and par in (nvec * NS * 2, nvec * NS * 4))
    L = smem_layout(RT, NS, S, G, tpr, ntensors, backward, C, par)
    # staged parameters: fp32 float4 [param][half][chunk] or bf16 uint4
    # [param][chunk]; the highest 16-byte word read is inside the region
    if par:
        words = nvec * nsc * (2 if par == nvec * NS * 4 else 1)
        assert L["params"] + words * 16 <= L["stats"]
    assert smem == L["total"] <= smem_optin, "shared memory over the opt-in limit"
    assert L["stage"] < TX_LIMIT
    assert L["bar"] % 8 == 0 and L["stats"] % 16 == 0 and L["red"] % 16 == 0
    if backward:
        nparts = 2 if mode == 1 else 1
        # column partial fold reuses the ring: nparts * G * NS floats
        assert nparts * G * NS * 4 <= S * L["stage"]
    # per CTA slice
    for crank in range(C):
        col0 = crank * NS
        nsc_me = min(nsc, nc - crank * nsc)
        assert nsc_me >= 1, "a CTA of the cluster owns no column"
        assert col0 + nsc_me * 8 <= N
        assert (col0 * 2) % 16 == 0
        # chunk ownership: thread t, k < K -> c = t + k*tpr; valid iff c < nsc_me
        owned = sorted(t + k * tpr for t in range(tpr) for k in range(K) if t + k * tpr < nsc_me)
        assert owned == list(range(nsc_me)), "chunks not owned exactly once"
        # smem reads of a row slot: r * NS*2 + c*16 + 16 <= tensor bytes
        assert (RT - 1) * NS * 2 + (nsc_me - 1) * 16 + 16 <= L["tensor"]
        # bulk copy sizes / alignment
        if C == 1:
            max_bytes = RT * N * 2
            assert max_bytes <= L["tensor"] and max_bytes % 16 == 0
            # every tensor of the stage lies inside the stage
            assert ntensors * L["tensor"] == L["stage"]
        else:
            assert nsc_me * 16 <= NS * 2 and (NS * 2) % 16 == 0
        if backward:
            nparts = 2 if mode == 1 else 1
            last = ((nparts - 1) * P + (P - 1)) * N + col0 + nsc_me * 8
            assert last <= nparts * P * N, "partial row write out of the workspace"
    # tiles: every tile visited exactly once across clusters; rows in range
    seen = 0
    for cid in range(P):
        it = 0
        while True:
            tile = cid + it * P
            if tile >= ntiles:
                break
            row0 = tile * RT
            nrows = min(RT, M - row0)
            assert 1 <= nrows <= RT
            assert (row0 + nrows) * N <= M * N
            assert ((row0 * N) * 2) % 16 == 0
            if backward:
                assert (S - 1) * RT * 2 + 2 * (nrows - 1) + 1 < S * RT * 2
            seen += 1
            it += 1
    assert seen == ntiles
    # group scratch: slot (rpar*G + g)*W + w, 4 floats, rpar in {0, 1}
    if tpr > 32:
        W = tpr // 32
        hi = ((1 * G + (G - 1)) * W + (W - 1)) * 4 + 4
        assert L["red"] + hi * 4 <= L["xch"]
    if C > 1:
        # slot [buf][r][q] float4 for buf < 4, r < RT, q < C; then 4 mbarriers
        hi = (((XCH_BUFFERS - 1) * RT + (RT - 1)) * C + (C - 1)) * 4 + 4
        bars = L["xch"] + XCH_BUFFERS * RT * C * 16
        assert L["xch"] + hi * 4 <= bars and bars % 8 == 0
        assert bars + 8 * XCH_BUFFERS <= L["bar"]
    return True


def check_fp8_plan(p, M, N, scaling):
    """The E4M3-output forward on plan `p` (a norm_plan dict of the plain or
    fused-residual forward): codes and scales stay in their buffers and, for
    MX scaling, every 32-column block is 4 consecutive chunks held by 4
    consecutive lanes of one row group, owned (or not) together."""
    C, tpr, K = p["cluster"], p["threads_per_row"], p["chunks_per_thread"]
    nc = N // 8
    if C > 1 or p["long_rows"]:
        # long-row kernels: slices start on a 32-column block, tpr % 32 == 0
        nsc = p["cols_per_cta"] // 8
        assert nsc % 4 == 0 and tpr % 32 == 0 and (C - 1) * nsc < nc
        for crank in range(C):
            nsc_me = min(nsc, nc - crank * nsc)
            for c in range(0, nsc_me, 4):
                blk = (crank * nsc + c) // 4
                assert blk < N // 32 or scaling != "mx"
        return True
    for t in range(tpr):
        for k in range(K):
            c = t + k * tpr
            if c < nc:
                assert c * 8 + 8 <= N                   # 8 code bytes per chunk
    assert (M - 1) * N + N <= M * N
    if scaling == "mx":
        assert N % 32 == 0 and tpr % 4 == 0
        nb = N // 32
        for t0 in range(0, tpr, 4):
            for k in range(K):
                cs = [t0 + i + k * tpr for i in range(4)]
                own = [c < nc for c in cs]
                assert all(own) or not any(own), "a block is split between owners"
                if own[0]:
                    assert cs[0] % 4 == 0 and cs == list(range(cs[0], cs[0] + 4))
                    assert cs[0] // 4 < nb                # E8M0 byte inside the row
        # a quad never straddles a group: groups start at multiples of tpr
        assert (p["groups"] * tpr) % 4 == 0
    return True


REDUCE_WARPS = 32
REDUCE_BATCH = 8


def check_reduce(P, N, nparts):
    """Reduce kernel: grid (ceil(N/128), nparts), 32 warps, lane owns 4
    columns, warp w sums p in [P*w/32, P*(w+1)/32) in batches of 8 loads,
    each guarded by p < the range end."""
    assert N % 4 == 0
    gx = -(-N // 128)
    for bx in (0, gx - 1):
        for lane in range(32):
            col = (bx * 32 + lane) * 4
            if col < N:
                assert col + 4 <= N
                assert ((nparts - 1) * P + (P - 1)) * N + col + 4 <= nparts * P * N
    ranges = [(P * w // REDUCE_WARPS, P * (w + 1) // REDUCE_WARPS) for w in range(REDUCE_WARPS)]
    covered = []
    for a, b in ranges:
        for p in range(a, b, REDUCE_BATCH):
            covered += [p + u for u in range(REDUCE_BATCH) if p + u < b]
    assert covered == list(range(P))
    return True


SPLIT_FWD_STATS, SPLIT_FWD_OUT, SPLIT_BWD_DOTS, SPLIT_BWD_DX = range(4)


def split_layout(RT, NS, S, G, tpr, ntensors):
    """Same region order as the two-pass kernels' shared-memory layout."""
    tensor = RT * NS * 2
    stage = tensor * ntensors
    off = stage * S
    L = {"tensor": tensor, "stage": stage, "stats": off}
    off = _align16(off + S * RT * 4 * 4)
    L["red"] = off
    if tpr > 32:
        off = _align16(off + 2 * G * (tpr // 32) * 4 * 4)
    L["bar"] = off
    off = _align16(off + S * 8)
    L["flag"] = off
    off = _align16(off + 4 + 4 * S)
    L["total"] = off
    return L


def unit_ranges(U, grid):
    """[begin, end) of the units of each CTA: [U b / grid, U (b+1) / grid)."""
    return [(U * b // grid, U * (b + 1) // grid) for b in range(grid)]


def check_split_plan(p, M, N, mode, phase, smem_optin=232448):
    """The two-pass kernels on plan `p` (a norm_plan dict with
    split_segments > 0): every unit visited once, every bulk copy, shared
    memory slot, scratch and workspace index in bounds; for the dx pass,
    each (CTA, segment) slot is distinct and the reduction reads exactly
    the slots that the CTAs touching each segment wrote."""
    NS, tpr, K = p["cols_per_cta"], p["threads_per_row"], p["chunks_per_thread"]
    G, rpg, RT, S = p["groups"], p["rows_per_group"], p["rows_per_tile"], p["stages"]
    threads, smem, T, grid = p["threads"], p["smem_bytes"], p["tiles"], p["grid"]
    nseg = p["split_segments"]
    nc, nsc = N // 8, NS // 8
    assert p["cluster"] == 1 and nseg == -(-N // NS) and NS % 1024 == 0
    assert tpr * K * 8 == NS and tpr % 32 == 0 and threads == G * tpr <= MAX_THREADS
    assert G <= 16 and (tpr == 32 or G <= 15)
    assert RT == G * rpg and S >= 2 and T == -(-M // RT)
    ntensors = 2 if phase >= SPLIT_BWD_DOTS else 1
    L = split_layout(RT, NS, S, G, tpr, ntensors)
    assert smem == L["total"] <= smem_optin and L["stage"] < TX_LIMIT
    if tpr > 32:
        W = tpr // 32
        hi = ((1 * G + (G - 1)) * W + (W - 1)) * 4 + 4
        assert L["red"] + hi * 4 <= L["bar"]
    # stats slots [S][RT][4]
    assert L["stats"] + ((S - 1) * RT + RT - 1) * 16 + 16 <= L["red"]
    U = T * nseg
    assert 1 <= grid <= U
    ranges = unit_ranges(U, grid)
    assert ranges[0][0] == 0 and ranges[-1][1] == U
    assert all(a < b for a, b in ranges), "a CTA with no unit"
    assert all(ranges[i][1] == ranges[i + 1][0] for i in range(grid - 1))
    # per segment: chunks and copies
    for seg in {0, nseg - 1, nseg // 2}:
        nsc_me = min(nsc, nc - seg * nsc)
        assert 1 <= nsc_me <= nsc
        col0 = seg * NS
        assert col0 + nsc_me * 8 <= N and (col0 * 2) % 16 == 0
        owned = sorted(t + k * tpr for t in range(tpr) for k in range(K) if t + k * tpr < nsc_me)
        assert owned == list(range(nsc_me))
        assert (RT - 1) * NS * 2 + nsc_me * 16 <= L["tensor"]
        if phase == SPLIT_FWD_STATS:
            # partial of (row, seg) in y's row: float (RMS) or float2 (LN)
            assert (seg + 1) * (8 if mode == 1 else 4) <= 2 * N
    for rt in {0, T - 1}:
        row0 = rt * RT
        nrows = min(RT, M - row0)
        assert 1 <= nrows and (row0 + nrows - 1) * N + N <= M * N
    if phase == SPLIT_BWD_DOTS:
        assert (M - 1) * nseg + nseg - 1 < M * nseg      # rowp float2 index
    if phase == SPLIT_BWD_DX:
        nslots = grid + nseg
        slots = set()
        touch = [[] for _ in range(nseg)]
        for b, (u0, u1) in enumerate(ranges):
            for seg in range(u0 // T, (u1 - 1) // T + 1):
                assert 0 <= b + seg < nslots
                assert (b, seg) not in slots
                slots.add((b, seg))
                touch[seg].append(b)
        assert len({b + s for b, s in slots}) == len(slots), "two pairs share a slot"
        for seg in range(nseg):
            lo = ((seg * T + 1) * grid - 1) // U
            hi = ((seg + 1) * T * grid - 1) // U
            assert touch[seg] == list(range(lo, hi + 1)), "reduce reads other slots"
    return True
