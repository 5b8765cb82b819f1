"""A CPU model of the split plan that stage 1 and stage 2 derive on the device.

The device code (Sched and segment_pieces in gda_device.cuh) decides, from
kv_indptr alone, which CTA computes which (sequence, KV head, position range)
piece and where the piece's partial is stored.  This model restates the same
rules and checks their invariants over many random ragged batches: every KV
position is covered exactly once, piece ids are unique and within the workspace
capacity, and the list of pieces stage 2 merges for a segment is exactly the set
stage 1 wrote.  (The GPU parity tests check the device code itself.)"""
import random

AUTO_MAX_CTAS = 1024


STREAM_MIN_PER_CTA = 3072   # a BF16 cache; twice as many positions of an e4m3 cache


def uniform_splits(indptr, Hkv, grid, min_chunk, kv8=False):
    """The automatic split rule (Sched::auto_uniform_splits): S uniform splits, or 0
    for the stream schedule.  kv8: the e4m3 variant (the per-CTA bound for the stream
    doubled, S_opt from 16 S^2 > lmax instead of 4 S^2)."""
    B = len(indptr) - 1
    units1 = B * Hkv
    if units1 > grid:
        return 0
    if units1 == 0:
        return 1
    lmax = max([indptr[b + 1] - indptr[b] for b in range(B)] + [0])
    n = indptr[B]
    if Hkv * n >= STREAM_MIN_PER_CTA * (2 if kv8 else 1) * grid or 4 * lmax * B > 5 * n:
        return 0
    k = 16 if kv8 else 4
    s_opt = 1
    while k * s_opt * s_opt <= lmax:
        s_opt *= 2
    s = min(s_opt, max(1, -(-lmax // min_chunk)))
    s_wave = grid // units1
    if s >= s_wave:
        p2 = 1
        while 2 * p2 <= s_wave:
            p2 *= 2
        s = p2 if 5 * p2 * units1 >= 4 * grid else s_wave
        if 5 * s * units1 < 4 * grid:
            return 0
    return s


PIECE_COST = 300        # a BF16 cache
PIECE_COST_E4M3 = 600   # an e4m3 cache streams twice the positions per microsecond


def piece_cost(B, Hkv, grid, cost=PIECE_COST):
    """The cost of a segment start (the host's Stage1Params::piece_cost): `cost` with
    more segments than CTAs, else 0."""
    return cost if B * Hkv > grid else 0


def stream_cost(total, B, Hkv, X):
    """The stream's cost: one per position, X more per segment start after the first
    (Sched::stream_cost)."""
    return total + X * max(B * Hkv - 1, 0)


def position_at_cost(indptr, Hkv, X, t):
    """The first stream position whose cost is at least t (the stream's end past
    it): position p of segment sigma costs p + X * sigma.  A plain scan over the
    positions, not the device's search."""
    B = len(indptr) - 1
    for b in range(B):
        L = indptr[b + 1] - indptr[b]
        for k in range(Hkv):
            sigma = b * Hkv + k
            start = Hkv * indptr[b] + k * L
            if L > 0 and start + L - 1 + X * sigma >= t:
                return start + max(0, t - (start + X * sigma))
    return Hkv * indptr[B]


def stage1_pieces(indptr, Hkv, grid, min_chunk, S, cost=PIECE_COST):
    B = len(indptr) - 1
    if S <= 0:
        S = uniform_splits(indptr, Hkv, grid, min_chunk)
    out = []
    if S > 0:
        for c in range(grid):
            u = c
            while u < B * Hkv * S:
                sig, s = divmod(u, S)
                b = sig // Hkv
                L = indptr[b + 1] - indptr[b]
                cc = -(-L // S)
                j0, j1 = s * cc, min(L, s * cc + cc)
                if j0 < j1:
                    out.append((b, sig % Hkv, j0, j1, u))
                u += grid
        return out, S, None
    total = Hkv * indptr[B]
    X = piece_cost(B, Hkv, grid, cost)
    T = max(-(-stream_cost(total, B, Hkv, X) // grid), min_chunk)
    for c in range(grid):
        pos, end = position_at_cost(indptr, Hkv, X, c * T), position_at_cost(indptr, Hkv, X, c * T + T)
        if pos >= end:
            continue
        b = 0
        while pos < end:
            while Hkv * indptr[b + 1] <= pos:
                b += 1
            base = Hkv * indptr[b]
            L = indptr[b + 1] - indptr[b]
            kvh, j0 = divmod(pos - base, L)
            stop = min(end, base + (kvh + 1) * L)
            out.append((b, kvh, j0, j0 + stop - pos, c + b * Hkv + kvh))
            pos = stop
    return out, 0, T


def stage2_ids(indptr, Hkv, b, kvh, S, T, grid, cost=PIECE_COST):
    L = indptr[b + 1] - indptr[b]
    if L <= 0:
        return []
    sig = b * Hkv + kvh
    if S > 0:
        c = -(-L // S)
        return [sig * S + k for k in range(-(-L // c))]
    X = piece_cost(len(indptr) - 1, Hkv, grid, cost)
    start = Hkv * indptr[b] + kvh * L + X * sig  # the segment's first position's cost
    return [c + sig for c in range(start // T, (start + L - 1) // T + 1)]


def test_plan_invariants_random_batches():
    rng = random.Random(7)
    for _ in range(600):
        B = rng.randint(1, 120)
        lens = [rng.choice([0, 1, 2, 15, 16, 17, 64, 65, 300, 512, 700, 4096]) for _ in range(B)]
        indptr = [0]
        for L in lens:
            indptr.append(indptr[-1] + L)
        Hkv = rng.choice([1, 2, 4])
        grid = rng.choice([1, 7, 152, 1024])
        min_chunk = rng.choice([1, 16, 64])
        S_user = rng.choice([0, 0, 0, 1, 3, 8])
        cost = rng.choice([PIECE_COST, PIECE_COST_E4M3])
        pieces, S, T = stage1_pieces(indptr, Hkv, grid, min_chunk, S_user, cost)
        ids = [p[4] for p in pieces]
        assert len(ids) == len(set(ids))
        cap = B * Hkv * S_user if S_user > 0 else AUTO_MAX_CTAS + B * Hkv
        assert all(0 <= i < cap for i in ids)
        cover = {}
        for b, kvh, j0, j1, _ in pieces:
            for j in range(j0, j1):
                cover[(b, kvh, j)] = cover.get((b, kvh, j), 0) + 1
        assert all(cover.get((b, kvh, j)) == 1 for b in range(B) for kvh in range(Hkv) for j in range(lens[b]))
        assert sum(cover.values()) == Hkv * sum(lens)
        for b in range(B):
            for kvh in range(Hkv):
                mine = sorted(p[4] for p in pieces if p[0] == b and p[1] == kvh)
                assert stage2_ids(indptr, Hkv, b, kvh, S, T, grid, cost) == mine


def test_split_rule_on_measured_buckets():
    # the choices the GB300 sweeps found best (Hkv = 2, 152 CTAs, equal lengths)
    eq = lambda B, L: [L * i for i in range(B + 1)]
    want = {(1, 512): 8, (1, 2048): 32, (1, 8192): 64, (1, 32768): 64, (2, 2048): 32, (2, 32768): 32, (4, 2048): 16,
            (4, 32768): 16, (8, 2048): 8, (16, 512): 4, (24, 8192): 3, (32, 2048): 2, (64, 512): 1,
            (64, 2048): 1, (64, 3072): 1,
            # stream schedule: >= 3072 positions per CTA, < 80 % of the CTAs busy, more than a wave
            (64, 4096): 0, (16, 32768): 0, (8, 131072): 0, (48, 4096): 0, (128, 512): 0}
    for (B, L), S in want.items():
        assert uniform_splits(eq(B, L), 2, 152, 64) == S, (B, L)
    # an e4m3 cache: the per-CTA bound doubled (one-wave uniform splits won at 3450 ..
    # 5174 positions per CTA, tied at 6899 and lost from ~13800), a wave that leaves
    # < 80 % of the CTAs busy still takes the stream; at small batches half the BF16
    # count (the e4m3 sweep: B1 L2048 best at 16, B1 L8192 at 32, B2 L2048 at 16)
    want8 = {(64, 4096): 1, (64, 6144): 1, (64, 8192): 0, (32, 8192): 2, (32, 32768): 0, (16, 16384): 4,
             (8, 131072): 0, (4, 65536): 16, (24, 16384): 3, (48, 4096): 0, (40, 8192): 0, (128, 512): 0,
             (1, 2048): 16, (1, 8192): 32, (1, 32768): 64, (2, 2048): 16, (2, 8192): 32, (4, 2048): 16,
             (8, 2048): 8}
    for (B, L), S in want8.items():
        assert uniform_splits(eq(B, L), 2, 152, 64, kv8=True) == S, (B, L)
    # far from equal lengths: the stream schedule balances them
    assert uniform_splits([0, 8000, 8100, 8200, 30000], 2, 152, 64) == 0
    assert uniform_splits([0], 2, 152, 64) == 1 and uniform_splits([0, 0, 0], 2, 152, 64) == 1


def test_small_batches_get_one_piece_per_cta():
    # B=4 ragged 512/495/478/461 at Hkv=2: uniform 8 splits, 64 units on 152 CTAs
    indptr = [0, 512, 1007, 1485, 1946]
    assert uniform_splits(indptr, 2, 152, 64) == 8
    # B=64 x 4096 does not fit: the stream schedule balances it instead
    indptr = [4096 * i for i in range(65)]
    assert uniform_splits(indptr, 2, 152, 64) == 0
    pieces, S, T = stage1_pieces(indptr, 2, 152, 64, 0)
    # fewer segments (128) than CTAs: equal positions per CTA
    per_cta = {}
    for b, kvh, j0, j1, pid in pieces:
        c = pid - (b * 2 + kvh)
        per_cta[c] = per_cta.get(c, 0) + (j1 - j0)
    assert max(per_cta.values()) - min(per_cta.values()) <= T
    assert max(per_cta.values()) == T
    # more segments than CTAs (a ragged batch of 224): equal cost ranges per CTA; its
    # positions plus the piece cost per piece after its first leave out the parts of a
    # segment-start gap at either end of its range, at most twice the piece cost
    rng = random.Random(3)
    indptr = [0]
    for _ in range(224):
        indptr.append(indptr[-1] + rng.randint(1, 6142))
    for X in (PIECE_COST, PIECE_COST_E4M3):
        pieces, S, T = stage1_pieces(indptr, 2, 152, 64, 0, X)
        cost = {}
        for b, kvh, j0, j1, pid in pieces:
            c = pid - (b * 2 + kvh)
            cost[c] = cost.get(c, -X) + (j1 - j0) + X
        assert max(cost.values()) - min(cost.values()) <= 2 * X
        assert max(cost.values()) == T and len(cost) == 152


def team_size(npass):
    """Groups of 8 per piece on the MMA kernel: 1 for one pass, pairs for 2 or 4
    passes, threes otherwise (3 passes: one read instead of two; 5 .. 6: two instead of
    three)."""
    return 1 if npass <= 1 else 2 if npass in (2, 4) else 3


def test_team_size_reads_every_row_fewest_times():
    # reads of every K/V row per KV head = ceil(npass / team); teams of three never
    # read more often than pairs, and pairs are kept where they read as rarely
    for npass in range(1, 17):
        t = team_size(npass)
        reads = -(-npass // t)
        assert reads == min(-(-npass // 2), -(-npass // 3)) or npass == 1
        if npass in (2, 4):
            assert t == 2 and reads == -(-npass // 3)
    assert [-(-n // team_size(n)) for n in (2, 3, 4, 5, 6, 7)] == [1, 1, 2, 2, 2, 3]


def test_team_partials_fit_the_workspace():
    # G > 8 on the MMA kernel: the npass groups of 8 query heads of a KV head go in
    # nteam = ceil(npass / team) teams; pieces are scheduled per (sequence, KV head,
    # team) and the partial of (piece, group of the team) sits at piece * team + group.
    # The workspace holds max(team x the pieces of that schedule, the pieces of the
    # per-virtual-head schedule of the other kernels); stage 2 finds exactly stage 1's
    # slots for every query-head group.
    rng = random.Random(11)
    for _ in range(300):
        B = rng.randint(1, 80)
        lens = [rng.choice([0, 1, 16, 17, 65, 700, 4096]) for _ in range(B)]
        indptr = [0]
        for L in lens:
            indptr.append(indptr[-1] + L)
        Hkv = rng.choice([1, 2, 4])
        npass = rng.choice([2, 2, 3, 3, 4, 5, 7])
        team = team_size(npass)
        nteam = -(-npass // team)
        grid = rng.choice([7, 152, 1024])
        S_user = rng.choice([0, 0, 2, 8])
        heads = Hkv * nteam
        pieces, S, T = stage1_pieces(indptr, heads, grid, 64, S_user)
        num_pieces = lambda vh: B * vh * S_user if S_user > 0 else AUTO_MAX_CTAS + B * vh
        cap = max(team * num_pieces(heads), num_pieces(Hkv * npass))
        slots = [p[4] * team + g for p in pieces for g in range(team)]
        assert len(slots) == len(set(slots)) and all(0 <= s < cap for s in slots)
        for b in range(B):
            for kvh in range(Hkv):
                for gp in range(npass):  # query-head group gp of KV head kvh
                    sched_h, g = kvh * nteam + gp // team, gp % team
                    want = sorted(p[4] * team + g for p in pieces if p[0] == b and p[1] == sched_h)
                    assert [i * team + g for i in stage2_ids(indptr, heads, b, sched_h, S, T, grid)] == want


def test_team_kernel_tile_arithmetic():
    # The team stage-1 loop (NG groups per piece on NW warps: pairs on 8, threes on 6):
    # warp w loads tiles w + NW k of a piece (16 positions each); it is member w // WPG
    # of team w % WPG (WPG = NW / NG) and owns group w // WPG.  All members run the
    # step count of the team's first warp (w % WPG), and at step k warp w takes its own
    # tile and each partner's (when k < that warp's tile count) for its own group.
    # Every tile is loaded once, every group sees every tile once, and the shared step
    # count covers all members' tiles.
    for NW, NG in ((8, 2), (6, 3)):
        WPG = NW // NG

        def nmine(w, length):
            ntiles = (length + 15) // 16
            return (ntiles - w + NW - 1) // NW if ntiles > w else 0

        def tile_n(w, k, length):
            return min(16, length - 16 * (w + NW * k)) if k < nmine(w, length) else 0

        for length in list(range(0, 700)) + [1023, 1024, 1025, 4096, 3449, 5000]:
            ntiles = (length + 15) // 16
            loaded = [0] * ntiles
            seen = {g: [0] * ntiles for g in range(NG)}
            positions = {g: 0 for g in range(NG)}
            for w in range(NW):
                team, grp = w % WPG, w // WPG
                members = [team + WPG * j for j in range(NG)]
                # tile order of a step: own first, then the partners in member order
                order = [w] + [m for m in members if m != w]
                steps = nmine(team, length)
                assert all(steps >= nmine(m, length) for m in members)
                for k in range(nmine(w, length)):
                    loaded[w + NW * k] += 1
                for k in range(steps):
                    for owner in order:
                        n = tile_n(owner, k, length)
                        if n > 0:
                            seen[grp][owner + NW * k] += 1
                            positions[grp] += n
            assert loaded == [1] * ntiles
            assert all(seen[g] == [1] * ntiles for g in range(NG))
            assert all(positions[g] == length for g in range(NG))


def test_cluster_kernel_partition_and_merge_slots():
    # The one-kernel path: a cluster of C CTAs per (sequence, KV head).  CTA r takes
    # positions [min(L, r c), min(L, r c + c)), c = ceil(L / C), and stores its state
    # of query head h (h < G <= 8) in slot (h // C) * C + r of CTA h % C; CTA r'
    # finalises heads r' + C k, reading slots k C + x for x < C.  Every state lands in
    # a distinct slot of one of 8, and each finaliser reads exactly its head's C states.
    for C in (1, 2, 4, 8):
        for L in list(range(0, 300)) + [1023, 1024, 1025]:
            c = (L + C - 1) // C
            got = []
            for r in range(C):
                lo = min(L, r * c)
                got.extend(range(lo, min(L, lo + c)))
            assert got == list(range(L))
        for G in range(1, 9):
            slots = {}
            for r in range(C):
                for h in range(G):
                    key = (h % C, (h // C) * C + r)
                    assert key not in slots and key[1] < 8
                    slots[key] = (h, r)
            for rp in range(C):
                k = 0
                while rp + C * k < G:
                    h = rp + C * k
                    assert [slots[(rp, k * C + x)] for x in range(C)] == [(h, x) for x in range(C)]
                    k += 1


def test_device_closed_forms_equal_the_loops():
    # The device evaluates the rule with closed forms (Sched::auto_uniform_splits):
    # s_opt = 2^(h / 2) with h the index of lmax's top bit, and the largest power of
    # two <= s_wave from its top bit.  The host rule and this model use the loops; the
    # two agree everywhere.
    def s_opt_loop(lmax):
        p = 1
        while 4 * p * p <= lmax:
            p *= 2
        return p

    def s_opt_closed(lmax, kv8=False):
        if lmax <= 0:
            return 1
        h = lmax.bit_length() - 1
        return 1 << max(0, (h >> 1) - (1 if kv8 else 0))

    def s_opt_loop8(lmax):
        p = 1
        while 16 * p * p <= lmax:
            p *= 2
        return p

    def p2_loop(w):
        p = 1
        while 2 * p <= w:
            p *= 2
        return p

    rng = random.Random(3)
    cases = list(range(0, 1 << 15)) + [rng.randrange(0, 2 ** 31) for _ in range(20000)] + [2 ** 31 - 1]
    for lmax in cases:
        assert s_opt_closed(lmax) == s_opt_loop(lmax), lmax
        assert s_opt_closed(lmax, kv8=True) == s_opt_loop8(lmax), lmax
    for w in range(1, 4096):
        assert (1 << (w.bit_length() - 1)) == p2_loop(w), w
