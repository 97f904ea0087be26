"""A CPU model of the split-KV attention kernel's work partition and of its
cross-CTA combine protocol, run under random CTA interleavings.

The kernel (fp8_paged_kv_gb300/csrc/decode_attn.cu, partition rules in
csrc/attn_plan.cuh) lays all (request, kv head) segments end to end as a list
of 16-token tiles, cuts it into W splits of equal tile count and gives each
CTA a run of consecutive splits, which it walks piece by piece (a piece stays
inside one segment and one split).  A piece that covers its whole segment
writes the output; any other writes its split's partial and counts one
arrival on an arrival counter, a CTA's consecutive arrivals on one counter in
one atomic.  The arrival that completes a counter combines: all of a
segment's partials up to 16 of them, else groups of about sqrt(n) first and
then the groups.

This model restates those rules and checks, for thousands of random shapes and
arrival orders, what the combine's correctness rests on: every tile is read
exactly once; every slot a combine reads was written in this call before the
arrival that released it; every segment is combined exactly once, from all of
its tiles; every counter is back at zero afterwards.  Tiles stand in for the
partial results: a slot holds the set of tiles its partial covers.
"""
import math
import random

import pytest

K_DIRECT = 16


def worker_of(x, T, W):
    return ((x + 1) * W - 1) // T


class Shape:
    def __init__(self, tiles, Hkv, W, nctas, aligned_csz=0):
        self.tiles = tiles            # tiles per request
        self.B = len(tiles)
        self.Hkv = Hkv
        self.T = sum(tiles) * Hkv
        self.aligned = aligned_csz > 0
        if self.aligned:
            # every non-empty segment cut into splits of csz tiles, one per CTA
            self.csz = aligned_csz
            self.W = sum(Hkv * -(-n // aligned_csz) for n in tiles)
            self.nctas = max(nctas, self.W)
        else:
            self.W = W
            self.nctas = nctas

    def seg_start(self, r, h):
        return sum(self.tiles[:r]) * self.Hkv + h * self.tiles[r]


def next_piece(c, sh):
    """The next piece of a cursor: the longest run inside one segment and one
    split (the kernel's next_piece)."""
    if c["remaining"] <= 0:
        return None
    T, W = sh.T, sh.W
    s = c["split"] if c["split"] >= 0 else worker_of(c["x"], T, W)
    split_end = c["x"] + c["remaining"] if c["split"] >= 0 else (s + 1) * T // W
    take = min(c["n"] - c["t"], c["remaining"], split_end - c["x"])
    assert take > 0
    p = dict(s=s, r=c["r"], h=c["h"], t0=c["t"], t1=c["t"] + take, n=c["n"], x0=c["x"])
    c["remaining"] -= take
    c["x"] += take
    c["t"] += take
    if c["remaining"] > 0 and c["t"] == c["n"]:
        c["t"] = 0
        c["h"] += 1
        if c["h"] == sh.Hkv:
            c["h"] = 0
            while True:
                c["r"] += 1
                c["n"] = sh.tiles[c["r"]] if c["r"] < sh.B else 1
                if c["n"] > 0:
                    break
            assert c["r"] < sh.B
    return p


def start_cursor(sh, w):
    if sh.aligned:
        k = 0
        for r, n in enumerate(sh.tiles):
            m = -(-n // sh.csz)
            for h in range(sh.Hkv):
                for j in range(m):
                    if k == w:
                        t0 = j * sh.csz
                        return dict(r=r, h=h, t=t0, n=n, x=sh.seg_start(r, h) + t0,
                                    remaining=min(n, t0 + sh.csz) - t0, split=w,
                                    first=k - j, m=m)
                    k += 1
        return None
    s0, s1 = w * sh.W // sh.nctas, (w + 1) * sh.W // sh.nctas
    b0, b1 = s0 * sh.T // sh.W, s1 * sh.T // sh.W
    if b0 >= b1:
        return None
    base = 0
    for r, n in enumerate(sh.tiles):
        span = n * sh.Hkv
        if b0 < base + span:
            off = b0 - base
            return dict(r=r, h=off // n, t=off % n, n=n, x=b0, remaining=b1 - b0, split=-1)
        base += span
    raise AssertionError("start past the tiles")


def pending_of(sh, p, seg, cur0):
    """Counter, member list and destination of a piece's arrival (the
    kernel's pending_of)."""
    T, W = sh.T, sh.W
    xseg = p["x0"] - p["t0"]
    if sh.aligned:
        w0, w1 = cur0["first"], cur0["first"] + cur0["m"] - 1
    else:
        w0, w1 = worker_of(xseg, T, W), worker_of(xseg + p["n"] - 1, T, W)
    dense = sh.aligned or T >= W
    nsl = w1 - w0 + 1 if dense else p["n"]
    me = p["s"] - w0 if dense else p["t0"]

    def slot(i):
        return seg + (w0 + i if dense else worker_of(xseg + i, T, W))

    q = dict(seg=seg, slot=slot, i0=0, stride=1, ctr=("seg", seg), n=nsl, dst=None, K=1, ng=1)
    if nsl > K_DIRECT:
        K = int(math.sqrt(nsl))
        while K * K < nsl:
            K += 1
        gi = me // K
        q.update(K=K, ng=-(-nsl // K), i0=gi * K, n=min(K, nsl - gi * K))
        q["dst"] = slot(q["i0"])
        q["ctr"] = ("grp", q["dst"])
    return q


class World:
    def __init__(self, sh):
        self.sh = sh
        self.slots = {}       # slot -> frozenset of (seg, tile) | "empty"
        self.ctr = {}
        self.out = {}         # seg -> tiles combined into the output
        self.events = 0

    def write(self, slot, val):
        self.slots[slot] = val

    def combine(self, q):
        got = []
        for k in range(q["n"]):
            sl = q["slot"](q["i0"] + k * q["stride"])
            assert sl in self.slots, f"combine reads slot {sl}, not written in this call"
            v = self.slots[sl]
            if v != "empty":
                got.extend(v)
        assert len(got) == len(set(got)), "a tile reached the combine twice"
        if q["dst"] is None:
            assert q["seg"] not in self.out, "segment combined twice"
            self.out[q["seg"]] = got
        else:
            self.slots[q["dst"]] = frozenset(got) if got else "empty"


def cta_program(world, sh, w):
    """Generator: one CTA's shared-memory steps, in program order."""
    cur = start_cursor(sh, w)
    if cur is None:
        return
    cur0 = dict(cur)
    pend = None  # (piece, seg, counter key, k)

    def flush(q, arrivals):
        while True:
            key = q["ctr"]
            old = world.ctr.get(key, 0)
            world.ctr[key] = old + arrivals
            yield
            if old + arrivals != q["n"]:
                return
            world.combine(q)
            world.ctr[key] = 0
            yield
            if q["dst"] is None:
                return
            q = dict(q, ctr=("seg", q["seg"]), n=q["ng"], dst=None, i0=0, stride=q["K"])
            arrivals = 1

    p = next_piece(cur, sh)
    while p is not None:
        seg = p["r"] * sh.Hkv + p["h"]
        tiles = frozenset((seg, t) for t in range(p["t0"], p["t1"]))
        if p["t0"] == 0 and p["t1"] == p["n"]:
            assert seg not in world.out
            world.out[seg] = list(tiles)
            yield
        else:
            world.write(seg + p["s"], tiles)
            yield
            key = pending_of(sh, p, seg, cur0)["ctr"]
            if pend is not None and pend[2] != key:
                q = pending_of(sh, pend[0], pend[1], cur0)
                yield from flush(q, pend[3])
                pend = None
            pend = (p, seg, key, 1) if pend is None else (pend[0], pend[1], key, pend[3] + 1)
        p = next_piece(cur, sh)
    if pend is not None:
        yield from flush(pending_of(sh, pend[0], pend[1], cur0), pend[3])


def run_shape(sh, rng):
    world = World(sh)
    progs = [cta_program(world, sh, w) for w in range(sh.nctas)]
    live = list(range(len(progs)))
    while live:
        i = rng.randrange(len(live))
        try:
            next(progs[live[i]])
        except StopIteration:
            live.pop(i)
    for r, n in enumerate(sh.tiles):
        for h in range(sh.Hkv):
            seg = r * sh.Hkv + h
            if n == 0:
                assert seg not in world.out
                continue
            assert seg in world.out, f"segment {seg} never combined"
            assert sorted(world.out[seg]) == [(seg, t) for t in range(n)]
    assert all(v == 0 for v in world.ctr.values()), "a counter is left non-zero"


def random_shape(rng):
    B = rng.randint(1, 6)
    tiles = [rng.choice([0, 1, 2, 3, 5, 8, 17, 40, 64, 130]) for _ in range(B)]
    if sum(tiles) == 0:
        tiles[0] = rng.randint(1, 50)
    Hkv = rng.choice([1, 2, 3, 8])
    T = sum(tiles) * Hkv
    kind = rng.random()
    if kind < 0.15:
        return Shape(tiles, Hkv, 0, rng.randint(1, 40), aligned_csz=rng.randint(1, 40))
    nctas = rng.randint(1, 48)
    if kind < 0.45:
        W = rng.randint(1, nctas)                    # at most one split per CTA
    elif kind < 0.85:
        W = rng.randint(nctas, 6 * nctas)            # consecutive splits per CTA
    else:
        W = rng.randint(T, 3 * T + 1)                # more splits than tiles
    return Shape(tiles, Hkv, W, nctas)


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes_and_orders(seed):
    rng = random.Random(1000 + seed)
    for _ in range(250):
        sh = random_shape(rng)
        for _ in range(2):
            run_shape(sh, rng)


def test_long_segments_two_level_groups():
    # 64 splits per segment over 7-split CTAs: a CTA's arrivals straddle the sqrt groups
    rng = random.Random(7)
    for nctas in (9, 10, 37, 73):
        sh = Shape([512, 512], 4, 2 * 4 * 64, nctas)
        for _ in range(3):
            run_shape(sh, rng)


def test_whole_segment_pieces_take_no_ticket():
    # one split per segment, two segments per CTA
    sh = Shape([8, 8, 8, 8], 2, 8, 4)
    world = World(sh)
    for w in range(sh.nctas):
        for _ in cta_program(world, sh, w):
            pass
    assert sorted(world.out) == list(range(8))
    assert not world.ctr and not world.slots


def test_model_catches_a_dropped_partial():
    # the model must fail when a piece's partial is never written
    rng = random.Random(3)
    sh = Shape([300], 1, 40, 5)
    orig = World.write
    dropped = []

    def drop_one(self, slot, val):
        if dropped:
            orig(self, slot, val)
        else:
            dropped.append(slot)

    World.write = drop_one
    try:
        with pytest.raises(AssertionError, match="not written in this call"):
            run_shape(sh, rng)
    finally:
        World.write = orig


def test_model_catches_a_wrong_group_size():
    # a CTA that takes one split more than its share double-counts a tile
    rng = random.Random(4)
    sh = Shape([200, 90], 2, 30, 7)
    orig = start_cursor

    def greedy(sh2, w):
        c = orig(sh2, w)
        if c is not None and w == 2:
            c["remaining"] += 1
        return c

    g = globals()
    g["start_cursor"] = greedy
    try:
        with pytest.raises(AssertionError):
            run_shape(sh, rng)
    finally:
        g["start_cursor"] = orig
