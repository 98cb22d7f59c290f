"""A CPU model of the staged mixed-phase kernel's index arithmetic
(`fused_stage_kernel` in csrc/ar_stage.cuh), checked before any change to it
runs on a GPU.

The model follows the kernel step by step on a byte-exact memory: the tiles
of each segment, the aligned 16-byte words staged per rank (one slot per rank
up to eight, eight slots streamed beyond that, one for the gather form), the
4-byte frame words read from a slot at a rank's offset, the fold in the
schedule's position order, the shifted result copies (four word shifts, four
more moved by one 2-byte element; the gather form of up to 8 ranks builds
one copy per destination, in two buffers used in turn), and the stores: one bulk copy of whole
entries per destination plus the two partial edge words, or, for 2- and
4-rank rows of 2-byte elements, words shifted in registers.  The fold step is
a stand-in operation that is neither commutative nor associative, so any
change of order or operand shows.  Blocks run in a random order, and before
each block every byte of the row outside the block's tile is overwritten
with noise, so a block that read another tile's bytes would store a wrong
value.  Checked: every staged word overlaps the tile's own words, every
shared-memory access lies inside the launch's dynamic allocation, every
global write is a byte of the block's own tile, each destination element is
written exactly once, and the result equals the fold written out per
element.  None of this runs CUDA; the GPU parity tests check the kernel
itself against the oracle."""
import random

import numpy as np
import pytest

TV, BLOCK = 512, 256                 # frame vectors per tile, threads per block
SLOT = TV * 16 + 16                  # one rank's staged words
COPY = (TV + 2) * 16                 # one shifted copy of the result
M32 = (1 << 32) - 1


def slots(nr, gather, es):
    """Rank slots: one per rank up to 8 (4-byte elements of 6 to 8 ranks:
    five, streamed), eight streamed beyond; the gather form one."""
    return 1 if gather else 5 if es == 4 and 5 < nr <= 8 else nr if nr < 8 else 8


def gather_form(nr):
    """1: a copy per destination in two buffers used in turn (up to 8 ranks);
    2: all shifted copies at once (more ranks)."""
    return 1 if nr <= 8 else 2


def copies(es, nr, gather):
    if gather and gather_form(nr) == 1:
        return 2
    return 8 if es == 2 and (gather or slots(nr, gather, es) == 8) else 4


def smem_bytes(nr, es, gather):
    if gather and gather_form(nr) == 1:  # the slot, then the two copy buffers
        return SLOT + 2 * COPY
    return max(slots(nr, gather, es) * SLOT, copies(es, nr, gather) * COPY)


def fshr(lo, hi, sh):
    return ((hi << 32 | lo) >> sh) & M32


def fshl(lo, hi, sh):
    return ((hi << 32 | lo) << sh >> 32) & M32


def op_elem(a, b, es):
    """Stand-in fold step: neither commutative nor associative."""
    return (a * 3 + b + 1) & ((1 << 8 * es) - 1)


def op_word(a, b, es):
    if es == 4:
        return op_elem(a, b, 4)
    return (op_elem(a >> 16, b >> 16, 2) << 16) | op_elem(a & 0xFFFF, b & 0xFFFF, 2)


def inorder_root(lo, hi):
    return lo if lo == hi else hi & ~((1 << ((lo ^ hi).bit_length() - 1)) - 1)


def inorder_fold(xs, lo, hi, f):
    """Double binary tree over positions lo..hi (xs[p - 1] at position p)."""
    r = inorder_root(lo, hi)
    acc = xs[r - 1]
    if lo < r:
        acc = f(inorder_fold(xs, lo, r - 1, f), acc)
    if r < hi:
        acc = f(acc, inorder_fold(xs, r + 1, hi, f))
    return acc


def tree_fold(xs, f):
    xs = list(xs)
    w = 1
    while w < len(xs):
        for i in range(0, len(xs), 2 * w):
            xs[i] = f(xs[i], xs[i + w])
        w *= 2
    return xs[0]


def fold(order, vals, c, nr, f):
    """vals[r] = rank r's value; the schedule's fold for chunk c."""
    if order == "ring":
        acc = vals[(c + 1) % nr]
        for p in range(1, nr):
            acc = f(acc, vals[(c + 1 + p) % nr])
        return acc
    if order == "tree":
        return tree_fold(vals, f)
    shift = 1 if c else 0  # double binary tree: tree B is tree A over the ranks moved by one
    return inorder_fold([vals[(p + shift) % nr] for p in range(nr)], 1, nr, f)


class Memory:
    def __init__(self):
        self.blocks = []

    def alloc(self, base, size):
        self.blocks.append((base, np.zeros(size, np.uint8)))

    def _at(self, addr, n):
        for base, a in self.blocks:
            if base <= addr and addr + n <= base + len(a):
                return a, addr - base
        raise AssertionError(f"{n} bytes at {addr:#x} outside every allocation")

    def read(self, addr, n):
        a, o = self._at(addr, n)
        return a[o:o + n].copy()

    def write(self, addr, data):
        a, o = self._at(addr, len(data))
        a[o:o + len(data)] = data


def words(b):
    return b.view("<u4").astype(np.uint64)


def run(rng, nr, es, order, owner_only=False, gather=False, root=0, counts=(1000,), mutation=None, phase=None):
    """phase: every buffer at this address modulo 16 (else each at its own);
    mutation: a planted mistake in the modelled kernel (see the last test)."""
    vec = 16 // es
    mem = Memory()
    ptrs, valid, orig = [], [], []
    for t, cnt in enumerate(counts):
        for r in range(nr):
            base = 0x4000000 * (1 + len(ptrs))
            mem.alloc(base, cnt * es + 64)
            p = base + (rng.randrange(0, 16 // es) * es if phase is None else phase) + 16 * rng.randrange(0, 2)
            data = np.frombuffer(rng.randbytes(cnt * es), np.uint8)
            mem.write(p, data)
            ptrs.append(p)
            valid.append((p, p + cnt * es))
            orig.append(data.view("<u2" if es == 2 else "<u4").astype(np.int64))
    # segments and tiles as the host builds them
    segs = []
    for t, cnt in enumerate(counts):
        if gather and order == "broadcast":
            bounds = [(root, 0, cnt)]
        elif order == "dbtree":
            bounds = [(0, 0, cnt // 2), (1, cnt // 2, cnt)]
        else:
            bounds = [(c, c * cnt // nr, (c + 1) * cnt // nr) for c in range(nr)]
        segs += [dict(tensor=t, chunk=c, begin=b, end=e) for c, b, e in bounds if e > b]
    ntiles = 0
    for sg in segs:
        sg["tile_begin"] = ntiles
        shift = (ptrs[sg["tensor"] * nr] & 15) // es
        vb, ve = (sg["begin"] + shift + vec - 1) // vec, (sg["end"] + shift) // vec
        units = max(ve - vb, 0)
        extra = (sg["end"] - sg["begin"]) - units * vec
        tiles = (units + TV - 1) // TV
        ntiles += tiles if tiles or not extra else 1
    smem = smem_bytes(nr, es, gather)
    nfold = 1 if gather else nr
    ns = slots(nr, gather, es)
    written = {}
    for tile in rng.sample(range(ntiles), ntiles):
        sg = max((s for s in segs if s["tile_begin"] <= tile), key=lambda s: s["tile_begin"])
        P = ptrs[sg["tensor"] * nr:(sg["tensor"] + 1) * nr]
        V = valid[sg["tensor"] * nr:(sg["tensor"] + 1) * nr]
        c = sg["chunk"]
        shift = (P[0] & 15) // es
        vb, ve = (sg["begin"] + shift + vec - 1) // vec, (sg["end"] + shift) // vec
        if ve > vb:
            head, tail = vb * vec - shift - sg["begin"], sg["end"] - (ve * vec - shift)
        else:
            ve, head, tail = vb, sg["end"] - sg["begin"], 0
        ti = tile - sg["tile_begin"]
        t0 = vb + ti * TV
        nv = min(ve - t0, TV)
        base = t0 * 16 - shift * es
        scalars = [sg["begin"] + k if k < head else ve * vec - shift + (k - head)
                   for k in range(head + tail)] if ti == 0 else []
        own = [set() for _ in range(nr)]
        for r in range(nr):
            if nv > 0:
                own[r].update(range(P[r] + base, P[r] + base + 16 * nv))
            for e in scalars:
                own[r].update(range(P[r] + e * es, P[r] + (e + 1) * es))
        # noise on every byte of the row near the tile that is not the tile's
        saved = []
        for r in range(nr):
            lo, hi = V[r]
            if nv > 0:
                lo, hi = max(lo - 16, P[r] + base - 64), min(hi + 16, P[r] + base + 16 * nv + 64)
            for addr in range(lo, hi):
                if addr not in own[r]:
                    try:
                        old = mem.read(addr, 1)
                    except AssertionError:
                        continue
                    saved.append((addr, old))
                    mem.write(addr, np.frombuffer(rng.randbytes(1), np.uint8))
        S = np.zeros(smem, np.uint8)
        stores = []
        if nv > 0:
            def rank_at(p):
                if gather:
                    return c
                if order == "ring":
                    return (c + (0 if mutation == "ring_from_owner" else 1) + p) % nr
                if order == "dbtree":
                    return (p + (1 if c else 0)) % nr
                return p

            def stage(p):
                r = rank_at(p)
                off = (P[r] - P[0]) & 15
                g = P[r] + base - off
                assert g % 16 == 0
                nw = nv + (off != 0)
                assert g < V[r][1] and g + 16 * nw > V[r][0], "staged words outside the buffer"
                assert g + 16 > P[r] + base and g + 16 * (nw - 1) < P[r] + base + 16 * nv, \
                    "staged words outside the tile's words"
                d = (p % ns) * SLOT
                assert d + 16 * nw <= smem
                S[d:d + 16 * nw] = mem.read(g, 16 * nw)

            def frame_words(p):
                r = rank_at(p)
                off = (P[r] - P[0]) & 15
                d = (p % ns) * SLOT + 4 * (off >> 2)
                assert d + 4 * (4 * TV + 1) <= smem
                w = words(S[d:d + 4 * (4 * TV + 1)])
                return w[:4 * TV] if es == 4 else fshr(w[:4 * TV], w[1:], (off & 2) * 8)

            vals = []
            for p in range(min(nfold, ns)):
                stage(p)
            for p in range(nfold):
                vals.append(frame_words(p))
                if p + ns < nfold:
                    stage(p + ns)  # the kernel refills after the next barrier, still before its fold
            f = np.vectorize(lambda a, b: op_word(int(a), int(b), es), otypes=[np.uint64])
            if gather:
                F = vals[0]
            else:
                F = fold(order, [vals[(p - (c + 1)) % nr] if order == "ring" else
                                 vals[(p - (1 if c else 0)) % nr] if order == "dbtree" else vals[p]
                                 for p in range(nr)], c, nr, f)
            if gather and gather_form(nr) == 1:
                for idx, r0 in enumerate(r for r in range(nr) if r != c):
                    off = (P[r0] - P[0]) & 15
                    k, h = off >> 2, es == 2 and off & 2
                    cb = SLOT + (idx & 1) * COPY
                    assert cb + COPY <= smem
                    buf = words(S[cb:cb + COPY]).copy()
                    if h:
                        below = np.concatenate(([F[0]], F[:-1]))  # m = 0: a value no stored byte uses
                        buf[k + 4:k + 4 + 4 * TV] = fshl(below, F, 16)
                        buf[k + 4 + 4 * TV] = fshl(F[-1], np.uint64(0), 16)
                    else:
                        buf[k + 4:k + 4 + 4 * TV] = F
                    S[cb:cb + COPY] = buf.astype("<u4").view(np.uint8)
                    for r in (r0,):
                        g = P[r] + base - off
                        lo = 1 if off else 0
                        if nv > lo:
                            stores.append((g + 16 * lo, S[cb + 16 * (lo + 1):cb + 16 * (nv + 1)].copy()))
                        if off:
                            stores.append((g + off, S[cb + 16:cb + 32][off:].copy()))
                            stores.append((g + 16 * nv, S[cb + 16 * (nv + 1):cb + 16 * (nv + 2)][:off].copy()))
            # the shifted copies: copy k holds frame word m at word index m + k + 4
            form1 = gather and gather_form(nr) == 1
            C = [] if form1 else [words(S[k * COPY:(k + 1) * COPY]).copy() for k in range(copies(es, nr, gather))]
            for k in range(len(C) and 4):
                C[k][k + 4:k + 4 + 4 * TV] = F
            if len(C) == 8:
                below = np.concatenate(([C[0][3]], F[:-1]))   # lane 0 reads copy 0's word below
                Hw = fshl(below, F, 16)
                for k in range(4):
                    C[4 + k][k + 4:k + 4 + 4 * TV] = Hw
                    if mutation != "no_word_past_tile":
                        C[4 + k][k + 4 + 4 * TV] = fshl(F[-1], np.uint64(0), 16)
            for k, ck in enumerate(C):
                S[k * COPY:(k + 1) * COPY] = ck.astype("<u4").view(np.uint8)
            dests = [] if form1 else [r for r in range(nr) if r != c] if gather else [c] if owner_only else range(nr)
            for r in dests:
                off = (P[r] - P[0]) & 15
                k, hs = off >> 2, off & 2
                g = P[r] + base - off
                nw = nv + (off != 0)
                half = len(C) == 8 and hs
                cp = ((4 if half else 0) + k) * COPY
                entry = lambda i: S[cp + 16 * i:cp + 16 * i + 16]
                if es == 4 or hs == 0 or half:
                    lo = 1 if off else 0
                    if nv > lo:
                        assert cp + 16 * (nv + 1) <= smem
                        first = lo + (2 if mutation == "bulk_one_entry_late" else 1)
                        stores.append((g + 16 * lo, S[cp + 16 * first:cp + 16 * (first + nv - lo)].copy()))
                    if off:
                        stores.append((g + off, entry(1)[off:].copy()))
                        stores.append((g + 16 * nv, entry(nv + 1)[:off].copy()))
                    continue
                for i in range(nw):
                    ic = min(i, TV)
                    cur = words(entry(ic + 1))
                    prev = words(entry(ic))[3]
                    v = np.array([fshl(prev, cur[0], 16), fshl(cur[0], cur[1], 16),
                                  fshl(cur[1], cur[2], 16), fshl(cur[2], cur[3], 16)]).astype("<u4").view(np.uint8)
                    lo_b, hi_b = (off, 16) if i == 0 else (0, off) if i == nv else (0, 16)
                    stores.append((g + 16 * i + lo_b, v[lo_b:hi_b].copy()))
        for e in scalars:
            el = [int.from_bytes(mem.read(P[r] + e * es, es).tobytes(), "little") for r in range(nr)]
            if gather:
                v, dests = el[c], [r for r in range(nr) if r != c]
            else:
                v = fold(order, el, c, nr, lambda a, b: op_elem(a, b, es))
                dests = [c] if owner_only else range(nr)
            for r in dests:
                stores.append((P[r] + e * es, np.frombuffer(v.to_bytes(es, "little"), np.uint8)))
        for addr, old in saved:
            mem.write(addr, old)
        for addr, data in stores:
            r = next(i for i in range(nr) if V[i][0] - 16 <= addr < V[i][1] + 16)
            for j in range(len(data)):
                assert addr + j in own[r], f"write outside the block's own bytes at {addr + j:#x}"
                written[addr + j] = written.get(addr + j, 0) + 1
            mem.write(addr, data)
    # the whole result
    for t, cnt in enumerate(counts):
        xs = orig[t * nr:(t + 1) * nr]
        for e in range(cnt):
            if gather:
                c = root if order == "broadcast" else min(cc for cc in range(nr) if e < (cc + 1) * cnt // nr)
            elif order == "dbtree":
                c = 0 if e < cnt // 2 else 1
            else:
                c = min(cc for cc in range(nr) if e < (cc + 1) * cnt // nr)
            if gather:
                want = [int(xs[c][e])] * nr
                dest = [r != c for r in range(nr)]
            else:
                v = fold(order, [int(x[e]) for x in xs], c, nr, lambda a, b: op_elem(a, b, es))
                dest = [(not owner_only) or r == c for r in range(nr)]
                want = [v if dest[r] else int(xs[r][e]) for r in range(nr)]
            for r in range(nr):
                a = ptrs[t * nr + r] + e * es
                got = int.from_bytes(mem.read(a, es).tobytes(), "little")
                assert got == want[r], (t, r, e, got, want[r])
                assert written.get(a, 0) == (1 if dest[r] else 0), (t, r, e)
    return ntiles


CASES = [
    # (ranks, element bytes, order, owner only, gather, counts per tensor)
    (8, 2, "ring", False, False, (2 * 512 * 8 * 8 + 37,)),
    (8, 4, "tree", True, False, (512 * 4 * 8 + 5, 301)),
    (8, 2, "dbtree", False, False, (3 * 512 * 8 + 11,)),
    (4, 2, "ring", False, False, (2 * 512 * 8 * 4 - 3,)),
    (2, 2, "tree", False, False, (512 * 8 * 2 + 9, 17)),
    (3, 4, "ring", True, False, (512 * 4 * 3 + 77,)),
    (5, 2, "ring", False, False, (3001,)),
    (16, 2, "tree", False, False, (16 * 8 * 300 + 5,)),
    (16, 4, "dbtree", False, False, (1200 * 4 + 3,)),
    (16, 2, "ring", True, False, (16 * 8 * 100 + 1, 7)),
    (8, 2, "ring", False, True, (512 * 8 * 8 + 21,)),
    (5, 4, "broadcast", False, True, (512 * 4 + 999,)),
    (8, 2, "broadcast", False, True, (3, 5000)),
    (16, 2, "ring", False, True, (16 * 8 * 60 + 3,)),
    (16, 4, "broadcast", False, True, (7000,)),
    (7, 2, "dbtree", False, False, (2 * 512 * 8 + 301,)),
    (3, 4, "dbtree", False, False, (3 * 512 * 4 + 6, 9)),
    (12, 2, "dbtree", False, False, (2 * 512 * 8 + 1001,)),
    (8, 4, "ring", False, False, (2 * 512 * 4 * 8 + 19,)),
    (7, 4, "dbtree", False, False, (512 * 4 * 7 + 3001,)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_staged_kernel_index_model(case):
    nr, es, order, owner_only, gather, counts = CASES[case]
    rng = random.Random(1000 + case)
    root = rng.randrange(nr)
    tiles = run(rng, nr, es, order, owner_only, gather, root, counts)
    assert tiles >= len(counts)


@pytest.mark.parametrize("nr,es,phase", [(5, 2, 6), (7, 4, 0), (3, 2, 0)])
def test_staged_kernel_index_model_one_phase(nr, es, phase):
    """Double binary trees of 3, 5 and 7 ranks take the staged kernel even
    when every buffer sits at the same address modulo 16."""
    rng = random.Random(nr * 100 + es)
    run(rng, nr, es, "dbtree", counts=(2 * 512 * 16 // es + 77, 5), phase=phase)


def level_counter_fold(xs, f, mutation=None):
    """The double binary tree's fold as the staged kernel takes it for a rank
    count known at run time: positions arrive in order; position q sits at
    level tz(q) of the in-order tree; a leaf (odd q) completes at once and,
    while the subtree it completes is a right child (the bits of q above bit
    0 are ones), completes its parents, whose held values take it in; node q
    of level l >= 1 holds (its left subtree) (+) x_q; at the end the held
    values fold in right-nested from the lowest level up."""
    hold, cur, pend, opn = [None] * 7, None, False, 0
    for q in range(1, len(xs) + 1):
        if q & 1:
            casc = ((~(q >> 1)) & -(~(q >> 1))).bit_length() - 1  # ones above bit 0
            cur = xs[q - 1]
            for lv in range(1, casc + 1):
                cur = f(hold[lv], cur)
            opn &= ~((2 << casc) - 2)
            pend = True
        else:
            t = (q & -q).bit_length() - 1
            hold[t] = f(cur, xs[q - 1]) if mutation != "operands_swapped" else f(xs[q - 1], cur)
            opn |= 1 << t
            pend = False
    levels = range(1, 7) if mutation != "end_from_the_top" else range(6, 0, -1)
    for lv in levels:
        if opn & (1 << lv):
            cur = f(hold[lv], cur) if pend else hold[lv]
            pend = True
    return cur


def test_dbtree_level_counter_rule():
    """The run-time double binary tree fold equals the recursive in-order
    definition for every rank count up to 64 (a step that keeps its operands
    as text shows any change of order or grouping), and two planted
    mistakes make it differ."""
    f = lambda a, b: f"({a}.{b})"
    for n in range(1, 65):
        xs = [f"x{q}" for q in range(1, n + 1)]
        assert level_counter_fold(xs, f) == inorder_fold(xs, 1, n, f), n
    for mutation in ("operands_swapped", "end_from_the_top"):
        assert any(level_counter_fold([f"x{q}" for q in range(1, n + 1)], f, mutation)
                   != inorder_fold([f"x{q}" for q in range(1, n + 1)], 1, n, f) for n in range(1, 65)), mutation


@pytest.mark.parametrize("mutation", ["ring_from_owner", "no_word_past_tile", "bulk_one_entry_late"])
def test_model_catches_planted_mistakes(mutation):
    """Pins of the model itself: a ring folded from the owner instead of the
    rank after it, the element-moved word one past a full tile left out (the
    bug the model caught before any GPU run), and a bulk copy one entry late
    each make it fail."""
    rng = random.Random(7)
    with pytest.raises(AssertionError):
        run(rng, 8, 2, "ring", False, False, 0, (2 * 512 * 8 * 8,), mutation=mutation)
