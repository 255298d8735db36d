"""Model of the synchronisation of the fused forward on CTA pairs (`fwd_tc2.cu`):
its four-CTA form (d_v = 512, QUAD) and its two-CTA form (`roles_pair`).  Test
infrastructure, no arithmetic of the method.

Every role of one cluster of four CTAs (two pairs over the same query rows) is
a generator that yields the steps the kernel takes on its mbarriers and named
barriers, in the kernel's order, with the kernel's arrival counts, and follows
the kernel's exit logic when a wait gives up:
  ok = yield ('wait', key, k)     bounded wait for phase k of barrier `key`
  yield ('arrive', key)           one arrival
  yield ('nb', key, n)            named barrier of n warps
  ok = yield ('red', key, n, p)   reducing named barrier: every warp gets the AND
  yield ('use', buf, op, x)       an access to a buffer (checked for overlaps)
Copies and MMAs complete at once; only the order of steps matters here.  A
wait that gives up raises its CTA's abort flag, after which every wait of that
CTA that finds its phase incomplete gives up at once (a phase already complete
still passes), as in the kernel.

A scheduler runs the roles in random interleavings and reports
  - deadlock: no role can take a step and some have not finished (a wait can
    always give up, so this means warps stranded at a named barrier);
  - overrun: a wait for phase k finds k + 2 or more phases completed, or k - 1
    (a parity wait cannot tell phase k from k + 2, and passes at k - 1);
  - hazards on the buffers that the barriers protect (only while nothing has
    given up: an aborted launch's results are discarded): the pair's O
    accumulator (the epilogue's reads against the next item's first O
    product); each S buffer in TMEM (the S product writing it against the
    pair's own P stored over it and read by the O product); and each CTA's
    shared-memory P buffer (the other pair's P writes against this pair's O
    product that consumes them and against the epilogue, which stages its
    output through the same buffer).

`mutation` plants one mistake (tests check that each is caught).
"""
import random
from collections import defaultdict

BM = 128          # query rows per CTA, keys per tile


def cluster_items(n_clusters, c, B, H, T, nsplit=1):
    """Work items of cluster c in the kernel's serpentine longest-first order:
    (head, number of key tiles); nsplit d_v slices per query block (two-CTA
    form at d_v = 512 without the exchange)."""
    per = B * H * nsplit
    npairs = ((T + BM - 1) // BM + 1) // 2
    n_items = npairs * per
    out, r = [], 0
    while r * n_clusters < n_items:
        w = r * n_clusters + ((n_clusters - 1 - c) if (r & 1) else c)
        if w < n_items:
            pair = npairs - 1 - w // per
            out.append(((w % per) // nsplit, (min(T, (2 * pair + 2) * BM) - 1) // BM + 1))
        r += 1
    return out


def roles(items, nkg=4, nk=2, nv=2, mutation=None):
    """The cluster's roles as (name, cta, generator).  nkg: K granules per key
    tile (d_qk / 128); nk, nv: ring granules; every tile takes two V granules
    of each CTA."""
    counts = {}
    NS = 2                                   # S buffers

    def own(pr, g):                          # tile g of the sequence belongs to pair g & 1
        return (g & 1) == pr

    for cta in range(4):
        counts[(cta, 'QFull')] = 4           # two producers in each CTA of the pair
        counts[(cta, 'QEmpty')] = 1
        for b in range(NS):
            counts[(cta, f'SFull{b}')] = 1
            counts[(cta, f'SEmpty{b}')] = 1  # the own-tile O product
            counts[(cta, f'PFull{b}')] = 16  # eight gating warps in each CTA of the pair
        counts[(cta, 'PEmpty')] = 1
        counts[(cta, 'OFull')] = 1
        counts[(cta, 'BxFull')] = 2 if mutation == 'bx_count' else 4
        counts[(cta, 'EpiDone')] = 1
        counts[(cta, 'ODrained')] = 2
        counts[(cta, 'PRx')] = 8 if mutation == 'prx_count' else 16
        for s in range(nk + nv):
            counts[(cta, f'Full{s}')] = 2    # the loads of both CTAs of the pair
            counts[(cta, f'Empty{s}')] = 1

    def pfull(buf):
        return 'PFull0' if mutation == 'single_pfull' else f'PFull{buf}'

    def pfull_phase(gs):
        return gs if mutation == 'single_pfull' else gs // NS

    def producer(cta, pi):
        lead, pr = cta & ~1, cta >> 1
        base, n = (0, nk) if pi == 0 else (nk, nv)
        st, g0, fills = 0, 0, defaultdict(int)
        ok = True
        for qi, (_, nkv) in enumerate(items):
            if qi > 0:
                ok = yield ('wait', (cta, 'QEmpty'), qi - 1)
                if not ok:
                    break
            yield ('arrive', (lead, 'QFull'))
            for j in range(nkv):
                if pi == 0 and not own(pr, g0 + j):
                    continue                 # the K ring carries this pair's tiles only
                for _ in range(nkg if pi == 0 else 2):
                    s = base + st
                    ok = yield ('wait', (cta, f'Empty{s}'), fills[s] - 1)
                    if not ok:
                        break
                    fills[s] += 1
                    yield ('arrive', (lead, f'Full{s}'))
                    st = (st + 1) % n
                if not ok:
                    break
            g0 += nkv
            if not ok:
                break

    def s_issuer(cta):
        pr, pm = cta >> 1, (cta, cta + 1)
        st, uses, gs, gt = 0, defaultdict(int), 0, 0
        for qi, (_, nkv) in enumerate(items):
            ok = yield ('wait', (cta, 'QFull'), qi)
            for _ in range(nkv):
                if not ok:
                    break
                g, gt = gt, gt + 1
                if not own(pr, g):
                    continue
                buf, u = gs % NS, gs // NS
                if mutation != 'no_sempty':
                    ok = yield ('wait', (cta, f'SEmpty{buf}'), u - 1)
                    if not ok:
                        break
                yield ('use', ('S', cta, buf), 's_write', g)
                for _ in range(nkg):
                    ok = yield ('wait', (cta, f'Full{st}'), uses[st])
                    if not ok:
                        break
                    uses[st] += 1
                    for c in pm:
                        yield ('arrive', (c, f'Empty{st}'))
                    st = (st + 1) % nk
                if not ok:
                    break
                for c in pm:
                    yield ('arrive', (c, f'SFull{buf}'))
                gs += 1
            if not ok:
                break
            for c in pm:
                yield ('arrive', (c, 'QEmpty'))

    def o_issuer(cta):
        pr, pm, xm = cta >> 1, (cta, cta + 1), (cta ^ 2, (cta ^ 2) + 1)
        st, uses, gs, go, gt = 0, defaultdict(int), 0, 0, 0
        ok = True
        for qi, (_, nkv) in enumerate(items):
            if qi > 0 and mutation != 'no_odrained':
                ok = yield ('wait', (cta, 'ODrained'), qi - 1)
            for j in range(nkv):
                if not ok:
                    break
                g, gt = gt, gt + 1
                mine = own(pr, g)
                if mine:
                    buf = gs % NS
                    ok = yield ('wait', (cta, pfull(buf)), pfull_phase(gs))
                    gs += 1
                else:
                    ok = yield ('wait', (cta, 'PRx'), go)
                    go += 1
                if not ok:
                    break
                got = []
                for _ in range(2):
                    s = nk + st
                    ok = yield ('wait', (cta, f'Full{s}'), uses[s])
                    if not ok:
                        break
                    uses[s] += 1
                    got.append(s)
                    st = (st + 1) % nv
                if not ok:
                    break
                if j == 0:
                    yield ('use', ('O', cta), 'write', None)
                if mine:
                    yield ('use', ('S', cta, buf), 'p_consume', g)
                else:
                    for c in pm:
                        yield ('use', ('P', c), 'consume', g)
                for s in got:
                    for c in pm:
                        yield ('arrive', (c, f'Empty{s}'))
                for c in (pm if mine else xm):
                    yield ('arrive', (c, f'SEmpty{buf}' if mine else 'PEmpty'))
            if not ok:
                break
            for c in pm:
                yield ('arrive', (c, 'OFull'))

    def gating(cta, gw):
        lead, pr, x = cta & ~1, cta >> 1, cta ^ 2
        half = gw >> 2
        gs, gt = 0, 0
        ok = True
        for qi, (_, nkv) in enumerate(items):
            partner_free = qi == 0
            for j in range(0 if own(pr, gt) else 1, nkv, 2):
                buf, u = gs % NS, gs // NS
                ok = yield ('wait', (cta, f'SFull{buf}'), u)
                if not ok:
                    break
                yield ('use', ('S', lead, buf), 'p_store', gt + j)
                yield ('arrive', (lead, pfull(buf)))          # own P in TMEM
                if not partner_free:
                    if mutation != 'no_epidone':
                        ok = yield ('wait', (cta, 'EpiDone'), qi - 1)
                        if not ok:
                            break
                    partner_free = True
                if mutation != 'no_pempty':
                    ok = yield ('wait', (cta, 'PEmpty'), gs - 1)
                    if not ok:
                        break
                yield ('use', ('P', x), 'write', gt + j)        # remote stores
                yield ('arrive', (x & ~1, 'PRx'))
                gs += 1
            if not ok and mutation == 'exit_early':
                return                                          # leaves without the group
            if ok and not partner_free and mutation != 'no_idle_epidone':
                ok = yield ('wait', (cta, 'EpiDone'), qi - 1)
            gt += nkv
            ok = yield ('red', (cta, 'sums', qi), 8, ok)         # all eight leave together, or none
            if not ok:
                break
            if half == 0:
                yield ('arrive', (x, 'BxFull'))                  # row sums to the other pair
            ok = yield ('wait', (cta, 'OFull'), qi)
            if ok:
                ok = yield ('wait', (cta, 'BxFull'), qi)
            if mutation == 'exit_unreduced':
                yield ('nb', (cta, 'epi', qi), 8)
            else:
                ok = yield ('red', (cta, 'epi', qi), 8, ok)
            if not ok:
                break
            yield ('use', ('O', lead), 'read_begin', (cta, gw))
            yield ('use', ('P', cta), 'stage_begin', gw)
            yield ('nb', (cta, 'half', half, qi), 4)            # the epilogue's per-half barriers
            yield ('use', ('P', cta), 'stage_end', gw)
            yield ('use', ('O', lead), 'read_end', (cta, gw))
            yield ('nb', (cta, 'end', qi), 8)
            if gw == 5:
                yield ('arrive', (lead, 'ODrained'))
                yield ('arrive', (x, 'EpiDone'))

    out = []
    for cta in range(4):
        out.append((f'producer K {cta}', cta, producer(cta, 0)))
        out.append((f'producer V {cta}', cta, producer(cta, 1)))
        if cta % 2 == 0:
            out.append((f'S issuer {cta}', cta, s_issuer(cta)))
            out.append((f'O issuer {cta}', cta, o_issuer(cta)))
        for gw in range(8):
            out.append((f'gating {cta}.{gw}', cta, gating(cta, gw)))
    return counts, out


def roles_pair(items, nsbuf=1, nkg=3, nk=3, nv=3, vpt=3, mutation=None):
    """The two-CTA form's roles as (name, cta, generator): one pair, every key
    tile its own; S in nsbuf TMEM buffers that the gating warps release once
    they have read S; P through the CTA's shared-memory P buffer; vpt V
    granules per tile."""
    counts = {}
    for cta in range(2):
        counts[(cta, 'QFull')] = 4
        counts[(cta, 'QEmpty')] = 1
        for b in range(nsbuf):
            counts[(cta, f'SFull{b}')] = 1
            counts[(cta, f'SEmpty{b}')] = 8 if mutation == 'pair_sempty_count' else 16   # both CTAs' gating warps
        counts[(cta, 'PFull')] = 16
        counts[(cta, 'PEmpty')] = 1
        counts[(cta, 'OFull')] = 1
        for s in range(nk + nv):
            counts[(cta, f'Full{s}')] = 2
            counts[(cta, f'Empty{s}')] = 1

    def producer(cta, pi):
        base, n = (0, nk) if pi == 0 else (nk, nv)
        st, fills = 0, defaultdict(int)
        ok = True
        for qi, (_, nkv) in enumerate(items):
            if qi > 0:
                ok = yield ('wait', (cta, 'QEmpty'), qi - 1)
                if not ok:
                    break
            yield ('arrive', (0, 'QFull'))
            for _ in range(nkv):
                for _ in range(nkg if pi == 0 else vpt):
                    s = base + st
                    ok = yield ('wait', (cta, f'Empty{s}'), fills[s] - 1)
                    if not ok:
                        break
                    fills[s] += 1
                    yield ('arrive', (0, f'Full{s}'))
                    st = (st + 1) % n
                if not ok:
                    break
            if not ok:
                break

    def s_issuer():
        st, uses, gt = 0, defaultdict(int), 0
        for qi, (_, nkv) in enumerate(items):
            ok = yield ('wait', (0, 'QFull'), qi)
            for _ in range(nkv):
                if not ok:
                    break
                g, gt = gt, gt + 1
                buf, u = g % nsbuf, g // nsbuf
                ok = yield ('wait', (0, f'SEmpty{buf}'), u - 1)
                if not ok:
                    break
                yield ('use', ('S', 0, buf), 's_write', g)
                for _ in range(nkg):
                    ok = yield ('wait', (0, f'Full{st}'), uses[st])
                    if not ok:
                        break
                    uses[st] += 1
                    for c in (0, 1):
                        yield ('arrive', (c, f'Empty{st}'))
                    st = (st + 1) % nk
                if not ok:
                    break
                for c in (0, 1):
                    yield ('arrive', (c, f'SFull{buf}'))
            if not ok:
                break
            for c in (0, 1):
                yield ('arrive', (c, 'QEmpty'))

    def o_issuer():
        st, uses, gt = 0, defaultdict(int), 0
        ok = True
        for qi, (_, nkv) in enumerate(items):
            for j in range(nkv):
                g, gt = gt, gt + 1
                ok = yield ('wait', (0, 'PFull'), g)
                if not ok:
                    break
                got = []
                for _ in range(vpt):
                    s = nk + st
                    ok = yield ('wait', (0, f'Full{s}'), uses[s])
                    if not ok:
                        break
                    uses[s] += 1
                    got.append(s)
                    st = (st + 1) % nv
                if not ok:
                    break
                if j == 0:
                    yield ('use', ('O', 0), 'write', None)
                for c in (0, 1):
                    yield ('use', ('P', c), 'consume', g)
                for s in got:
                    for c in (0, 1):
                        yield ('arrive', (c, f'Empty{s}'))
                for c in (0, 1):
                    yield ('arrive', (c, 'PEmpty'))
            if not ok:
                break
            for c in (0, 1):
                yield ('arrive', (c, 'OFull'))

    def gating(cta, gw):
        gt = 0
        ok = True
        for qi, (_, nkv) in enumerate(items):
            for j in range(nkv):
                g = gt + j
                buf, u = g % nsbuf, g // nsbuf
                ok = yield ('wait', (cta, f'SFull{buf}'), u)
                if not ok:
                    break
                yield ('use', ('S', 0, buf), 's_read', g)
                yield ('arrive', (0, f'SEmpty{buf}'))
                ok = yield ('wait', (cta, 'PEmpty'), g - 1)
                if not ok:
                    break
                yield ('use', ('P', cta), 'write', g)
                yield ('arrive', (0, 'PFull'))
            if not ok and mutation == 'pair_exit_early':
                return
            gt += nkv
            if ok:
                ok = yield ('wait', (cta, 'OFull'), qi)
            ok = yield ('red', (cta, 'epi', qi), 8, ok)
            if not ok:
                break
            yield ('use', ('O', 0), 'read_begin', (cta, gw))
            yield ('use', ('P', cta), 'stage_begin', gw)
            yield ('nb', (cta, 'half', gw >> 2, qi), 4)
            yield ('use', ('P', cta), 'stage_end', gw)
            yield ('use', ('O', 0), 'read_end', (cta, gw))
            yield ('nb', (cta, 'end', qi), 8)

    out = []
    for cta in range(2):
        out.append((f'producer K {cta}', cta, producer(cta, 0)))
        out.append((f'producer V {cta}', cta, producer(cta, 1)))
        for gw in range(8):
            out.append((f'gating {cta}.{gw}', cta, gating(cta, gw)))
    out.append(('S issuer', 0, s_issuer()))
    out.append(('O issuer', 0, o_issuer()))
    return counts, out


class _State:
    def __init__(self, counts):
        self.counts = counts
        self.pending = {}
        self.done = defaultdict(int)
        self.named = defaultdict(dict)         # named barrier -> {member: predicate}
        self.abort = [False] * 4
        self.errors = []
        self.o_readers = defaultdict(set)      # O accumulator (pair leader) -> open epilogue reads
        self.stage = defaultdict(set)          # CTA -> warps staging through its P buffer
        self.rx = {}                           # CTA -> [tile held, writes landed, consumed]
        self.sbuf = {}                         # (pair leader, buffer) -> [tile, P stores, consumed]

    def arrive(self, key):
        c = self.counts[key]
        p = self.pending.get(key, c) - 1
        if p == 0:
            self.done[key] += 1
            p = c
        self.pending[key] = p

    def ready(self, key, k):
        # the kernel's waits compare parities: phase k looks complete whenever
        # the number of completed phases differs from k in parity
        d = self.done[key]
        if not any(self.abort):
            if d >= k + 2:
                self.errors.append(f'overrun: {key} wanted phase {k}, {d} completed')
            elif d < k and (k - d) % 2 == 1:
                self.errors.append(f'early pass: {key} wanted phase {k}, only {d} completed')
        return d >= k + 1

    def hazard(self, msg):
        if not any(self.abort):
            self.errors.append('hazard: ' + msg)

    def use(self, buf, op, x):
        kind, cta = buf[0], buf[1]
        if kind == 'S':
            sb = self.sbuf.setdefault(buf, [None, 0, True])
            if op == 's_write':
                if not sb[2]:
                    self.hazard(f'S product of tile {x} overwrites unconsumed P of tile {sb[0]}')
                self.sbuf[buf] = [x, 0, False]
            elif op == 'p_store':
                if sb[0] != x:
                    self.hazard(f'P of tile {x} stored over S of tile {sb[0]}')
                sb[1] += 1
            elif op == 'p_consume':
                if sb[0] != x or sb[1] != 16:
                    self.hazard(f'O product reads P of tile {x} from {sb[:2]}')
                sb[2] = True
            elif op == 's_read':                       # two-CTA form: S read out, then released
                if sb[0] != x:
                    self.hazard(f'S of tile {x} read from a buffer holding tile {sb[0]}')
                sb[1] += 1
                sb[2] = sb[1] == 16
            return
        if kind == 'O':
            if op == 'write' and self.o_readers[cta]:
                self.hazard(f'O of pair {cta} overwritten while the epilogue reads it')
            elif op == 'read_begin':
                self.o_readers[cta].add(x)
            elif op == 'read_end':
                self.o_readers[cta].discard(x)
            return
        rx = self.rx.setdefault(cta, [None, 0, True])
        if op == 'write':
            if self.stage[cta]:
                self.hazard(f'P written into CTA {cta} while its epilogue stages there')
            if rx[0] != x:
                if not rx[2]:
                    self.hazard(f'P of tile {x} overwrites unconsumed tile {rx[0]} in CTA {cta}')
                self.rx[cta] = [x, 1, False]
            else:
                rx[1] += 1
        elif op == 'consume':
            if rx[0] != x or rx[1] != 8:
                self.hazard(f'O product reads tile {x} in CTA {cta} holding {rx[:2]}')
            rx[2] = True
        elif op == 'stage_begin':
            if not rx[2]:
                self.hazard(f'epilogue stages over unconsumed P in CTA {cta}')
            self.stage[cta].add(x)
        elif op == 'stage_end':
            self.stage[cta].discard(x)
            self.rx[cta] = [None, 0, True]


def run(items, seed, give_up_at=None, form='quad', **kw):
    """Runs one random interleaving; returns (status, errors, steps) with
    status 'ok' or 'deadlock'.  A blocked wait gives up whenever nothing else
    can move, and (a spin budget running out) at the first step from
    `give_up_at` on where some wait is blocked."""
    counts, rl = (roles_pair if form == 'pair' else roles)(items, **kw)
    st = _State(counts)
    rng = random.Random(seed)
    gens = {name: g for name, _, g in rl}
    cta_of = {name: c for name, c, _ in rl}
    cur = {name: next(g, None) for name, _, g in rl}

    def step(n, value):
        try:
            cur[n] = gens[n].send(value)
        except StopIteration:
            cur[n] = None

    steps = 0
    while True:
        steps += 1
        live = [n for n in cur if cur[n] is not None]
        if not live:
            return 'ok', st.errors, steps
        rng.shuffle(live)
        blocked_waits = []
        moved = False
        for n in live:
            a = cur[n]
            if a[0] == 'wait':
                if a[2] < 0 or st.ready(a[1], a[2]):
                    step(n, True)
                elif st.abort[cta_of[n]]:
                    step(n, False)
                else:
                    blocked_waits.append(n)
                    continue
            elif a[0] == 'arrive':
                st.arrive(a[1])
                step(n, None)
            elif a[0] in ('nb', 'red'):
                members = st.named[a[1]]
                members.setdefault(n, a[3] if a[0] == 'red' else True)
                if len(members) < a[2]:
                    continue
                step(n, all(members.values()) if a[0] == 'red' else None)
            elif a[0] == 'use':
                st.use(a[1], a[2], a[3])
                step(n, None)
            moved = True
            break
        if blocked_waits and (not moved or (give_up_at is not None and steps >= give_up_at)):
            n = rng.choice(blocked_waits)       # this wait runs out of its budget
            st.abort[cta_of[n]] = True
            give_up_at = None
            step(n, False)
            continue
        if not moved:
            return 'deadlock', st.errors + [f'blocked: {n} at {cur[n]}' for n in sorted(live)], steps
