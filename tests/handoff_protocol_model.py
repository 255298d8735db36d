"""Model of the synchronisation of the parallel-to-recurrent hand-off kernel
(`final_state.cu`, tensor-core form): test infrastructure, no arithmetic of
the method.

One CTA walks `nu` units (64 tokens of one head) through a ring of `nst` stages;
a piece is a run of units of one head, ending at the head's last chunk or at
the CTA's last unit.  Roles, as in the kernel:
  - three TMA producers fill each stage once it is empty;
  - the MMA issuer adds the stage's product once the V warps have scaled it,
    and at a piece's start waits until the previous piece's epilogue has read
    the accumulator;
  - twelve weighting warps (eight V warps, four n warps) meet at named barrier
    1 for every unit; the V warps scale the stage, the n warps read its K; at a
    piece's end all twelve agree at reducing barrier 4 that the accumulator is
    complete, and the V warps run the epilogue (a named barrier per column
    half) and release the accumulator.
A warp whose wait gives up leaves the unit loop and makes up, in order, barrier
1 of every unit it skipped and barrier 4 (reporting failure) at every piece
end among them; the twelve meet once more at the end (reducing barrier 1).

Steps, scheduler and checks are those of `quad_protocol_model.py`; the buffers
checked here are the stages (a load into a stage that some role still reads)
and the accumulator (a piece's first product while the previous epilogue
reads it).  `mutation` plants one mistake.
"""
import random
from collections import defaultdict


def roles(nu, nchunk, c0, nst, mutation=None):
    counts = {}
    for s in range(nst):
        counts[('Full', s)] = 3                          # the three producers' boxes
        counts[('Scaled', s)] = 8                        # the V warps
        counts[('Empty', s)] = 1 if mutation == 'empty_count' else 1 + 4   # the MMA commit, the n warps
    counts[('AccFull',)] = 1
    counts[('AccEmpty',)] = 8                            # the V warps
    units = [((c0 + i) % nchunk) for i in range(nu)]
    pend = [i == nu - 1 or units[i] == nchunk - 1 for i in range(nu)]
    pstart = [i == 0 or units[i] == 0 for i in range(nu)]

    def producer(q):
        for i in range(nu):
            s, u = i % nst, i // nst
            ok = yield ('wait', ('Empty', s), u - 1)
            if not ok:
                break
            yield ('use', ('stage', s), 'load', (i, q))
            yield ('arrive', ('Full', s))

    def mma():
        piece = 0
        for i in range(nu):
            s, u = i % nst, i // nst
            ok = yield ('wait', ('Scaled', s), u)
            if not ok:
                break
            if pstart[i] and piece > 0:
                ok = yield ('wait', ('AccEmpty',), piece - 1)
                if not ok:
                    break
            yield ('use', ('acc',), 'write' if pstart[i] else 'add', piece)
            yield ('use', ('stage', s), 'mma', i)
            yield ('arrive', ('Empty', s))
            if pend[i]:
                yield ('arrive', ('AccFull',))
                piece += 1

    def weighting(w):
        vw = w < 8
        ok, done, piece = True, 0, 0
        for i in range(nu):
            s, u = i % nst, i // nst
            ok = yield ('wait', ('Full', s), u)
            if not ok:
                break
            yield ('nb', ('bar1', i), 12)
            done += 1
            if vw:
                yield ('use', ('stage', s), 'scale', (i, w))
                yield ('arrive', ('Scaled', s))
            else:
                yield ('use', ('stage', s), 'readk', (i, w))
                yield ('arrive', ('Empty', s))
            if not pend[i]:
                continue
            acc_ok = yield ('wait', ('AccFull',), piece)
            if mutation == 'acc_plain':
                yield ('nb', ('bar4', i), 12)
                ok = acc_ok
            else:
                ok = yield ('red', ('bar4', i), 12, acc_ok)
            if not ok:
                break
            if not vw:
                piece += 1
                continue
            yield ('use', ('acc',), 'read_begin', w)
            yield ('nb', ('half', w // 4, i), 4)
            yield ('use', ('acc',), 'read_end', w)
            yield ('arrive', ('AccEmpty',))
            piece += 1
        if mutation != 'no_debt':
            for j in range(done, nu):
                yield ('nb', ('bar1', j), 12)
                if pend[j] and mutation != 'debt_no_piece':
                    yield ('red', ('bar4', j), 12, False)
        yield ('red', ('final',), 12, ok)

    out = [(f'producer {q}', producer(q)) for q in range(3)]
    out.append(('mma', mma()))
    out += [(f'weighting {w}', weighting(w)) for w in range(12)]
    return counts, out


class _State:
    def __init__(self, counts):
        self.counts = counts
        self.pending = {}
        self.done = defaultdict(int)
        self.named = defaultdict(dict)
        self.abort = False
        self.errors = []
        self.stage = defaultdict(lambda: {'unit': None, 'loads': 0, 'scaled': 0, 'readk': 0, 'mma': False})
        self.acc_readers = set()

    def arrive(self, key):
        c = self.counts[key]
        p = self.pending.get(key, c) - 1
        if p == 0:
            self.done[key] += 1
            p = c
        self.pending[key] = p

    def ready(self, key, k):
        d = self.done[key]
        if not self.abort:
            if d >= k + 2:
                self.errors.append(f'overrun: {key} wanted phase {k}, {d} completed')
            elif d < k and (k - d) % 2 == 1:
                self.errors.append(f'early pass: {key} wanted phase {k}, only {d} completed')
        return d >= k + 1

    def hazard(self, msg):
        if not self.abort:
            self.errors.append('hazard: ' + msg)

    def use(self, buf, op, x):
        if buf[0] == 'acc':
            if op == 'write' and self.acc_readers:
                self.hazard('a piece overwrites the accumulator while the previous epilogue reads it')
            elif op == 'read_begin':
                self.acc_readers.add(x)
            elif op == 'read_end':
                self.acc_readers.discard(x)
            return
        st = self.stage[buf[1]]
        if op == 'load':
            i = x[0]
            if st['unit'] != i:
                if st['unit'] is not None and not (st['scaled'] == 8 and st['readk'] == 4 and st['mma']):
                    self.hazard(f'unit {i} loads into stage {buf[1]} still in use by unit {st["unit"]}')
                st.update(unit=i, loads=0, scaled=0, readk=0, mma=False)
            st['loads'] += 1
        elif op in ('scale', 'readk'):
            if st['unit'] != x[0] or st['loads'] != 3:
                self.hazard(f'unit {x[0]} reads stage {buf[1]} holding unit {st["unit"]} ({st["loads"]} loads)')
            st['scaled' if op == 'scale' else 'readk'] += 1
        elif op == 'mma':
            if st['unit'] != x or st['scaled'] != 8:
                self.hazard(f'unit {x} multiplies stage {buf[1]} before it is scaled')
            st['mma'] = True


def run(nu, nchunk, c0, nst, seed, give_up_at=None, **kw):
    """One random interleaving: (status, errors, steps); a blocked wait gives
    up when nothing else can move, and at the first step from `give_up_at` on
    where some wait is blocked."""
    counts, rl = roles(nu, nchunk, c0, nst, **kw)
    st = _State(counts)
    rng = random.Random(seed)
    gens = dict(rl)
    cur = {name: next(g, None) for name, g in rl}

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
        blocked_waits, moved = [], False
        for n in live:
            a = cur[n]
            if a[0] == 'wait':
                if a[2] < 0 or st.ready(a[1], a[2]):
                    step(n, True)
                elif st.abort:
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
            n = rng.choice(blocked_waits)
            st.abort = True
            give_up_at = None
            step(n, False)
            continue
        if not moved:
            return 'deadlock', st.errors + [f'blocked: {n} at {cur[n]}' for n in sorted(live)], steps
