"""A model of the indexer kernel's mbarrier protocol, run under random schedules.

The score kernel is warp-specialised: two producers issue TMA copies of the
key blocks of alternate slots into a ring of `stages` buffers (and the first,
at each query-group change, the group's query rows), two MMA issuers take
alternate slots into a ring of
`nacc` tensor-memory accumulators, and epilogue groups drain alternate
accumulators.  Copies land and MMAs complete asynchronously; a commit
arrives once the issuing thread's earlier MMAs are done.  With FP8 keys the
epilogue also quantises each group's query rows (q8full) and reads the key
scales that travel with each stage (sempty releases them).

An mbarrier parity wait passes when the barrier's current phase has the other
parity, so a waiter must never get a full phase ahead of the barrier.  The
kernel sizes each ring as a multiple of the roles that share it, so that a
stage, like an accumulator, always belongs to one issuer and one epilogue
group: two groups with an even number of accumulators, three groups with
six; FP8 stages a multiple of 2 x groups (the epilogue reads their scales).
With two groups, a third group's warps still enter every query group (they
quantise their share of the query rows) but drain nothing.  This test runs
the protocol (as the kernel runs it) under thousands of random
interleavings: with such rings no schedule deadlocks or reads a stale stage,
accumulator or query block; with an odd ring, or accumulators shared between
groups, some schedule does.
"""
import random


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.done = name, count, count, 0, 0

    def passes(self, parity):
        return self.done % 2 != parity

    def arrive(self):
        self.pending -= 1
        if self.pending < 0:
            raise AssertionError(f"{self.name}: more arrivals than the phase expects")
        self._complete()

    def expect_tx(self, n):
        self.tx += n
        self.arrive()

    def land(self, n):
        self.tx -= n
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count


def simulate(slots, stages, nacc, groups, f8, seed, idle=0):
    """One random schedule of one CTA over `slots` ((query group, block)
    pairs); `groups` epilogue groups drain, `idle` more only enter the query
    groups.  Returns (finished, errors)."""
    rnd = random.Random(seed)
    bars = {}

    def bar(name, count):
        bars[name] = Barrier(name, count)

    for i in range(stages):
        bar(f"full{i}", 1)
        bar(f"empty{i}", 1)
        bar(f"sempty{i}", 4)
    for i in range(nacc):
        bar(f"tfull{i}", 1)
        bar(f"tempty{i}", 4)
    bar("qfull", 1)
    bar("qempty", 2)
    bar("q8full", 4 * (groups + idle))
    bar("done0", 1)
    bar("done1", 1)
    copies = []
    mma_queue = {0: [], 1: []}
    mem = {"q": None, "q8": None, "stage": [None] * stages, "acc": [None] * nacc}
    errors = []

    def producer(par):
        st = ph = it = qloads = 0
        loaded = None
        for grp, blk in slots:
            if grp != loaded:
                if par == 0:
                    if qloads:
                        yield "qempty", (qloads - 1) & 1
                    bars["qfull"].expect_tx(1)
                    copies.append(lambda g=grp: (mem.__setitem__("q", g), bars["qfull"].land(1)))
                    qloads += 1
                loaded = grp
            if it % 2 != par:
                it += 1
                st += 1
                if st == stages:
                    st, ph = 0, ph ^ 1
                continue
            if it >= stages:
                yield f"empty{st}", ph ^ 1
                if f8:
                    yield f"sempty{st}", ph ^ 1
            bars[f"full{st}"].expect_tx(1)
            copies.append(lambda s=st, v=(grp, blk): (mem["stage"].__setitem__(s, v),
                                                      bars[f"full{s}"].land(1)))
            it += 1
            st += 1
            if st == stages:
                st, ph = 0, ph ^ 1

    def issuer(par):
        st = ph = it = qn = 0
        loaded = None
        for grp, blk in slots:
            if grp != loaded:
                if qn:
                    mma_queue[par].append(("commit", "qempty"))
                yield ("q8full" if f8 else "qfull"), qn & 1
                qn += 1
                loaded = grp
            acc = it % nacc
            if it % 2 == par:
                if it >= nacc:
                    yield f"tempty{acc}", ((it // nacc) + 1) & 1
                yield f"full{st}", ph
                mma_queue[par] += [("mma", st, acc, (grp, blk)), ("commit", f"empty{st}"),
                                   ("commit", f"tfull{acc}")]
            it += 1
            st += 1
            if st == stages:
                st, ph = 0, ph ^ 1
        mma_queue[par].append(("commit", f"done{par}"))
        yield f"done{par}", 0

    def epilogue(g, w):
        it = qn = st = ph = 0
        seen = None
        for grp, blk in slots:
            if grp != seen:
                if f8:
                    yield "qfull", qn & 1
                    if mem["q"] != grp:
                        errors.append(f"epilogue quantised the query rows of {mem['q']} for {grp}")
                    mem["q8"] = grp
                    bars["q8full"].arrive()
                    yield "q8full", qn & 1
                    qn += 1
                seen = grp
            sst, sph = st, ph
            st += 1
            if st == stages:
                st, ph = 0, ph ^ 1
            if g >= groups or it % groups != g:
                it += 1
                continue
            acc = it % nacc
            yield f"tfull{acc}", (it // nacc) & 1
            if mem["acc"][acc] != (grp, blk):
                errors.append(f"slot {it} drained accumulator {acc} holding {mem['acc'][acc]}")
            if f8:
                yield f"full{sst}", sph
                if mem["stage"][sst] != (grp, blk):
                    errors.append(f"slot {it} read the scales of {mem['stage'][sst]}")
                bars[f"sempty{sst}"].arrive()
            bars[f"tempty{acc}"].arrive()
            it += 1

    roles = {"producer0": producer(0), "producer1": producer(1), "mma0": issuer(0),
             "mma1": issuer(1)}
    for g in range(groups + idle):
        for w in range(4):
            roles[f"epilogue{g}.{w}"] = epilogue(g, w)
    waiting = dict.fromkeys(roles)
    finished = set()

    def run_role(name):
        wait = waiting[name]
        if wait is not None and not bars[wait[0]].passes(wait[1]):
            return False
        waiting[name] = None
        try:
            waiting[name] = next(roles[name])
        except StopIteration:
            finished.add(name)
        return True

    def run_mma(par):
        if not mma_queue[par]:
            return False
        op = mma_queue[par].pop(0)
        if op[0] == "mma":
            _, st, acc, want = op
            if mem["stage"][st] != want:
                errors.append(f"MMA of {want} read stage {st} holding {mem['stage'][st]}")
            q = mem["q8"] if f8 else mem["q"]
            if q != want[0]:
                errors.append(f"MMA of {want} read the query rows of {q}")
            mem["acc"][acc] = want
        else:
            bars[op[1]].arrive()
        return True

    while True:
        actions = ([("role", n) for n in roles if n not in finished] + [("mma", 0), ("mma", 1)] +
                   [("copy", i) for i in range(len(copies))])
        rnd.shuffle(actions)
        moved = False
        for kind, x in actions:
            if kind == "role":
                moved = run_role(x)
            elif kind == "mma":
                moved = rnd.random() < 0.5 and run_mma(x)
            elif x < len(copies) and rnd.random() < 0.3:
                copies.pop(x)()
                moved = True
            if moved:
                break
        if not moved:
            if copies:
                copies.pop(0)()
            elif not (run_mma(0) or run_mma(1)):
                return len(finished) == len(roles), errors
        if len(finished) == len(roles) and not copies and not any(mma_queue.values()):
            return True, errors


def _slots(seed):
    r = random.Random(seed)
    return ([(0, i) for i in range(r.randint(0, 12))] + [(1, i) for i in range(r.randint(1, 30))]
            + [(2, i) for i in range(r.randint(0, 10))])


def test_even_rings_never_deadlock_or_read_stale_data():
    for stages in (2, 4, 6, 10, 12):
        for nacc in (2, 4):
            for seed in range(120):
                ok, errors = simulate(_slots(seed), stages, nacc, 2, seed % 2 == 1, seed)
                assert ok and not errors, (stages, nacc, seed, errors[:2])


def test_one_epilogue_group_is_safe_too():
    for stages in (4, 6):
        for seed in range(100):
            ok, errors = simulate(_slots(seed), stages, 2, 1, seed % 2 == 1, seed)
            assert ok and not errors, (stages, seed, errors[:2])


def test_an_odd_ring_with_two_epilogue_groups_fails():
    """The failure the even ring rules out: with five stages a stage
    alternates between the issuers, one issuer can get a lap ahead, and its
    parity wait on a stage whose previous load is still in flight passes."""
    failures = 0
    for seed in range(400):
        try:
            ok, errors = simulate(_slots(seed), 5, 4, 2, False, seed)
        except AssertionError:
            ok, errors = False, ["barrier accounting broken"]
        failures += (not ok) or bool(errors)
    assert failures > 0


def test_three_epilogue_groups_with_six_accumulators():
    """Six accumulators (slot s to accumulator s % 6 and group s % 3); FP8
    stage rings a multiple of six, bf16 rings even (the epilogue does not
    read those stages)."""
    for f8, rings in ((True, (6, 12)), (False, (2, 4, 8))):
        for stages in rings:
            for seed in range(100):
                ok, errors = simulate(_slots(seed), stages, 6, 3, f8, seed)
                assert ok and not errors, (f8, stages, seed, errors[:2])


def test_two_draining_groups_and_an_idle_one():
    for stages in (4, 12):
        for seed in range(100):
            ok, errors = simulate(_slots(seed), stages, 4, 2, seed % 2 == 1, seed, idle=1)
            assert ok and not errors, (stages, seed, errors[:2])


def test_accumulators_shared_between_three_groups_fail():
    """Four accumulators and three groups: accumulator s % 4 passes from
    group to group, and a group that runs ahead waits on the parity of a use
    whose predecessor is still pending."""
    failures = 0
    for seed in range(400):
        try:
            ok, errors = simulate(_slots(seed), 4, 4, 3, False, seed)
        except AssertionError:
            ok, errors = False, ["barrier accounting broken"]
        failures += (not ok) or bool(errors)
    assert failures > 0
