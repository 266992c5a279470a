"""A model of the attention kernel's S/P-buffer protocol, run under random schedules.

Per 64-key tile i the kernel runs three roles in a pipeline over kNSB
tensor-memory S/P buffers (buffer i % kNSB):
  QK issuer (two warps, alternate tiles): waits until PV of tile i - kNSB has
    released the buffer (s_free), issues S(i) = Q K(i)^T, commits s_full;
  softmax (the row warps): waits s_full(i), writes P(i) over S(i), arrives on
    the P-ready barrier;
  PV issuer: waits for P(i), issues O += P(i) V(i), commits s_free(i).
MMAs complete asynchronously, in issue order per issuing thread.

An mbarrier parity wait passes when the barrier's phase count has the other
parity, so a waiter must never fall a full phase behind it.  With one P-ready
barrier for all buffers, the softmax can complete P(i + 1) (it needs only
S(i + 1), that is PV(i + 1 - kNSB)) before the PV issuer has waited for P(i).
The PV issuer's wait for phase i then sees phase i + 2's parity, blocks until
phase i + 2, and every later wait slips a phase: at the end it waits for a
phase that never comes.  With one P-ready barrier per buffer, the softmax of
tile i + kNSB needs S(i + kNSB), whose QK waited for PV(i), so no phase is
skipped.  This test runs both variants under random schedules.
"""
import random


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.done = count, count, 0

    def passes(self, parity):
        return self.done % 2 != parity

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.done += 1
            self.pending = self.count


def simulate(nt, nsb, per_buffer, seed):
    """One random schedule of one CTA over nt tiles.  Returns (finished, errors)."""
    rnd = random.Random(seed)
    s_full = [Barrier(1) for _ in range(nsb)]
    s_free = [Barrier(1) for _ in range(nsb)]
    p_full = [Barrier(1) for _ in range(nsb if per_buffer else 1)]
    queue = {0: [], 1: [], "pv": []}  # MMAs issued, not yet complete, per issuing thread
    buf = [None] * nsb                # what each S/P buffer holds: ("S", i) or ("P", i)
    errors = []

    def qk(par):
        for i in range(par, nt, 2):
            sb = i % nsb
            if i >= nsb:
                yield s_free[sb], ((i // nsb) - 1) & 1
            queue[par].append(("S", i, sb))

    def softmax():
        for i in range(nt):
            sb = i % nsb
            yield s_full[sb], (i // nsb) & 1
            if buf[sb] != ("S", i):
                errors.append(f"softmax of tile {i} read {buf[sb]}")
            buf[sb] = ("P", i)
            if per_buffer:
                p_full[sb].arrive()
            else:
                p_full[0].arrive()

    def pv():
        for i in range(nt):
            sb = i % nsb
            if per_buffer:
                yield p_full[sb], (i // nsb) & 1
            else:
                yield p_full[0], i & 1
            if buf[sb] != ("P", i):
                errors.append(f"PV of tile {i} read {buf[sb]}")
            queue["pv"].append(("PV", i, sb))

    roles = {"qk0": qk(0), "qk1": qk(1), "softmax": softmax(), "pv": pv()}
    waiting = dict.fromkeys(roles)
    finished = set()

    def run_role(name):
        w = waiting[name]
        if w is not None and not w[0].passes(w[1]):
            return False
        waiting[name] = None
        try:
            waiting[name] = next(roles[name])
        except StopIteration:
            finished.add(name)
        return True

    def complete(q):
        if not queue[q]:
            return False
        kind, i, sb = queue[q].pop(0)
        if kind == "S":
            buf[sb] = ("S", i)
            s_full[sb].arrive()
        else:
            s_free[sb].arrive()
        return True

    steps = 0
    while steps < 100000:
        steps += 1
        acts = [("role", n) for n in roles if n not in finished] + [("mma", q) for q in queue]
        rnd.shuffle(acts)
        moved = False
        for kind, x in acts:
            if kind == "role":
                # the PV issuer is sometimes slow to get its turn
                if x == "pv" and rnd.random() < 0.7:
                    continue
                moved = run_role(x)
            else:
                moved = rnd.random() < 0.5 and complete(x)
            if moved:
                break
        if not moved:
            # no random pick moved: try every role and MMA queue in turn
            moved = any(run_role(n) for n in roles if n not in finished) or any(
                complete(q) for q in queue)
        if not moved:
            # nothing can move: done, or a wait that never passes
            return len(finished) == len(roles), errors
    return False, errors


def test_one_p_ready_barrier_per_buffer_is_exact():
    for nsb in (2, 3):
        for nt in (1, 2, 5, 9, 16):
            for seed in range(150):
                ok, errors = simulate(nt, nsb, True, seed)
                assert ok and not errors, (nsb, nt, seed, errors[:2])


def test_a_shared_p_ready_barrier_can_skip_a_phase():
    """With three buffers and one P-ready barrier, some schedule lets the
    softmax run two tiles ahead of the PV issuer's wait, and the PV issuer
    then waits on a phase that has already passed."""
    failures = 0
    for seed in range(300):
        ok, errors = simulate(9, 3, False, seed)
        failures += (not ok) or bool(errors)
    assert failures > 0
