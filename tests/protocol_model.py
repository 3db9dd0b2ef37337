"""Building blocks of the CPU models of the kernels' barrier protocols (test infrastructure).

An mbarrier completes a phase when its arrival count and its transaction count both reach
zero; a wait on parity P passes while the barrier's current phase parity differs from P, as
mbarrier.try_wait.parity does.  `schedule` runs roles (generators that yield the
(barrier, parity) they wait on) together with asynchronous events: copies that may land in
any order, and per-issuer queues of tensor-core completions that finish in issue order.  At
each step it picks at random among the roles whose wait has passed and the events that may
happen next.
"""


class Violation(Exception):
    pass


class Bar:
    """An mbarrier: `count` arrivals and a zero transaction count complete a phase."""

    def __init__(self, count):
        self.count, self.pending, self.tx, self.done = count, count, 0, 0

    def arrive(self, n=1, tx=0):
        self.tx += tx
        self.pending -= n
        if self.pending < 0:
            raise Violation("more arrivals than the barrier's count in one phase")
        self._step()

    def complete_tx(self, n):
        self.tx -= n
        self._step()

    def _step(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count

    def passed(self, parity):
        return (self.done & 1) != parity


def schedule(roles, copies, queues, rng):
    """Run `roles` to completion.  copies: list of pending landings (callables, any order);
    queues: lists of pending completions (callables), each finishing in order."""
    waits = [None] * len(roles)

    def advance(i):
        try:
            waits[i] = next(roles[i])
        except StopIteration:
            waits[i] = "done"

    for i in range(len(roles)):
        advance(i)
    while True:
        cands = [("role", i) for i, w in enumerate(waits) if w != "done" and w[0].passed(w[1])]
        cands += [("copy", k) for k in range(len(copies))]
        cands += [("queue", k) for k, q in enumerate(queues) if q]
        if not cands:
            if all(w == "done" for w in waits):
                return
            raise Violation("deadlock: every role waits and nothing is in flight")
        kind, k = rng.choice(cands)
        if kind == "role":
            advance(k)
        elif kind == "copy":
            copies.pop(k)()
        else:
            queues[k].pop(0)()
