"""A small discrete-event simulator for the barrier protocols of the prefill kernels (host logic
only: it runs no kernel). Roles are generators that yield parity waits; mbarriers have arrival
counts and transaction bytes; asynchronous completions (copies, MMA commits) land after random
delays, copies in any order and the MMAs of one issuing thread in issue order. A run fails on
a deadlock, on a wait issued more than one phase ahead of its barrier (a parity wait would
return early), and on a waiter left two phases behind (a parity wait could hang). Models add
their own checks that each buffer holds what its reader expects."""
import random

class Err(Exception):
    pass

class Bar:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending, self.tx, self.done = count, 0, 0
        self.waiters = []  # (role, n)
    def _maybe_complete(self, sim):
        while self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count
            for (role, n) in self.waiters:
                if n <= self.done - 2:
                    raise Err(f"{role.name} waiting {self.name} phase {n} missed it (done={self.done})")
            sim.wake(self)
            break
    def arrive(self, sim, k=1):
        self.pending -= k
        if self.pending < 0:
            raise Err(f"{self.name}: too many arrivals")
        self._maybe_complete(sim)
    def expect_tx(self, sim, b):
        self.tx += b
        self.arrive(sim)
    def complete_tx(self, sim, b):
        self.tx -= b
        self._maybe_complete(sim)

class Role:
    def __init__(self, name, gen):
        self.name, self.gen, self.blocked, self.finished = name, gen, None, False

class Sim:
    def __init__(self, seed):
        self.rng = random.Random(seed)
        self.roles, self.asyncs = [], []
        self.t = 0
        self.seq = 0
    def wake(self, bar):
        pass
    def later(self, fn, lo=1, hi=6, queue=None):
        """An asynchronous completion. Ops of one queue (the MMAs and commits one thread issued)
        complete in issue order; copies complete in any order."""
        self.asyncs.append((self.t + self.rng.randint(lo, hi), fn, queue, self.seq))
        self.seq += 1
    def run(self, max_steps=200000):
        for _ in range(max_steps):
            runnable = [r for r in self.roles if not r.finished and self.ready(r)]
            heads = {}
            for a in self.asyncs:
                if a[2] is not None and (a[2] not in heads or a[3] < heads[a[2]][3]):
                    heads[a[2]] = a
            due = [a for a in self.asyncs if a[2] is None or heads[a[2]] is a]
            if not runnable and not due:
                if all(r.finished for r in self.roles):
                    return
                blocked = [(r.name, r.blocked[0].name, r.blocked[1], r.blocked[0].done) for r in self.roles if not r.finished]
                raise Err(f"deadlock: {blocked[:8]}")
            self.t += 1
            # pick an async op or a role at random
            if due and (not runnable or self.rng.random() < 0.4):
                a = min(due, key=lambda x: x[0] + self.rng.random() * 3)
                self.asyncs.remove(a)
                a[1]()
            else:
                r = self.rng.choice(runnable)
                self.step(r)
        raise Err("too many steps")
    def ready(self, r):
        if r.blocked is None:
            return True
        bar, n = r.blocked
        if bar.done >= n + 1:
            if bar.done > n + 1:
                raise Err(f"{r.name} resumed on {bar.name} phase {n} with done={bar.done} (parity wait would hang)")
            return True
        return False
    def step(self, r):
        if r.blocked is not None:
            bar, n = r.blocked
            bar.waiters.remove((r, n))
            r.blocked = None
        try:
            act = next(r.gen)
        except StopIteration:
            r.finished = True
            return
        if act is None:
            return
        kind, bar, n = act
        assert kind == "wait"
        if bar.done < n:
            raise Err(f"{r.name} waits {bar.name} phase {n} while done={bar.done} (early parity return)")
        if bar.done >= n + 1:
            if bar.done > n + 1:
                raise Err(f"{r.name} waits {bar.name} phase {n} with done={bar.done} (parity wait would hang)")
            return
        r.blocked = (bar, n)
        bar.waiters.append((r, n))

