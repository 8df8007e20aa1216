"""A small discrete scheduler for checking mbarrier protocols on the CPU.

Each kernel role (TMA producer, MMA issuer, elementwise warps, ...) is a
Python generator that yields the waits it would make on an mbarrier.  A
seeded random scheduler interleaves the roles with the completion of
asynchronous work: TMA loads (landing in any order), the tensor pipe
(executing its MMAs and commits strictly in issue order) and bulk reductions
(reading shared memory at random times).  Every buffer (a shared-memory slot,
a TMEM region) carries a version tag; every read asserts the tag it expects,
so a write that lands before its reader is done fails, and a state in which
nothing can move is reported as a deadlock.
"""
import random


class Bar:
    """An mbarrier: `count` arrivals plus transaction bytes complete a phase."""

    def __init__(self, name, count):
        self.name, self.count = name, count
        self.arr = self.tx = self.phase = 0

    def arrive(self, n=1, tx=0):
        self.arr += n
        self.tx += tx
        self._check()

    def complete_tx(self, tx):
        self.tx -= tx
        self._check()

    def _check(self):
        assert self.arr <= self.count, (self.name, self.arr)
        if self.arr == self.count and self.tx == 0:
            self.phase += 1
            self.arr = 0

    def done(self, parity):
        """The wait on `parity` passes (the phase of that parity completed)."""
        return (self.phase & 1) != parity


class Engine:
    def __init__(self, seed):
        self.rnd = random.Random(seed)
        self.bars = {}
        self.mem = {}
        self.loads = []     # (resource, tag, barrier)
        self.pipe = []      # ("mma", reads, writes) | ("commit", barrier)
        self.reduces = []   # (resource, tag, group id)
        self.read_done = set()
        self.roles = {}

    def bar(self, name, count):
        self.bars[name] = Bar(name, count)

    def expect(self, res, tag):
        got = self.mem.get(res)
        assert got == tag, f"{res}: expected {tag}, found {got}"

    def load(self, res, tag, bar_name):
        self.loads.append((res, tag, bar_name))

    def mma(self, reads, writes):
        self.pipe.append(("mma", list(reads), list(writes)))

    def commit(self, bar_name):
        self.pipe.append(("commit", bar_name))

    def run(self):
        pending = {name: None for name in self.roles}
        finished = set()

        def ready(act):
            if act is None:
                return True
            if act[0] == "wait":
                return self.bars[act[1]].done(act[2])
            if act[0] == "until":
                return act[1]()
            return True

        while True:
            cands = [("role", n) for n in self.roles if n not in finished and ready(pending[n])]
            if self.loads:
                cands.append(("load", None))
            if self.pipe:
                cands.append(("pipe", None))
            if self.reduces:
                cands.append(("reduce", None))
            if not cands:
                if len(finished) == len(self.roles):
                    return
                stuck = {n: pending[n] for n in self.roles if n not in finished}
                raise AssertionError(f"deadlock: {stuck}")
            kind, name = self.rnd.choice(cands)
            if kind == "role":
                try:
                    pending[name] = next(self.roles[name])
                except StopIteration:
                    finished.add(name)
            elif kind == "load":
                res, tag, b = self.loads.pop(self.rnd.randrange(len(self.loads)))
                self.mem[res] = tag
                self.bars[b].complete_tx(1)
            elif kind == "pipe":
                op = self.pipe.pop(0)
                if op[0] == "mma":
                    for res, tag in op[1]:
                        if callable(tag):
                            tag = tag()
                        self.expect(res, tag)
                    for res, tag in op[2]:
                        self.mem[res] = tag
                else:
                    self.bars[op[1]].arrive(1)
            else:
                i = 0 if self.rnd.random() < 0.7 else self.rnd.randrange(len(self.reduces))
                res, tag, gid = self.reduces.pop(i)
                self.expect(res, tag)
                self.read_done.add(gid)
