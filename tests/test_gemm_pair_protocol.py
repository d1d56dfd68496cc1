"""An exhaustive model of the SM-pair GEMM kernel's hand-off protocol.

Two CTAs of a cluster (rank 0, the leader, and rank 1) compute each output tile
together: an M = 256 pair MMA reads operand stage s of both CTAs' shared
memory and writes both CTAs' tensor memory.  In the kernel:

* each CTA's producer waits for its own stage's empty barrier and issues its
  TMA load; the leader also arrives on its own full barrier with the pair's
  expected byte count; every load, the follower's included, completes its
  bytes on the LEADER's full barrier (so the count may go below zero when the
  follower's bytes land before the leader's arrival);
* the leader's MMA thread waits for its full barrier, issues the stage's MMAs
  and commits the empty barrier of both CTAs (one multicast commit), and after
  a tile's last stage the accumulator's full barrier of both CTAs;
* each CTA's epilogue warps wait for their own accumulator-full barrier, read
  their half of the accumulator and arrive on the leader's accumulator-empty
  barrier (count = the epilogue warps of both CTAs).

Every interleaving is explored (loads land in any order, the tensor pipe runs
in issue order, a commit arrives once every earlier operation has completed),
checking that an MMA reads both CTAs' data of its own (tile, k-block), that no
load overwrites a stage an MMA has yet to read, that each CTA's epilogue reads
an accumulator only once every MMA of its tile has run and before any MMA of
the tile two later writes it, and that nothing deadlocks.  Planted mistakes
(each CTA expecting and completing only its own bytes, the leader counting
only its own epilogue warps, a commit that reaches only the leader) show up.
"""

from collections import deque

import pytest


class TxBarrier:
    """An mbarrier with a transaction count: the in-progress phase completes
    when its expected arrivals have arrived and its byte count is zero."""

    __slots__ = ("count", "pending", "tx", "phase")

    def __init__(self, count):
        self.count, self.pending, self.tx, self.phase = count, count, 0, 0

    def key(self):
        return (self.pending, self.tx, self.phase)

    def copy(self):
        c = TxBarrier(self.count)
        c.pending, c.tx, c.phase = self.pending, self.tx, self.phase
        return c

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, expect_tx=0):
        self.tx += expect_tx
        self.pending -= 1
        self._complete()

    def complete_tx(self, n=1):
        self.tx -= n
        self._complete()

    def passed(self, parity):
        return (self.phase & 1) != parity


def explore(n_tiles, k_blocks, stages, epi_warps, mutant=None):
    items = [(t, kb) for t in range(n_tiles) for kb in range(k_blocks)]
    # producer of CTA r: one load per (tile, k-block) into its own stage
    prods = []
    for r in range(2):
        prog = []
        for i, it in enumerate(items):
            s, use = i % stages, i // stages
            prog += [("wait_empty", (s, use))]
            if r == 0:
                prog += [("arrive_expect", s)]
            prog += [("load", (s, it))]
        prods.append(prog)
    # the leader's MMA thread
    mma = []
    i = 0
    for t in range(n_tiles):
        acc, use = t % 2, t // 2
        mma.append(("wait_tempty", (acc, use)))
        for kb in range(k_blocks):
            s, u = i % stages, i // stages
            mma += [("wait_full", (s, u)), ("mma", (s, (t, kb), acc)), ("commit", "empty%d" % s)]
            i += 1
        mma.append(("commit", "tfull%d" % acc))
    # epilogue warps of each CTA
    epi = []
    for t in range(n_tiles):
        acc, use = t % 2, t // 2
        epi += [("wait_tfull", (acc, use)), ("read", t), ("arrive_tempty", acc)]

    def fresh():
        b = {}
        for r in range(2):
            for s in range(stages):
                b[(r, "full%d" % s)], b[(r, "empty%d" % s)] = TxBarrier(1), TxBarrier(1)
            for a in range(2):
                drained = epi_warps if mutant == "tempty_local_only" else 2 * epi_warps
                b[(r, "tfull%d" % a)], b[(r, "tempty%d" % a)] = TxBarrier(1), TxBarrier(drained)
        return b

    def clone(bars):
        return {k: v.copy() for k, v in bars.items()}

    W = 2 * epi_warps  # epilogue warps of both CTAs: warp w belongs to CTA w // epi_warps
    # state: producer pcs, mma pc, epilogue pcs, loads in flight (cta, stage, item), tensor pipe,
    # barriers, stage contents per CTA, MMAs executed per tile, epilogue reads per (cta, tile)
    start = ((0, 0), 0, (0,) * W, frozenset(), (), fresh(), ((None,) * stages, (None,) * stages), (0,) * n_tiles,
             ((0,) * n_tiles, (0,) * n_tiles))
    seen, queue, viol = set(), deque([start]), set()
    while queue:
        st = queue.popleft()
        ppcs, mpc, epcs, loads, pipe, bars, sdata, mmas_done, reads = st
        key = (ppcs, mpc, epcs, loads, pipe, tuple(sorted((k, v.key()) for k, v in bars.items())), sdata, mmas_done,
               reads)
        if key in seen:
            continue
        seen.add(key)
        nexts = []
        # producers
        for r in range(2):
            pc = ppcs[r]
            if pc >= len(prods[r]):
                continue
            kind, a = prods[r][pc]
            adv = ppcs[:r] + (pc + 1,) + ppcs[r + 1:]
            if kind == "wait_empty":
                s, use = a
                if bars[(r, "empty%d" % s)].passed((use & 1) ^ 1):
                    nexts.append((adv, mpc, epcs, loads, pipe, bars, sdata, mmas_done, reads))
            elif kind == "arrive_expect":
                nb = clone(bars)
                # both CTAs' bytes (the planted mistake: each CTA for itself)
                nb[(0, "full%d" % a)].arrive(expect_tx=1 if mutant == "follower_own_full" else 2)
                nexts.append((adv, mpc, epcs, loads, pipe, nb, sdata, mmas_done, reads))
            else:
                s, it = a
                nexts.append((adv, mpc, epcs, loads | {(r, s, it)}, pipe, bars, sdata, mmas_done, reads))
        # a load in flight lands (any of them): data into its own CTA, bytes on the leader's barrier
        for ld in loads:
            r, s, it = ld
            nb = clone(bars)
            target = r if mutant == "follower_own_full" else 0
            nb[(target, "full%d" % s)].complete_tx()
            prev = sdata[r][s]
            if prev is not None and prev[1] is False:
                viol.add("load overwrites a stage not yet read")
            row = sdata[r][:s] + ((it, False),) + sdata[r][s + 1:]
            sd = sdata[:r] + (row,) + sdata[r + 1:]
            nexts.append((ppcs, mpc, epcs, loads - {ld}, pipe, nb, sd, mmas_done, reads))
        # the leader's MMA thread
        if mpc < len(mma):
            kind, a = mma[mpc]
            if kind == "wait_tempty":
                acc, use = a
                if bars[(0, "tempty%d" % acc)].passed((use & 1) ^ 1):
                    nexts.append((ppcs, mpc + 1, epcs, loads, pipe, bars, sdata, mmas_done, reads))
            elif kind == "wait_full":
                s, use = a
                if bars[(0, "full%d" % s)].passed(use & 1):
                    nexts.append((ppcs, mpc + 1, epcs, loads, pipe, bars, sdata, mmas_done, reads))
            else:
                nexts.append((ppcs, mpc + 1, epcs, loads, pipe + ((kind, a),), bars, sdata, mmas_done, reads))
        # the tensor pipe completes its oldest operation
        if pipe:
            kind, a = pipe[0]
            nb, sd, md = bars, sdata, mmas_done
            if kind == "mma":
                s, it, acc = a
                t = it[0]
                for r in range(2):
                    if sd[r][s] is None or sd[r][s][0] != it:
                        viol.add("MMA reads the wrong stage data")
                    else:
                        row = sd[r][:s] + ((it, True),) + sd[r][s + 1:]
                        sd = sd[:r] + (row,) + sd[r + 1:]
                if t >= 2 and min(reads[0][t - 2], reads[1][t - 2]) < epi_warps:
                    viol.add("MMA overwrites an accumulator not yet drained")
                md = md[:t] + (md[t] + 1,) + md[t + 1:]
            else:
                nb = clone(bars)
                targets = (0,) if mutant == "commit_leader_only" else (0, 1)
                for r in targets:
                    nb[(r, a)].arrive()
            nexts.append((ppcs, mpc, epcs, loads, pipe[1:], nb, sd, md, reads))
        # epilogue warps
        for w in range(W):
            r = w // epi_warps
            pc = epcs[w]
            if pc >= len(epi):
                continue
            kind, a = epi[pc]
            adv = epcs[:w] + (pc + 1,) + epcs[w + 1:]
            if kind == "wait_tfull":
                acc, use = a
                if bars[(r, "tfull%d" % acc)].passed(use & 1):
                    nexts.append((ppcs, mpc, adv, loads, pipe, bars, sdata, mmas_done, reads))
            elif kind == "read":
                t = a
                if mmas_done[t] != k_blocks:
                    viol.add("epilogue reads an unfinished accumulator")
                if t + 2 < n_tiles and mmas_done[t + 2] > 0:
                    viol.add("epilogue reads an overwritten accumulator")
                row = reads[r][:t] + (reads[r][t] + 1,) + reads[r][t + 1:]
                rd = reads[:r] + (row,) + reads[r + 1:]
                nexts.append((ppcs, mpc, adv, loads, pipe, bars, sdata, mmas_done, rd))
            else:
                nb = clone(bars)
                target = r if mutant == "tempty_local_only" else 0
                nb[(target, "tempty%d" % a)].arrive()
                nexts.append((ppcs, mpc, adv, loads, pipe, nb, sdata, mmas_done, reads))
        done = (all(pc == len(p) for pc, p in zip(ppcs, prods)) and mpc == len(mma) and
                all(p == len(epi) for p in epcs) and not loads and not pipe)
        if not nexts and not done:
            viol.add("deadlock")
        queue.extend(nexts)
    return viol


@pytest.mark.parametrize("n_tiles,k_blocks,stages,epi_warps", [(3, 2, 2, 1), (4, 1, 2, 1), (3, 1, 3, 1),
                                                               (2, 1, 2, 2)])
def test_pair_protocol_is_safe(n_tiles, k_blocks, stages, epi_warps):
    assert explore(n_tiles, k_blocks, stages, epi_warps) == set()


@pytest.mark.parametrize("mutant,expect", [
    ("follower_own_full", "MMA reads the wrong stage data"),
    ("tempty_local_only", "MMA overwrites an accumulator not yet drained"),
    ("commit_leader_only", "deadlock"),
])
def test_planted_pair_mistakes_are_caught(mutant, expect):
    assert expect in explore(3, 1, 2, 1, mutant=mutant)
