"""An exhaustive model of the prefill attention kernel's hand-off protocol.

The kernel's MMA thread and softmax warps pass tiles through mbarriers: the
MMA thread issues S(j) into TMEM buffer j % 2, the softmax warps wait for it,
write P(j) over it and arrive at a P-ready barrier, and the MMA thread then
issues P V(j); O is read once every P V has completed.  This module models
that protocol: mbarriers with expected counts, phases and parity waits (a
parity wait passes when the in-progress phase's parity differs from the one
asked for), an in-order tensor pipe in which a commit arrives once every
earlier operation has completed, one MMA thread and two softmax warps.  It
explores every interleaving, with and without the rescale of O a softmax warp
makes when a row maximum grows (it waits for P V(j-1) by parity on o_done),
and checks that P V(j) only ever reads a complete P(j), that O is rescaled
only after P V(j-1) and read only after the last P V, and that nothing
deadlocks.

It pins the reasoning behind the kernel's barriers:
* one P-ready barrier for all tiles lets a warp that finished tile j run
  through tile j+1 and arrive again before the other warp arrived for tile j,
  so tile j's phase completes with P(j) incomplete (and a later phase can be
  left an arrival short);
* waiting for the last P V by parity on the per-tile o_done barrier lets a
  warp that finished the last tile early pass while P V of the tile before is
  pending;
* one P-ready barrier per S buffer and the final read after the once-only
  drain barrier are safe in every interleaving (and neither fix alone is).
"""

from collections import deque

import pytest


class Barrier:
    """An mbarrier: `count` arrivals complete the in-progress phase."""

    __slots__ = ("count", "pending", "phase")

    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def key(self):
        return (self.pending, self.phase)

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def passed(self, parity):
        # try_wait.parity: the phase with this parity has completed when the
        # in-progress phase has the other parity
        return (self.phase & 1) != parity


def explore(n_tiles, per_buffer_p, final_on_drain, warps=2):
    """Every interleaving of the protocol; returns the set of violations seen."""
    # programs: lists of steps; a step is (kind, args)
    mma = [("issue_s", 0)]
    for j in range(n_tiles):
        if j + 1 < n_tiles:
            mma.append(("issue_s", j + 1))
        mma.append(("wait_p", j))
        mma.append(("issue_pv", j))
    mma.append(("commit_drain", None))
    soft = []
    for j in range(n_tiles):
        soft += [("wait_s", j)]
        if j > 0:  # the rescale of O when a row maximum grows (data-dependent: either branch)
            soft += [("maybe_rescale", j), ("rescale", j)]
        soft += [("write_p", j), ("arrive_p", j)]
    soft += [("wait_final", None), ("read_o", None)]

    def fresh_barriers():
        b = {"s0": Barrier(1), "s1": Barrier(1), "o_done": Barrier(1), "drain": Barrier(1)}
        if per_buffer_p:
            b["p0"], b["p1"] = Barrier(warps), Barrier(warps)
        else:
            b["p"] = Barrier(warps)
        return b

    def p_barrier(j):
        return ("p%d" % (j & 1), (j >> 1) & 1) if per_buffer_p else ("p", j & 1)

    # state: (mma pc, warp pcs, pipe, barriers, written P, completed P V)
    def key(st):
        mpc, wpcs, pipe, bars, written, pv_done = st
        return (mpc, wpcs, pipe, tuple(sorted((k, v.key()) for k, v in bars.items())), written, pv_done)

    def clone_bars(bars):
        out = {}
        for k, v in bars.items():
            c = Barrier(v.count)
            c.pending, c.phase = v.pending, v.phase
            out[k] = c
        return out

    start = (0, (0,) * warps, (), fresh_barriers(), frozenset(), frozenset())
    seen, queue, violations = set(), deque([start]), set()
    while queue:
        st = queue.popleft()
        k = key(st)
        if k in seen:
            continue
        seen.add(k)
        mpc, wpcs, pipe, bars, written, pv_done = st
        nexts = []
        # the MMA thread
        if mpc < len(mma):
            kind, j = mma[mpc]
            if kind == "issue_s":
                nexts.append((mpc + 1, wpcs, pipe + (("S", j), ("commit", "s%d" % (j & 1))), bars, written,
                              pv_done))
            elif kind == "wait_p":
                name, parity = p_barrier(j)
                if bars[name].passed(parity):
                    nexts.append((mpc + 1, wpcs, pipe, bars, written, pv_done))
            elif kind == "issue_pv":
                nexts.append((mpc + 1, wpcs, pipe + (("PV", j), ("commit", "o_done")), bars, written, pv_done))
            elif kind == "commit_drain":
                nexts.append((mpc + 1, wpcs, pipe + (("commit", "drain"),), bars, written, pv_done))
        # the tensor pipe completes its oldest operation
        if pipe:
            op, arg = pipe[0]
            nb, nw, npv = bars, written, pv_done
            if op == "PV":
                if any((arg, w) not in written for w in range(warps)):
                    violations.add("P V reads an incomplete P")
                npv = pv_done | {arg}
            elif op == "commit":
                nb = clone_bars(bars)
                nb[arg].arrive()
            nexts.append((mpc, wpcs, pipe[1:], nb, nw, npv))
        # the softmax warps
        for w in range(warps):
            pc = wpcs[w]
            if pc >= len(soft):
                continue
            kind, j = soft[pc]
            adv = wpcs[:w] + (pc + 1,) + wpcs[w + 1:]
            if kind == "wait_s":
                if bars["s%d" % (j & 1)].passed((j >> 1) & 1):
                    nexts.append((mpc, adv, pipe, bars, written, pv_done))
            elif kind == "maybe_rescale":
                nexts.append((mpc, adv, pipe, bars, written, pv_done))  # rescale
                nexts.append((mpc, wpcs[:w] + (pc + 2,) + wpcs[w + 1:], pipe, bars, written, pv_done))  # skip
            elif kind == "rescale":
                # waits for P V(j-1) by parity on o_done, then reads and writes O
                if bars["o_done"].passed((j - 1) & 1):
                    if (j - 1) not in pv_done:
                        violations.add("O rescaled before P V(j-1)")
                    nexts.append((mpc, adv, pipe, bars, written, pv_done))
            elif kind == "write_p":
                if j >= 2 and (j - 2) not in pv_done:
                    violations.add("P overwrites a P not yet read")
                nexts.append((mpc, adv, pipe, bars, written | {(j, w)}, pv_done))
            elif kind == "arrive_p":
                nb = clone_bars(bars)
                nb[p_barrier(j)[0]].arrive()
                nexts.append((mpc, adv, pipe, nb, written, pv_done))
            elif kind == "wait_final":
                ok = bars["drain"].passed(0) if final_on_drain else bars["o_done"].passed((n_tiles - 1) & 1)
                if ok:
                    nexts.append((mpc, adv, pipe, bars, written, pv_done))
            elif kind == "read_o":
                if len(pv_done) != n_tiles:
                    violations.add("O read before the last P V")
                nexts.append((mpc, adv, pipe, bars, written, pv_done))
        if not nexts and not (mpc == len(mma) and all(pc == len(soft) for pc in wpcs) and not pipe):
            violations.add("deadlock")
        queue.extend(nexts)
    return violations


@pytest.mark.parametrize("n_tiles,warps", [(3, 2), (4, 2), (5, 2), (3, 3)])
def test_per_buffer_p_ready_and_drain_final_wait_are_safe(n_tiles, warps):
    # the protocol the kernel uses
    assert explore(n_tiles, per_buffer_p=True, final_on_drain=True, warps=warps) == set()


def test_one_p_ready_barrier_mixes_tiles():
    # a warp's early arrival completes another tile's phase: P V(j) may read an
    # incomplete P(j), and the shifted count can leave the last phase one
    # arrival short (in the kernel the bounded wait then gives up)
    v = explore(4, per_buffer_p=False, final_on_drain=True)
    assert v == {"P V reads an incomplete P", "deadlock"}


def test_parity_wait_for_the_last_p_v_can_pass_early():
    v = explore(4, per_buffer_p=True, final_on_drain=False)
    assert v == {"O read before the last P V"}


def test_single_tile_is_safe_either_way():
    assert explore(1, per_buffer_p=False, final_on_drain=False) == set()
    assert explore(1, per_buffer_p=True, final_on_drain=True) == set()
