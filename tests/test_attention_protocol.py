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

A second model adds the K and V shared-memory rings and their TMA producers
(one thread for both, or one each as the kernel runs them), loads landing in
any order: no stage is overwritten before the MMA that reads it completes, S
and P V read the tiles they expect, and the V rows past the context are zeroed
after V lands and before P V reads them.

A third model has the MMAs issued by two threads, as the kernel does: S from
one, P V from the other, each thread's MMAs and commits in its own in-order
queue with no order assumed between the queues.  S(j) then waits for a
per-buffer P V-done barrier (P V(j-2) has completed) before it overwrites the
buffer P(j-2) was written to; without that wait, or with the commit queued
ahead of P V, the model finds S overwriting a P that P V has not read.
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


# ---------------------------------------------------------------------------
# The same protocol with the K and V rings and their TMA producers
# ---------------------------------------------------------------------------


def explore_with_loads(n_tiles, split_producers, warps=2, mistake=None, k_stages=2, v_stages=2, s_bufs=2):
    """Every interleaving of the kernel's protocol including the K and V
    shared-memory rings (k_stages K stages, two V stages) and their producers.
    K(j) goes to stage j % k_stages, V(j) to stage j % 2; a producer waits for
    the stage's empty barrier (parity ((j // stages) & 1) ^ 1), issues the TMA
    load, and the load lands at any later
    point, in any order with the other loads in flight, arriving at the
    stage's full barrier.  The MMA thread waits for K(j)'s full barrier before
    S(j) and frees the K stage by a commit after it; it waits for P(j) and
    V(j) before P V(j) and frees the V stage by a commit after it.  On the last
    tile the softmax warps wait for V's full barrier and zero the V rows past
    the context before they arrive with P.

    split_producers: K from one thread and V from another (the kernel), or
    both from one thread in the order K(0), V(0), K(1), V(1), ...
    s_bufs: S buffers in tensor memory.  With two, S(j+1) is issued before the
    MMA thread waits for P(j); with one (128-key tiles), after P V(j), which
    reads P(j) out of that buffer.
    mistake: plant one error to show the model catches it:
      "no_v_empty_wait"  the V producer does not wait for the stage to be free
      "no_k_empty_wait"  the K producer does not wait for the stage to be free
      "s_ahead"          with one S buffer, S(j+1) issued before P V(j)
      "k_freed_late"     the K stage is freed after P V instead of after S
                         (safe, only slower: no violation expected)
      "no_v_full_wait"   the MMA thread issues P V without waiting for V
      "zero_before_load" the softmax warps zero V rows without waiting for V
    Returns the set of violations seen."""
    last = n_tiles - 1
    mma = [("wait_k", 0), ("issue_s", 0)]
    for j in range(n_tiles):
        if (s_bufs > 1 or mistake == "s_ahead") and j + 1 < n_tiles:
            mma += [("wait_k", j + 1), ("issue_s", j + 1)]
        mma += [("wait_p", j)]
        if mistake != "no_v_full_wait":
            mma += [("wait_v", j)]
        mma += [("issue_pv", j)]
        if s_bufs == 1 and mistake != "s_ahead" and j + 1 < n_tiles:
            mma += [("wait_k", j + 1), ("issue_s", j + 1)]
    mma.append(("commit_drain", None))
    soft = []
    for j in range(n_tiles):
        soft += [("wait_s", j)]
        if j > 0:
            soft += [("maybe_rescale", j), ("rescale", j)]
        soft += [("write_p", j)]
        if j == last:
            if mistake != "zero_before_load":
                soft += [("wait_v_last", j)]
            soft += [("zero_v", j)]
        soft += [("arrive_p", j)]
    soft += [("wait_final", None), ("read_o", None)]

    def prod(kinds):
        out = []
        for j in range(n_tiles):
            for kind in kinds:
                skip_wait = (kind == "V" and mistake == "no_v_empty_wait") or \
                    (kind == "K" and mistake == "no_k_empty_wait")
                if not skip_wait:
                    out.append(("wait_empty", (kind, j)))
                out.append(("load", (kind, j)))
        return out

    producers = [prod("K"), prod("V")] if split_producers else [prod("KV")]

    def fresh_barriers():
        b = {"o_done": Barrier(1), "drain": Barrier(1)}
        for i in range(s_bufs):
            b["s%d" % i], b["p%d" % i] = Barrier(1), Barrier(warps)
        for i in range(v_stages):
            b["vf%d" % i], b["ve%d" % i] = Barrier(1), Barrier(1)
        for i in range(k_stages):
            b["kf%d" % i], b["ke%d" % i] = Barrier(1), Barrier(1)
        return b

    def clone_bars(bars):
        out = {}
        for k, v in bars.items():
            c = Barrier(v.count)
            c.pending, c.phase = v.pending, v.phase
            out[k] = c
        return out

    # state: mma pc, warp pcs, producer pcs, pipe, barriers, loads in flight,
    # K stage contents, V stage contents, P written, S done, P V done, V rows zeroed
    start = (0, (0,) * warps, (0,) * len(producers), (), fresh_barriers(), frozenset(), (None,) * k_stages,
             (None,) * v_stages, frozenset(), frozenset(), frozenset(), frozenset())

    def key(st):
        m, w, pp, pipe, bars, fl, ks, vs, wr, sd, pvd, zr = st
        return (m, w, pp, pipe, tuple(sorted((k, v.key()) for k, v in bars.items())), fl, ks, vs, wr, sd, pvd, zr)

    seen, queue, violations = set(), deque([start]), set()
    while queue:
        st = queue.popleft()
        k = key(st)
        if k in seen:
            continue
        seen.add(k)
        mpc, wpcs, ppcs, pipe, bars, flight, kst, vst, written, s_done, pv_done, zeroed = st
        nexts = []

        def with_(**kw):
            d = dict(mpc=mpc, wpcs=wpcs, ppcs=ppcs, pipe=pipe, bars=bars, flight=flight, kst=kst, vst=vst,
                     written=written, s_done=s_done, pv_done=pv_done, zeroed=zeroed)
            d.update(kw)
            return (d["mpc"], d["wpcs"], d["ppcs"], d["pipe"], d["bars"], d["flight"], d["kst"], d["vst"],
                    d["written"], d["s_done"], d["pv_done"], d["zeroed"])

        # the producers
        for i, prog in enumerate(producers):
            pc = ppcs[i]
            if pc >= len(prog):
                continue
            kind, (kv, j) = prog[pc]
            adv = ppcs[:i] + (pc + 1,) + ppcs[i + 1:]
            n = k_stages if kv == "K" else v_stages
            e = ("ke%d" if kv == "K" else "ve%d") % (j % n)
            if kind == "wait_empty":
                if bars[e].passed(((j // n) & 1) ^ 1):
                    nexts.append(with_(ppcs=adv))
            else:
                nexts.append(with_(ppcs=adv, flight=flight | {(kv, j)}))
        # a load in flight lands (any of them)
        for (kv, j) in flight:
            s = j % (k_stages if kv == "K" else v_stages)
            nb = clone_bars(bars)
            nb[("kf%d" if kv == "K" else "vf%d") % s].arrive()
            if kv == "K":
                if j >= k_stages and (j - k_stages) not in s_done:
                    violations.add("K load overwrites a tile S has not read")
                nexts.append(with_(bars=nb, flight=flight - {(kv, j)}, kst=kst[:s] + (j,) + kst[s + 1:]))
            else:
                if j >= v_stages and (j - v_stages) not in pv_done:
                    violations.add("V load overwrites a tile P V has not read")
                if j == last and zeroed:
                    violations.add("V load lands over the zeroed rows")
                nexts.append(with_(bars=nb, flight=flight - {(kv, j)}, vst=vst[:s] + (j,) + vst[s + 1:]))
        # the MMA thread
        if mpc < len(mma):
            kind, j = mma[mpc]
            s = (j or 0) % s_bufs
            ks = (j or 0) % k_stages
            vs = (j or 0) % v_stages
            if kind == "wait_k":
                if bars["kf%d" % ks].passed((j // k_stages) & 1):
                    nexts.append(with_(mpc=mpc + 1))
            elif kind == "issue_s":
                free_k = () if mistake == "k_freed_late" else (("commit", "ke%d" % ks),)
                nexts.append(with_(mpc=mpc + 1, pipe=pipe + (("S", j), ("commit", "s%d" % s)) + free_k))
            elif kind == "wait_p":
                if bars["p%d" % s].passed((j // s_bufs) & 1):
                    nexts.append(with_(mpc=mpc + 1))
            elif kind == "wait_v":
                if bars["vf%d" % vs].passed((j // v_stages) & 1):
                    nexts.append(with_(mpc=mpc + 1))
            elif kind == "issue_pv":
                free_k = (("commit", "ke%d" % ks),) if mistake == "k_freed_late" else ()
                nexts.append(with_(mpc=mpc + 1, pipe=pipe + (("PV", j), ("commit", "ve%d" % vs), ("commit", "o_done"))
                                   + free_k))
            elif kind == "commit_drain":
                nexts.append(with_(mpc=mpc + 1, pipe=pipe + (("commit", "drain"),)))
        # the tensor pipe completes its oldest operation
        if pipe:
            op, arg = pipe[0]
            if op == "S":
                if kst[arg % k_stages] != arg or any(f == ("K", arg) for f in flight):
                    violations.add("S reads a K stage that does not hold its tile")
                if arg >= s_bufs and (arg - s_bufs) not in pv_done:
                    violations.add("S overwrites a P that P V has not read")
                nexts.append(with_(pipe=pipe[1:], s_done=s_done | {arg}))
            elif op == "PV":
                if any((arg, w) not in written for w in range(warps)):
                    violations.add("P V reads an incomplete P")
                if vst[arg % v_stages] != arg:
                    violations.add("P V reads a V stage that does not hold its tile")
                if arg == last and len(zeroed) != warps:
                    violations.add("P V reads V rows that are not zeroed")
                nexts.append(with_(pipe=pipe[1:], pv_done=pv_done | {arg}))
            else:
                nb = clone_bars(bars)
                nb[arg].arrive()
                nexts.append(with_(pipe=pipe[1:], bars=nb))
        # the softmax warps
        for w in range(warps):
            pc = wpcs[w]
            if pc >= len(soft):
                continue
            kind, j = soft[pc]
            adv = wpcs[:w] + (pc + 1,) + wpcs[w + 1:]
            if kind == "wait_s":
                if bars["s%d" % (j % s_bufs)].passed((j // s_bufs) & 1):
                    nexts.append(with_(wpcs=adv))
            elif kind == "maybe_rescale":
                nexts.append(with_(wpcs=adv))
                nexts.append(with_(wpcs=wpcs[:w] + (pc + 2,) + wpcs[w + 1:]))
            elif kind == "rescale":
                if bars["o_done"].passed((j - 1) & 1):
                    if (j - 1) not in pv_done:
                        violations.add("O rescaled before P V(j-1)")
                    nexts.append(with_(wpcs=adv))
            elif kind == "write_p":
                if j >= s_bufs and (j - s_bufs) not in pv_done:
                    violations.add("P overwrites a P not yet read")
                nexts.append(with_(wpcs=adv, written=written | {(j, w)}))
            elif kind == "wait_v_last":
                if bars["vf%d" % (j % v_stages)].passed((j // v_stages) & 1):
                    nexts.append(with_(wpcs=adv))
            elif kind == "zero_v":
                nexts.append(with_(wpcs=adv, zeroed=zeroed | {w}))
            elif kind == "arrive_p":
                nb = clone_bars(bars)
                nb["p%d" % (j % s_bufs)].arrive()
                nexts.append(with_(wpcs=adv, bars=nb))
            elif kind == "wait_final":
                if bars["drain"].passed(0):
                    nexts.append(with_(wpcs=adv))
            elif kind == "read_o":
                if len(pv_done) != n_tiles:
                    violations.add("O read before the last P V")
                nexts.append(with_(wpcs=adv))
        done = (mpc == len(mma) and all(pc == len(soft) for pc in wpcs) and not pipe and not flight and
                all(pc == len(prog) for pc, prog in zip(ppcs, producers)))
        if not nexts and not done:
            violations.add("deadlock")
        queue.extend(nexts)
    return violations


@pytest.mark.parametrize("n_tiles", [1, 2, 3])
@pytest.mark.parametrize("split", [False, True])
def test_k_and_v_rings_are_safe_with_one_or_two_producers(n_tiles, split):
    # K and V from separate producer threads, or (the earlier form) from one
    assert explore_with_loads(n_tiles, split_producers=split) == set()


@pytest.mark.parametrize("n_tiles", [1, 2, 3, 4])
def test_single_s_buffer_with_one_stage_rings_is_safe(n_tiles):
    # 128-key tiles: one S buffer (S(j+1) after P V(j)), one K and one V stage
    assert explore_with_loads(n_tiles, split_producers=True, k_stages=1, v_stages=1, s_bufs=1) == set()


def test_single_s_buffer_needs_s_after_p_v():
    # issuing S(j+1) ahead of P V(j) into the only buffer would overwrite P(j)
    v = explore_with_loads(3, split_producers=True, k_stages=2, v_stages=1, s_bufs=1, mistake="s_ahead")
    assert "S overwrites a P that P V has not read" in v or "P overwrites a P not yet read" in v


@pytest.mark.parametrize("n_tiles", [2, 4])
def test_three_stage_k_ring_is_safe(n_tiles):
    # the kernel's ring depth is a constant: three K stages (measured slower
    # than two on GB300) and two V stages, separate producers
    assert explore_with_loads(n_tiles, split_producers=True, k_stages=3) == set()



def test_planted_k_ring_mistake_with_three_stages():
    assert "K load overwrites a tile S has not read" in explore_with_loads(
        4, split_producers=True, k_stages=3, mistake="no_k_empty_wait")


@pytest.mark.parametrize("mistake,expected", [
    ("no_v_empty_wait", "V load overwrites a tile P V has not read"),
    ("no_v_full_wait", "P V reads a V stage that does not hold its tile"),
    ("zero_before_load", "V load lands over the zeroed rows"),
])
def test_planted_ring_mistakes_are_caught(mistake, expected):
    # each planted mistake shows up as its own violation (and may cause more)
    assert expected in explore_with_loads(3, split_producers=True, mistake=mistake)


def test_freeing_k_late_is_only_slower():
    assert explore_with_loads(3, split_producers=True, mistake="k_freed_late") == set()


# ---------------------------------------------------------------------------
# Two MMA issuers: S = Q K^T from one warp, P V from another
# ---------------------------------------------------------------------------


def explore_two_issuers(n_tiles, warps=2, s_bufs=2, mistake=None):
    """Every interleaving of the protocol with the MMAs issued by two threads.

    The S thread issues S(j) into buffer j % s_bufs once K(j) has landed and
    P V(j - s_bufs), which read P out of that buffer, has completed (its
    per-buffer P V-done barrier, committed by the P V thread); it frees the K
    stage by a commit.  The P V thread waits for V(j) and P(j), issues P V(j) and commits
    the V stage's empty barrier, o_done, the buffer's P V-done barrier and, after
    the last tile, the drain barrier.  Each thread's MMAs and commits run in its
    own in-order queue, and the two queues progress independently (no order
    between the threads' MMAs is assumed).  K and V come from their own
    producers through two-stage rings, loads landing in any order.

    mistake: plant one error to show the model catches it:
      "no_pv_done_wait"  S(j) issued without waiting for P V(j - s_bufs)
      "pv_done_early"    the P V-done commit queued before P V itself
    Returns the set of violations seen."""
    last, k_stages, v_stages = n_tiles - 1, 2, 2
    s_prog = []
    for j in range(n_tiles):
        s_prog.append(("wait_k", j))
        if j >= s_bufs and mistake != "no_pv_done_wait":
            s_prog.append(("wait_pvd", j))
        s_prog.append(("issue_s", j))
    pv_prog = []
    for j in range(n_tiles):
        pv_prog += [("wait_v", j), ("wait_p", j), ("issue_pv", j)]
    pv_prog.append(("commit_drain", None))
    soft = []
    for j in range(n_tiles):
        soft += [("wait_s", j)]
        if j > 0:
            soft += [("maybe_rescale", j), ("rescale", j)]
        soft += [("write_p", j)]
        if j == last:
            soft += [("wait_v_last", j), ("zero_v", j)]
        soft += [("arrive_p", j)]
    soft += [("wait_final", None), ("read_o", None)]
    producers = []
    for kv in ("K", "V"):
        prog = []
        for j in range(n_tiles):
            prog += [("wait_empty", (kv, j)), ("load", (kv, j))]
        producers.append(prog)

    def fresh_barriers():
        b = {"o_done": Barrier(1), "drain": Barrier(1)}
        for i in range(s_bufs):
            b["s%d" % i], b["p%d" % i], b["pvd%d" % i] = Barrier(1), Barrier(warps), Barrier(1)
        for i in range(2):
            b["vf%d" % i], b["ve%d" % i], b["kf%d" % i], b["ke%d" % i] = Barrier(1), Barrier(1), Barrier(1), Barrier(1)
        return b

    def clone_bars(bars):
        out = {}
        for k, v in bars.items():
            c = Barrier(v.count)
            c.pending, c.phase = v.pending, v.phase
            out[k] = c
        return out

    # state: S pc, P V pc, warp pcs, producer pcs, S queue, P V queue, barriers,
    # loads in flight, K stages, V stages, P written, S done, P V done, V zeroed
    start = (0, 0, (0,) * warps, (0, 0), (), (), fresh_barriers(), frozenset(), (None,) * k_stages,
             (None,) * v_stages, frozenset(), frozenset(), frozenset(), frozenset())
    names = ("spc", "vpc", "wpcs", "ppcs", "qs", "qv", "bars", "flight", "kst", "vst", "written", "s_done",
             "pv_done", "zeroed")

    def key(st):
        return tuple(tuple(sorted((k, v.key()) for k, v in x.items())) if i == 6 else x for i, x in enumerate(st))

    seen, queue, violations = set(), deque([start]), set()
    while queue:
        st = queue.popleft()
        k = key(st)
        if k in seen:
            continue
        seen.add(k)
        cur = dict(zip(names, st))
        bars = cur["bars"]
        nexts = []

        def with_(**kw):
            d = dict(cur)
            d.update(kw)
            return tuple(d[n] for n in names)

        def arrive(name):
            nb = clone_bars(bars)
            nb[name].arrive()
            return nb

        # producers
        for i, prog in enumerate(producers):
            pc = cur["ppcs"][i]
            if pc >= len(prog):
                continue
            kind, (kv, j) = prog[pc]
            adv = cur["ppcs"][:i] + (pc + 1,) + cur["ppcs"][i + 1:]
            e = ("ke%d" if kv == "K" else "ve%d") % (j % 2)
            if kind == "wait_empty":
                if bars[e].passed(((j // 2) & 1) ^ 1):
                    nexts.append(with_(ppcs=adv))
            else:
                nexts.append(with_(ppcs=adv, flight=cur["flight"] | {(kv, j)}))
        # loads land
        for (kv, j) in cur["flight"]:
            s = j % 2
            if kv == "K":
                if j >= 2 and (j - 2) not in cur["s_done"]:
                    violations.add("K load overwrites a tile S has not read")
                nexts.append(with_(bars=arrive("kf%d" % s), flight=cur["flight"] - {(kv, j)},
                                   kst=cur["kst"][:s] + (j,) + cur["kst"][s + 1:]))
            else:
                if j >= 2 and (j - 2) not in cur["pv_done"]:
                    violations.add("V load overwrites a tile P V has not read")
                if j == last and cur["zeroed"]:
                    violations.add("V load lands over the zeroed rows")
                nexts.append(with_(bars=arrive("vf%d" % s), flight=cur["flight"] - {(kv, j)},
                                   vst=cur["vst"][:s] + (j,) + cur["vst"][s + 1:]))
        # the S thread
        if cur["spc"] < len(s_prog):
            kind, j = s_prog[cur["spc"]]
            adv = cur["spc"] + 1
            if kind == "wait_pvd":
                if bars["pvd%d" % (j % s_bufs)].passed(((j - s_bufs) // s_bufs) & 1):
                    nexts.append(with_(spc=adv))
            elif kind == "wait_k":
                if bars["kf%d" % (j % 2)].passed((j // 2) & 1):
                    nexts.append(with_(spc=adv))
            else:
                nexts.append(with_(spc=adv, qs=cur["qs"] + (("S", j), ("commit", "s%d" % (j % s_bufs)),
                                                            ("commit", "ke%d" % (j % 2)))))
        # the P V thread
        if cur["vpc"] < len(pv_prog):
            kind, j = pv_prog[cur["vpc"]]
            adv = cur["vpc"] + 1
            if kind == "wait_p":
                if bars["p%d" % (j % s_bufs)].passed((j // s_bufs) & 1):
                    nexts.append(with_(vpc=adv))
            elif kind == "wait_v":
                if bars["vf%d" % (j % 2)].passed((j // 2) & 1):
                    nexts.append(with_(vpc=adv))
            elif kind == "issue_pv":
                pvd = ("commit", "pvd%d" % (j % s_bufs))
                ops = (("PV", j), ("commit", "ve%d" % (j % 2)), ("commit", "o_done"), pvd)
                if mistake == "pv_done_early":
                    ops = (pvd, ("PV", j), ("commit", "ve%d" % (j % 2)), ("commit", "o_done"))
                nexts.append(with_(vpc=adv, qv=cur["qv"] + ops))
            else:
                nexts.append(with_(vpc=adv, qv=cur["qv"] + (("commit", "drain"),)))
        # either queue completes its oldest operation
        for qn in ("qs", "qv"):
            q = cur[qn]
            if not q:
                continue
            op, arg = q[0]
            if op == "S":
                if cur["kst"][arg % 2] != arg or ("K", arg) in cur["flight"]:
                    violations.add("S reads a K stage that does not hold its tile")
                if arg >= s_bufs and (arg - s_bufs) not in cur["pv_done"]:
                    violations.add("S overwrites a P that P V has not read")
                nexts.append(with_(**{qn: q[1:], "s_done": cur["s_done"] | {arg}}))
            elif op == "PV":
                if any((arg, w) not in cur["written"] for w in range(warps)):
                    violations.add("P V reads an incomplete P")
                if cur["vst"][arg % 2] != arg:
                    violations.add("P V reads a V stage that does not hold its tile")
                if arg == last and len(cur["zeroed"]) != warps:
                    violations.add("P V reads V rows that are not zeroed")
                nexts.append(with_(**{qn: q[1:], "pv_done": cur["pv_done"] | {arg}}))
            else:
                nexts.append(with_(**{qn: q[1:], "bars": arrive(arg)}))
        # softmax warps
        wpcs = cur["wpcs"]
        for w in range(warps):
            pc = wpcs[w]
            if pc >= len(soft):
                continue
            kind, j = soft[pc]
            adv = wpcs[:w] + (pc + 1,) + wpcs[w + 1:]
            if kind == "wait_s":
                if bars["s%d" % (j % s_bufs)].passed((j // s_bufs) & 1):
                    nexts.append(with_(wpcs=adv))
            elif kind == "maybe_rescale":
                nexts.append(with_(wpcs=adv))
                nexts.append(with_(wpcs=wpcs[:w] + (pc + 2,) + wpcs[w + 1:]))
            elif kind == "rescale":
                if bars["o_done"].passed((j - 1) & 1):
                    if (j - 1) not in cur["pv_done"]:
                        violations.add("O rescaled before P V(j-1)")
                    nexts.append(with_(wpcs=adv))
            elif kind == "write_p":
                if j >= s_bufs and (j - s_bufs) not in cur["pv_done"]:
                    violations.add("P overwrites a P not yet read")
                nexts.append(with_(wpcs=adv, written=cur["written"] | {(j, w)}))
            elif kind == "wait_v_last":
                if bars["vf%d" % (j % 2)].passed((j // 2) & 1):
                    nexts.append(with_(wpcs=adv))
            elif kind == "zero_v":
                nexts.append(with_(wpcs=adv, zeroed=cur["zeroed"] | {w}))
            elif kind == "arrive_p":
                nexts.append(with_(wpcs=adv, bars=arrive("p%d" % (j % s_bufs))))
            elif kind == "wait_final":
                if bars["drain"].passed(0):
                    nexts.append(with_(wpcs=adv))
            elif kind == "read_o":
                if len(cur["pv_done"]) != n_tiles:
                    violations.add("O read before the last P V")
                nexts.append(with_(wpcs=adv))
        done = (cur["spc"] == len(s_prog) and cur["vpc"] == len(pv_prog) and all(pc == len(soft) for pc in wpcs)
                and not cur["qs"] and not cur["qv"] and not cur["flight"]
                and all(pc == len(prog) for pc, prog in zip(cur["ppcs"], producers)))
        if not nexts and not done:
            violations.add("deadlock")
        queue.extend(nexts)
    return violations


@pytest.mark.parametrize("n_tiles", [1, 2, 3, 4])
def test_two_mma_issuers_are_safe(n_tiles):
    # the kernel's protocol: S and P V from separate threads, S(j) after P V(j-2) has completed
    assert explore_two_issuers(n_tiles) == set()


@pytest.mark.parametrize("n_tiles", [1, 2, 3])
def test_two_mma_issuers_with_one_s_buffer_are_safe(n_tiles):
    # 128-key tiles: S(j) waits for P V(j-1)
    assert explore_two_issuers(n_tiles, s_bufs=1) == set()


@pytest.mark.parametrize("mistake", ["no_pv_done_wait", "pv_done_early"])
def test_two_mma_issuers_need_the_p_v_done_wait(mistake):
    # without the wait (or with the commit ahead of P V) S(j) can overwrite P(j-2) before P V(j-2) read it
    v = explore_two_issuers(3, mistake=mistake)
    assert "S overwrites a P that P V has not read" in v
