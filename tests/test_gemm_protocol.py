"""An exhaustive model of the persistent GEMM kernel's hand-off protocol.

One producer thread fills a ring of operand stages with TMA loads (each load
completes on its own, in any order, and arrives at the stage's full barrier);
one MMA thread waits for a stage, issues the stage's MMAs into one of two
tensor-memory accumulators and commits the stage's empty barrier, and after a
tile's last stage commits the accumulator's full barrier; several epilogue
warps wait for that, read the accumulator and arrive at its empty barrier
(count = the number of epilogue warps).  The tensor pipe runs in issue order
and a commit arrives once every earlier operation has completed.  Every
interleaving is explored, checking that an MMA reads the stage data of its own
(tile, k-block), that no load overwrites a stage an MMA has yet to read, that
the epilogue reads an accumulator only once every MMA of its tile has run and
before any MMA of the tile two later writes it, and that nothing deadlocks.
"""

from collections import deque

import pytest

from tests.test_attention_protocol import Barrier


def explore(n_tiles, k_blocks, stages, epi_warps, mutant=None):
    items = [(t, kb) for t in range(n_tiles) for kb in range(k_blocks)]
    # producer program: one load per (tile, k-block), stage = running index % stages
    prod = []
    for i, it in enumerate(items):
        s, use = i % stages, i // stages
        prod += [("wait_empty", (s, use)), ("load", (s, it))]
    # MMA program
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
    # epilogue program (every warp)
    epi = []
    for t in range(n_tiles):
        acc, use = t % 2, t // 2
        epi += [("wait_tfull", (acc, use)), ("read", t), ("arrive_tempty", acc)]

    def fresh():
        b = {}
        for s in range(stages):
            b["full%d" % s], b["empty%d" % s] = Barrier(1), Barrier(1)
        for a in range(2):
            drained = 1 if mutant == "tempty_count_1" else epi_warps  # arrivals that free an accumulator
            b["tfull%d" % a], b["tempty%d" % a] = Barrier(1), Barrier(drained)
        return b

    def clone(bars):
        out = {}
        for k, v in bars.items():
            c = Barrier(v.count)
            c.pending, c.phase = v.pending, v.phase
            out[k] = c
        return out

    # state: pcs, in-flight loads, tensor pipe, barriers, stage contents,
    # MMAs executed per tile, epilogue reads per tile
    start = (0, 0, (0,) * epi_warps, frozenset(), (), fresh(), (None,) * stages, (0,) * n_tiles, (0,) * n_tiles)
    seen, queue, viol = set(), deque([start]), set()
    while queue:
        st = queue.popleft()
        ppc, mpc, epcs, loads, pipe, bars, stage_data, mmas_done, reads = st
        key = (ppc, mpc, epcs, loads, pipe, tuple(sorted((k, v.key()) for k, v in bars.items())), stage_data,
               mmas_done, reads)
        if key in seen:
            continue
        seen.add(key)
        nexts = []
        # producer
        if ppc < len(prod):
            kind, a = prod[ppc]
            if kind == "wait_empty":
                s, use = a
                if mutant == "no_empty_wait" or bars["empty%d" % s].passed((use & 1) ^ 1):
                    nexts.append((ppc + 1, mpc, epcs, loads, pipe, bars, stage_data, mmas_done, reads))
            else:
                nexts.append((ppc + 1, mpc, epcs, loads | {a}, pipe, bars, stage_data, mmas_done, reads))
        # a load in flight lands (any of them)
        for ld in loads:
            s, it = ld
            nb = clone(bars)
            nb["full%d" % s].arrive()
            # an MMA still to read this stage's previous contents would lose them
            prev = stage_data[s]
            if prev is not None and prev[1] is False:
                viol.add("load overwrites a stage not yet read")
            sd = stage_data[:s] + ((it, False),) + stage_data[s + 1:]
            nexts.append((ppc, mpc, epcs, loads - {ld}, pipe, nb, sd, mmas_done, reads))
        # MMA thread
        if mpc < len(mma):
            kind, a = mma[mpc]
            if kind == "wait_tempty":
                acc, use = a
                if bars["tempty%d" % acc].passed((use & 1) ^ 1):
                    nexts.append((ppc, mpc + 1, epcs, loads, pipe, bars, stage_data, mmas_done, reads))
            elif kind == "wait_full":
                s, use = a
                if bars["full%d" % s].passed(use & 1):
                    nexts.append((ppc, mpc + 1, epcs, loads, pipe, bars, stage_data, mmas_done, reads))
            else:  # mma or commit: into the tensor pipe
                nexts.append((ppc, mpc + 1, epcs, loads, pipe + ((kind, a),), bars, stage_data, mmas_done, reads))
        # the tensor pipe completes its oldest operation
        if pipe:
            kind, a = pipe[0]
            nb, sd, md = bars, stage_data, mmas_done
            if kind == "mma":
                s, it, acc = a
                t = it[0]
                if sd[s] is None or sd[s][0] != it:
                    viol.add("MMA reads the wrong stage data")
                else:
                    sd = sd[:s] + ((it, True),) + sd[s + 1:]
                if t >= 2 and reads[t - 2] < epi_warps:
                    viol.add("MMA overwrites an accumulator not yet drained")
                md = md[:t] + (md[t] + 1,) + md[t + 1:]
            else:
                nb = clone(bars)
                nb[a].arrive()
            nexts.append((ppc, mpc, epcs, loads, pipe[1:], nb, sd, md, reads))
        # epilogue warps
        for w in range(epi_warps):
            pc = epcs[w]
            if pc >= len(epi):
                continue
            kind, a = epi[pc]
            adv = epcs[:w] + (pc + 1,) + epcs[w + 1:]
            if kind == "wait_tfull":
                acc, use = a
                if bars["tfull%d" % acc].passed(use & 1):
                    nexts.append((ppc, mpc, adv, loads, pipe, bars, stage_data, mmas_done, reads))
            elif kind == "read":
                t = a
                if mmas_done[t] != k_blocks:
                    viol.add("epilogue reads an unfinished accumulator")
                if t + 2 < n_tiles and mmas_done[t + 2] > 0:
                    viol.add("epilogue reads an overwritten accumulator")
                rd = reads[:t] + (reads[t] + 1,) + reads[t + 1:]
                nexts.append((ppc, mpc, adv, loads, pipe, bars, stage_data, mmas_done, rd))
            else:
                nb = clone(bars)
                nb["tempty%d" % a].arrive()
                nexts.append((ppc, mpc, adv, loads, pipe, nb, stage_data, mmas_done, reads))
        done = (ppc == len(prod) and mpc == len(mma) and all(p == len(epi) for p in epcs) and not loads
                and not pipe)
        if not nexts and not done:
            viol.add("deadlock")
        queue.extend(nexts)
    return viol


@pytest.mark.parametrize("n_tiles,k_blocks,stages,epi_warps", [(3, 2, 2, 2), (4, 1, 2, 2), (3, 3, 2, 2),
                                                               (3, 2, 3, 3)])
def test_gemm_protocol_is_safe(n_tiles, k_blocks, stages, epi_warps):
    assert explore(n_tiles, k_blocks, stages, epi_warps) == set()


@pytest.mark.parametrize("mutant,expect", [
    ("tempty_count_1", "MMA overwrites an accumulator not yet drained"),
    ("no_empty_wait", "load overwrites a stage not yet read"),
])
def test_planted_protocol_mistakes_are_caught(mutant, expect):
    # the model is not vacuous: a released-too-early accumulator or a producer
    # that does not wait for its stage to drain shows up
    assert expect in explore(3, 2, 2, 2, mutant=mutant)
