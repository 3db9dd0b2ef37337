"""A model of the W4A16 decode kernel's barrier protocol (csrc/w4dec.cuh), run on the CPU.

The kernel's roles talk only through mbarriers.  A code producer and an activation producer
fill two rings of shared-memory stages by TMA.  G converter groups take the code stages of
their chunks (chunk q goes to group q % G) and write the decoded weights into their TMEM
slot.  G MMA warps take the activation stages and the slots and accumulate into a pair of
TMEM buffers, and the epilogue drains the buffers.

The model keeps each barrier's arrival count, transaction count and completed phases.  A
wait on parity P passes when the barrier's current phase parity differs from P, as
mbarrier.try_wait.parity does.  Copies land and MMAs complete at random later times (copies
in any order, each MMA warp's commits in issue order), and the roles advance in random
order.  Each read checks that the stage, slot or accumulator holds what the reader expects,
landed and not yet overwritten.  A run must also end with every role done (no deadlock),
and no phase may receive more arrivals than the barrier's count.

The stage and group counts come from w4dec.cuh.  With the counts the kernel uses, no run
reads early.  With the five-stage activation ring that its first build had at G = 3, the
model finds the early read that build showed on the GPU.
"""
import os
import random
import re

import pytest

from protocol_model import Bar, Violation, schedule

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "nvfp4_latentmoe_fwd_02_b300", "csrc", "w4dec.cuh")


def kernel_config(nt):
    """(G, code stages, activation stages) of w4_decode_kernel<nt>, read from its source."""
    text = open(HDR).read()

    def pick(name):
        m = re.search(r"\b" + name + r" = NT == 16 \? (\d+) : (\d+);", text)
        assert m, name
        return int(m.group(1) if nt == 16 else m.group(2))

    return pick("G"), pick("kStagesC"), pick("kStagesA")


def run(G, SC, SA, nch, ntiles, rng):
    """One randomly scheduled run of one CTA over `ntiles` tiles of `nch` chunks each."""
    fullc = [Bar(1) for _ in range(SC)]
    emptyc = [Bar(4) for _ in range(SC)]        # the group's four converter warps
    fulla = [Bar(1) for _ in range(SA)]
    emptya = [Bar(1) for _ in range(SA)]        # the MMA commit
    aready = [Bar(4) for _ in range(G)]
    afree = [Bar(1) for _ in range(G)]
    tfull = [Bar(G) for _ in range(2)]
    tempty = [Bar(4) for _ in range(2)]         # the four epilogue warps
    code, act = [None] * SC, [None] * SA        # stage -> (chunk, landed)
    slot = [None] * G                           # group -> chunk decoded into its TMEM slot
    acc = {}                                    # (group, buffer) -> tile it accumulates
    done = set()                                # chunks whose MMAs completed
    tma, mmaq = [], [[] for _ in range(G)]
    total = nch * ntiles

    def fill(ring, bars, s, q):
        ring[s] = (q, False)
        bars[s].arrive(1, tx=1)

        def land():
            if ring[s] != (q, False):
                raise Violation(f"stage {s} was reissued while chunk {q} was landing")
            ring[s] = (q, True)
            bars[s].complete_tx(1)
        tma.append(land)

    def read(ring, s, q, what):
        if ring[s] != (q, True):
            raise Violation(f"{what} stage {s} read for chunk {q} holds {ring[s]}")

    def takes_part(it, g):
        return any(q % G == g for q in range(it * nch, (it + 1) * nch))

    def code_producer():
        npre = min(SC, nch)                     # the first tile's first ring pass, before the wait
        for q in range(npre):
            fill(code, fullc, q, q)
        for q in range(npre, total):
            s = q % SC
            yield emptyc[s], ((q // SC) & 1) ^ 1
            fill(code, fullc, s, q)

    def act_producer():
        for q in range(total):
            s = q % SA
            yield emptya[s], ((q // SA) & 1) ^ 1
            fill(act, fulla, s, q)

    def converters(g):
        for q in range(g, total, G):
            s = q % SC
            yield fullc[s], (q // SC) & 1
            read(code, s, q, "code")
            emptyc[s].arrive(4)                 # codes in registers: the stage goes back
            yield afree[g], ((q // G) & 1) ^ 1
            slot[g] = q
            aready[g].arrive(4)

    def mma(g):
        for it in range(ntiles):
            a = it & 1
            yield tempty[a], ((it >> 1) & 1) ^ 1
            issued = False
            for q in range(it * nch, (it + 1) * nch):
                if q % G != g:
                    continue
                s = q % SA
                yield fulla[s], (q // SA) & 1
                yield aready[g], (q // G) & 1
                read(act, s, q, "activation")
                if slot[g] != q:
                    raise Violation(f"slot {g} holds chunk {slot[g]} when chunk {q} issues")
                acc[(g, a)] = it
                issued = True

                def complete(q=q, s=s, g=g):
                    read(act, s, q, "activation (MMA in flight)")
                    if slot[g] != q:
                        raise Violation(f"slot {g} rewritten under the MMA of chunk {q}")
                    done.add(q)
                    emptya[s].arrive(1)
                    afree[g].arrive(1)
                mmaq[g].append(complete)
            if issued:
                mmaq[g].append(lambda a=a: tfull[a].arrive(1))
            else:
                tfull[a].arrive(1)

    def epilogue():
        for it in range(ntiles):
            a = it & 1
            yield tfull[a], (it >> 1) & 1
            missing = [q for q in range(it * nch, (it + 1) * nch) if q not in done]
            if missing:
                raise Violation(f"tile {it} read before chunks {missing} completed")
            for g in range(G):
                if takes_part(it, g) and acc.get((g, a)) != it:
                    raise Violation(f"buffer ({g}, {a}) holds tile {acc.get((g, a))}, not {it}")
            tempty[a].arrive(4)

    roles = [code_producer(), act_producer()] + [converters(g) for g in range(G)] + \
            [mma(g) for g in range(G)] + [epilogue()]
    schedule(roles, tma, mmaq, rng)


@pytest.mark.parametrize("nt", [16, 32])
def test_kernel_rings_never_read_early(nt):
    G, SC, SA = kernel_config(nt)
    assert SC % G == 0 and SA % G == 0
    rng = random.Random(nt)
    for nch in (1, 2, 3, 4, 8):
        for ntiles in (1, 2, 5):
            for _ in range(60):
                run(G, SC, SA, nch, ntiles, rng)


def test_model_finds_the_shared_stage_race():
    # the first build: three groups sharing a five-stage activation ring
    G, SC, _ = kernel_config(16)
    rng = random.Random(5)
    found = None
    for _ in range(2000):
        try:
            run(G, SC, 5, 8, 4, rng)
        except Violation as v:
            found = str(v)
            break
    assert found is not None
    assert "activation" in found or "deadlock" in found or "arrivals" in found, found
