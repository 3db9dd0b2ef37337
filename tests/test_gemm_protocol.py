"""A model of the grouped / dense GEMM kernel's barrier protocol (gemm_kernel, csrc/gemm.cuh),
run on the CPU with the building blocks of protocol_model.

Roles, one per warp group of the kernel:
  * the producer fills stage s of the ring by TMA (activations A, weights B; in the NVFP4
    kernel also the scale atoms, on a barrier of their own).  At decode, the weights of the
    first tile's first ring pass go out before the grid-dependency wait, and those stages'
    arrivals count the activation bytes still to come;
  * NVFP4: two copier warps move the A and B scale atoms of a stage into TMEM (tcgen05.cp,
    completed by a commit) and signal the stage's scale barrier;
    W4A16 above decode / fp32 A at decode: two converter warps turn the stage's raw operand into
    the MMA's operand in the same stage and signal that barrier;
  * the MMA warp waits for the stage (and its scales or converted operand), issues, and
    releases the stage by a commit; at a tile's end it commits the accumulator buffer;
  * the epilogue warps wait for the buffer, load it and release it.
Copies land in any order; the MMA warp's and each copier's commits complete in issue order.
Every read checks that the stage, the scales in TMEM or the accumulator hold the expected
k-tile or tile, landed and not yet overwritten; every run must finish.  The stage counts are
those the library launches with (read from lmoe_api.cu); the accumulator count is one for
the 256-column NVFP4 tiles and two otherwise.
"""
import os
import random
import re

import pytest

from protocol_model import Bar, Violation, schedule

API = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "nvfp4_latentmoe_fwd_02_b300", "csrc", "lmoe_api.cu")


def launch_stage_counts():
    text = open(API).read()
    counts = {int(v) for v in re.findall(r"\bkStages\w* = (\d+)", text)}
    assert counts, "no stage constants found"
    return sorted(counts)


def run(stages, ktiles, ntiles, num_acc, mode, preload, rng, skip_scale_wait=False):
    full = [Bar(1) for _ in range(stages)]
    empty = [Bar(1) for _ in range(stages)]          # the MMA commit
    sffull = [Bar(1) for _ in range(stages)]         # NVFP4 scale atoms
    sfready = [Bar(2) for _ in range(stages)]        # two copier / converter warps
    tfull = [Bar(1) for _ in range(num_acc)]
    tempty = [Bar(4) for _ in range(num_acc)]        # the epilogue warps
    stage = [None] * stages                          # s -> dict(key, landed parts)
    sf_tmem = {"A": [None] * stages, "B": [None] * stages}
    conv = [[None] * stages, [None] * stages]        # converter warp -> stage -> key written
    acc = [None] * num_acc
    done = set()
    copies, queues = [], [[], [], []]                # queues: MMA warp, copier A, copier B
    keys = [(it, kt) for it in range(ntiles) for kt in range(ktiles)]
    npre = min(stages, ktiles) if preload else 0
    nvf4 = mode == "nvf4"

    def new_stage(s, key):
        stage[s] = {"key": key, "A": False, "B": False, "sfA": not nvf4, "sfB": not nvf4}

    def issue(s, key, parts, bar):
        for p in parts:
            def land(p=p):
                st = stage[s]
                if st is None or st["key"] != key:
                    raise Violation(f"stage {s} reissued while {p} of {key} was landing")
                st[p] = True
                bar.complete_tx(1)
            copies.append(land)

    def check_stage(s, key, what):
        st = stage[s]
        if st is None or st["key"] != key or not all(st[p] for p in ("A", "B", "sfA", "sfB")):
            raise Violation(f"{what}: stage {s} for {key} holds {st}")

    def producer():
        for i in range(npre):                        # before the grid-dependency wait
            new_stage(i, keys[i])
            if nvf4:
                sffull[i].arrive(1, tx=2)
                issue(i, keys[i], ["sfB"], sffull[i])
            full[i].arrive(1, tx=2)
            issue(i, keys[i], ["B"], full[i])
        for i, key in enumerate(keys):
            s, ph = i % stages, (i // stages) & 1
            yield empty[s], ph ^ 1
            pre = i < npre
            if not pre:
                new_stage(s, key)
            if nvf4:
                if not pre:
                    sffull[s].arrive(1, tx=2)
                issue(s, key, ["sfA"] if pre else ["sfA", "sfB"], sffull[s])
            if not pre:
                full[s].arrive(1, tx=2)
            issue(s, key, ["A"] if pre else ["A", "B"], full[s])

    def copier(which, qi):
        for i, key in enumerate(keys):
            s, ph = i % stages, (i // stages) & 1
            yield sffull[s], ph
            st = stage[s]
            if st is None or st["key"] != key or not st["sf" + which]:
                raise Violation(f"copier {which}: stage {s} for {key} holds {st}")

            def complete(s=s, key=key):
                st = stage[s]
                if st is None or st["key"] != key:
                    raise Violation(f"scale atoms of stage {s} overwritten under their copy")
                sf_tmem[which][s] = key
                sfready[s].arrive(1)
            queues[qi].append(complete)

    def converter(w):
        for i, key in enumerate(keys):
            s, ph = i % stages, (i // stages) & 1
            yield full[s], ph
            check_stage(s, key, f"converter {w}")
            conv[w][s] = key
            sfready[s].arrive(1)

    def mma():
        for it in range(ntiles):
            a = it & 1 if num_acc == 2 else 0
            aph = ((it >> 1) & 1) if num_acc == 2 else (it & 1)
            yield tempty[a], aph ^ 1
            for kt in range(ktiles):
                i, key = it * ktiles + kt, (it, kt)
                s, ph = i % stages, (i // stages) & 1
                yield full[s], ph
                if mode != "plain" and not skip_scale_wait:
                    yield sfready[s], ph
                check_stage(s, key, "MMA")
                if nvf4 and (sf_tmem["A"][s] != key or sf_tmem["B"][s] != key):
                    raise Violation(f"MMA of {key}: scales in TMEM are {sf_tmem['A'][s]}, {sf_tmem['B'][s]}")
                if mode == "conv" and (conv[0][s] != key or conv[1][s] != key):
                    raise Violation(f"MMA of {key}: converted operand is {conv[0][s]}, {conv[1][s]}")
                acc[a] = it

                def complete(s=s, key=key):
                    check_stage(s, key, "MMA in flight")
                    if nvf4 and (sf_tmem["A"][s] != key or sf_tmem["B"][s] != key):
                        raise Violation(f"scales of {key} overwritten under its MMA")
                    done.add(key)
                    empty[s].arrive(1)
                queues[0].append(complete)
            queues[0].append(lambda a=a: tfull[a].arrive(1))

    def epilogue():
        for it in range(ntiles):
            a = it & 1 if num_acc == 2 else 0
            aph = ((it >> 1) & 1) if num_acc == 2 else (it & 1)
            yield tfull[a], aph
            missing = [kt for kt in range(ktiles) if (it, kt) not in done]
            if missing or acc[a] != it:
                raise Violation(f"tile {it} read with k-tiles {missing} outstanding, buffer holds {acc[a]}")
            tempty[a].arrive(4)

    roles = [producer(), mma(), epilogue()]
    if nvf4:
        roles += [copier("A", 1), copier("B", 2)]
    elif mode == "conv":
        roles += [converter(0), converter(1)]
    schedule(roles, copies, queues, rng)


@pytest.mark.parametrize("mode", ["nvf4", "conv", "plain"])
def test_gemm_pipeline_never_reads_early(mode):
    rng = random.Random({"nvf4": 1, "conv": 2, "plain": 3}[mode])
    for stages in launch_stage_counts():
        for num_acc in (1, 2):
            for preload in (False, True):
                for ktiles in (1, 3, 8):
                    for ntiles in (1, 4):
                        for _ in range(8):
                            run(stages, ktiles, ntiles, num_acc, mode, preload, rng)


def test_model_catches_an_mma_that_skips_the_scale_barrier():
    rng = random.Random(3)
    found = None
    for _ in range(500):
        try:
            run(4, 8, 4, 2, "nvf4", True, rng, skip_scale_wait=True)
        except Violation as v:
            found = str(v)
            break
    assert found is not None and "scales" in found, found
