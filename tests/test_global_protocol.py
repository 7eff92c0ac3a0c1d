"""The barrier protocol of the global (K==V) prefill kernel (csrc/g4_prefill_global.cu), modelled
on the CPU.

One unit per 4-CTA cluster. Score CTAs 0-1: warp 0 copies the roped Q (into K stages 1-2 and the
first bytes of the P staging) and the K tiles (3 stages; tiles 1 and 2 wait until Q has moved
into tensor memory); warp 1 issues QK^T (rank 0) or relays ring landings (rank 1); warps 2-5
move Q, run the softmax into one of two S buffers, write P into the staging and copy it to the
output CTA of their head (one P slot of two). Output CTAs 2-3: warp 0 copies V (4 stages); warp 1
checks V and issues P.V (rank 2); warps 2-5 read alpha, rescale O and write the output (a full
tile staged in the V ring once the last P.V is done); warp 6 hands P slots back. The model keeps
the kernel's barriers, counts and phase arithmetic and checks at every MMA and read that the
buffer holds the expected tile. A planted mistake (a wait removed) must make it fail."""
import random

import pytest

from protocol_sim import Bar, Err, Role, Sim

NK, NV, NP = 3, 4, 2


def model(seed, n, mut=""):
    S = Sim(seed)
    rng = S.rng
    sc, oc = {}, {}
    for X in (0, 1):
        d = {}
        for s in range(NK):
            for nm in ("k_full", "k_empty", "k_peer"):
                d[f"{nm}{s}"] = Bar(f"S{X}.{nm}{s}", 1)
        for s in range(NP):
            d[f"s_full{s}"] = Bar(f"S{X}.s_full{s}", 1)
            d[f"s_free{s}"] = Bar(f"S{X}.s_free{s}", 8)
            d[f"p_free{s}"] = Bar(f"S{X}.p_free{s}", 1)
        d["q_full"] = Bar(f"S{X}.q_full", 1)
        d["q_moved"] = Bar(f"S{X}.q_moved", 4)
        d["q_pair"] = Bar(f"S{X}.q_pair", 8)
        d["stg_free"] = Bar(f"S{X}.stg_free", 1)
        sc[X] = d
    for Y in (2, 3):
        d = {}
        for s in range(NV):
            for nm in ("v_full", "v_empty", "v_ready"):
                d[f"{nm}{s}"] = Bar(f"O{Y}.{nm}{s}", 1)
        for s in range(NP):
            d[f"p_full{s}"] = Bar(f"O{Y}.p_full{s}", 1)
            d[f"o_ready{s}"] = Bar(f"O{Y}.o_ready{s}", 8)
            d[f"pv_done{s}"] = Bar(f"O{Y}.pv_done{s}", 1)
        d["ep_staged"] = Bar(f"O{Y}.ep_staged", 4)
        oc[Y] = d
    # data state
    kstage = {X: [None] * NK for X in (0, 1)}
    kpend = {X: [0] * NK for X in (0, 1)}         # tiles issued into the stage, not yet read by QK^T
    qstage = {X: None for X in (0, 1)}            # "Q" once landed, None after it is overwritten
    qmoved = {X: 0 for X in (0, 1)}               # softmax warps that moved their rows of Q
    qtmem = {X: False for X in (0, 1)}
    sbuf = {X: [None] * NP for X in (0, 1)}
    sreads = {}
    stg_busy = {X: 0 for X in (0, 1)}             # P copies in flight from the staging
    stg_tile = {X: None for X in (0, 1)}          # the tile those copies belong to
    pslot = {Y: [None] * NP for Y in (2, 3)}
    pparts = {Y: [0] * NP for Y in (2, 3)}
    vstage = {Y: [None] * NV for Y in (2, 3)}
    o_steps = {Y: 0 for Y in (2, 3)}
    pv_left = {"n": 2 * n}                        # P.V steps not yet executed (both CTAs)

    def chk(c, m):
        if not c:
            raise Err(m)

    def producer(X):
        sc[X]["q_full"].expect_tx(S, 1)

        def land_q(X=X):
            qstage[X] = "Q"
            sc[X]["q_full"].complete_tx(S, 1)
        S.later(land_q, 2, 10)
        for j in range(n):
            s = j % NK
            if j in (1, 2):
                if mut != "no_qmoved":
                    yield ("wait", sc[X]["q_moved"], 0)
            elif j >= NK:
                yield ("wait", sc[X][f"k_empty{s}"], j // NK - 1)
            if s in (1, 2):
                chk(qmoved[X] == 4, f"S{X} K tile {j} over Q not yet moved by every warp")
                qstage[X] = None
            chk(kpend[X][s] == 0, f"S{X} K tile {j} over stage {s} not yet read")
            kpend[X][s] = 1
            kstage[X][s] = None
            sc[X][f"k_full{s}"].expect_tx(S, 1)

            def land_k(X=X, s=s, j=j):
                kstage[X][s] = j
                sc[X][f"k_full{s}"].complete_tx(S, 1)
            S.later(land_k, 2, 10)

    def relay():
        for j in range(n):
            s = j % NK
            yield ("wait", sc[1][f"k_full{s}"], j // NK)
            sc[0][f"k_peer{s}"].arrive(S)

    def issuer():
        yield ("wait", sc[0]["q_pair"], 0)
        for j in range(n):
            s, sb = j % NK, j % NP
            yield ("wait", sc[0][f"k_full{s}"], j // NK)
            yield ("wait", sc[0][f"k_peer{s}"], j // NK)
            if j >= NP and mut != "no_sfree":
                yield ("wait", sc[0][f"s_free{sb}"], (j - NP) // NP)

            def mma(s=s, sb=sb, j=j):
                for X in (0, 1):
                    chk(kstage[X][s] == j, f"QK {j}: S{X} stage {s} holds {kstage[X][s]}")
                    chk(qtmem[X], f"QK {j}: S{X} Q not in tensor memory")
                    chk(sbuf[X][sb] is None, f"QK {j}: S{X} S buffer {sb} still holds {sbuf[X][sb]}")
                    sbuf[X][sb] = j
                for X in (0, 1):
                    kpend[X][s] = 0
                    sc[X][f"s_full{sb}"].arrive(S)
                    sc[X][f"k_empty{s}"].arrive(S)
            S.later(mma, 2, 8, queue="qk")

    def softmax(X, w):
        yield ("wait", sc[X]["q_full"], 0)
        chk(qstage[X] == "Q", f"S{X}.w{w} reads Q staging that holds {qstage[X]}")
        qmoved[X] += 1
        qtmem[X] = True
        sc[X]["q_moved"].arrive(S)
        sc[0]["q_pair"].arrive(S)
        for j in range(n):
            sb = j % NP
            yield ("wait", sc[X][f"s_full{sb}"], j // NP)
            chk(sbuf[X][sb] == j, f"S{X}.w{w} reads S {sb} holding {sbuf[X][sb]}")
            key = (X, j)
            sreads[key] = sreads.get(key, 0) + 1
            if sreads[key] == 4:
                sbuf[X][sb] = None
            sc[0][f"s_free{sb}"].arrive(S)
            if j > 0 and mut != "no_stgfree":
                yield ("wait", sc[X]["stg_free"], j - 1)
            # each warp copies its own rows, so only copies of an earlier tile would clash
            chk(stg_busy[X] == 0 or stg_tile[X] == j, f"S{X}.w{w} writes P {j} into staging still being copied")
            # the staging's first bytes hold the end of Q until every warp of both CTAs moved it
            chk(qmoved[0] == 4 and qmoved[1] == 4, f"S{X}.w{w} writes P over Q not yet moved")
            if j >= NP:
                yield ("wait", sc[X][f"p_free{sb}"], (j - NP) // NP)
            Y = X + 2
            stg_busy[X] += 1
            stg_tile[X] = j

            def land_p(X=X, Y=Y, sb=sb, j=j):
                if pparts[Y][sb] == 0:
                    chk(pslot[Y][sb] is None, f"P {j} lands in O{Y} slot {sb} still holding {pslot[Y][sb]}")
                pparts[Y][sb] += 1
                if pparts[Y][sb] == 4:
                    pslot[Y][sb], pparts[Y][sb] = j, 0
                stg_busy[X] -= 1
                oc[Y][f"p_full{sb}"].complete_tx(S, 1)
            S.later(land_p, 2, 9)

    def vprod(Y):
        for c in range(2 * n):
            s = c % NV
            if c >= NV:
                yield ("wait", oc[Y][f"v_empty{s}"], c // NV - 1)
            vstage[Y][s] = None
            oc[Y][f"v_full{s}"].expect_tx(S, 1)

            def land_v(Y=Y, s=s, c=c):
                vstage[Y][s] = c
                oc[Y][f"v_full{s}"].complete_tx(S, 1)
            S.later(land_v, 2, 10)

    def vcheck(Y):
        for c in range(2 * n):
            s, j, e = c % NV, c // 2, c % 2
            yield ("wait", oc[Y][f"v_full{s}"], c // NV)
            chk(vstage[Y][s] == c, f"O{Y} V stage {s} holds {vstage[Y][s]}")
            if Y == 3:
                oc[2][f"v_ready{s}"].arrive(S)
                continue
            yield ("wait", oc[2][f"v_ready{s}"], c // NV)
            if e == 0 and mut != "no_oready":
                yield ("wait", oc[2][f"o_ready{j % NP}"], j // NP)

            def pv(s=s, c=c, j=j, e=e):
                for Yy in (2, 3):
                    chk(vstage[Yy][s] == c, f"PV {c}: O{Yy} V stage holds {vstage[Yy][s]}")
                    chk(pslot[Yy][j % NP] == j, f"PV {c}: O{Yy} P slot holds {pslot[Yy][j % NP]}")
                    o_steps[Yy] += 1
                pv_left["n"] -= 1
                for Yy in (2, 3):
                    oc[Yy][f"v_empty{s}"].arrive(S)
                    if e == 1:
                        oc[Yy][f"pv_done{j % NP}"].arrive(S)
            S.later(pv, 2, 8, queue="pv")

    def alpha(Y, w):
        for j in range(n):
            sb = j % NP
            yield ("wait", oc[Y][f"p_full{sb}"], j // NP)
            chk(pslot[Y][sb] == j, f"O{Y}.w{w} alpha of tile {j}: slot holds {pslot[Y][sb]}")
            if w == 0 and j + 1 < n:
                sc[Y - 2]["stg_free"].arrive(S)
            if j > 0 and rng.random() < 0.5:
                yield ("wait", oc[Y][f"pv_done{(j - 1) % NP}"], (j - 1) // NP)
                chk(o_steps[Y] == 2 * j, f"O{Y}.w{w} rescales O with {o_steps[Y]} steps in, not {2 * j}")
            oc[2][f"o_ready{sb}"].arrive(S)
        jl = n - 1
        if mut != "no_pvdone_epilogue":
            yield ("wait", oc[Y][f"pv_done{jl % NP}"], jl // NP)
        # the epilogue stages O in the V ring: every P.V must have read its V stage
        chk(pv_left["n"] == 0 and o_steps[Y] == 2 * n, f"O{Y}.w{w} stages O in the V ring with P.V steps pending")
        oc[Y]["ep_staged"].arrive(S)

    def handback(Y):
        for j in range(n):
            yield ("wait", oc[Y][f"pv_done{j % NP}"], j // NP)
            if j + NP < n:
                pslot[Y][j % NP] = None
                oc[Y][f"p_full{j % NP}"].expect_tx(S, 4)
                sc[Y - 2][f"p_free{j % NP}"].arrive(S)

    for Y in (2, 3):
        for s in range(min(NP, n)):
            oc[Y][f"p_full{s}"].expect_tx(S, 4)
    for X in (0, 1):
        S.roles.append(Role(f"S{X}.prod", producer(X)))
        for w in range(4):
            S.roles.append(Role(f"S{X}.soft{w}", softmax(X, w)))
    S.roles.append(Role("S1.relay", relay()))
    S.roles.append(Role("S0.issuer", issuer()))
    for Y in (2, 3):
        S.roles.append(Role(f"O{Y}.vprod", vprod(Y)))
        S.roles.append(Role(f"O{Y}.vcheck", vcheck(Y)))
        for w in range(4):
            S.roles.append(Role(f"O{Y}.alpha{w}", alpha(Y, w)))
        S.roles.append(Role(f"O{Y}.handback", handback(Y)))
    S.run()


def run_many(count, mut="", base=7000):
    failures = []
    for seed in range(count):
        n = random.Random(base + seed).randint(1, 12)
        try:
            model(seed, n, mut)
        except Err as e:
            failures.append((seed, n, str(e)))
    return failures


def test_global_protocol_has_no_deadlock_aliasing_or_hazard():
    """300 random runs (1 to 12 key tiles per unit) end with every check passing."""
    failures = run_many(300)
    assert not failures, failures[:3]


@pytest.mark.parametrize("mut", ["no_qmoved", "no_sfree", "no_stgfree", "no_oready", "no_pvdone_epilogue"])
def test_global_protocol_model_catches_a_missing_wait(mut):
    """Control: each of these waits guards a hazard the model can see, so removing it fails."""
    assert run_many(100, mut)
