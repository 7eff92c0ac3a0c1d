"""The barrier protocol of the persistent global (K==V) prefill kernel (csrc/g4_prefill_global.cu),
modelled on the CPU.

A 4-CTA cluster computes a sequence of units (query tile, head pair), each of some number of key
tiles; every barrier phase continues across units. Score CTAs 0-1: warp 0 copies K tiles into 3
stages (each unit starts at stage 0; its tile 1, and so tile 2, waits until the unit's Q, staged in
stages 1-2, has moved into tensor memory; a unit of one tile waits for nothing of the kind, yet the
warp never runs two phases of that barrier ahead); warp 7 copies each unit's Q once every QK^T of
the earlier unit is done (q_free, committed by the issuer after a unit's last tile); warp 6 of rank 0
waits for each tile's operands (the unit's Q in place, both K halves, the S buffer read) and hands
the tile to the issuer through one of two barriers; warp 1 issues QK^T (rank 0) or relays ring
landings (rank 1); warps 2-5 move Q, run the softmax into one of two S buffers, write P into the
staging and copy it to the output CTA of their head (one P slot of two). Output CTAs 2-3: warp 0
copies V (4 stages); warp 7 of rank 2 (warp 1 of rank 3) checks V and, on rank 2, waits for the
rest of each step's operands (rank 3's half, alpha applied, a unit's first step only once both
CTAs have read the earlier unit's O out) and hands the step to the P.V issuer (warp 1) through the
barrier of its V stage; warps 2-5 read alpha, rescale O and write the output; warp 6 hands P slots
back. The model keeps the kernel's barriers, counts and phase arithmetic and checks at every MMA
and read that the buffer holds what its reader expects. Planted mistakes (a wait removed) must make
it fail."""
import random

import pytest

from protocol_sim import Bar, Err, Role, Sim

NK, NV, NP = 3, 4, 2


def model(seed, units, mut=""):
    S = Sim(seed)
    rng = S.rng
    total = sum(units)
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
        d["q_free"] = Bar(f"S{X}.q_free", 1)
        for b in range(2):
            d[f"go{b}"] = Bar(f"S{X}.go{b}", 1)
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
        d["o_free"] = Bar(f"O{Y}.o_free", 8)
        for s in range(NV):
            d[f"go_pv{s}"] = Bar(f"O{Y}.go_pv{s}", 1)
        oc[Y] = d

    # data state
    kstage = {X: [None] * NK for X in (0, 1)}     # (unit, tile) landed in a K stage, or "Q"
    kpend = {X: [0] * NK for X in (0, 1)}         # copies issued into the stage, not yet read by QK^T
    qland = {X: None for X in (0, 1)}             # unit whose Q has landed in the staging
    qmoved = {X: {} for X in (0, 1)}              # unit -> softmax warps that moved their rows
    qrows = {X: [None] * 4 for X in (0, 1)}       # unit whose Q each warp's rows hold in tensor memory
    qk_pending = {"n": 0}                         # QK^T issued and not yet complete
    qk_done = {"unit": -1}                        # last unit whose QK^T are all complete
    sbuf = {X: [None] * NP for X in (0, 1)}
    sreads = {}
    stg_busy = {X: 0 for X in (0, 1)}             # P copies in flight from the staging
    stg_tile = {X: None for X in (0, 1)}
    pslot = {Y: [None] * NP for Y in (2, 3)}
    pparts = {Y: [0] * NP for Y in (2, 3)}
    vstage = {Y: [None] * NV for Y in (2, 3)}
    ounit = {Y: [None, 0] for Y in (2, 3)}        # unit whose O is accumulating, P.V steps done
    oread = {Y: {} for Y in (2, 3)}               # unit -> epilogue warps that read O out

    def chk(c, m):
        if not c:
            raise Err(m)

    def q_moved_all(X, u):
        return qmoved[X].get(u, 0) == 4

    def producer(X):
        kuse = [0] * NK
        for ui, n in enumerate(units):
            for j in range(n):
                s = j % NK
                if j == 1:
                    if mut != "no_qmoved":
                        yield ("wait", sc[X]["q_moved"], ui)
                elif j != 2 and kuse[s] > 0:
                    yield ("wait", sc[X][f"k_empty{s}"], kuse[s] - 1)
                if s in (1, 2):
                    chk(q_moved_all(X, ui), f"S{X} K tile {ui}.{j} over the Q of unit {ui} not yet moved")
                chk(kpend[X][s] == 0, f"S{X} K tile {ui}.{j} over stage {s} not yet read")
                kpend[X][s] = 1
                kstage[X][s] = None

                def land_k(X=X, s=s, ui=ui, j=j):
                    kstage[X][s] = (ui, j)
                    sc[X][f"k_full{s}"].complete_tx(S, 1)
                sc[X][f"k_full{s}"].expect_tx(S, 1)
                S.later(land_k, 2, 10)
                kuse[s] += 1

    def relay():
        kuse = [0] * NK
        for ui, n in enumerate(units):
            for j in range(n):
                s = j % NK
                yield ("wait", sc[1][f"k_full{s}"], kuse[s])
                sc[0][f"k_peer{s}"].arrive(S)
                kuse[s] += 1

    def helper():
        kuse = [0] * NK
        tc = 0
        for ui, n in enumerate(units):
            yield ("wait", sc[0]["q_pair"], ui)
            for j in range(n):
                s, gt = j % NK, tc + j
                sb = gt % NP
                yield ("wait", sc[0][f"k_full{s}"], kuse[s])
                yield ("wait", sc[0][f"k_peer{s}"], kuse[s])
                if gt >= NP and mut != "no_sfree":
                    yield ("wait", sc[0][f"s_free{sb}"], (gt - NP) // NP)
                sc[0][f"go{gt % 2}"].arrive(S)
                kuse[s] += 1
            tc += n

    def issuer():
        tc = 0
        for ui, n in enumerate(units):
            for j in range(n):
                s, gt = j % NK, tc + j
                sb = gt % NP
                if mut != "no_go":
                    yield ("wait", sc[0][f"go{gt % 2}"], gt // 2)
                qk_pending["n"] += 1

                def mma(s=s, sb=sb, gt=gt, ui=ui, j=j):
                    for X in (0, 1):
                        chk(kstage[X][s] == (ui, j), f"QK {ui}.{j}: S{X} stage {s} holds {kstage[X][s]}")
                        chk(all(q == ui for q in qrows[X]), f"QK {ui}.{j}: S{X} Q rows hold units {qrows[X]}")
                        chk(sbuf[X][sb] is None, f"QK {gt}: S{X} S buffer {sb} still holds {sbuf[X][sb]}")
                        sbuf[X][sb] = gt
                    qk_pending["n"] -= 1
                    for X in (0, 1):
                        kpend[X][s] = 0
                        sc[X][f"s_full{sb}"].arrive(S)
                        sc[X][f"k_empty{s}"].arrive(S)
                S.later(mma, 2, 8, queue="qk")

            def qfree(ui=ui):
                qk_done["unit"] = ui
                for X in (0, 1):
                    sc[X]["q_free"].arrive(S)
            S.later(qfree, 1, 3, queue="qk")   # the commit after the unit's last tile
            tc += n

    def qcopier(X):
        for ui, n in enumerate(units):
            if ui > 0 and mut != "no_qfree":
                yield ("wait", sc[X]["q_free"], ui - 1)
            chk(kpend[X][1] == 0 and kpend[X][2] == 0, f"S{X} Q of unit {ui} over K tiles not yet read")
            chk(qk_done["unit"] >= ui - 1, f"S{X} Q of unit {ui} while unit {ui - 1}'s QK^T still read stages 1-2")
            kstage[X][1] = kstage[X][2] = "Q"

            def land_q(X=X, ui=ui):
                qland[X] = ui
                sc[X]["q_full"].complete_tx(S, 1)
            sc[X]["q_full"].expect_tx(S, 1)
            S.later(land_q, 2, 10)
        if units:
            yield ("wait", sc[X]["q_free"], len(units) - 1)

    def softmax(X, w):
        kq = [0] * NK
        tc = 0
        for ui, n in enumerate(units):
            for j in range(n):
                kq[j % NK] += 1
            yield ("wait", sc[X]["q_full"], ui)
            chk(qland[X] == ui and kstage[X][1] == "Q" and kstage[X][2] == "Q",
                f"S{X}.w{w} moves Q of unit {ui}: staging holds {qland[X]}, {kstage[X][1:]}")
            chk(qk_pending["n"] == 0 or all(q == ui for q in qrows[1 - X]) or qrows[X][w] is None or
                _no_qk_reads(X), f"S{X}.w{w} replaces Q while QK^T reads it")
            qrows[X][w] = ui
            qmoved[X][ui] = qmoved[X].get(ui, 0) + 1
            sc[X]["q_moved"].arrive(S)
            sc[0]["q_pair"].arrive(S)
            for j in range(n):
                gt = tc + j
                sb = gt % NP
                yield ("wait", sc[X][f"s_full{sb}"], gt // NP)
                chk(sbuf[X][sb] == gt, f"S{X}.w{w} reads S {sb} holding {sbuf[X][sb]}, not {gt}")
                key = (X, gt)
                sreads[key] = sreads.get(key, 0) + 1
                if sreads[key] == 4:
                    sbuf[X][sb] = None
                sc[0][f"s_free{sb}"].arrive(S)
                if gt > 0 and mut != "no_stgfree":
                    yield ("wait", sc[X]["stg_free"], gt - 1)
                chk(stg_busy[X] == 0 or stg_tile[X] == gt, f"S{X}.w{w} writes P {gt} into staging still being copied")
                chk(q_moved_all(0, ui) and q_moved_all(1, ui), f"S{X}.w{w} writes P over Q not yet moved")
                if gt >= NP:
                    yield ("wait", sc[X][f"p_free{sb}"], (gt - NP) // NP)
                Y = X + 2
                stg_busy[X] += 1
                stg_tile[X] = gt

                def land_p(X=X, Y=Y, sb=sb, gt=gt):
                    if pparts[Y][sb] == 0:
                        chk(pslot[Y][sb] is None, f"P {gt} lands in O{Y} slot {sb} still holding {pslot[Y][sb]}")
                    pparts[Y][sb] += 1
                    if pparts[Y][sb] == 4:
                        pslot[Y][sb], pparts[Y][sb] = gt, 0
                    stg_busy[X] -= 1
                    oc[Y][f"p_full{sb}"].complete_tx(S, 1)
                S.later(land_p, 2, 9)
            tc += n

    def _no_qk_reads(X):
        return qk_pending["n"] == 0

    def vprod(Y):
        vc = 0
        for ui, n in enumerate(units):
            for c in range(2 * n):
                s = vc % NV
                if vc >= NV:
                    yield ("wait", oc[Y][f"v_empty{s}"], vc // NV - 1)
                vstage[Y][s] = None

                def land_v(Y=Y, s=s, vc=vc):
                    vstage[Y][s] = vc
                    oc[Y][f"v_full{s}"].complete_tx(S, 1)
                oc[Y][f"v_full{s}"].expect_tx(S, 1)
                S.later(land_v, 2, 10)
                vc += 1

    def vcheck(Y):
        vc, tc = 0, 0
        for ui, n in enumerate(units):
            for c in range(2 * n):
                s, j, e = vc % NV, c // 2, c % 2
                gt = tc + j
                yield ("wait", oc[Y][f"v_full{s}"], vc // NV)
                chk(vstage[Y][s] == vc, f"O{Y} V stage {s} holds {vstage[Y][s]}, not {vc}")
                if Y == 3:
                    oc[2][f"v_ready{s}"].arrive(S)
                    vc += 1
                    continue
                yield ("wait", oc[2][f"v_ready{s}"], vc // NV)
                if e == 0 and mut != "no_oready":
                    yield ("wait", oc[2][f"o_ready{gt % NP}"], gt // NP)
                if c == 0 and ui > 0 and mut != "no_ofree":
                    yield ("wait", oc[2]["o_free"], ui - 1)

                oc[2][f"go_pv{s}"].arrive(S)
                vc += 1
            tc += n

    def pv_issuer():
        vc, tc = 0, 0
        for ui, n in enumerate(units):
            for c in range(2 * n):
                s, j, e = vc % NV, c // 2, c % 2
                gt = tc + j
                if mut != "no_gopv":
                    yield ("wait", oc[2][f"go_pv{s}"], vc // NV)

                def pv(s=s, vc=vc, gt=gt, e=e, c=c, ui=ui):
                    for Yy in (2, 3):
                        chk(vstage[Yy][s] == vc, f"PV {vc}: O{Yy} V stage holds {vstage[Yy][s]}")
                        chk(pslot[Yy][gt % NP] == gt, f"PV {vc}: O{Yy} P slot holds {pslot[Yy][gt % NP]}")
                        if c == 0:
                            chk(ui == 0 or oread[Yy].get(ui - 1, 0) == 4,
                                f"PV of unit {ui} overwrites O{Yy} before unit {ui - 1} was read out")
                            ounit[Yy] = [ui, 0]
                        chk(ounit[Yy][0] == ui, f"PV of unit {ui}: O{Yy} holds unit {ounit[Yy][0]}")
                        ounit[Yy][1] += 1
                    for Yy in (2, 3):
                        oc[Yy][f"v_empty{s}"].arrive(S)
                        if e == 1:
                            oc[Yy][f"pv_done{gt % NP}"].arrive(S)
                S.later(pv, 2, 8, queue="pv")
                vc += 1
            tc += n

    def alpha(Y, w):
        tc = 0
        for ui, n in enumerate(units):
            for j in range(n):
                gt = tc + j
                sb = gt % NP
                yield ("wait", oc[Y][f"p_full{sb}"], gt // NP)
                chk(pslot[Y][sb] == gt, f"O{Y}.w{w} alpha of tile {gt}: slot holds {pslot[Y][sb]}")
                if w == 0:
                    sc[Y - 2]["stg_free"].arrive(S)
                if j > 0 and rng.random() < 0.5:
                    yield ("wait", oc[Y][f"pv_done{(gt - 1) % NP}"], (gt - 1) // NP)
                    chk(ounit[Y] == [ui, 2 * j], f"O{Y}.w{w} rescales O of unit {ui} with state {ounit[Y]}")
                oc[2][f"o_ready{sb}"].arrive(S)
            gl = tc + n - 1
            if mut != "no_pvdone_epilogue":
                yield ("wait", oc[Y][f"pv_done{gl % NP}"], gl // NP)
            chk(ounit[Y] == [ui, 2 * n], f"O{Y}.w{w} reads O of unit {ui} out with state {ounit[Y]}")
            oread[Y][ui] = oread[Y].get(ui, 0) + 1
            oc[2]["o_free"].arrive(S)
            tc += n

    def handback(Y):
        for gt in range(total):
            yield ("wait", oc[Y][f"pv_done{gt % NP}"], gt // NP)
            if gt + NP < total:
                pslot[Y][gt % NP] = None
                oc[Y][f"p_full{gt % NP}"].expect_tx(S, 4)
                sc[Y - 2][f"p_free{gt % NP}"].arrive(S)

    for Y in (2, 3):
        for s in range(min(NP, total)):
            oc[Y][f"p_full{s}"].expect_tx(S, 4)
    for X in (0, 1):
        S.roles.append(Role(f"S{X}.prod", producer(X)))
        for w in range(4):
            S.roles.append(Role(f"S{X}.soft{w}", softmax(X, w)))
    S.roles.append(Role("S1.relay", relay()))
    S.roles.append(Role("S0.issuer", issuer()))
    S.roles.append(Role("S0.helper", helper()))
    for X in (0, 1):
        S.roles.append(Role(f"S{X}.qcopy", qcopier(X)))
    S.roles.append(Role("O2.pv_issuer", pv_issuer()))
    for Y in (2, 3):
        S.roles.append(Role(f"O{Y}.vprod", vprod(Y)))
        S.roles.append(Role(f"O{Y}.vcheck", vcheck(Y)))
        for w in range(4):
            S.roles.append(Role(f"O{Y}.alpha{w}", alpha(Y, w)))
        S.roles.append(Role(f"O{Y}.handback", handback(Y)))
    S.run(max_steps=400000)


def unit_mix(seed):
    """1 to 6 units of 1 to 10 key tiles each; one tile is common (a sequence's first query tile)."""
    r = random.Random(seed)
    return [1 if r.random() < 0.35 else r.randint(2, 10) for _ in range(r.randint(1, 6))]


def run_many(count, mut="", base=7000):
    failures = []
    for seed in range(count):
        units = unit_mix(base + seed)
        try:
            model(seed, units, mut)
        except Err as e:
            failures.append((seed, units, str(e)))
    return failures


def test_global_protocol_has_no_deadlock_aliasing_or_hazard():
    """300 random unit sequences end with every check passing."""
    failures = run_many(300)
    assert not failures, failures[:3]


def test_runs_of_single_tile_units():
    """Several units of one tile in a row: the K producer, which waits on no Q move in them, still
    never waits on a phase of that barrier two ahead of the last completed one."""
    for seed in range(40):
        model(seed, [1, 1, 1, 3, 1, 1, 2, 1])


@pytest.mark.parametrize("mut", ["no_qmoved", "no_sfree", "no_stgfree", "no_oready",
                                 "no_pvdone_epilogue", "no_qfree", "no_go", "no_gopv"])
def test_global_protocol_model_catches_a_missing_wait(mut):
    """Control: each of these waits guards a hazard the model can see, so removing it fails."""
    assert run_many(150, mut)


def test_o_free_is_implied_by_the_first_o_ready():
    """The wait on o_free before a unit's first P.V is kept as an explicit guard, but it is also
    implied: the epilogue warps arrive on o_ready for a unit's first tile only after reading the
    earlier unit's O out, and the first P.V waits on that o_ready. So removing it is no hazard."""
    assert not run_many(150, "no_ofree")
