"""The barrier protocol of the sliding prefill kernel (csrc/g4_prefill.cu), modelled on the CPU.

A persistent 2-CTA cluster walks its units in order. Per CTA: warp 0 copies K tiles into a
two-stage ring and each unit's roped Q into its own buffers: dims 0-127 into a staging buffer,
dims 128-255 into one of two buffers by unit parity; unit 0's at the start, unit u + 1's after
unit u's second key tile, once unit u's Q has left the staging buffer. Warp 6 copies V; warp 1
issues QK^T (even CTA) or relays ring landings (odd CTA); warp 7 checks V and issues P.V (even
CTA); eight softmax warps, two per row quarter (one per half of the columns), rotate Q in shared
memory (meeting on a barrier), move dims 0-127 into tensor memory, run the softmax, write P and
the epilogue, and meet their row partner on a barrier of their quarter once per key tile (the
row max) and once per unit (the sums). The model keeps the kernel's barriers, counts and phase
arithmetic, and checks at every MMA and every read that the buffer holds the expected tile or
unit: K slots, the Q buffers, tensor-memory Q, the single S and P buffers, the V stages, O and
the partner's posted half.

The random unit sequences are lists of key-tile counts; a planted mistake (a wait removed) must
make the model fail."""
import random

import pytest

from protocol_sim import Bar, Err, Role, Sim

NK, NV = 2, 2
SMX = 8   # softmax warps per CTA: two per row quarter (w and w + 4 here), one per column half


def model(seed, units, mut=""):
    S = Sim(seed)
    rng = S.rng
    B = {}
    for X in (0, 1):
        d = {}
        for s in range(NK):
            d[f"k_full{s}"] = Bar(f"C{X}.k_full{s}", 1)
            d[f"k_empty{s}"] = Bar(f"C{X}.k_empty{s}", 1)
            d[f"k_peer{s}"] = Bar(f"C{X}.k_peer{s}", 1)
        for s in range(NV):
            d[f"v_full{s}"] = Bar(f"C{X}.v_full{s}", 1)
            d[f"v_empty{s}"] = Bar(f"C{X}.v_empty{s}", 1)
            d[f"v_ready{s}"] = Bar(f"C{X}.v_ready{s}", 1)
        for nm, cnt in (("s_full", 1), ("s_free", 2 * SMX), ("p_full", 2 * SMX), ("pv_done", 1), ("q_full", 1),
                        ("q_pair", 2 * SMX), ("q_free", 1), ("o_free", 2 * SMX), ("q_read", SMX), ("q_rot", SMX)):
            d[nm] = Bar(f"C{X}.{nm}", cnt)
        for q in range(4):
            d[f"xchg{q}"] = Bar(f"C{X}.xchg{q}", 2)
        B[X] = d
    c0s = [0]
    for n in units:
        c0s.append(c0s[-1] + n)
    jt0s = [0]
    for n in units:
        jt0s.append(jt0s[-1] + n)
    # data state
    kring = {X: [None] * NK for X in (0, 1)}       # ("K", jt) landed
    kpend = {X: [0] * NK for X in (0, 1)}          # issued, not yet released
    qlo = {X: None for X in (0, 1)}                # unit whose Q dims 0-127 sit in the staging buffer
    qhi = {X: [None, None] for X in (0, 1)}        # unit whose Q dims 128-255 sit in qhi[0], qhi[1]
    qlo_read = {X: {} for X in (0, 1)}             # unit -> softmax warps that moved their share of qlo
    rots = {X: {} for X in (0, 1)}                 # unit -> softmax warps that rotated their share
    tq = {X: [None] * SMX for X in (0, 1)}         # unit whose Q dims 0-127 each warp's share of tensor memory holds
    sbuf = {X: None for X in (0, 1)}
    sreads = {X: 0 for X in (0, 1)}
    pbuf = {X: None for X in (0, 1)}
    vring = {X: [None] * NV for X in (0, 1)}
    o_own = {X: None for X in (0, 1)}
    o_steps = {X: 0 for X in (0, 1)}
    o_reads = {X: SMX for X in (0, 1)}
    xposted = {}                                   # (CTA, quarter, exchange) -> halves posted
    qk_done_unit = {"last": -1}
    def chk(c, m):
        if not c:
            raise Err(m)
    def producer_k(X):
        def issue_q(ui):
            chk(ui == 0 or qlo_read[X].get(ui - 1, 0) == SMX, f"C{X} Q of unit {ui} over qlo not yet moved")
            chk(qk_done_unit["last"] >= ui - 2, f"C{X} Q of unit {ui} over qhi{ui & 1} still read by unit {ui - 2}'s QK")
            qlo[X] = None
            qhi[X][ui & 1] = None
            B[X]["q_full"].expect_tx(S, 2)
            def land_ql(X=X, ui=ui):
                qlo[X] = ui
                B[X]["q_full"].complete_tx(S, 1)
            def land_qh(X=X, ui=ui):
                qhi[X][ui & 1] = ui
                B[X]["q_full"].complete_tx(S, 1)
            S.later(land_ql, 2, 10)
            S.later(land_qh, 2, 10)
        if units:
            issue_q(0)
        for ui, n in enumerate(units):
            for j in range(n):
                c = c0s[ui] + j
                s = c % NK
                if c >= NK:
                    yield ("wait", B[X][f"k_empty{s}"], c // NK - 1)
                chk(kpend[X][s] == 0, f"C{X} slot {s} reloaded before release")
                kpend[X][s] = 1
                kring[X][s] = None
                jt = jt0s[ui] + j
                B[X][f"k_full{s}"].expect_tx(S, 1)
                def land_k(X=X, s=s, jt=jt):
                    kring[X][s] = ("K", jt)
                    B[X][f"k_full{s}"].complete_tx(S, 1)
                S.later(land_k, 2, 10)
                if ui + 1 < len(units) and j == min(1, n - 1):   # the next unit's Q
                    if mut != "no_qread":
                        yield ("wait", B[X]["q_read"], ui)
                    issue_q(ui + 1)
    def producer_v(X):
        vc = 0
        for ui, n in enumerate(units):
            for i in range(n):
                s = vc % NV
                if vc >= NV:
                    yield ("wait", B[X][f"v_empty{s}"], vc // NV - 1)
                vring[X][s] = None
                B[X][f"v_full{s}"].expect_tx(S, 1)
                def land_v(X=X, s=s, vc=vc):
                    vring[X][s] = vc
                    B[X][f"v_full{s}"].complete_tx(S, 1)
                S.later(land_v, 2, 10)
                vc += 1
    def relay():
        for ui, n in enumerate(units):
            for idx in range(n):
                c = c0s[ui] + idx
                s = c % NK
                yield ("wait", B[1][f"k_full{s}"], c // NK)
                B[0][f"k_peer{s}"].arrive(S)
    def issuer():
        for ui, n in enumerate(units):
            yield ("wait", B[0]["q_pair"], ui)
            for j in range(n):
                jt = jt0s[ui] + j
                c = c0s[ui] + j
                s = c % NK
                yield ("wait", B[0][f"k_full{s}"], c // NK)
                yield ("wait", B[0][f"k_peer{s}"], c // NK)
                if jt > 0 and mut != "no_sfree":
                    yield ("wait", B[0]["s_free"], jt - 1)
                def mma(s=s, jt=jt, ui=ui):
                    for X in (0, 1):
                        chk(kring[X][s] == ("K", jt), f"QK {jt}: C{X} slot {s} holds {kring[X][s]}")
                        chk(all(q == ui for q in tq[X]), f"QK {jt}: C{X} TMEM Q holds units {tq[X]}")
                        chk(qhi[X][ui & 1] == ui, f"QK {jt}: C{X} qhi{ui & 1} holds unit {qhi[X][ui & 1]}")
                        chk(sbuf[X] is None, f"QK {jt}: C{X} S still holds {sbuf[X]}")
                        sbuf[X] = jt
                        sreads[X] = 0
                    for X in (0, 1):
                        kpend[X][s] = 0
                        B[X]["s_full"].arrive(S)
                        B[X][f"k_empty{s}"].arrive(S)
                S.later(mma, 2, 8, queue="qk")
            def qfree(ui=ui):
                qk_done_unit["last"] = ui
                for X in (0, 1):
                    B[X]["q_free"].arrive(S)
            S.later(qfree, 1, 3, queue="qk")
    def vpv(X):
        cv = 0
        for ui, n in enumerate(units):
            for i in range(n):
                jt = jt0s[ui] + i
                s = cv % NV
                yield ("wait", B[X][f"v_full{s}"], cv // NV)
                chk(vring[X][s] == cv, f"C{X} V stage {s} holds {vring[X][s]} not {cv}")
                if X == 1:
                    B[0][f"v_ready{s}"].arrive(S)
                    cv += 1
                    continue
                yield ("wait", B[0]["p_full"], jt)
                yield ("wait", B[0][f"v_ready{s}"], cv // NV)
                if i == 0 and ui > 0 and mut != "no_ofree":
                    yield ("wait", B[0]["o_free"], ui - 1)
                def pv(s=s, cv=cv, jt=jt, i=i, ui=ui):
                    for Y in (0, 1):
                        chk(vring[Y][s] == cv, f"PV {jt}: C{Y} V stage holds {vring[Y][s]}")
                        chk(pbuf[Y] == jt, f"PV {jt}: C{Y} P holds {pbuf[Y]}")
                        if i == 0:
                            chk(o_reads[Y] == SMX, f"PV of unit {ui} overwrites C{Y} O before it is read out")
                            o_own[Y], o_steps[Y], o_reads[Y] = ui, 0, 0
                        else:
                            chk(o_own[Y] == ui, f"PV {jt} of unit {ui} into C{Y} O of {o_own[Y]}")
                        o_steps[Y] += 1
                        pbuf[Y] = ("read", jt)
                    for Y in (0, 1):
                        B[Y]["pv_done"].arrive(S)
                        B[Y][f"v_empty{s}"].arrive(S)
                S.later(pv, 2, 8, queue="pv")
                cv += 1
    pwrites = {}   # (CTA, tile): softmax warps that have written their rows of P
    def softmax(X, w):
        q = w % 4
        xn = [0]   # exchanges of this row quarter so far
        def exchange():
            """Post this half's value, wait for the partner's (the kernel's xchg barrier)."""
            n = xn[0]
            key = (X, q, n)
            xposted[key] = xposted.get(key, 0) + 1
            B[X][f"xchg{q}"].arrive(S)
            if mut != "no_xchg":
                yield ("wait", B[X][f"xchg{q}"], n)
            chk(xposted.get(key, 0) == 2, f"C{X}.w{w} reads its row partner's half of exchange {n} before it was posted")
            xn[0] += 1
        def move_q(ui):
            yield ("wait", B[X]["q_full"], ui)
            chk(qlo[X] == ui and qhi[X][ui & 1] == ui,
                f"C{X}.w{w} rotates Q of unit {ui}: qlo holds {qlo[X]}, qhi{ui & 1} holds {qhi[X][ui & 1]}")
            rots[X][ui] = rots[X].get(ui, 0) + 1
            B[X]["q_rot"].arrive(S)
            if mut != "no_qrot":
                yield ("wait", B[X]["q_rot"], ui)
            chk(rots[X].get(ui, 0) == SMX, f"C{X}.w{w} moves Q of unit {ui} before every warp rotated its share")
            if ui > 0 and mut != "no_qfree":
                yield ("wait", B[X]["q_free"], ui - 1)
            chk(qk_done_unit["last"] >= ui - 1, f"C{X}.w{w} replaces tensor-memory Q while unit {ui - 1}'s QK^T read it")
            chk(qlo[X] == ui, f"C{X}.w{w} moves Q of unit {ui}: qlo holds {qlo[X]}")
            tq[X][w] = ui
            qlo_read[X][ui] = qlo_read[X].get(ui, 0) + 1
            B[0]["q_pair"].arrive(S)
            B[X]["q_read"].arrive(S)
        if not units:
            return
        yield from move_q(0)
        for ui, n in enumerate(units):
            for j in range(n):
                jt = jt0s[ui] + j
                yield ("wait", B[X]["s_full"], jt)
                chk(sbuf[X] == jt, f"C{X}.w{w} reads S holding {sbuf[X]} not {jt}")
                sreads[X] += 1
                if sreads[X] == SMX:
                    sbuf[X] = None
                B[0]["s_free"].arrive(S)
                yield from exchange()   # the row max
                if jt > 0:
                    yield ("wait", B[X]["pv_done"], jt - 1)
                    if j > 0 and rng.random() < 0.5:
                        chk(o_own[X] == ui, f"C{X}.w{w} rescales O of {o_own[X]} in unit {ui}")
                chk(pbuf[X] is None or pbuf[X] == ("read", jt - 1) or pbuf[X] == jt,
                    f"C{X}.w{w} writes P {jt} over {pbuf[X]}")
                key = (X, jt)
                pwrites[key] = pwrites.get(key, 0) + 1
                if pwrites[key] == SMX:
                    pbuf[X] = jt
                B[0]["p_full"].arrive(S)
            if ui + 1 < len(units):
                yield from move_q(ui + 1)
            jl = jt0s[ui] + n - 1
            yield from exchange()   # the halves' sums
            yield ("wait", B[X]["pv_done"], jl)
            chk(o_own[X] == ui and o_steps[X] == n, f"C{X}.w{w} epilogue of unit {ui}: O of {o_own[X]}, {o_steps[X]} steps")
            o_reads[X] += 1
            B[0]["o_free"].arrive(S)
    for X in (0, 1):
        S.roles.append(Role(f"C{X}.prodK", producer_k(X)))
        S.roles.append(Role(f"C{X}.prodV", producer_v(X)))
        S.roles.append(Role(f"C{X}.vpv", vpv(X)))
        for w in range(SMX):
            S.roles.append(Role(f"C{X}.soft{w}", softmax(X, w)))
    S.roles.append(Role("C1.relay", relay()))
    S.roles.append(Role("C0.issuer", issuer()))
    S.run()

def run_many(n, mut="", base=5000):
    failures = []
    for seed in range(n):
        r = random.Random(base + seed)
        units = [r.randint(1, 10) for _ in range(r.randint(1, 6))]
        try:
            model(seed, units, mut)
        except Err as e:
            failures.append((seed, units, str(e)))
    return failures


def test_sliding_protocol_has_no_deadlock_aliasing_or_hazard():
    """300 random unit sequences (1 to 6 units of 1 to 10 key tiles) run to the end with every
    check passing."""
    failures = run_many(300)
    assert not failures, failures[:3]


def test_runs_of_single_tile_units():
    """Units of one key tile in a row (a sequence's first query tiles): the next unit's Q copy
    then follows the unit's only key tile."""
    for seed in range(40):
        model(seed, [1, 1, 1, 2, 1, 1, 3, 1])


@pytest.mark.parametrize("mut", ["no_sfree", "no_qread", "no_xchg", "no_qrot"])
def test_sliding_protocol_model_catches_a_missing_wait(mut):
    """Control: each of these waits guards a hazard the model can see, so removing it fails. (The
    P.V issuer's wait for O to be read out is implied as well by its wait for the next unit's
    first P: the same warps read O out before they write that P, so removing it alone cannot
    fail.)"""
    assert run_many(100, mut)


def test_q_free_before_the_move_is_implied():
    """The softmax warps wait for the earlier unit's QK^T to be done (q_free) before they write the
    next unit's Q into tensor memory. The wait is kept as an explicit guard, but it is implied: the
    same warps read the earlier unit's last S first, which lands only after its last QK^T (and the
    QK^T of one issuer complete in order). So removing it is no hazard."""
    assert not run_many(100, "no_qfree")
