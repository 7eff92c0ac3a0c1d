"""The barrier protocol of the sliding prefill kernel (csrc/g4_prefill.cu), modelled on the CPU.

A persistent 2-CTA cluster walks its units in order. Per CTA: warp 0 copies K tiles and each
unit's roped Q (dims 0-127 into the K ring slot after the unit's first tile, dims 128-255 into
their own buffer, once the previous unit's last QK^T is done); warp 6 copies V; warp 1 issues
QK^T (even CTA) or relays ring landings (odd CTA); warp 7 checks V and issues P.V (even CTA);
eight softmax warps, two per row quarter (one per half of the columns), move Q into tensor
memory, run the softmax, write P and the epilogue, and meet their row partner on a barrier of
their quarter once per key tile (the row max) and once per unit (the sums). The model keeps the
kernel's barriers, counts and phase arithmetic, and checks at every MMA and every read that the
buffer holds the expected tile or unit: K slots, the Q buffers, the single S and P buffers in
tensor memory, the V stages, O and the partner's posted half.

The random unit sequences are lists of key-tile counts; a planted mistake (a wait removed) must
make the model fail."""
import random

import pytest

from protocol_sim import Bar, Err, Role, Sim

NK, NV, QAFTER = 2, 2, 1
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
                        ("q_pair", 2 * SMX), ("q_free", 1), ("o_free", 2 * SMX), ("q_read", SMX)):
            d[nm] = Bar(f"C{X}.{nm}", cnt)
        for q in range(4):
            d[f"xchg{q}"] = Bar(f"C{X}.xchg{q}", 2)
        B[X] = d
    qpos = [min(QAFTER, n) for n in units]
    def kslot(ui, j):
        return j + (1 if j >= qpos[ui] else 0)
    c0s = [0]
    for n in units:
        c0s.append(c0s[-1] + n + 1)
    jt0s = [0]
    for n in units:
        jt0s.append(jt0s[-1] + n)
    # data state
    kring = {X: [None] * NK for X in (0, 1)}       # ("K", jt) or ("Q", ui) landed
    kpend = {X: [0] * NK for X in (0, 1)}          # issued, not yet released
    qhi = {X: None for X in (0, 1)}
    tq = {X: None for X in (0, 1)}                 # unit whose Q dims 0-127 are in tensor memory
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
        for ui, n in enumerate(units):
            for idx in range(n + 1):
                c = c0s[ui] + idx
                s = c % NK
                is_q = idx == qpos[ui]
                j = idx if idx < qpos[ui] else idx - 1
                if c >= NK:
                    yield ("wait", B[X][f"k_empty{s}"], c // NK - 1)
                if is_q and ui > 0 and mut != "no_qfree":
                    yield ("wait", B[X]["q_free"], ui - 1)
                chk(kpend[X][s] == 0, f"C{X} slot {s} reloaded before release")
                kpend[X][s] = 1
                kring[X][s] = None
                if is_q:
                    chk(qk_done_unit["last"] >= ui - 1, f"C{X} Q of unit {ui} over qhi still read by unit {ui-1}'s QK")
                    B[X][f"k_full{s}"].expect_tx(S, 1)
                    B[X]["q_full"].expect_tx(S, 1)
                    qhi[X] = None
                    def land_ql(X=X, s=s, ui=ui):
                        kring[X][s] = ("Q", ui)
                        B[X][f"k_full{s}"].complete_tx(S, 1)
                    def land_qh(X=X, ui=ui):
                        qhi[X] = ui
                        B[X]["q_full"].complete_tx(S, 1)
                    S.later(land_ql, 2, 10)
                    S.later(land_qh, 2, 10)
                else:
                    jt = jt0s[ui] + j
                    B[X][f"k_full{s}"].expect_tx(S, 1)
                    def land_k(X=X, s=s, jt=jt):
                        kring[X][s] = ("K", jt)
                        B[X][f"k_full{s}"].complete_tx(S, 1)
                    S.later(land_k, 2, 10)
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
            for idx in range(n + 1):
                c = c0s[ui] + idx
                s = c % NK
                yield ("wait", B[1][f"k_full{s}"], c // NK)
                B[0][f"k_peer{s}"].arrive(S)
    def issuer():
        for ui, n in enumerate(units):
            cq = c0s[ui] + qpos[ui]
            yield ("wait", B[0][f"k_full{cq % NK}"], cq // NK)
            yield ("wait", B[0][f"k_peer{cq % NK}"], cq // NK)
            yield ("wait", B[0]["q_pair"], ui)
            for j in range(n):
                jt = jt0s[ui] + j
                c = c0s[ui] + kslot(ui, j)
                s = c % NK
                yield ("wait", B[0][f"k_full{s}"], c // NK)
                yield ("wait", B[0][f"k_peer{s}"], c // NK)
                if jt > 0 and mut != "no_sfree":
                    yield ("wait", B[0]["s_free"], jt - 1)
                def mma(s=s, jt=jt, ui=ui):
                    for X in (0, 1):
                        chk(kring[X][s] == ("K", jt), f"QK {jt}: C{X} slot {s} holds {kring[X][s]}")
                        chk(tq[X] == ui, f"QK {jt}: C{X} TMEM Q holds unit {tq[X]}")
                        chk(qhi[X] == ui, f"QK {jt}: C{X} qhi holds unit {qhi[X]}")
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
            cq = c0s[ui] + qpos[ui]
            s = cq % NK
            yield ("wait", B[X][f"k_full{s}"], cq // NK)
            yield ("wait", B[X]["q_full"], ui)
            chk(kring[X][s] == ("Q", ui), f"C{X}.w{w} moves Q of unit {ui} from slot holding {kring[X][s]}")
            tq[X] = ui
            B[0]["q_pair"].arrive(S)
            B[X]["q_read"].arrive(S)
            if w == 0:
                if mut != "no_qread":
                    yield ("wait", B[X]["q_read"], ui)
                # the slot goes back to the ring only once all four warps have read it
                chk(B[X]["q_read"].done >= ui + 1, f"C{X} Q slot released before all warps read it")
                kpend[X][s] = 0
                B[X][f"k_empty{s}"].arrive(S)
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
    """300 random unit sequences (1 to 6 units of 1 to 10 key tiles, the Q slot at each position
    it can take) run to the end with every check passing."""
    failures = run_many(300)
    assert not failures, failures[:3]


@pytest.mark.parametrize("mut", ["no_qfree", "no_sfree", "no_qread", "no_xchg"])
def test_sliding_protocol_model_catches_a_missing_wait(mut):
    """Control: each of these waits guards a hazard the model can see, so removing it fails. (The
    P.V issuer's wait for O to be read out is implied as well by its wait for the next unit's
    first P: the same warps read O out before they write that P, so removing it alone cannot
    fail.)"""
    assert run_many(100, mut)
