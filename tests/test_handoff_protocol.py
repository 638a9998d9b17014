"""Exhaustive check of the named-barrier hand-off protocol (host model, no GPU).

The ring forward hands P to each unit's MMA issuer, and the dK/dV kernel hands P^T and dS^T
to its MMA warp, on hardware named barriers, which cannot time out.  This test explores every
interleaving of a small model of that protocol and checks that the waiting side can never be
left in its `bar.sync` for good, and that no barrier phase gets two arrivals from one warp.

Model (n tiles, W arriving warps, one issuer):
  * named barrier: counts arrivals; the issuer's `bar.sync` is one of them; when the count
    reaches W + 1 the phase completes, the count starts again from 0, and an issuer whose
    arrival was in that phase goes on;
  * issuer, per tile j: check the abort flag (leave if set), `bar.sync` (a separate step: the
    flag may rise between the two), then queue the gating MMA of tile j + 1 (S(j+1) for
    P(j+1));
  * each arriving warp, per tile j: wait for MMA j to complete, then arrive.  It gives up only
    when its own time limit runs out, which can happen only while MMA j was never queued, and
    raises the abort flag when it does;
  * environment: a queued MMA eventually completes; some other role may raise the abort flag
    at any moment.

The dK/dV kernel's two barriers (P^T gated by S^T, dS^T gated by dP^T) each follow this
pattern on their own.

The same model with the earlier rule -- the arriving warps also give up when the flag is set,
and every way out after an abort adds one more arrival -- must deadlock somewhere; the test
checks that the exploration finds that state.
"""
from __future__ import annotations

from collections import deque


def _explore(n_tiles: int, n_warps: int, old_rule: bool):
    """Return (deadlocks, double_arrivals, states, whether the all-done state is reachable)."""
    E = n_warps + 1
    # state: (flag, iss_tile, iss_stage, queued, done, warps, count, iss_in, arrived)
    #   iss_stage: 0 check the flag, 5 flag found clear (the bar.sync is the next instruction,
    #   so the flag may rise in between), 1 waiting in bar.sync, 2 queue next, 3 left, 4 finished
    #   warps: tuple of (tile, stage) with stage 0 wait, 1 arrive, 2 left, 3 finished
    #   arrived: frozenset of warps that arrived in the current phase
    init = (False, 0, 0, (True,) + (False,) * (n_tiles - 1), (False,) * n_tiles,
            tuple((0, 0) for _ in range(n_warps)), 0, False, frozenset())
    seen = {init}
    todo = deque([init])
    deadlocks = []
    doubles = []
    finished = False

    def arrive(count, iss_in, arrived, who):
        """One arrival (who = warp index, or -1 for the issuer). Returns the new
        (count, iss_in, arrived, issuer_released, double)."""
        double = who >= 0 and who in arrived
        count += 1
        arrived = arrived | {who}
        if who == -1:
            iss_in = True
        if count == E:
            return 0, False, frozenset(), iss_in, double
        return count, iss_in, arrived, False, double

    while todo:
        st = todo.popleft()
        flag, it, ist, queued, done, warps, count, iss_in, arrived = st
        succ = []
        # environment: a queued MMA completes
        for j in range(n_tiles):
            if queued[j] and not done[j]:
                d = list(done)
                d[j] = True
                succ.append((flag, it, ist, queued, tuple(d), warps, count, iss_in, arrived))
        # environment: another role raises the abort flag
        if not flag:
            succ.append((True, it, ist, queued, done, warps, count, iss_in, arrived))
        # issuer
        if ist == 0:
            succ.append((flag, it, 3 if flag else 5, queued, done, warps, count, iss_in, arrived))
        elif ist == 5:
            c, ii, ar, rel, _ = arrive(count, iss_in, arrived, -1)
            succ.append((flag, it, 2 if rel else 1, queued, done, warps, c, ii and not rel, ar))
        elif ist == 2:
            q = list(queued)
            if it + 1 < n_tiles:
                q[it + 1] = True
                succ.append((flag, it + 1, 0, tuple(q), done, warps, count, iss_in, arrived))
            else:
                succ.append((flag, it, 4, tuple(q), done, warps, count, iss_in, arrived))
        # arriving warps
        for w, (wt, wst) in enumerate(warps):
            def with_warp(new, f=flag, c=count, ii=iss_in, ar=arrived, iss_stage=ist):
                ws = list(warps)
                ws[w] = new
                return (f, it, iss_stage, queued, done, tuple(ws), c, ii, ar)
            if wst == 0:
                if done[wt]:
                    succ.append(with_warp((wt, 1)))
                gives_up = (not queued[wt]) or (old_rule and flag)
                if gives_up:
                    if old_rule:  # one more arrival on the way out
                        c, ii, ar, rel, dbl = arrive(count, iss_in, arrived, w)
                        if dbl:
                            doubles.append(st)
                        stage = 2 if (rel and ist == 1) else ist
                        succ.append(with_warp((wt, 2), True, c, ii and not rel, ar, stage))
                    else:
                        succ.append(with_warp((wt, 2), True))
            elif wst == 1:
                c, ii, ar, rel, dbl = arrive(count, iss_in, arrived, w)
                if dbl:
                    doubles.append(st)
                stage = 2 if (rel and ist == 1) else ist
                nxt = (wt + 1, 0) if wt + 1 < n_tiles else (wt, 3)
                succ.append(with_warp(nxt, flag, c, ii and not rel, ar, stage))
        if not succ and ist == 1:
            deadlocks.append(st)
        if ist == 4 and all(ws == 3 for _, ws in warps):
            finished = True
        for s in succ:
            if s not in seen:
                seen.add(s)
                todo.append(s)
    return deadlocks, doubles, len(seen), finished


def test_protocol_as_built_never_strands_the_issuer():
    for n_tiles, n_warps in ((3, 1), (3, 2), (4, 2)):
        deadlocks, doubles, states, finished = _explore(n_tiles, n_warps, old_rule=False)
        assert states > 50 and finished
        assert not deadlocks, deadlocks[:3]
        assert not doubles, doubles[:3]


def test_earlier_abort_arrival_rule_can_strand_the_issuer():
    deadlocks, doubles, _, _ = _explore(3, 2, old_rule=True)
    assert deadlocks and doubles


def _explore_two(n_tiles: int, n_warps: int, early_queue: bool = False):
    """The dK/dV kernel's sequence with its two barriers.  Issuer per tile t: check, sync on
    barrier P (P^T(t)), queue S^T(t+1); check, sync on barrier D (dS^T(t)), queue dP^T(t+1).
    Each warp per tile t: wait S^T(t), arrive on P; wait dP^T(t), arrive on D.  Waits give up
    only on their own limit (possible only while the product was never queued).
    `early_queue` plants an ordering mistake: S^T(t+1) queued before the sync on P(t).
    Returns (deadlocks, double arrivals, states, whether the all-done state is reachable)."""
    E = n_warps + 1
    # state: (flag, it, ist, sq, sd, dq, dd, warps, bars)
    #   ist: 0 check P, 1 sync P pending (flag found clear), 2 waiting on P, 3 queue S^T(t+1),
    #        4 check D, 5 sync D pending, 6 waiting on D, 7 queue dP^T(t+1), 8 left, 9 finished
    #   sq/sd: S^T queued/done per tile; dq/dd: dP^T queued/done per tile
    #   warps: (tile, stage) stage 0 wait S^T, 1 arrive P, 2 wait dP^T, 3 arrive D, 4 left, 5 done
    #   bars: ((count, issuer_in, arrived), (count, issuer_in, arrived)) for P and D
    zero = (0, False, frozenset())
    f0 = (False,) * n_tiles
    first = (True,) + (False,) * (n_tiles - 1)
    init = (False, 0, 0, first, f0, first, f0, tuple((0, 0) for _ in range(n_warps)), (zero, zero))
    seen = {init}
    todo = deque([init])
    deadlocks, doubles = [], []
    finished = False

    def arrive(bar, who):
        count, iss_in, arrived = bar
        double = who >= 0 and who in arrived
        count += 1
        arrived = arrived | {who}
        iss_in = iss_in or who == -1
        if count == E:
            return zero, iss_in, double
        return (count, iss_in, arrived), False, double

    while todo:
        st = todo.popleft()
        flag, it, ist, sq, sd, dq, dd, warps, bars = st
        succ = []
        for j in range(n_tiles):
            if sq[j] and not sd[j]:
                x = list(sd); x[j] = True
                succ.append((flag, it, ist, sq, tuple(x), dq, dd, warps, bars))
            if dq[j] and not dd[j]:
                x = list(dd); x[j] = True
                succ.append((flag, it, ist, sq, sd, dq, tuple(x), warps, bars))
        if not flag:
            succ.append((True, it, ist, sq, sd, dq, dd, warps, bars))
        # issuer
        if ist == 0 and early_queue and it + 1 < n_tiles and not sq[it + 1]:
            x = list(sq)
            x[it + 1] = True
            succ.append((flag, it, ist, tuple(x), sd, dq, dd, warps, bars))
        elif ist in (0, 4):
            succ.append((flag, it, 8 if flag else ist + 1, sq, sd, dq, dd, warps, bars))
        elif ist in (1, 5):
            k = 0 if ist == 1 else 1
            nb, rel, _ = arrive(bars[k], -1)
            b2 = list(bars); b2[k] = nb
            succ.append((flag, it, ist + 2 if rel else ist + 1, sq, sd, dq, dd, warps, tuple(b2)))
        elif ist == 3:
            x = list(sq)
            if it + 1 < n_tiles:
                x[it + 1] = True
            succ.append((flag, it, 4, tuple(x), sd, dq, dd, warps, bars))
        elif ist == 7:
            x = list(dq)
            if it + 1 < n_tiles:
                x[it + 1] = True
                succ.append((flag, it + 1, 0, sq, sd, tuple(x), dd, warps, bars))
            else:
                succ.append((flag, it, 9, sq, sd, tuple(x), dd, warps, bars))
        # warps
        for w, (wt, wst) in enumerate(warps):
            def put(new, f=flag, b=bars, i=ist):
                ws = list(warps); ws[w] = new
                return (f, it, i, sq, sd, dq, dd, tuple(ws), b)
            if wst == 0:
                if sd[wt]:
                    succ.append(put((wt, 1)))
                if not sq[wt]:
                    succ.append(put((wt, 4), True))
            elif wst == 2:
                if dd[wt]:
                    succ.append(put((wt, 3)))
                if not dq[wt]:
                    succ.append(put((wt, 4), True))
            elif wst in (1, 3):
                k = 0 if wst == 1 else 1
                nb, rel, dbl = arrive(bars[k], w)
                if dbl:
                    doubles.append(st)
                b2 = list(bars); b2[k] = nb
                i2 = ist
                if rel and ist == (2 if k == 0 else 6):
                    i2 = ist + 1
                if wst == 1:
                    nxt = (wt, 2)
                else:
                    nxt = (wt + 1, 0) if wt + 1 < n_tiles else (wt, 5)
                succ.append(put(nxt, flag, tuple(b2), i2))
        if not succ and ist in (2, 6):
            deadlocks.append(st)
        if ist == 9 and all(ws == 5 for _, ws in warps):
            finished = True
        for s in succ:
            if s not in seen:
                seen.add(s)
                todo.append(s)
    return deadlocks, doubles, len(seen), finished


def test_dkdv_two_barrier_sequence_never_strands_the_issuer():
    for n_tiles, n_warps in ((2, 1), (3, 1), (2, 2), (3, 2)):
        deadlocks, doubles, states, finished = _explore_two(n_tiles, n_warps)
        assert states > 50 and finished
        assert not deadlocks, deadlocks[:3]
        assert not doubles, doubles[:3]


def test_dkdv_model_catches_a_product_queued_before_its_sync():
    _, doubles, _, _ = _explore_two(3, 2, early_queue=True)
    assert doubles
