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
    """Return (deadlocks, double_arrivals, states) over all reachable states."""
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
        for s in succ:
            if s not in seen:
                seen.add(s)
                todo.append(s)
    return deadlocks, doubles, len(seen)


def test_protocol_as_built_never_strands_the_issuer():
    for n_tiles, n_warps in ((3, 1), (3, 2), (4, 2)):
        deadlocks, doubles, states = _explore(n_tiles, n_warps, old_rule=False)
        assert states > 50
        assert not deadlocks, deadlocks[:3]
        assert not doubles, doubles[:3]


def test_earlier_abort_arrival_rule_can_strand_the_issuer():
    deadlocks, doubles, _ = _explore(3, 2, old_rule=True)
    assert deadlocks and doubles
