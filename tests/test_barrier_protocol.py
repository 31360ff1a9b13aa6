"""Model check of the tensor-core kernel's mbarrier protocol on the CPU.

The kernel's warps wait on mbarriers with parity waits, which only distinguish the
current phase from the one before it.  This discrete-event model replays the kernel's
protocol (weight producer, A producer, MMA issuers, dequant warpgroups, asynchronous copy
and MMA completions with random latencies; one issuer's MMAs complete in order, the two
issuers' independently) and flags any wait whose intended phase is not the barrier's
current or immediately preceding phase, any weight slot, A slot or TMEM W buffer
rewritten while a warp or an MMA still reads it, and any deadlock.

Layout modelled (as in csrc/gemm_tc.cu): a weight ring wfull[s] / wempty[s] (a slot is
released by the warps that read it, once they have read it) and an A ring afull[s] /
aempty[s] (released by the MMA commits of its stage), each with its own producer and its
own depth; W buffers t with tfull[issuer][t] (count: the warps that write the tile) and
tempty[warpgroup][t] (one MMA commit).  Whole-block tiles: warpgroup w unpacks blocks
w, w + NWG, ...; shared-block tiles: every warpgroup unpacks every block.

Events carry their own times (the heap key), and every callback is given that time, so
the random latencies really reorder the agents; the earlier shared layout (one tfull and
one tempty per W buffer for both issuers and both warpgroups) is flagged by the model,
the per-party layout is not.
"""
import heapq
import itertools
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.ph = 0  # completed phases

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0
        if self.pending == 0:
            self.ph += 1
            self.pending = self.count


def simulate(kNMI, NWG, T, kps, SW, SA, nkb, rng, interleave, per_party=True,
             w_readers=None, one_producer=None, tempty_wait=True):
    """w_readers: arrivals that release a weight slot (default: the kernel's count, one
    per warp that reads the slot's blocks).  one_producer: one agent streams both rings
    (the kernel's choice for two blocks per stage, i.e. decode tiles), always issuing the
    copy whose slot is released first.  tempty_wait=False drops the dequant warps' wait
    for a W buffer's previous MMAs (for the sensitivity test of the W-buffer race
    check)."""
    if one_producer is None:
        one_producer = kps == 2
    nst = (nkb + kps - 1) // kps
    wfull = [Bar(1) for _ in range(SW)]
    if w_readers is None:
        w_readers = (4 if interleave else 4 * NWG) * kps
    wempty = [Bar(w_readers) for _ in range(SW)]
    afull = [Bar(1) for _ in range(SA)]
    aempty = [Bar(2 if (kNMI == 2 and kps == 2) else 1) for _ in range(SA)]
    n_tparty = kNMI if per_party else 1
    n_eparty = (NWG if interleave else 1) if per_party else 1
    tfull = [[Bar(4 if interleave else 4 * NWG) for _ in range(T)] for _ in range(n_tparty)]
    tempty = [[Bar(1) for _ in range(T)] for _ in range(n_eparty)]
    events, cnt, errors = [], itertools.count(), []
    # readers of each slot right now: a copy into a slot while someone reads it is a race
    reading = {"w": [0] * SW, "a": [0] * SA, "t": [0] * T}

    def at(t, f):
        heapq.heappush(events, (t, next(cnt), f))

    def producer(ring, depth, full, empty, lo, hi):
        for p in range(nst):
            if p >= depth:
                yield ("wait", empty[p % depth], p // depth - 1)
            yield ("write", ring, p % depth)
            yield ("async", rng.uniform(lo, hi), full[p % depth])

    mma_free = [0.0] * kNMI  # MMAs of one issuer complete in order; issuers independently

    def issuer(k):
        seen = [0] * T
        last_p = -1
        for i in range(k, nkb, kNMI):
            p = i // kps
            if p != last_p:
                yield ("wait", afull[p % SA], p // SA)
                last_p = p
            t = i % T
            party = k if per_party else 0
            q = seen[t] if per_party else i // T
            yield ("wait", tfull[party][t], q)
            seen[t] += 1
            yield ("delay", rng.uniform(0.01, 0.1))
            yield ("mma", k, i, p, kNMI == 2 or i % kps == kps - 1 or i == nkb - 1)

    def warp(w):
        seen = [0] * T
        last_p = -1
        blocks = range(w, nkb, NWG) if interleave else range(nkb)
        for i in blocks:
            p = i // kps
            if p != last_p:
                yield ("wait", wfull[p % SW], p // SW)
                last_p = p
            t = i % T
            if i >= T and tempty_wait:
                party = (w if interleave else 0) if per_party else 0
                q = seen[t] if per_party else i // T - 1
                yield ("wait", tempty[party][t], q)
                seen[t] += 1
            yield ("write", "t", t)  # the unpack stores into W buffer t
            yield ("read", "w", p % SW, +1)
            yield ("delay", rng.uniform(0.05, 0.8))
            yield ("read", "w", p % SW, -1)
            yield ("arrive", wempty[p % SW])  # the block's weights are read
            yield ("arrive", tfull[(i % kNMI) if per_party else 0][t])

    def both():
        wi = ai = 0
        while wi < nst and wi < SW:  # the weight stages that need no slot back
            yield ("write", "w", wi % SW)
            yield ("async", rng.uniform(0.2, 3.0), wfull[wi % SW])
            wi += 1
        while wi < nst or ai < nst:
            if wi < nst and (ai >= nst or wi - SW <= ai - SA):
                if wi >= SW:
                    yield ("wait", wempty[wi % SW], wi // SW - 1)
                yield ("write", "w", wi % SW)
                yield ("async", rng.uniform(0.2, 3.0), wfull[wi % SW])
                wi += 1
            else:
                if ai >= SA:
                    yield ("wait", aempty[ai % SA], ai // SA - 1)
                yield ("write", "a", ai % SA)
                yield ("async", rng.uniform(0.1, 1.5), afull[ai % SA])
                ai += 1

    if one_producer:
        agents = [both()]
    else:
        agents = [producer("w", SW, wfull, wempty, 0.2, 3.0),
                  producer("a", SA, afull, aempty, 0.1, 1.5)]
    agents += [issuer(k) for k in range(kNMI)]
    agents += [warp(w) for w in range(NWG) for _ in range(4)]
    waiting, finished = {}, set()

    def wake(now):
        for ai, (bar, q) in list(waiting.items()):
            if bar.ph > q:
                del waiting[ai]
                at(now, lambda n, ai=ai: step(ai, n))

    def step(ai, now):
        g = agents[ai]
        while True:
            try:
                act = next(g)
            except StopIteration:
                finished.add(ai)
                return
            kind = act[0]
            if kind == "wait":
                bar, q = act[1], act[2]
                if not (bar.ph - 1 <= q <= bar.ph):
                    errors.append(f"parity alias: wants phase {q}, barrier at {bar.ph}")
                    finished.add(ai)
                    return
                if bar.ph > q:
                    continue
                waiting[ai] = (bar, q)
                return
            if kind == "delay":
                at(now + act[1], lambda n, ai=ai: step(ai, n))
                return
            if kind == "arrive":
                act[1].arrive()
                wake(now)
                continue
            if kind == "read":
                reading[act[1]][act[2]] += act[3]
                continue
            if kind == "write":
                if reading[act[1]][act[2]]:
                    errors.append(f"race: {act[1]} slot {act[2]} refilled while being read")
                    finished.add(ai)
                    return
                continue
            if kind == "async":
                bar = act[2]
                at(now + act[1], lambda n, bar=bar: (bar.arrive(), wake(n)))
                continue
            if kind == "mma":
                k, i, p, release = act[1], act[2], act[3], act[4]
                fin = max(now, mma_free[k]) + rng.uniform(0.05, 0.8)
                mma_free[k] = fin
                reading["a"][p % SA] += 1  # the MMA reads its A stage until it completes
                reading["t"][i % T] += 1   # and its W buffer

                def done(n, i=i, p=p, release=release):
                    reading["a"][p % SA] -= 1
                    reading["t"][i % T] -= 1
                    party = ((i + T) % NWG if interleave else 0) if per_party else 0
                    tempty[party][i % T].arrive()
                    if release:
                        aempty[p % SA].arrive()
                    wake(n)
                at(fin, done)
                continue

    for ai in range(len(agents)):
        at(rng.uniform(0, 0.5), lambda n, ai=ai: step(ai, n))
    while events and not errors:
        t_ev, _, f = heapq.heappop(events)
        f(t_ev)
    if errors:
        return errors[0]
    if len(finished) != len(agents) or waiting:
        return "deadlock"
    return None


def configs(interleave):
    # (2, 2): decode tiles; (1, 1): the shared-block 64- to 256-row tiles (and a
    # single-issuer whole-block variant); (2, 1): 64- and 128-row whole-block tiles with
    # two issuers taking alternate blocks (one block per stage); (1, 2): a single-issuer
    # variant of the two-block stage
    for kNMI, kps in ((2, 2), (1, 1), (2, 1), (1, 2)):
        for T in (2, 3, 4, 6):
            for NWG in (1, 2, 4):
                if interleave and NWG % kps:  # the kernel's static rule for whole blocks
                    continue
                for SW in (2, 3, 4, 5, 6, 8):
                    # host rule: with whole blocks per group, the weight ring depth is a
                    # multiple of groups per stage
                    if interleave and NWG > kps and SW % (NWG // kps):
                        continue
                    for SA in (2, 3, 4, 5):
                        # host rule: two issuers with one block per stage each read
                        # every other A stage, so the A ring depth is even
                        if kNMI == 2 and kps == 1 and SA % 2:
                            continue
                        for nkb in (1, 2, 3, 5, 7, 11, 16):
                            yield kNMI, NWG, T, kps, SW, SA, nkb


@pytest.mark.parametrize("one_producer", [False, True], ids=["two_producers", "one_producer"])
@pytest.mark.parametrize("interleave", [True, False], ids=["whole_blocks", "all_chunks"])
def test_per_party_barriers_never_alias_or_deadlock(interleave, one_producer):
    bad = []
    for cfg in configs(interleave):
        for trial in range(2):
            rng = random.Random(hash((cfg, trial, interleave, one_producer)))
            e = simulate(*cfg, rng, interleave, one_producer=one_producer)
            if e:
                bad.append((cfg, e))
                break
    assert not bad, bad[:3]


def test_model_catches_a_ring_depth_that_breaks_the_rule():
    """Sensitivity of the model: four warpgroups taking whole blocks, one block per stage,
    and a weight ring depth (3 or 2) that is not a multiple of 4: each group skips phases
    of slots it shares with the others; the host forbids those depths, and the model must
    flag them."""
    for SW in (3, 2):
        hits = sum(1 for trial in range(20)
                   if simulate(1, 4, 2, 1, SW, 3, 16, random.Random(trial), interleave=True))
        assert hits > 0, SW


def test_model_catches_a_weight_slot_released_too_early():
    """Sensitivity of the race check: if a weight slot were released after fewer
    arrivals than the warps that read it (here: one warpgroup's four where every group
    reads every block), the producer refills it while the other groups still read it; the
    model must flag that, and must not with the kernel's count."""
    hits = clean = 0
    for trial in range(30):
        e = simulate(1, 2, 3, 1, 4, 3, 16, random.Random(trial), False, w_readers=4)
        hits += e is not None and e.startswith("race")
        clean += simulate(1, 2, 3, 1, 4, 3, 16, random.Random(trial), False) is not None
    assert hits > 0 and clean == 0, (hits, clean)


def test_model_catches_an_odd_a_ring_with_two_issuers_of_single_block_stages():
    """Two issuers taking alternate blocks of one block per stage share the A slots of an
    odd-depth ring between them (two waiting parties per barrier); the host keeps that
    depth even, and the model must flag the odd depths."""
    hits = 0
    for SA in (3, 5):
        for trial in range(30):
            e = simulate(2, 4, 4, 1, 8, SA, 16, random.Random(trial), True, one_producer=False)
            hits += e is not None
    assert hits > 0, hits


def test_model_reproduces_the_shared_layout_failure():
    """The first layout of whole-block warpgroups shared one tfull[t] / tempty[t] per W
    buffer between both MMA issuers and both warpgroups; on the GPU it ran into the
    bounded-wait timeout in about one decode run of two.  The interleaving: with three W
    buffers and two issuers, buffer t holds blocks b, b + 3, ... written by alternating
    warpgroups and consumed by alternating issuers.  When block b + 1 (other group) is
    finished before block b, the issuer of b + 1 moves on to b + 3 and parity-waits on
    tfull[t] for phase j + 1 while phase j (block b) is still open; that parity is the
    one of the completed phase j - 1, so the wait returns at once and the MMA reads a
    buffer that block b is still being written into.  The model must flag it (decode-tile
    parameters: 2 issuers, 2 warpgroups, 3 W buffers, 2 blocks per stage), and must not
    flag the per-party layout with the same parameters and seeds."""
    shared = per_party = 0
    for S in (2, 4, 6):
        for trial in range(40):
            e = simulate(2, 2, 3, 2, S, S, 16, random.Random(trial), True, per_party=False)
            shared += e is not None and e.startswith("parity alias")
            per_party += simulate(2, 2, 3, 2, S, S, 16, random.Random(trial), True) is not None
    assert shared > 20, shared
    assert per_party == 0, per_party


def exchange_model(ranks, rng, exit_barrier, limit=10.0, late_rank=None):
    """Split-K exchange of one cluster: every rank finishes its K slice at a random time,
    pushes its partial of every other rank's slice (each push lands after a random
    latency), waits for the pushes into its own receive area with a bounded wait, and
    exits.  With exit_barrier the ranks meet at a cluster barrier before exiting (a rank
    arrives once its pushes have been read out) and then wait, bounded again, for any
    push still landing.  `late_rank` finishes after the others' waits have run out.
    Returns the number of pushes that land in a rank after it has exited."""
    done = [rng.uniform(0.0, 2.0) for _ in range(ranks)]
    if late_rank is not None:
        done[late_rank] = 3.0 * limit
    land = {(src, dst): done[src] + rng.uniform(0.05, 0.5)
            for src in range(ranks) for dst in range(ranks) if src != dst}
    read_out = [done[r] + 0.05 for r in range(ranks)]  # source reads of its pushes done
    recv_end = []
    for r in range(ranks):
        arrivals = [land[(s, r)] for s in range(ranks) if s != r]
        start = done[r] + 0.05
        recv_end.append(min(max(arrivals), start + limit))
    if not exit_barrier:
        exit_t = recv_end
    else:
        release = max(max(recv_end[r], read_out[r]) for r in range(ranks))
        exit_t = []
        for r in range(ranks):
            arrivals = [land[(s, r)] for s in range(ranks) if s != r]
            exit_t.append(max(release, min(max(arrivals), release + limit)))
    return sum(1 for (s, d), t in land.items() if t > exit_t[d])


def test_split_k_exit_waits_for_every_push():
    """With the exit barrier no push ever lands in a rank that has left, also when one
    rank is so late that the others' receive waits run out; without it, such a late
    rank's pushes land in exited ranks (the undefined case the barrier removes)."""
    for ranks in (2, 3, 8):
        for trial in range(50):
            rng = random.Random(trial)
            assert exchange_model(ranks, rng, exit_barrier=True) == 0
            late = trial % ranks
            assert exchange_model(ranks, random.Random(trial), True, late_rank=late) == 0
    assert sum(exchange_model(3, random.Random(t), False, late_rank=0) for t in range(20)) > 0



def test_model_catches_a_w_buffer_rewritten_under_its_mma():
    """Sensitivity of the W-buffer race check: if the dequant warps did not wait for the
    MMAs that last read a W buffer before unpacking the next block into it, they would
    overwrite operands an MMA still reads; the model must flag that, and must not with
    the kernel's wait."""
    hits = clean = 0
    for trial in range(30):
        e = simulate(2, 2, 3, 2, 4, 4, 16, random.Random(trial), True, one_producer=True,
                     tempty_wait=False)
        hits += e is not None and "race: t" in e
        clean += simulate(2, 2, 3, 2, 4, 4, 16, random.Random(trial), True,
                          one_producer=True) is not None
    assert hits > 0 and clean == 0, (hits, clean)
