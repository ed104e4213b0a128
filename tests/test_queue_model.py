"""CPU models of the work queues in the pack and combine kernels.

The kernels take a fixed first share of the work and then claim the rest in
increasing order from a counter that the routing kernel resets.  These tests
restate, step by step, the control flow each kernel's single issuing thread
follows (csrc/dispatch_pack.cu: dispatch_pack_bulk_queue; csrc/combine.cu:
combine_bulk_queue_kernel; csrc/dispatch_fp8.cu:
dispatch_pack_fp8_queue_kernel), run many CTAs as interleaved generators
against one shared counter, and check the protocol's invariants:

  - every unit (or token) is processed exactly once, whatever the interleaving;
  - the pack's stage ring: a stage is refilled only after the unit in it has
    been consumed, every issued load is consumed, and the destination rows
    loaded one unit ahead always belong to the CTA's next unit;
  - claims stop at the first value past the end, so the counter grows by at
    most the claimed work plus a few claims per CTA.

The per-group stage ring of route_pack_fp8 (csrc/route_pack_fp8.cu) is
modelled the same way, with mbarrier phases as counts: every wait is
satisfied by the phase of its own token's load, never an older one.
"""
import random

import pytest


def _run(gens, seed):
    rng = random.Random(seed)
    live = list(gens)
    while live:
        g = rng.choice(live)
        try:
            next(g)
        except StopIteration:
            live.remove(g)


def _pack_cta(b, G, units, stages, depth, counter, seq, lookahead):
    """dispatch_pack_bulk_queue: prologue of `stages` static units, then one
    claim in flight; the stage of sequence r = i-depth+1 is refilled with
    sequence r+stages at iteration i."""
    static_end = stages * G
    static_units = min(units, static_end)
    nstatic = (static_units - b + G - 1) // G if static_units > b else 0
    ring = [b + i * G if i < nstatic else -1 for i in range(stages)]
    loads = {i: (i, ring[i]) for i in range(stages) if ring[i] >= 0}
    claiming = units > static_end
    claim = None
    if claiming:
        claim = counter[0]
        counter[0] += 1
        yield
    i = 0
    u_cur = ring[0]
    while u_cur >= 0:
        s = i % stages
        assert loads.get(s) == (i, u_cur), "the stage holds this sequence's unit"
        del loads[s]
        seq.append(u_cur)
        lookahead.append(ring[(i + 1) % stages])
        r = i - depth + 1
        if r >= 0:
            u = -1
            if claiming:
                c = static_end + claim
                if c < units:
                    u = c
                    claim = counter[0]
                    counter[0] += 1
                    yield
                else:
                    claiming = False
            slot = (r + stages) % stages
            assert slot not in loads, "refill over a stage not yet consumed"
            ring[slot] = u
            if u >= 0:
                loads[slot] = (r + stages, u)
        i += 1
        u_cur = ring[i % stages]
        yield
    assert not loads, "a load was issued and never consumed"
    assert not claiming


@pytest.mark.parametrize("units", [0, 1, 5, 64, 65, 257, 2003])
@pytest.mark.parametrize("G", [1, 3, 16])
@pytest.mark.parametrize("stages", [2, 3, 8, 16])
def test_pack_unit_queue(units, G, stages):
    for depth in range(1, stages):
        for seed in range(3):
            counter = [0]
            seqs = [[] for _ in range(G)]
            looks = [[] for _ in range(G)]
            _run([_pack_cta(b, G, units, stages, depth, counter, seqs[b], looks[b]) for b in range(G)], seed)
            assert sorted(u for s in seqs for u in s) == list(range(units))
            for s, look in zip(seqs, looks):
                assert look[:-1] == s[1:], "the rows loaded ahead are the next unit's"
                if s:
                    assert look[-1] == -1
            assert counter[0] <= max(0, units - stages * G) + G


def _token_cta(b, G, T, P, counter, seen):
    """combine_bulk_queue_kernel (P pieces per token) and, with P = 1, the fp8
    pack's token sequence: token b, then tokens claimed whole, two claims in
    flight."""
    claiming = T > G
    q = []
    if claiming:
        for _ in range(2):
            q.append(counter[0])
            counter[0] += 1
            yield
    first, tok, j = True, -1, P
    while True:
        if j >= P:
            if first:
                first = False
                tok = b if b < T else -1
            elif not claiming:
                tok = -1
            else:
                c = G + q.pop(0)
                if c >= T:
                    claiming = False
                    tok = -1
                else:
                    tok = c
                    q.append(counter[0])
                    counter[0] += 1
            j = 0
            if tok < 0:
                break
        seen.append(tok * P + j)
        j += 1
        yield


@pytest.mark.parametrize("T", [0, 1, 2, 5, 64, 100, 1000])
@pytest.mark.parametrize("P", [1, 2, 4, 7])
@pytest.mark.parametrize("G", [1, 3, 16, 64])
def test_combine_token_queue(T, P, G):
    for seed in range(3):
        counter = [0]
        seen = []
        _run([_token_cta(b, G, T, P, counter, seen) for b in range(G)], seed)
        assert sorted(seen) == list(range(T * P))
        assert counter[0] <= max(0, T - G) + 2 * G


def _fp8_cta(b, G, T, stages, counter, seen):
    """dispatch_pack_fp8_queue_kernel: tokens b, b+G, ..., b+(stages-1)G, then
    tokens claimed from stages*G on, one claim in flight; token -1 ends."""
    static_end = stages * G
    static_tok = min(T, static_end)
    nstatic = (static_tok - b + G - 1) // G if static_tok > b else 0
    claiming = T > static_end
    claim = None
    if claiming:
        claim = counter[0]
        counter[0] += 1
        yield
    i = 0
    while True:
        if i < stages:
            t = b + i * G if i < nstatic else -1
        else:
            t = -1
            if claiming:
                c = static_end + claim
                if c < T:
                    t = c
                    claim = counter[0]
                    counter[0] += 1
                else:
                    claiming = False
        if t < 0:
            break
        seen.append(t)
        i += 1
        yield


@pytest.mark.parametrize("T", [0, 1, 7, 64, 65, 1000])
@pytest.mark.parametrize("G", [1, 3, 16])
@pytest.mark.parametrize("stages", [2, 3, 5, 8])
def test_fp8_token_queue(T, G, stages):
    for seed in range(3):
        counter = [0]
        seen = []
        _run([_fp8_cta(b, G, T, stages, counter, seen) for b in range(G)], seed)
        assert sorted(seen) == list(range(T))


def _fused_fp8_group(stages, mine, rng, seen):
    """route_pack_fp8, one group of 128 threads: its first thread loads tokens
    0..stages-1 of the group into its own ring before the routing; per token
    i the group waits on stage i % stages with parity (i / stages) & 1,
    quantises, synchronises, and refills the stage with token i + stages.
    Loads land after random delays; the mbarrier of a stage is modelled by
    its count of completed phases (try_wait with parity P succeeds once the
    count's parity differs from P)."""
    completed = [0] * stages           # phases completed per stage
    in_flight = []                     # (stage, token) loads not landed yet
    content = [None] * stages          # token whose row a landed load left in the stage
    for i in range(min(stages, mine)):
        in_flight.append((i % stages, i))

    def land_some():
        rng.shuffle(in_flight)
        for _ in range(rng.randint(0, len(in_flight))):
            s, t = in_flight.pop()
            content[s] = t
            completed[s] += 1

    for i in range(mine):
        s, parity = i % stages, (i // stages) & 1
        while (completed[s] & 1) == parity:  # try_wait.parity fails: not landed yet
            land_some()
            yield
        # The phase that satisfied the wait is this token's load, not an older one.
        assert completed[s] == i // stages + 1
        assert content[s] == i
        seen.append(i)
        if i + stages < mine:
            assert all(st != s for st, _ in in_flight), "a stage is refilled only once it is free"
            in_flight.append((s, i + stages))
        yield
    assert not in_flight


@pytest.mark.parametrize("stages,mine", [(1, 5), (2, 2), (2, 7), (3, 4), (3, 3), (7, 30), (16, 40), (4, 0)])
def test_fused_fp8_stage_ring(stages, mine):
    for seed in range(300):
        rng = random.Random(seed)
        seen = []
        _run([_fused_fp8_group(stages, mine, rng, seen)], seed)
        assert seen == list(range(mine))
