"""Work lists of the persistent Newton-Schulz launch, checked on the host (no GPU).

The launch is deadlock-free when every cluster is resident and the lists admit one global order
that keeps each cluster's list order and puts every item after all items of its matrix's earlier
stages. These tests rebuild the expected tiles independently, then check that exact cover, the
counter targets, and that the combined order graph has no cycle.
"""
from collections import Counter, defaultdict, deque

import pytest

import workloads as wl
from muon_newton_schulz_09_b300 import launch_choice, persistent_schedule

GRAM, GRAM_AA, COMB = 0, 1, 2
FIRST, LAST, ODD = 1, 2, 4


def groups_of(shapes):
    """Oriented shapes (n <= m) in order of first appearance, with their matrix counts."""
    order, count = [], Counter()
    for r, c in shapes:
        if r == 0 or c == 0:
            continue
        key = (min(r, c), max(r, c))
        if key not in count:
            order.append(key)
        count[key] += 1
    return [(n, m, count[(n, m)]) for n, m in order]


def expected_items(shapes, steps, with_c):
    """Every (kind, group, flags, matrix, row, col, counter target) the iterations need."""
    out = Counter()
    for g, (n, m, cnt) in enumerate(groups_of(shapes)):
        nt, gt2, mt = -(-n // 128), -(-n // 256), -(-m // 256)
        for b in range(cnt):
            halves = 0
            for it in range(steps):
                flags = (FIRST if it == 0 else 0) | (LAST if it == steps - 1 else 0) | (ODD if it % 2 else 0)
                kinds = [GRAM, GRAM_AA, COMB] if with_c else [GRAM, COMB]
                for kind in kinds:
                    if kind == COMB:
                        tiles = [(i, j) for i in range(0, nt, 2) for j in range(mt)]
                    else:
                        tiles = [(i, j) for j in range(gt2) for i in range(0, min(2 * j + 2, nt), 2)]
                    for i, j in tiles:
                        out[(kind, g, flags, b, i, j, halves)] += 1
                    halves += 4 * len(tiles)
    return out


def decode(item):
    x, b, z, w = item
    return (x & 3, (x >> 2) & 1023, x >> 12, b, z & 0xFFFF, z >> 16, w)


def check(shapes, steps, with_c, clusters):
    items, begin = persistent_schedule(shapes, steps, with_c, clusters)
    assert begin[0] == 0 and begin[-1] == len(items) and all(a <= b for a, b in zip(begin, begin[1:]))
    got = Counter(decode(it) for it in items)
    assert got == expected_items(shapes, steps, with_c)
    # Nodes: items, plus one node per (matrix, stage) that all its items feed and the next stage's
    # items depend on. Edges: consecutive items of a cluster list, item -> its stage node, previous
    # stage node -> item. Kahn's algorithm must visit every node.
    dec = [decode(it) for it in items]
    stages = defaultdict(set)
    for k, g, f, b, i, j, w in dec:
        stages[(g, b)].add(w)
    rank = {key: sorted(ws) for key, ws in stages.items()}
    n_items = len(dec)
    sid = {}
    for key, ws in rank.items():
        for s in range(len(ws)):
            sid[(key, s)] = n_items + len(sid)
    adj = defaultdict(list)
    indeg = [0] * (n_items + len(sid))

    def edge(a, b):
        adj[a].append(b)
        indeg[b] += 1

    for c in range(clusters):
        for t in range(begin[c], begin[c + 1] - 1):
            edge(t, t + 1)
    for t, (k, g, f, b, i, j, w) in enumerate(dec):
        s = rank[(g, b)].index(w)
        edge(t, sid[((g, b), s)])
        if s > 0:
            edge(sid[((g, b), s - 1)], t)
    q = deque(v for v in range(len(indeg)) if indeg[v] == 0)
    seen = 0
    while q:
        v = q.popleft()
        seen += 1
        for u in adj[v]:
            indeg[u] -= 1
            if indeg[u] == 0:
                q.append(u)
    assert seen == len(indeg), "the lists and the stage order form a cycle"
    return items, begin


def test_gpt2_124m_step_lists_cover_every_tile_and_are_acyclic():
    items, begin = check(wl.GPT2_124M.shapes, 5, False, 74)
    assert len(items) == 5 * (48 * (6 + 9) + 24 * (6 + 36))
    # balanced: the heaviest list within 30% of the mean, counting k-blocks per tile
    def kblocks(it):
        k, g, f, b, i, j, w = decode(it)
        n, m = (768, 768) if g == 0 else (768, 3072)
        return (m if k == GRAM else n) // 64
    loads = [sum(kblocks(items[t]) for t in range(begin[c], begin[c + 1])) for c in range(74)]
    assert max(loads) <= 1.3 * sum(loads) / 74, loads


@pytest.mark.parametrize("shapes,steps,with_c,clusters", [
    ([(130, 70), (70, 130), (1, 5), (0, 4), (513, 1000), (300, 300)], 3, False, 7),
    ([(256, 768), (768, 256), (384, 384)], 4, True, 5),
    ([(1024, 1024)] * 6, 16, False, 74),
    ([(4096, 16384)], 2, False, 74),
    ([(64, 64)], 1, True, 1),
])
def test_ragged_and_quintic_lists(shapes, steps, with_c, clusters):
    check(shapes, steps, with_c, clusters)


def test_bad_arguments_are_rejected():
    from muon_newton_schulz_09_b300 import MuonError
    for steps, clusters in [(0, 4), (17, 4), (2, 0)]:
        with pytest.raises(MuonError):
            persistent_schedule([(64, 64)], steps, False, clusters)


def test_more_shape_groups_than_an_item_can_name_is_refused():
    """A work item names its shape group in 10 bits; 1025 distinct shapes are refused here, and the
    library runs such calls with the per-phase launches instead."""
    from muon_newton_schulz_09_b300 import MuonError, MUON_ERR_UNSUPPORTED
    persistent_schedule([(1, k) for k in range(1, 1025)], 1, False, 4)
    with pytest.raises(MuonError) as e:
        persistent_schedule([(1, k) for k in range(1, 1026)], 1, False, 4)
    assert e.value.status == MUON_ERR_UNSUPPORTED


def kblocks_per_cluster(shapes, with_c, clusters=74):
    """One iteration's 64-wide k-blocks of 256 x 256 pair tiles per cluster, rebuilt from the tiles:
    Gram pairs reaching the upper triangle (K = m), the A A pass (K = n), the combine (K = n)."""
    kb = 0
    for n, m, cnt in groups_of(shapes):
        nt, gt2, mt = -(-n // 128), -(-n // 256), -(-m // 256)
        gram = sum(len(range(0, min(2 * J + 2, nt), 2)) for J in range(gt2))
        comb = len(range(0, nt, 2)) * mt
        kb += cnt * (gram * -(-m // 64) + (gram * -(-n // 64) if with_c else 0) + comb * -(-n // 64))
    return kb / clusters


@pytest.mark.parametrize("name,persistent", [
    ("gpt2_124m_hidden", True), ("gpt2_124m_hidden_quintic", True), ("square_64x1024", True),
    ("single_128x256_f32", True), ("gpt2_350m_hidden", False), ("illcond_4096x16384", False)])
def test_default_launch_choice_by_work_per_cluster(name, persistent):
    """The default handle runs the persistent launch below 800 k-blocks per cluster per iteration and
    the per-phase launches from there on: the GPT-2 124M sets (350, 420 with the A A pass) and the
    1024^2 batch (360) persistent, the GPT-2 350M set (1619) and the 4096 x 16384 matrix (1356) not."""
    w = wl.WORKLOADS[name]
    with_c = w.coeffs[2] != 0
    use, kb = launch_choice(w.shapes, with_c)
    assert use == persistent
    assert kb == pytest.approx(kblocks_per_cluster(w.shapes, with_c), rel=1e-12)
    assert (kb < 800) == persistent
    # explicit choices are taken as given
    assert launch_choice(w.shapes, with_c, persistent=True)[0] is True
    assert launch_choice(w.shapes, with_c, persistent=False)[0] is False


def test_launch_choice_thresholds_and_bad_arguments():
    from muon_newton_schulz_09_b300 import MuonError
    assert launch_choice(wl.GPT2_124M.shapes)[1] == pytest.approx(25920 / 74)
    # fewer clusters: more work each, so the same set crosses over
    assert launch_choice(wl.GPT2_124M.shapes, clusters=32)[0] is False
    # beyond 1024 shape groups every mode runs the per-phase launches
    assert launch_choice([(1, k) for k in range(1, 1026)], persistent=True)[0] is False
    for kw in ({"clusters": 0},):
        with pytest.raises(MuonError):
            launch_choice([(64, 64)], **kw)
