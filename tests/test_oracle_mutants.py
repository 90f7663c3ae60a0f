"""Planted mistakes: each test compiles a copy of the oracle with one plausible bug and checks
that the pins (brute force, closed forms, the worked example, a textbook core algorithm,
networkx) catch it.  The unmodified source is the control and must pass the same battery.

Mistakes are planted in a temporary copy of the oracle source on the CPU only.
"""
import os
import subprocess
import sys
import textwrap

import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

BATTERY = textwrap.dedent("""
    import sys, numpy as np
    sys.path.insert(0, %(root)r)
    import oracle as O
    from maximal_clique_enumeration_gb300 import graphs as G
    from tests import pins
    o = O.Oracle(sys.argv[1])
    n, edges, cliques, info = pins.load_golden("fig1_example.txt")
    g = G.csr_from_edges(n, *zip(*edges))
    assert sorted(o.enumerate_cliques(g)) == cliques
    assert o.count(g).key() == pins.summary(cliques)
    for seed in range(2):
        for p in (0.3, 0.6, 0.9):
            g = G.er_graph(10, p, seed)
            ex = pins.brute_subsets(g)
            assert sorted(o.enumerate_cliques(g)) == ex
            assert o.count(g).key() == pins.summary(ex)
    for g, cnt, k in [(G.moon_moser(4), 81, 4), (G.complete_graph(6), 1, 6),
                      (G.empty_graph(5), 5, 1), (G.path_graph(5), 4, 2)]:
        r = o.count(g)
        assert r.count == cnt and r.key()[2] == tuple([0] * k + [cnt])
        r = o.count(g, variant=O.ALG4_TOMITA)
        assert r.count == cnt and r.key()[2] == tuple([0] * k + [cnt])
    for seed in range(2):
        for p in (0.3, 0.6, 0.9):
            g = G.er_graph(10, p, seed)
            assert sorted(o.enumerate_cliques(g, variant=O.ALG4_TOMITA)) == pins.brute_subsets(g)
    for fx in ("peel_fig1.txt", "peel_k4_tails.txt"):
        n, edges, expect, info = pins.load_peel_golden(fx)
        core, rnd, rank, d = o.peel(G.csr_from_edges(n, *zip(*edges)))
        assert d == info["degeneracy"] and int(rnd.max()) + 1 == info["rounds"]
        assert all((int(rnd[v]), int(core[v]), int(rank[v])) == e for v, e in expect.items())
    import networkx as nx
    for name in ("er200", "rmat_s9"):
        g = G.config_graph(name, 1)
        core, rnd, rank, d = o.peel(g)
        assert np.array_equal(core, O.core_bz(g))
        key = rnd.astype(np.int64) * g.n + np.arange(g.n)
        assert np.array_equal(np.argsort(key, kind="stable"), np.argsort(rank, kind="stable"))
        h = nx.Graph(); h.add_nodes_from(range(g.n))
        h.add_edges_from(zip(*[x.tolist() for x in G.edges_of(g)]))
        ex = [tuple(sorted(c)) for c in nx.find_cliques(h)]
        assert o.count(g).key() == pins.summary(ex)
    print("battery passed")
""") % {"root": ROOT}

MUTANTS = {
    "report_without_X_check": ("if (nx == 0) report(c);", "report(c);"),
    "branch_on_pivot_neighbours": ("if (!contains_sorted(np_, dp, P[i])) cand[nc++] = P[i];",
                                   "if (contains_sorted(np_, dp, P[i])) cand[nc++] = P[i];"),
    "X_not_extended": ("        curX[at] = v;\n        ncx++;", "        curX[at] = v;\n"),
    "P_not_reduced": ("if (curP[i] != v) curP[w++] = curP[i];", "curP[w++] = curP[i];"),
    "first_level_drops_X": ("bk(c, nv + split, dv - split, nv, split);",
                            "bk(c, nv + split, dv - split, nv, 0);"),
    "first_level_all_neighbours_in_P": ("bk(c, nv + split, dv - split, nv, split);",
                                        "bk(c, nv, dv, NULL, 0);"),
    "merge_advances_wrong_side": ("else if (a[i] > b[j]) ++j;", "else if (a[i] > b[j]) ++i;"),
    "hash_xor_instead_of_sum": ("s += oracle_vertex_key(ids[i]);", "s ^= oracle_vertex_key(ids[i]);"),
    "vertex_key_off_by_one": ("((uint64_t)(uint32_t)id + 1ULL)", "((uint64_t)(uint32_t)id)"),
    "hist_index_off_by_one": ("else c->hist[k]++;", "else c->hist[k - 1]++;"),
    "peel_strict_threshold": ("if (curdeg[alive[i]] <= k) batch[nb++] = alive[i];",
                              "if (curdeg[alive[i]] < k) batch[nb++] = alive[i];"),
    "core_is_round_not_level": ("rnd[batch[i]] = r; core[batch[i]] = k;",
                                "rnd[batch[i]] = r; core[batch[i]] = r;"),
    # a level's vertices removed one at a time in id order (each removal updating its
    # neighbours at once, so a neighbour later in the sweep can join the same round)
    "peel_one_at_a_time_within_a_round": (
        "        for (int32_t i = 0; i < n_alive; ++i)\n"
        "            if (curdeg[alive[i]] <= k) batch[nb++] = alive[i];\n"
        "        if (nb == 0) { ++k; continue; }\n"
        "        for (int32_t i = 0; i < nb; ++i) { rnd[batch[i]] = r; core[batch[i]] = k; }\n"
        "        for (int32_t i = 0; i < nb; ++i) {\n"
        "            int32_t v = batch[i];\n"
        "            for (int64_t e = offs[v]; e < offs[v + 1]; ++e)\n"
        "                if (rnd[adj[e]] < 0) curdeg[adj[e]]--;\n"
        "        }\n",
        "        for (int32_t i = 0; i < n_alive; ++i) {\n"
        "            int32_t v = alive[i];\n"
        "            if (curdeg[v] > k) continue;\n"
        "            batch[nb++] = v; rnd[v] = r; core[v] = k;\n"
        "            for (int64_t e = offs[v]; e < offs[v + 1]; ++e)\n"
        "                if (rnd[adj[e]] < 0) curdeg[adj[e]]--;\n"
        "        }\n"
        "        if (nb == 0) { ++k; continue; }\n"),
    "rank_counting_sort_shift": ("for (int32_t v = 0; v < n; ++v) start[rnd[v] + 1]++;",
                                 "for (int32_t v = 0; v < n; ++v) start[rnd[v]]++;"),
    "second_level_X_split_at_first_vertex": ("while (split < k && common[split] < q) ++split;",
                                             "while (split < k && common[split] < p) ++split;"),
    "second_level_drops_X": ("bk(c, common + split, k - split, common, split);",
                             "bk(c, common + split, k - split, common, 0);"),
    "second_level_misses_isolated": ("        bk(c, NULL, 0, NULL, 0);\n", "\n"),
}


def _build_variant(tmp_path, name, mutation):
    src = open(os.path.join(ROOT, "oracle", "mce_oracle.c")).read()
    if mutation is not None:
        old, new = mutation
        assert src.count(old) == 1, f"mutation anchor for {name} not unique/absent"
        src = src.replace(old, new)
    path = tmp_path / f"{name}.c"
    path.write_text(src)
    return O.build(force=True, src=str(path), out=str(tmp_path / f"lib{name}.so"))


def _battery(lib):
    return subprocess.run([sys.executable, "-c", BATTERY, lib], capture_output=True, text=True,
                          timeout=300, cwd=ROOT)


def test_unmutated_oracle_passes_battery(tmp_path):
    r = _battery(_build_variant(tmp_path, "control", None))
    assert r.returncode == 0, r.stderr[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    r = _battery(_build_variant(tmp_path, name, MUTANTS[name]))
    assert r.returncode != 0, f"mutant {name} survived the pins"
