"""Expert-sharing batch planner (host code in libmoe_ffn.so, no GPU): the
oracle's metric and greedy pinned against hand counts, closed forms and a
known optimum; the library bit-exact against the oracle; the benefit on
synthetic clustered routing (alike sequences route alike)."""
import itertools

import numpy as np
import pytest

import fp4_block_scaled_gb300 as moe
import oracle
import synth


def _lib_or_skip():
    try:
        moe.lib()
    except Exception as e:  # the library needs nvcc to build; the planner itself needs no GPU
        pytest.skip(f"library not available: {e}")


# ----------------------------------------------------------- oracle pins

def test_distinct_hand_counts():
    # 4 sequences, 1 layer, top-2: {0,1} {0,2} {3,4} {3,5}
    r = np.array([[[0, 1]], [[0, 2]], [[3, 4]], [[3, 5]]])
    assert oracle.batch_distinct(r, [0, 1, 2, 3], 2).tolist() == [[3], [3]]
    assert oracle.batch_distinct(r, [0, 2, 1, 3], 2).tolist() == [[4], [4]]
    assert oracle.batch_distinct(r, [0, 1, 2, 3], 4).tolist() == [[6]]
    assert oracle.batch_distinct(r, [3, 2, 1], 2).tolist() == [[3], [2]]      # ragged last batch
    # -1 is no expert; a repeated id counts once
    r2 = np.array([[[7, -1]], [[7, 7]]])
    assert oracle.batch_distinct(r2, [0, 1], 2).tolist() == [[1]]


def test_distinct_closed_forms():
    rng = np.random.default_rng(0)
    N, L, k, B = 12, 3, 4, 4
    same = np.tile(rng.permutation(50)[:k], (N, L, 1))
    assert np.all(oracle.batch_distinct(same, np.arange(N), B) == k)          # identical rows: k
    disjoint = np.arange(N * L * k).reshape(N, L, k)
    assert np.all(oracle.batch_distinct(disjoint, np.arange(N), B) == B * k)  # disjoint rows: B k


def test_greedy_recovers_disjoint_clusters():
    """C clusters with disjoint expert supports, B sequences each, shuffled:
    the optimum puts each cluster in one batch (distinct = the cluster's
    support per layer), and the greedy reaches it."""
    rng = np.random.default_rng(1)
    C, B, L, k, per = 4, 5, 3, 2, 6
    rows, cl = [], []
    for c in range(C):
        for _ in range(B):
            rows.append([rng.choice(np.arange(c * per, (c + 1) * per), k, replace=False) for _ in range(L)])
            cl.append(c)
    perm = rng.permutation(C * B)
    sig = np.array(rows)[perm]
    order = oracle.batch_plan_greedy(sig, B)
    assert sorted(order.tolist()) == list(range(C * B))
    clusters = np.array(cl)[perm][order].reshape(C, B)
    assert all(len(set(row)) == 1 for row in clusters)
    union = [[len(set(sig[order[b * B:(b + 1) * B], l].ravel())) for l in range(L)] for b in range(C)]
    assert np.array_equal(oracle.batch_distinct(sig, order, B), np.array(union))


def test_greedy_never_worse_than_brute_force_bound_on_tiny_cases():
    """On 6 sequences in batches of 3 the greedy's total is between the
    optimum over all partitions (brute force) and the worst one."""
    rng = np.random.default_rng(2)
    for trial in range(20):
        sig = rng.integers(0, 8, size=(6, 2, 2))
        totals = []
        for first in itertools.combinations(range(1, 6), 2):
            a = [0, *first]
            b = [i for i in range(6) if i not in a]
            totals.append(oracle.batch_distinct(sig, a + b, 3).sum())
        g = oracle.batch_distinct(sig, oracle.batch_plan_greedy(sig, 3), 3).sum()
        assert min(totals) <= g <= max(totals)


# ------------------------------------------------- library vs the oracle

@pytest.mark.parametrize("N,L,k,E,B", [(1, 1, 1, 4, 1), (7, 2, 3, 10, 3), (40, 5, 6, 64, 8), (33, 4, 2, 16, 5)])
def test_library_plan_and_metric_equal_oracle_on_random_rows(N, L, k, E, B):
    _lib_or_skip()
    rng = np.random.default_rng(N * 7 + B)
    sig = rng.integers(-1, E, size=(N, L, k)).astype(np.int32)    # includes -1 and repeats
    order = moe.moe_batch_plan(sig, E, B)
    assert np.array_equal(order, oracle.batch_plan_greedy(sig, B))
    nxt = rng.integers(-1, E, size=(N, L, k)).astype(np.int32)
    assert np.array_equal(moe.moe_batch_distinct(nxt, order, E, B), oracle.batch_distinct(nxt, order, B))


def test_library_plan_equals_oracle_on_clustered_routing():
    _lib_or_skip()
    r0, _ = synth.routing_clustered(64, 8, 384, 6, seed=3, step=0)
    for B in (8, 16, 32):
        assert np.array_equal(moe.moe_batch_plan(r0, 384, B), oracle.batch_plan_greedy(r0, B))


def test_library_rejects_bad_arguments():
    _lib_or_skip()
    sig = np.zeros((4, 1, 2), np.int32)
    sig[1, 0, 0] = 9
    with pytest.raises(moe.MoeError):
        moe.moe_batch_plan(sig, 8, 2)                        # id out of range
    with pytest.raises(moe.MoeError):
        moe.moe_batch_distinct(np.zeros((4, 1, 2), np.int32), [0, 1, 1, 3], 8, 2)   # not a permutation
    assert moe.moe_batch_plan(np.zeros((0, 1, 2), np.int32), 8, 2).size == 0


def test_planning_on_one_step_cuts_the_next_steps_distinct_experts():
    """256 sequences of 8 clusters, 40 layers, top-6 of 384, batches of 32:
    planned on step 0's routing and counted on step 1's, the batches touch
    far fewer experts per layer than batches in arrival order, and as few as
    batches formed by the (hidden) clusters themselves."""
    _lib_or_skip()
    N, L, E, k, B = 256, 40, 384, 6, 32
    r0, cl = synth.routing_clustered(N, L, E, k, seed=0, step=0)
    r1, _ = synth.routing_clustered(N, L, E, k, seed=0, step=1)
    planned = moe.moe_batch_distinct(r1, moe.moe_batch_plan(r0, E, B), E, B).mean()
    arrival = moe.moe_batch_distinct(r1, np.arange(N, dtype=np.int32), E, B).mean()
    by_cluster = moe.moe_batch_distinct(r1, np.argsort(cl, kind="stable").astype(np.int32), E, B).mean()
    print(f"distinct experts per layer: arrival {arrival:.1f}, planned {planned:.1f}, clusters {by_cluster:.1f}")
    assert planned < 0.85 * arrival
    assert planned <= 1.02 * by_cluster
