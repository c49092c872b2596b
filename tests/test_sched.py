"""Expert-sharing batch planner (host code in libmoe_ffn.so, no GPU): the
oracle's metric and greedy pinned against hand counts, closed forms and a
known optimum; the library bit-exact against the oracle; the benefit on
synthetic clustered routing (alike sequences route alike)."""
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


# Hand-worked plans.  Each case is built so that one plausible misreading of
# the greedy rule gives a different order than the rule itself: a batch
# starts from the lowest-numbered unplaced sequence; the next member is the
# unplaced sequence adding the fewest experts not yet in the batch, counted
# per layer and summed over the layers; ties go to the lower number.
HAND_PLANS = [
    # tie-break: from seed 0 {0,1}, sequences 2 {0,5} and 3 {1,6} both add one
    # expert (1 adds two); the lower number, 2, joins.  (Ties to the higher
    # number would give 0 3 1 2.)
    ("ties go to the lower number", [[[0, 1]], [[2, 3]], [[0, 5]], [[1, 6]]], 2, [0, 2, 1, 3]),
    # per-layer sets: sequence 1 routes to {2} then {1}, sequence 2 to {1}
    # then {3}.  Counted per layer, 1 adds two experts and 2 adds one, so 2
    # joins; pooling the ids of all layers into one set would make 1 add
    # nothing and join first (0 1 2).
    ("experts are counted per layer", [[[1], [2]], [[2], [1]], [[1], [3]]], 2, [0, 2, 1]),
    # summed over layers: 1 adds {2,3} in layer 0 and nothing in layer 1 (sum
    # 2, largest layer 2); 2 adds {4} and {12} (sum 2, largest layer 1).  The
    # sums tie and the lower number, 1, joins; taking the largest layer's count
    # instead would pick 2.
    ("costs are summed over the layers", [[[0, 1], [10, 11]], [[2, 3], [10, 11]], [[0, 4], [10, 12]]], 3, [0, 1, 2]),
    # the second batch starts from the lowest unplaced sequence (2), not from
    # the best remaining pair: 1 and 3 share {2,3}, but 1 already sits in the
    # first batch, so the greedy pays 4 + 4 where 0 2 | 1 3 would pay 4 + 2.
    ("each batch starts from the lowest unplaced number", [[[0, 1]], [[2, 3]], [[4, 5]], [[2, 3]]], 2, [0, 1, 2, 3]),
    # growth uses the batch's union so far, not the seed alone: after 0 {0,1}
    # takes 1 {0,2} (adds 1; 2 {3,4} and 3 {2,5} add 2), sequence 3 adds only
    # {5} to {0,1,2} while 2 adds {3,4}, so 3 joins before 2.
    ("growth counts against the batch so far", [[[0, 1]], [[0, 2]], [[3, 4]], [[2, 5]]], 3, [0, 1, 3, 2]),
    # -1 is no expert: 2 {9,-1} adds one expert, 1 {9,10} two, so 2 joins
    # (counting -1 as an expert would tie them and take 1)
    ("-1 is no expert", [[[7, 8]], [[9, 10]], [[9, -1]]], 2, [0, 2, 1]),
    # a repeated id adds once: 2 {9,9} adds one expert, 1 {9,10} two
    ("a repeated id counts once", [[[7, 8]], [[9, 10]], [[9, 9]]], 2, [0, 2, 1]),
]


@pytest.mark.parametrize("what,sig,B,order", HAND_PLANS, ids=[h[0] for h in HAND_PLANS])
def test_greedy_hand_worked_plans(what, sig, B, order):
    assert oracle.batch_plan_greedy(np.array(sig), B).tolist() == order, what


@pytest.mark.parametrize("what,sig,B,order", HAND_PLANS, ids=[h[0] for h in HAND_PLANS])
def test_library_greedy_hand_worked_plans(what, sig, B, order):
    _lib_or_skip()
    sig = np.array(sig, np.int32)
    E = int(sig.max()) + 1
    assert moe.moe_batch_plan(sig, E, B).tolist() == order, what


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
