"""The expert cache's slot policy (host only, no GPU) against an independent model:
experts visited in order of first appearance, a hit refreshes its use time, a miss
takes the lowest free slot or evicts the least recently used expert the pass does not
need; a call with more distinct experts than slots runs in passes of at most that many
experts, those resident at the start of the call first; an id outside [0, E) is
refused."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__

    __graft_entry__._builder().build()
    import mixture_experts_layer_scan_gb300 as m

    return m


def lru_model(E, S, calls):
    slot_expert = [-1] * S
    expert_slot = {}
    last = [0] * S
    clock = hits = misses = 0
    slot_ids, loaded = [], []
    for ids in calls:
        needed = list(dict.fromkeys(int(e) for e in ids))
        if len(needed) <= S:
            passes = [needed]
        else:
            order = [e for e in needed if e in expert_slot] + [e for e in needed if e not in expert_slot]
            passes = [order[i:i + S] for i in range(0, len(order), S)]
        ld = [-1] * S
        sl_of = {}
        for group in passes:
            for e in group:
                if e in expert_slot:
                    hits += 1
                    s = expert_slot[e]
                else:
                    misses += 1
                    free = [c for c in range(S) if slot_expert[c] < 0]
                    if free:
                        s = free[0]
                    else:
                        s = min((c for c in range(S) if slot_expert[c] not in group), key=lambda c: last[c])
                        del expert_slot[slot_expert[s]]
                    slot_expert[s] = e
                    expert_slot[e] = s
                    ld[s] = e
                clock += 1
                last[s] = clock
            for e in group:
                sl_of[e] = expert_slot[e]
        slot_ids.append([sl_of[int(e)] for e in ids])
        loaded.append(ld)
    return np.array(slot_ids, dtype=np.int32), np.array(loaded, dtype=np.int32), hits, misses


def _zipf_calls(E, n_calls, T, k, seed, s=1.1):
    g = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** s
    p /= p.sum()
    perm = g.permutation(E)
    calls = []
    for _ in range(n_calls):
        rows = [perm[g.choice(E, size=k, replace=False, p=p)] for _ in range(T)]
        calls.append(np.concatenate(rows))
    return np.stack(calls).astype(np.int32)


@pytest.mark.parametrize("E,S,T,k,seed", [(16, 6, 1, 2, 0), (128, 48, 4, 8, 1), (64, 40, 4, 8, 2), (8, 8, 3, 2, 3),
                                          (32, 4, 2, 2, 4), (64, 12, 4, 8, 5), (128, 48, 16, 8, 6), (16, 3, 3, 2, 7)])
def test_policy_matches_model(moe, E, S, T, k, seed):
    calls = _zipf_calls(E, 40, T, k, seed)
    got = moe.moe_cache_lru_plan(E, S, calls)
    want = lru_model(E, S, calls)
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1], want[1])
    assert got[2:] == want[2:]
    if all(len(set(c.tolist())) <= S for c in calls):
        # one pass per call: no slot holds two experts within a call
        for ids, sl in zip(calls, got[0]):
            m = {}
            for e, s in zip(ids, sl):
                assert m.setdefault(int(s), int(e)) == int(e)


def test_hits_plus_misses_count_distinct_experts(moe):
    calls = _zipf_calls(64, 25, 4, 8, 9)
    _, loaded, hits, misses = moe.moe_cache_lru_plan(64, 32, calls)
    assert hits + misses == sum(len(set(c.tolist())) for c in calls)
    assert misses == int((loaded >= 0).sum())


def test_more_experts_than_slots_run_in_passes(moe):
    # 2 of 3 slots hold experts 5 and 6; the next call needs 0, 1, 5, 2, 6: passes [5, 6, 0], [1, 2]
    calls = np.array([[5, 6, 5, 5, 6, 6], [0, 1, 5, 2, 6, 0]], dtype=np.int32)
    slot_ids, loaded, hits, misses = moe.moe_cache_lru_plan(16, 3, calls)
    # call 0: 5 -> slot 0, 6 -> slot 1.  call 1, pass 1: 5, 6 hit, 0 -> free slot 2;
    # pass 2: 1 evicts the oldest of {5, 6} (5, slot 0), 2 evicts 6 (slot 1)
    assert slot_ids[1].tolist() == [2, 0, 0, 1, 1, 2]
    assert loaded[1].tolist() == [1, 2, 0]
    assert (hits, misses) == (2, 5)


def test_policy_refusals(moe):
    with pytest.raises(moe.MoeError) as e:
        moe.moe_cache_lru_plan(16, 8, np.array([[0, 16]], dtype=np.int32))
    assert e.value.code == moe.MOE_ERR_DEVICE_INDEX
