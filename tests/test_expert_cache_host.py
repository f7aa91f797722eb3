"""The expert cache's slot policy on the host (no GPU): least recently used
replacement keyed by (layer, expert), never evicting a slot the same call
needs, and a refused call (more distinct experts than slots) leaving nothing
marked resident that was not copied."""
from collections import OrderedDict

import numpy as np
import pytest

import bit_quantized_moe_bias_b300 as B

sim = B.ds4g_expert_lru_simulate


def test_hand_worked_sequence():
    # 6 empty slots are handed out from the last one down
    slots, miss = sim(6, [[1, 2, 3, 4, 5, 6], [1, 7, -1, 1], [8, 9]])
    assert slots[0] == [5, 4, 3, 2, 1, 0] and all(miss[0])
    # 1 is resident; 7 evicts the least recently used key (2, slot 4); a
    # skipped key has no slot; the repeat of 1 is not copied again
    assert slots[1] == [5, 4, -1, 5] and miss[1] == [False, True, False, False]
    # then 3 (slot 3) and 4 (slot 2) are the least recent
    assert slots[2] == [3, 2] and miss[2] == [True, True]


def _key_model(n, calls):
    """Misses of an LRU over keys: a call's keys become most recent in the
    order of their first appearance in it; a missing key evicts the least
    recent key that the call has not used (None if there is none: the call
    is refused)."""
    lru = OrderedDict()   # key -> None, least recent first
    out = []
    for keys in calls:
        used, flags, placed = set(), [], []
        ok = True
        for k in keys:
            if k < 0:
                flags.append(False)
                continue
            if k in lru:
                if k not in used:
                    lru.move_to_end(k)
                flags.append(False)
            else:
                if len(lru) >= n:
                    victim = next((v for v in lru if v not in used), None)
                    if victim is None:
                        ok = False
                        break
                    del lru[victim]
                lru[k] = None
                placed.append(k)
                flags.append(True)
            used.add(k)
        if not ok:
            for k in placed:   # nothing was copied for them
                del lru[k]
            flags = None
        out.append(flags)
    return out


@pytest.mark.parametrize("seed", range(5))
def test_random_calls_match_an_lru_over_keys(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(6, 12))
    calls = []
    for _ in range(60):
        size = int(rng.integers(1, 2 * n))
        keys = rng.integers(-1, 3 * n, size).tolist()      # repeats and skipped keys included
        calls.append([int(k) for k in keys])
    slots, miss = sim(n, calls)
    model = _key_model(n, calls)
    holder = {}   # slot -> key it holds
    for keys, s, m, ref in zip(calls, slots, miss, model):
        if ref is None:   # refused: the slots it had taken are empty again (the model forgets those keys)
            assert all(v == -2 for v in s)
            continue
        assert m == ref
        seen = {}
        for k, sl in zip(keys, s):
            if k < 0:
                assert sl == -1
                continue
            assert 0 <= sl < n
            assert seen.setdefault(k, sl) == sl         # one slot per key within a call
            if not m[keys.index(k)]:
                assert holder.get(sl) == k              # a hit finds its own slot
        assert len(set(seen.values())) == len(seen)     # distinct keys, distinct slots
        for k, sl in seen.items():
            holder[sl] = k


def test_refused_call_forgets_what_it_placed():
    # 6 slots; the second call needs 7 distinct keys: refused after it had
    # evicted 0, 1, 2 for 6, 7, 8, so 3..8 are forgotten and 0..2 are gone
    slots, miss = sim(6, [[0, 1, 2], [3, 4, 5, 6, 7, 8, 9], [0], [3], [1, 2]])
    assert slots[1] == [-2] * 7
    assert miss[2] == [True] and miss[3] == [True] and miss[4] == [True, True]
    # a refused call that had only hits changes nothing
    slots, miss = sim(6, [[0, 1, 2, 3, 4, 5], [0, 1, 2, 3, 4, 5, 6], [5, 4, 3, 2, 1, 0]])
    assert slots[1] == [-2] * 7 and not any(miss[2])


def test_keys_are_per_layer():
    # the same expert id of two layers is two keys (key = layer * 256 + e)
    slots, miss = sim(6, [[0 * 256 + 7], [1 * 256 + 7], [0 * 256 + 7]])
    assert miss == [[True], [True], [False]]
    assert slots[0] == slots[2] != slots[1]


def test_host_checks_before_any_cuda_call():
    L = B.lib()
    assert L.ds4g_expert_cache_pool_bytes(0, 2, 8) == 0          # IQ2 + Q4_K: unsupported
    assert L.ds4g_expert_cache_pool_bytes(0, 1, 0) == 0
    q2 = L.ds4g_expert_cache_pool_bytes(0, 1, 8)
    q4 = L.ds4g_expert_cache_pool_bytes(2, 2, 8)
    # slots, the [3][256] pointer table (6 KB) and 256 B of ready flags
    assert q2 == 8 * (2 * 2162688 + 2752512) + 6144 + 256 and q4 == 8 * 3 * 4718592 + 6144 + 256
    import ctypes as C
    h = C.c_void_p()
    fake = 0x10000000
    assert L.ds4g_expert_cache_create(0, 1, 5, 1, fake, q2, C.byref(h)) == 1      # fewer than 6 slots
    assert L.ds4g_expert_cache_create(0, 1, 8, 0, fake, q2, C.byref(h)) == 1      # max_tokens < 1
    assert L.ds4g_expert_cache_create(0, 2, 8, 1, fake, q2, C.byref(h)) == 5
    assert L.ds4g_expert_cache_create(0, 1, 8, 1, fake + 8, q2, C.byref(h)) == 2
    assert L.ds4g_expert_cache_create(0, 1, 8, 1, fake, q2 - 1, C.byref(h)) == 3
    assert L.ds4g_expert_cache_destroy(None) == 1
    assert L.ds4g_moe_forward_streamed(fake, 1, 0, None, fake, fake, fake, fake, fake, fake, fake, None, fake,
                                       1 << 30, None) == 1
