"""The adapter slot manager's policy (no GPU: the manager runs without device
stores and only tracks the assignment).  vLLM offline multi-LoRA page, step 2:
max_loras GPU slots and max_cpu_loras host-cached adapters; "limits": a rank
above the slot rank cannot load."""
import numpy as np
import pytest

from lora_serving_gb300 import abi

H_IN, WIDTH = [64, 32], [48, 16]


def _adapter(rng, r):
    A = [rng.integers(0, 1 << 16, (r, h), dtype=np.uint16) & 0x3FFF for h in H_IN]
    B = [rng.integers(0, 1 << 16, (w, r), dtype=np.uint16) & 0x3FFF for w in WIDTH]
    return A, B


def _manager(n_slots=3, r_slot=16, max_cpu=6, n_adapters=5, seed=0):
    abi.load()
    m = abi.SlotManager(H_IN, WIDTH, n_slots, r_slot, max_cpu)
    rng = np.random.default_rng(seed)
    for k in range(n_adapters):
        A, B = _adapter(rng, 8 + k)
        m.register(k, A, B, 8 + k, 2.0 * (8 + k))
    return m


def test_rank_above_slot_rank_rejected_and_nothing_changes():
    m = _manager()
    before = m.stats()
    A, B = _adapter(np.random.default_rng(1), 24)
    with pytest.raises(abi.LoraError) as e:
        m.register(99, A, B, 24, 48.0)
    assert e.value.name == "LORA_ERR_RANK_EXCEEDS_SLOT"
    assert m.stats() == before and m.slot_of(99) == -1


def test_batch_maps_ids_to_distinct_slots_and_base_stays_base():
    m = _manager()
    slots = m.acquire([0, 1, -1, 0, 1])
    assert slots[2] == -1 and slots[0] == slots[3] and slots[1] == slots[4] and slots[0] != slots[1]
    assert set(slots[[0, 1]]) <= {0, 1, 2}
    st = m.stats()
    assert st["loads"] == 2 and st["hits"] == 0


def test_resident_adapters_are_hits_without_reload():
    m = _manager()
    first = m.acquire([0, 1])
    again = m.acquire([1, 0, 1])
    assert again[0] == first[1] and again[1] == first[0]
    st = m.stats()
    assert st["loads"] == 2 and st["hits"] == 2


def test_free_slots_then_least_recently_used_slot():
    m = _manager(n_slots=3)
    m.acquire([0])
    m.acquire([1])
    m.acquire([2])                   # all three slots taken, 0 least recently used
    s3 = m.acquire([3])[0]
    assert m.slot_of(0) == -1 and s3 >= 0       # 0 gave up its slot
    assert m.slot_of(1) >= 0 and m.slot_of(2) >= 0
    assert m.stats()["slot_evictions"] == 1


def test_never_evicts_an_adapter_the_batch_needs():
    m = _manager(n_slots=3)
    m.acquire([0, 1, 2])
    m.acquire([1])                   # 0 and 2 now older than 1
    slots = m.acquire([4, 0, 2])     # 4 must take 1's slot, the only one the batch does not name
    assert len(set(slots.tolist())) == 3
    assert m.slot_of(1) == -1 and m.slot_of(0) >= 0 and m.slot_of(2) >= 0


def test_too_many_adapters_or_unknown_id_rejected_unchanged():
    m = _manager(n_slots=3)
    m.acquire([0, 1])
    state = [m.slot_of(k) for k in range(5)]
    before = m.stats()
    with pytest.raises(abi.LoraError) as e:
        m.acquire([0, 1, 2, 3])
    assert e.value.name == "LORA_ERR_SLOT_RANGE"
    with pytest.raises(abi.LoraError) as e:
        m.acquire([0, 42])
    assert e.value.name == "LORA_ERR_INVALID_ARG"
    assert [m.slot_of(k) for k in range(5)] == state and m.stats() == before


def test_host_cache_drops_least_recently_used_non_resident_adapter():
    m = _manager(n_slots=2, max_cpu=4, n_adapters=4)
    m.acquire([0, 1])                # 0 and 1 resident
    A, B = _adapter(np.random.default_rng(5), 8)
    m.register(10, A, B, 8, 16.0)    # full: drops 2 (oldest not resident)
    assert m.stats()["host_evictions"] == 1
    with pytest.raises(abi.LoraError) as e:
        m.acquire([2])               # no longer registered
    assert e.value.name == "LORA_ERR_INVALID_ARG"
    assert m.slot_of(0) >= 0 and m.slot_of(1) >= 0
    m.acquire([10, 3])               # the newcomer and 3 can still load


def test_cache_full_of_resident_adapters_rejects_register():
    m = _manager(n_slots=2, max_cpu=2, n_adapters=2)
    m.acquire([0, 1])
    A, B = _adapter(np.random.default_rng(6), 8)
    with pytest.raises(abi.LoraError) as e:
        m.register(7, A, B, 8, 16.0)
    assert e.value.name == "LORA_ERR_SLOT_RANGE"


def test_reregistering_a_resident_adapter_reloads_it_in_place():
    m = _manager()
    s = m.acquire([3])[0]
    A, B = _adapter(np.random.default_rng(7), 4)
    m.register(3, A, B, 4, 8.0)
    assert m.acquire([3])[0] == s
    st = m.stats()
    assert st["loads"] == 2 and st["hits"] == 0


def test_create_validates_arguments():
    abi.load()
    with pytest.raises(abi.LoraError):
        abi.SlotManager(H_IN, WIDTH, n_slots=4, r_slot=16, max_cpu=3)      # cache smaller than the slots
    with pytest.raises(abi.LoraError) as e:
        abi.SlotManager(H_IN, WIDTH, n_slots=2, r_slot=136, max_cpu=4)
    assert e.value.name == "LORA_ERR_RANK_EXCEEDS_SLOT"
    with pytest.raises(abi.LoraError) as e:
        abi.SlotManager([60], [16], n_slots=2, r_slot=16, max_cpu=4)        # h_in not a multiple of 8
    assert e.value.name == "LORA_ERR_ALIGNMENT"
