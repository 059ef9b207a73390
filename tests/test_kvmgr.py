"""The host-side block manager (pkv_kvmgr_*): its C++ implementation against
the oracle's plain Python model of the same policies, operation by operation
(every output and the whole state), and the model pinned by invariants that
follow from what a block table is (reference counts equal the holders,
free = unreferenced, slots address the table's blocks, prefix reuse returns
cached content, copy-on-write never writes a shared block)."""

import numpy as np
import pytest

from oracle.kvmgr_model import BS, NO_BLOCKS, OK, UNKNOWN_SEQ, BlockManagerModel
from paged_kv_decode_14_gb300 import _native as nat


def _random_ops(seed, n_ops, n_prompts=4):
    """A seeded stream of operations on conversations that share prompts."""
    rng = np.random.default_rng(seed)
    bases = [rng.integers(0, 50, size=int(rng.integers(20, 90))).tolist() for _ in range(n_prompts)]
    live, next_id, ops = [], 0, []
    for _ in range(n_ops):
        r = rng.random()
        if r < 0.3 or not live:
            base = bases[int(rng.integers(0, n_prompts))]
            cut = int(rng.integers(1, len(base) + 1))
            prompt = base[:cut] + rng.integers(0, 50, size=int(rng.integers(0, 40))).tolist()
            ops.append(("add", next_id, prompt))
            live.append(next_id)
            next_id += 1
        elif r < 0.65:
            s = live[int(rng.integers(0, len(live)))]
            ops.append(("append", s, rng.integers(0, 50, size=int(rng.choice([1, 1, 1, 5]))).tolist()))
        elif r < 0.78:
            ops.append(("commit", live[int(rng.integers(0, len(live)))], None))
        elif r < 0.86:
            ops.append(("fork", live[int(rng.integers(0, len(live)))], next_id))
            live.append(next_id)
            next_id += 1
        else:
            s = live.pop(int(rng.integers(0, len(live))))
            ops.append(("release", s, None))
    return ops


def _apply(m, model, op):
    kind, a, b = op
    if kind == "add":
        st = model.add_sequence(a, b)
        try:
            got = m.add_sequence(a, b)
        except nat.PagedKVError as e:
            assert e.status == st[0] != OK
            return False
        assert st[0] == OK and got[0] == st[1] and list(got[1]) == st[2]
        return True
    if kind == "append":
        st = model.append(a, b)
        try:
            slots, copy = m.append(a, b)
            assert st[0] == OK and list(slots) == st[1] and copy == st[2]
        except nat.PagedKVError as e:
            assert e.status == st[0] != OK
        return True
    if kind == "commit":
        assert model.commit(a) == OK
        m.commit(a)
        return True
    if kind == "fork":
        st = model.fork(a, b)
        try:
            m.fork(a, b)
            assert st == OK
            return True
        except nat.PagedKVError as e:
            assert e.status == st != OK
            return False
    assert model.release(a) == OK
    m.release(a)
    return True


def _check_state(m, model):
    assert m.num_free() == model.num_free()
    assert m.num_cached() == model.num_cached()
    assert [m.refcount(b) for b in range(model.num_blocks)] == model.ref
    live = sorted(model.seqs)
    if live:
        mb = max(len(s["blocks"]) for s in model.seqs.values()) or 1
        bt, lens = m.tables(live, mb)
        rows, mlens = model.tables(live, mb)
        assert bt.tolist() == rows and lens.tolist() == mlens


def _check_invariants(model):
    """What a block table means, independent of how the model gets there."""
    holders = [0] * model.num_blocks
    for s in model.seqs.values():
        assert len(s["blocks"]) == -(-len(s["tokens"]) // BS)
        for b in s["blocks"]:
            holders[b] += 1
    tree = model.tree_blocks()
    for b in range(model.num_blocks):
        assert model.ref[b] == holders[b] + (1 if b in tree else 0)
    assert sorted(model.free) == [b for b in range(model.num_blocks) if model.ref[b] == 0]
    assert len(set(model.free)) == len(model.free)


@pytest.mark.parametrize("seed,pool", [(1, 48), (2, 200), (3, 24), (4, 96)])
def test_cpp_manager_matches_model(seed, pool):
    m = nat.KVManager(pool)
    model = BlockManagerModel(pool)
    live = set()
    for op in _random_ops(seed, 500):
        kind, a, b = op
        if kind in ("append", "commit", "release", "fork") and a not in live:
            continue
        ok = _apply(m, model, op)
        if kind == "add" and ok:
            live.add(a)
        if kind == "fork" and ok:
            live.add(b)
        if kind == "release":
            live.discard(a)
        _check_state(m, model)
        _check_invariants(model)


def test_model_prefix_reuse_returns_cached_content():
    """A prompt that extends a committed sequence's tokens reuses exactly its
    full blocks (leaving one token to compute), and the reused blocks are the
    ones holding those tokens."""
    model = BlockManagerModel(64)
    prompt = list(range(100, 150))                              # 50 tokens: 3 full blocks + 2
    st, cached, slots = model.add_sequence(0, prompt)
    assert st == OK and cached == 0 and len(slots) == 50
    model.commit(0)
    st, cached, _ = model.add_sequence(1, prompt + [7, 8, 9])
    assert st == OK and cached == 48
    assert model.seqs[1]["blocks"][:3] == model.seqs[0]["blocks"][:3]
    # an exactly block-aligned cached prompt still leaves its last token to compute
    st, cached, _ = model.add_sequence(2, prompt[:48])
    assert cached == 32
    # a prompt that differs inside block 1 reuses only block 0
    other = prompt[:20] + [999] + prompt[21:]
    st, cached, _ = model.add_sequence(3, other)
    assert cached == 16 and model.seqs[3]["blocks"][0] == model.seqs[0]["blocks"][0]
    _check_invariants(model)


def test_model_copy_on_write_never_writes_a_shared_block():
    model = BlockManagerModel(16)
    model.add_sequence(0, list(range(20)))                     # block 0 full, block 1 holds 4 tokens
    model.fork(0, 1)
    last = model.seqs[0]["blocks"][-1]
    st, slots, copy = model.append(1, [5])
    assert st == OK and copy == (last, model.seqs[1]["blocks"][-1]) and copy[1] != last
    assert slots[0] // BS == copy[1]                           # the new token lands in the copy
    assert model.seqs[0]["blocks"][-1] == last                 # the parent keeps the original
    st, slots, copy = model.append(0, [6])                     # now held by the parent alone
    assert copy is None and slots[0] // BS == last
    _check_invariants(model)


def test_model_eviction_order_and_exhaustion():
    """Pool of 4: a committed, released sequence leaves blocks 0 and 1 cached;
    a new 48-token prompt takes the two free blocks and evicts the chain's
    leaf (block 1), the next block evicts block 0, and once nothing is left an
    append fails without changing anything."""
    model = BlockManagerModel(4)
    assert model.add_sequence(0, list(range(33)))[0] == OK     # blocks 0, 1, 2
    model.commit(0)                                            # full blocks 0, 1 -> tree
    model.release(0)                                           # block 2 freed; 0 and 1 stay cached
    assert model.num_free() == 2 and model.tree_blocks() == {0, 1}
    st, cached, _ = model.add_sequence(1, list(range(500, 548)))
    assert st == OK and cached == 0
    assert model.seqs[1]["blocks"] == [2, 3, 1] and model.tree_blocks() == {0}
    st, slots, _ = model.append(1, [1])                         # a 4th block: evicts block 0
    assert st == OK and slots == [0 * BS] and model.tree_blocks() == set()
    assert model.append(1, list(range(15)))[0] == OK           # fills block 0
    before = (list(model.free), list(model.ref), list(model.seqs[1]["blocks"]), len(model.seqs[1]["tokens"]))
    assert model.append(1, [2])[0] == NO_BLOCKS
    assert before == (list(model.free), list(model.ref), list(model.seqs[1]["blocks"]), len(model.seqs[1]["tokens"]))
    _check_invariants(model)
    # the library agrees step by step
    m = nat.KVManager(4)
    m.add_sequence(0, list(range(33)))
    m.commit(0)
    m.release(0)
    m.add_sequence(1, list(range(500, 548)))
    m.append(1, [1])
    m.append(1, list(range(15)))
    with pytest.raises(nat.PagedKVError) as e:
        m.append(1, [2])
    assert e.value.status == NO_BLOCKS
    bt, lens = m.tables([1], 4)
    assert bt.tolist() == [[2, 3, 1, 0]] and lens.tolist() == [64]


def test_unknown_and_duplicate_ids():
    m = nat.KVManager(8)
    with pytest.raises(nat.PagedKVError) as e:
        m.append(3, [1])
    assert e.value.status == UNKNOWN_SEQ
    m.add_sequence(1, [1, 2, 3])
    with pytest.raises(nat.PagedKVError) as e:
        m.add_sequence(1, [4])
    assert e.value.status == UNKNOWN_SEQ
    with pytest.raises(nat.PagedKVError) as e:
        m.fork(1, 1)
    assert e.value.status == UNKNOWN_SEQ
