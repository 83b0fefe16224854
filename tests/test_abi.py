"""The C ABI without a GPU: exported symbols, blob sizes and bytes against the oracle's own
writer, argument checks, and the bounded pool's slot policy against a brute-force simulator."""
import ctypes
import os
import re

import numpy as np
import pytest

from int4_routed_expert_05_b300 import moe, synth
from int4_routed_expert_05_b300.resident import moe_shape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from int4_routed_expert_05_b300 import _build
    _build.build()
    return moe.load()


def _declared_functions(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions("moe.h")
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(moe.ENTRY_POINTS)


def test_exports_every_hybrid_symbol(lib):
    headers = sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))
    assert headers == ["hybrid.h", "moe.h"]
    names = _declared_functions("hybrid.h")
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(moe.HYBRID_ENTRY_POINTS)


def test_hybrid_host_checks_without_a_gpu(lib):
    # shape and argument checks run on the host before any CUDA call
    bad = moe.GdnShape(16, 32, 64, 128)
    with pytest.raises(moe.MoeError) as e:
        moe.gdn_step(bad, 1, *([16] * 10), 1.0, 16)
    assert e.value.status == moe.E_SHAPE
    good = moe.GdnShape(16, 32, 128, 128)
    with pytest.raises(moe.MoeError) as e:
        moe.gdn_step(good, 1, *([16] * 9), 8, 1.0, 16)   # misaligned norm weight pointer
    assert e.value.status == moe.E_INVALID
    sh = moe.GqaShape(16, 2, 256, 8192)
    assert moe.gqa_workspace_bytes(sh, 1, 8192) == 2 * 74 * 8 * (256 + 2) * 4
    assert moe.gqa_workspace_bytes(sh, 1, 8193) == 0
    assert moe.gqa_workspace_bytes(moe.GqaShape(16, 2, 96, 64), 1, 8) == 0
    assert moe.gqa_workspace_bytes(moe.GqaShape(12, 2, 256, 64), 1, 8) == 0   # 6 query heads per K/V head
    with pytest.raises(moe.MoeError) as e:
        moe.gqa_decode(sh, 1, 8192, *([16] * 7), 1.0, 16, 100, 16, 16)
    assert e.value.status == moe.E_NOMEM


@pytest.mark.parametrize("sh", [synth.TINY, synth.TINY.with_bits(8), synth.S80, synth.S35.with_bits(8)])
def test_blob_sizes_match_oracle(lib, orc, sh):
    ms = moe_shape(sh)
    assert moe.expert_bytes(ms) == orc.blob_bytes(sh)
    assert moe.expert_stride(ms) == orc.blob_stride(sh)
    assert moe.expert_stride(ms, shared=True) == orc.blob_stride(sh, shared=True)


@pytest.mark.parametrize("sh", [synth.TINY, synth.TINY.with_bits(8), synth.S80])
def test_pack_matches_oracle_writer(lib, orc, sh):
    """The library's packer and the oracle's own writer produce the same bytes."""
    for e, shared in ((3, False), (synth.SHARED_EXPERT, True)):
        t = synth.expert_tensors(sh, 9, 1, e)
        a = moe.pack_expert(moe_shape(sh), t, shared=shared)
        b = orc.pack(sh, t, shared=shared)
        assert np.array_equal(a, b)


def test_shape_and_argument_errors(lib):
    bad = moe.make_shape(300, 16, 2, 64, 64)
    with pytest.raises(moe.MoeError) as ei:
        moe.pack_expert(bad, synth.expert_tensors(synth.TINY, 0, 0, 0))
    assert ei.value.status == moe.E_SHAPE
    t = synth.expert_tensors(synth.TINY, 0, 0, 0)
    t["gate_q"] = t["gate_q"].copy()
    t["gate_q"][0, 0] = 16
    with pytest.raises(moe.MoeError) as ei:
        moe.pack_expert(moe_shape(synth.TINY), t)
    assert ei.value.status == moe.E_INVALID
    for args in [(17, 16, 2, 64, 64), (256, 16, 17, 64, 64), (256, 513, 2, 64, 64), (256, 16, 2, 96, 64)]:
        with pytest.raises(moe.MoeError):
            moe.Pool(moe.make_shape(*args), 1, 4)
    assert moe.workspace_bytes(moe_shape(synth.S80), 48) > 0


def _host_pool(n_slots, layers=4, experts=16):
    sh = moe.make_shape(256, experts, 2, 64, 64)
    return moe.Pool(sh, layers, n_slots)


def test_policy_matches_bruteforce_simulator(lib):
    from oracle.pool_sim import PoolSim
    rng = np.random.default_rng(0)
    for n_slots, trace_kind in [(6, "uniform"), (12, "zipf"), (3, "zipf")]:
        pool = _host_pool(n_slots)
        pool.set_copy_hook(lambda slot, blob, n: 0)
        sim = PoolSim(n_slots)
        blob = np.zeros(16, np.uint8)
        for step in range(300):
            layer = int(rng.integers(0, 4))
            if trace_kind == "uniform":
                ex = rng.choice(16, size=2, replace=False)
            else:
                p = 1.0 / np.arange(1, 17) ** 1.1
                ex = rng.choice(16, size=2, replace=False, p=p / p.sum())
            got = list(pool.lookup(layer, ex))
            want = sim.lookup(layer, ex)
            assert got == want, (step, got, want)
            for e, s in zip(ex, got):
                if s < 0:
                    ws = sim.load(layer, int(e))
                    if ws is None:
                        with pytest.raises(moe.MoeError) as ei:
                            pool.load_slot(layer, int(e), blob)
                        assert ei.value.status == moe.E_POOL_FULL
                    else:
                        assert pool.load_slot(layer, int(e), blob) == ws
            for l in range(4):
                for e in range(16):
                    k = sim.slot_of((l, e))
                    assert pool.slot_of(l, e) == k
            pool.release()
            sim.release()
        hits, misses, nbytes = pool.stats()
        assert hits + misses == 600


def test_pool_full_when_everything_pinned(lib):
    pool = _host_pool(2)
    pool.set_copy_hook(lambda slot, blob, n: 0)
    blob = np.zeros(16, np.uint8)
    pool.lookup(0, [1, 2, 3])
    assert pool.load_slot(0, 1, blob) == 0
    assert pool.load_slot(0, 2, blob) == 1
    with pytest.raises(moe.MoeError) as ei:
        pool.load_slot(0, 3, blob)
    assert ei.value.status == moe.E_POOL_FULL
    pool.release()
    assert pool.load_slot(0, 3, blob) in (0, 1)


def test_injected_copy_failure_leaves_pool_unchanged(lib):
    pool = _host_pool(4)
    blob = np.zeros(16, np.uint8)
    calls = []
    pool.set_copy_hook(lambda slot, b, n: calls.append(slot) or 0)
    pool.lookup(1, [5])
    s = pool.load_slot(1, 5, blob)
    pool.release()
    before = [[pool.slot_of(l, e) for e in range(16)] for l in range(4)]
    pool.set_copy_hook(lambda slot, b, n: 1)
    pool.lookup(2, [7])
    with pytest.raises(moe.MoeError) as ei:
        pool.load_slot(2, 7, blob)
    assert ei.value.status == moe.E_CUDA
    after = [[pool.slot_of(l, e) for e in range(16)] for l in range(4)]
    assert before == after and pool.slot_of(1, 5) == s and calls == [s]


def test_batched_workspace_bytes(lib):
    """The batched workspace query is host-only: zero for no tokens, grows with the token count,
    and holds at least the token-major buffers the layout names (input rows and h rows in
    assignment order, logits)."""
    ms = moe_shape(synth.S80)
    assert moe.batched_workspace_bytes(ms, 0) == 0
    assert moe.batched_workspace_bytes(ms, -3) == 0
    sizes = [moe.batched_workspace_bytes(ms, t) for t in (1, 8, 64, 512, 4096)]
    assert all(b % 256 == 0 for b in sizes)
    assert sizes == sorted(sizes) and len(set(sizes)) == len(sizes)
    H, E, k, Imax = synth.S80.hidden, synth.S80.n_experts, synth.S80.top_k, synth.S80.inter
    for t, b in zip((1, 8, 64, 512, 4096), sizes):
        a = t * (k + 1)
        assert b >= 2 * a * H + 2 * a * Imax + 4 * t * E


@pytest.mark.parametrize("Hq,Hkv,D", [(16, 2, 256), (4, 4, 128), (16, 1, 128), (8, 2, 256)])
@pytest.mark.parametrize("batch", [1, 3, 64])
@pytest.mark.parametrize("max_pos", [1, 31, 32, 33, 1000, 8192, 32768])
def test_gqa_split_policy_invariants(lib, Hq, Hkv, D, batch, max_pos):
    # the ranges the workspace is sized for: at least one, at most one per SM of a 148-SM part over
    # the (sequence, K/V head) pairs (or one), none empty, together covering every position
    sh = moe.GqaShape(Hq, Hkv, D, 32768)
    wb = moe.gqa_workspace_bytes(sh, batch, max_pos)
    G = Hq // Hkv
    per_range = batch * Hkv * G * (D + 2) * 4
    assert wb > 0 and wb % per_range == 0
    n_split = wb // per_range
    assert 1 <= n_split <= max(1, 148 // (batch * Hkv))
    assert n_split <= -(-max_pos // 32)                 # never more ranges than 32-position chunks
    per = -(-max_pos // n_split)
    assert (n_split - 1) * per < max_pos <= n_split * per  # no empty range, all positions covered


def test_gqa_and_gdn_argument_checks(lib):
    sh = moe.GqaShape(16, 2, 256, 128)
    wb = moe.gqa_workspace_bytes(sh, 1, 64)
    args = lambda **kw: dict(dict(k_cache=16, v_cache=16, pos=16, q=16, k=16, v=16, gate=16, work=16, y=16,
                                  status=16), **kw)

    def call(shape=sh, batch=1, max_pos=64, work_bytes=wb, **kw):
        a = args(**kw)
        moe.gqa_decode(shape, batch, max_pos, a["k_cache"], a["v_cache"], a["pos"], a["q"], a["k"], a["v"],
                       a["gate"], 1.0, a["work"], work_bytes, a["y"], a["status"])

    for kw, want in [(dict(max_pos=129), moe.E_INVALID), (dict(max_pos=0), moe.E_INVALID),
                     (dict(batch=0), moe.E_INVALID), (dict(batch=70000), moe.E_INVALID),
                     (dict(status=None), moe.E_INVALID), (dict(y=8), moe.E_INVALID),
                     (dict(k_cache=None), moe.E_INVALID),
                     (dict(shape=moe.GqaShape(12, 4, 256, 128)), moe.E_SHAPE),   # 3 query heads per K/V head
                     (dict(shape=moe.GqaShape(32, 2, 256, 128)), moe.E_SHAPE),   # 16 per K/V head at D 256
                     (dict(shape=moe.GqaShape(16, 2, 64, 128)), moe.E_SHAPE),
                     (dict(work_bytes=wb - 1), moe.E_NOMEM)]:
        with pytest.raises(moe.MoeError) as e:
            call(**kw)
        assert e.value.status == want, kw
    gs = moe.GdnShape(16, 32, 128, 128)
    ok = [16] * 10
    for shape, batch, ptrs, want in [(moe.GdnShape(16, 24, 128, 128), 1, ok, moe.E_SHAPE),   # Hv % Hk
                                     (moe.GdnShape(16, 32, 128, 96), 1, ok, moe.E_SHAPE),
                                     (moe.GdnShape(0, 32, 128, 128), 1, ok, moe.E_SHAPE),
                                     (gs, 0, ok, moe.E_INVALID),
                                     (gs, 1, [None] + ok[1:], moe.E_INVALID)]:
        with pytest.raises(moe.MoeError) as e:
            moe.gdn_step(shape, batch, *ptrs, 1.0, 16)
        assert e.value.status == want, (shape.n_key_heads, shape.n_value_heads, shape.value_dim, batch)
