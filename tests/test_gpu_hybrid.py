"""GPU parity of the two hybrid-layer decode steps (include/hybrid.h) against the CPU oracle.

Tolerances. Both kernels compute in fp32 from the same bf16/fp32 inputs the oracle reads exactly
in double. Gated DeltaNet: a state element takes a few roundings per step (2^-24 each) and the two
128-term dot products add about sqrt(128) 2^-24 relative; the decay alpha = exp(-A sp) carries
about |A sp| 2^-24 (|A sp| < 50 here). Over 16 steps (alpha <= 1 does not amplify) that stays
below 1e-5 relative; 2e-5 is asserted on the state, o and y. GQA decode: the scores are 256-term
dot products (|s| error about 2^-24 |q||k| scale), the running softmax and the weighted sums of
up to 32768 positions add random-sign roundings of about sqrt(n) 2^-24 (5.4e-6 at 8K, 1.1e-5 at
32K); 2e-5 is asserted on o and y. The cache rows a step appends are bf16 values widened to fp32: bit-exact.
"""
import numpy as np
import pytest
import torch

from int4_routed_expert_05_b300 import moe
from int4_routed_expert_05_b300 import synth_hybrid as SH
from int4_routed_expert_05_b300.synth import bf16_value
from oracle import hybrid as OH

pytestmark = pytest.mark.gpu

TOL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_routed_expert_05_b300 import _build
    _build.build()
    assert torch.cuda.is_available()


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


# ---------------------------------------------------------------- Gated DeltaNet


class GdnCase:
    def __init__(self, sh: SH.GdnShape, seed: int, batch: int):
        self.sh, self.seed, self.batch = sh, seed, batch
        self.shape = moe.GdnShape(sh.n_key_heads, sh.n_value_heads, sh.key_dim, sh.value_dim)
        self.S0 = SH.gdn_state(sh, seed, 0, batch)
        self.P = SH.gdn_params(sh, seed, 0)
        self.state = _dev(self.S0)
        self.dP = {k: _dev(v) for k, v in self.P.items()}
        self.scale = sh.key_dim ** -0.5

    def gpu_step(self, inp):
        B, Hv, dv = self.batch, self.sh.n_value_heads, self.sh.value_dim
        d = {k: _dev(v) for k, v in inp.items()}
        y = torch.empty(B, Hv, dv, device="cuda")
        o = torch.empty(B, Hv, dv, device="cuda")
        moe.gdn_step(self.shape, B, self.state, d["q"], d["k"], d["v"], d["z"], d["a"], d["b"], self.dP["A_log"],
                     self.dP["dt_bias"], self.dP["norm_w"], self.scale, y, o=o)
        torch.cuda.synchronize()
        return o.cpu().numpy(), y.cpu().numpy()

    def oracle_step(self, S, inp, i):
        f = lambda x: bf16_value(x[i]).astype(np.float64)
        return OH.gdn_step(S, f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["z"]), inp["a"][i], inp["b"][i],
                           self.P["A_log"], self.P["dt_bias"], self.P["norm_w"], np.float32(self.scale))


GDN_SHAPES = [SH.GdnShape(2, 4, 128, 32), SH.GdnShape(1, 3, 128, 64), SH.GdnShape(4, 8, 128, 256), SH.GDN80]


@pytest.mark.parametrize("sh", GDN_SHAPES, ids=lambda s: f"Hk{s.n_key_heads}Hv{s.n_value_heads}dv{s.value_dim}")
@pytest.mark.parametrize("batch", [1, 3])
def test_gdn_matches_oracle_over_steps(sh, batch):
    steps = 16 if sh == SH.GDN80 and batch == 1 else 4
    C = GdnCase(sh, 7, batch)
    S = [C.S0[i].astype(np.float64) for i in range(batch)]
    for t in range(steps):
        inp = SH.gdn_inputs(sh, 7, 0, t, batch)
        o, y = C.gpu_step(inp)
        for i in range(batch):
            S[i], ro, ry = C.oracle_step(S[i], inp, i)
            assert rel_l2(o[i], ro) < TOL, (t, i, rel_l2(o[i], ro))
            assert rel_l2(y[i], ry) < TOL, (t, i, rel_l2(y[i], ry))
    Sg = C.state.cpu().numpy()
    for i in range(batch):
        assert rel_l2(Sg[i], S[i]) < TOL, (i, rel_l2(Sg[i], S[i]))


def test_gdn_write_then_read_returns_value_on_gpu():
    # no decay (A_log = -1000), full write (b = 40), q = k, scale 1: o = v whatever the old state
    sh = SH.GdnShape(2, 4, 128, 128)
    C = GdnCase(sh, 3, 2)
    C.dP["A_log"].fill_(-1000.0)
    C.scale = 1.0
    inp = SH.gdn_inputs(sh, 3, 0, 0, 2)
    inp["q"] = inp["k"].copy()
    inp["b"][:] = 40.0
    o, _ = C.gpu_step(inp)
    v = bf16_value(inp["v"]).astype(np.float64)
    assert rel_l2(o, v) < 1e-6


def test_gdn_batch_rows_independent_and_deterministic():
    sh = SH.GdnShape(4, 8, 128, 128)
    inp = SH.gdn_inputs(sh, 5, 0, 0, 3)
    A = GdnCase(sh, 5, 3)
    o3, y3 = A.gpu_step(inp)
    B = GdnCase(sh, 5, 3)
    o3b, y3b = B.gpu_step(inp)
    np.testing.assert_array_equal(y3, y3b)
    np.testing.assert_array_equal(A.state.cpu().numpy(), B.state.cpu().numpy())
    # sequence 1 alone: the same bits as inside the batch
    one = GdnCase(sh, 5, 1)
    one.state = A.state.new_tensor(A.S0[1:2])
    sub = {k: v[1:2] for k, v in inp.items()}
    o1, y1 = one.gpu_step(sub)
    np.testing.assert_array_equal(y1[0], y3[1])
    np.testing.assert_array_equal(one.state.cpu().numpy()[0], A.state.cpu().numpy()[1])


# ---------------------------------------------------------------- gated GQA


class GqaCase:
    def __init__(self, sh: SH.GqaShape, seed: int, batch: int, max_len: int, filled):
        self.sh, self.seed, self.batch, self.max_len = sh, seed, batch, max_len
        self.shape = moe.GqaShape(sh.n_q_heads, sh.n_kv_heads, sh.head_dim, max_len)
        fill = max(filled)
        self.K0 = SH.gqa_cache(sh, seed, 0, max_len, fill, batch)
        self.V0 = SH.gqa_cache(sh, seed + 1, 0, max_len, fill, batch)
        self.kc, self.vc = _dev(self.K0), _dev(self.V0)
        self.pos = np.array(filled, np.int32)
        self.scale = sh.head_dim ** -0.5

    def gpu_step(self, inp, max_pos=None, pos=None):
        B, Hq, D = self.batch, self.sh.n_q_heads, self.sh.head_dim
        pos = self.pos if pos is None else np.asarray(pos, np.int32)
        max_pos = int(pos.max()) + 1 if max_pos is None else max_pos
        wb = moe.gqa_workspace_bytes(self.shape, B, max_pos)
        work = torch.empty(wb // 4 + 4, dtype=torch.float32, device="cuda")
        d = {k: _dev(v) for k, v in inp.items()}
        y = torch.empty(B, Hq, D, device="cuda")
        o = torch.empty(B, Hq, D, device="cuda")
        status = torch.zeros(4, dtype=torch.int32, device="cuda")
        moe.gqa_decode(self.shape, B, max_pos, self.kc, self.vc, _dev(pos), d["q"], d["k"], d["v"], d["gate"],
                       self.scale, work, wb, y, status, o=o)
        torch.cuda.synchronize()
        return o.cpu().numpy(), y.cpu().numpy(), int(status[0].item())


def _gqa_run(sh, batch, max_len, filled, steps, seed=11, max_pos_extra=0):
    C = GqaCase(sh, seed, batch, max_len, filled)
    Kc = [C.K0[i].astype(np.float64) for i in range(batch)]
    Vc = [C.V0[i].astype(np.float64) for i in range(batch)]
    for t in range(steps):
        inp = SH.gqa_inputs(sh, seed, 0, t, batch)
        mp = min(max_len, int(C.pos.max()) + 1 + max_pos_extra)
        o, y, st = C.gpu_step(inp, max_pos=mp)
        assert st == moe.OK
        for i in range(batch):
            f = lambda x: bf16_value(x[i]).astype(np.float64)
            Kc[i], Vc[i], ro, ry = OH.gqa_step(Kc[i], Vc[i], int(C.pos[i]), f(inp["q"]), f(inp["k"]), f(inp["v"]),
                                               f(inp["gate"]), np.float32(C.scale))
            assert rel_l2(o[i], ro) < TOL, (t, i, rel_l2(o[i], ro))
            assert rel_l2(y[i], ry) < TOL, (t, i, rel_l2(y[i], ry))
        C.pos += 1
    kc, vc = C.kc.cpu().numpy(), C.vc.cpu().numpy()
    for i in range(batch):
        n = int(C.pos[i])
        np.testing.assert_array_equal(kc[i][:, :n], Kc[i][:, :n].astype(np.float32))
        np.testing.assert_array_equal(vc[i][:, :n], Vc[i][:, :n].astype(np.float32))
    return C


GQA_SHAPES = [SH.GQA80, SH.GqaShape(4, 4, 128), SH.GqaShape(16, 1, 128), SH.GqaShape(8, 2, 256), SH.GqaShape(2, 1, 256)]


@pytest.mark.parametrize("sh", GQA_SHAPES, ids=lambda s: f"Hq{s.n_q_heads}Hkv{s.n_kv_heads}D{s.head_dim}")
@pytest.mark.parametrize("filled", [[0], [31], [32, 1], [33, 100], [1000, 7]])
def test_gqa_matches_oracle(sh, filled):
    # positions on both sides of chunk (32) and range boundaries, ragged batches, the empty cache
    _gqa_run(sh, len(filled), 1100, filled, steps=2)


def test_gqa_80b_full_8k_context():
    # the pages' 8K context: 8190 cached positions, two steps fill the cache to its capacity
    _gqa_run(SH.GQA80, 1, 8192, [8190], steps=2)


def test_gqa_80b_32k_context():
    # the pages' 32K context (about 1.5 GiB of cache over the 12 layers; one layer here): one step
    # at the last position, the ranges 886 positions long
    _gqa_run(SH.GQA80, 1, 32768, [32767], steps=1)


def test_gqa_split_count_changes_nothing_beyond_rounding():
    # a larger max_pos spreads the same positions over other ranges: same result within rounding
    _gqa_run(SH.GqaShape(8, 2, 256), 2, 4096, [700, 1500], steps=1, max_pos_extra=2500)


def test_gqa_deterministic():
    sh = SH.GQA80
    inp = SH.gqa_inputs(sh, 3, 0, 0, 1)
    A = GqaCase(sh, 3, 1, 2048, [2000])
    o1, y1, _ = A.gpu_step(inp)
    B = GqaCase(sh, 3, 1, 2048, [2000])
    o2, y2, _ = B.gpu_step(inp)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(o1, o2)


def test_gqa_large_scores_stay_finite():
    # scale 1 with inputs scaled by 8: scores of several hundred; the running maximum keeps exp finite
    sh = SH.GqaShape(8, 2, 256)
    C = GqaCase(sh, 9, 1, 512, [300])
    C.scale = 1.0
    from int4_routed_expert_05_b300.synth import bf16_bits
    inp = SH.gqa_inputs(sh, 9, 0, 0, 1)
    inp["q"] = bf16_bits(bf16_value(inp["q"]) * 8.0)
    o, y, st = C.gpu_step(inp)
    assert st == moe.OK and np.isfinite(y).all()
    f = lambda x: bf16_value(x[0]).astype(np.float64)
    _, _, ro, ry = OH.gqa_step(C.K0[0].astype(np.float64), C.V0[0].astype(np.float64), 300, f(inp["q"]), f(inp["k"]),
                               f(inp["v"]), f(inp["gate"]), 1.0)
    assert rel_l2(y[0], ry) < TOL


@pytest.mark.parametrize("bad", [-1, 64])
def test_gqa_position_outside_the_bound_sets_status(bad):
    # sequence 0 valid, sequence 1 at a position the kernel's own check rejects (max_pos = 64):
    # status MOE_E_RANGE, sequence 1's cache rows untouched, sequence 0 still computed
    sh = SH.GqaShape(4, 2, 128)
    C = GqaCase(sh, 4, 2, 128, [10, 10])
    inp = SH.gqa_inputs(sh, 4, 0, 0, 2)
    o, y, st = C.gpu_step(inp, max_pos=64, pos=[10, bad])
    assert st == moe.E_RANGE
    np.testing.assert_array_equal(C.kc.cpu().numpy()[1], C.K0[1])
    np.testing.assert_array_equal(C.vc.cpu().numpy()[1], C.V0[1])
    f = lambda x: bf16_value(x[0]).astype(np.float64)
    _, _, ro, ry = OH.gqa_step(C.K0[0].astype(np.float64), C.V0[0].astype(np.float64), 10, f(inp["q"]), f(inp["k"]),
                               f(inp["v"]), f(inp["gate"]), np.float32(C.scale))
    assert rel_l2(y[0], ry) < TOL
