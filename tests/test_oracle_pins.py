"""Pins of the CPU oracle to things other than itself (CPU only).

Each test fixes part of the oracle by what the pages state, by a closed form, by a special case
that reduces to a textbook computation done here independently (numpy from the raw generator
arrays, never through the oracle's blob reader), or by brute force on tiny inputs. Together they
fail on a dropped term, a wrong sign or index, a transposed operand, a swapped nibble, a missing
renormalisation or a wrong tie-break anywhere in the oracle.
"""
import json
import os

import numpy as np
import pytest
import torch

from int4_routed_expert_05_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _silu(z):
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def _textbook_dequant(t, name, group):
    """W = s*q + b straight from the generator arrays (numpy, float64)."""
    q = t[name + "_q"].astype(np.float64)
    s = np.repeat(synth.bf16_value(t[name + "_s"]).astype(np.float64), group, axis=1)
    b = np.repeat(synth.bf16_value(t[name + "_b"]).astype(np.float64), group, axis=1)
    return s * q + b


def _textbook_swiglu(t, u, group):
    Wg = _textbook_dequant(t, "gate", group)
    Wu = _textbook_dequant(t, "up", group)
    Wd = _textbook_dequant(t, "down", group)
    return Wd @ (_silu(Wg @ u) * (Wu @ u))


def _zero_tensors(shape, shared=False):
    t = synth.expert_tensors(shape, 0, 0, synth.SHARED_EXPERT if shared else 0)
    for k in t:
        t[k] = np.zeros_like(t[k])
    return t


# ---------------------------------------------------------------------------------------------
# blob format
# ---------------------------------------------------------------------------------------------

def test_blob_size_matches_page_arithmetic(orc):
    """[size]: 480 experts ~ 810 MiB per token at zero hits => 1,769,472 B per expert exactly,
    which is gate/up/down 2048x512 int4 plus bf16 scale+bias per 64-group. The same blob size
    reproduces the pages' disk footprints."""
    p = json.load(open(os.path.join(GOLDEN, "page_sizes.json")))
    blob = orc.blob_bytes(synth.S80)
    assert p["experts_per_token_80b_zero_hits"] == p["layers_80b"] * p["top_k_80b"]
    assert blob * p["experts_per_token_80b_zero_hits"] == p["logical_read_mib_80b_zero_hits"] * 2 ** 20
    assert orc.blob_stride(synth.S80) == blob  # already a multiple of 4096
    tol = p["tolerance_gb"] * 1e9
    gb35 = p["layers_35b"] * p["experts_35b"] * orc.blob_bytes(synth.S35)
    assert abs(gb35 - p["disk_gb_35b_int4"] * 1e9) < tol
    gb35_8 = p["layers_35b"] * p["experts_35b"] * orc.blob_bytes(synth.S35.with_bits(8))
    assert abs(gb35_8 - p["disk_gb_35b_int8"] * 1e9) < tol
    gb80 = p["layers_80b"] * p["experts_80b"] * blob
    # the 42 GB figure includes the dense (resident) weights, a few GB more than the experts
    assert 0.9 * p["disk_gb_80b_int4_incl_dense"] * 1e9 < gb80 < p["disk_gb_80b_int4_incl_dense"] * 1e9 * 1.1


def _layout_fixture():
    fx = json.load(open(os.path.join(GOLDEN, "blob_layout_h64_i64.json")))
    sh = synth.Shape(fx["shape"]["hidden"], 1, 1, fx["shape"]["inter"], fx["shape"]["inter"],
                     bits=fx["shape"]["bits"], group=fx["shape"]["group"])
    H, I = sh.hidden, sh.inter
    t = {}
    t["gate_q"] = np.zeros((I, H), np.uint8)
    t["gate_q"][0] = np.arange(H) % 16
    t["up_q"] = np.zeros((I, H), np.uint8)
    t["up_q"][0] = 15 - np.arange(H) % 16
    t["down_q"] = np.zeros((H, I), np.uint8)
    t["down_q"][1, 0], t["down_q"][1, 1] = 7, 9
    for m, (rows, cols) in (("gate", (I, H)), ("up", (I, H)), ("down", (H, I))):
        for sb in ("s", "b"):
            v = int(fx["bf16"][m + "_" + sb], 16)
            t[m + "_" + sb] = np.full((rows, cols // 64), v, np.uint16)
    return fx, sh, t


def test_blob_layout_golden(orc):
    """Hand-derived bytes of a tiny blob pin the section order and the nibble order (R2)."""
    fx, sh, t = _layout_fixture()
    assert orc.blob_bytes(sh) == fx["blob_bytes"]
    assert orc.blob_stride(sh) == fx["stride"]
    blob = orc.pack(sh, t)
    assert blob.shape[0] == fx["stride"]
    covered = np.zeros(fx["stride"], bool)
    for run in fx["runs"]:
        want = bytes.fromhex(run["hex"])
        got = blob[run["offset"]: run["offset"] + len(want)].tobytes()
        assert got == want, run["offset"]
        covered[run["offset"]: run["offset"] + len(want)] = True
    # everything not listed is zero (unset codes and the padding up to the stride)
    assert not blob[~covered].any()
    # the reader decodes the hand-built bytes back
    back = orc.unpack(sh, blob)
    for k in t:
        np.testing.assert_array_equal(back[k], t[k])


def test_blob_layout_dequant_values(orc):
    fx, sh, t = _layout_fixture()
    blob = orc.pack(sh, t)
    W = [orc.dequant(sh, blob, m) for m in range(3)]
    names = {"gate": 0, "up": 1, "down": 2}
    for key, val in fx["dequant"].items():
        m, rest = key.split("[", 1)
        r, c = [int(x) for x in rest.replace("]", " ").replace("[", " ").split()]
        assert W[names[m]][r, c] == val, key


@pytest.mark.parametrize("shape", [synth.TINY, synth.TINY.with_bits(8)])
def test_pack_unpack_roundtrip(orc, shape):
    t = synth.expert_tensors(shape, 3, 1, 5)
    back = orc.unpack(shape, orc.pack(shape, t))
    for k in t:
        np.testing.assert_array_equal(back[k], t[k])


# ---------------------------------------------------------------------------------------------
# bf16 values
# ---------------------------------------------------------------------------------------------

def test_bf16_round_matches_torch(orc):
    """The oracle's own round-to-nearest-even agrees with torch's float32 -> bfloat16 cast
    (values that are float32-exact, including exact ties and both signs)."""
    rng = np.random.default_rng(0)
    v = rng.standard_normal(4000).astype(np.float32) * np.float32(3.0)
    bits = v.view(np.uint32)
    ties = ((bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)  # exact halfway
    vals = np.concatenate([v, ties, np.float32([0.0, -0.0, 1.0, -1.5, 65504.0, 1e-30, 3e38])])
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.round_bf16(vals.astype(np.float64))
    np.testing.assert_array_equal(got, want)
    back = orc.bf16(want[:200])
    np.testing.assert_array_equal(back, torch.from_numpy(want[:200].view(np.int16)).view(torch.bfloat16).float().numpy())


# ---------------------------------------------------------------------------------------------
# dequantisation and the expert MLP
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [4, 8])
def test_dequant_identity_scale_one_bias_zero(orc, bits):
    """s = 1, b = 0 gives W = q exactly, and an integer GEMV is exact in double."""
    sh = synth.TINY.with_bits(bits)
    t = synth.expert_tensors(sh, 1, 0, 2)
    for m in ("gate", "up", "down"):
        t[m + "_s"] = np.full_like(t[m + "_s"], 0x3F80)
        t[m + "_b"] = np.zeros_like(t[m + "_b"])
    blob = orc.pack(sh, t)
    for i, m in enumerate(("gate", "up", "down")):
        W = orc.dequant(sh, blob, i)
        np.testing.assert_array_equal(W, t[m + "_q"].astype(np.float64))
    # an integer activation: Wg u is an exact integer; compare h with silu(g)*v from int64 sums
    rng = np.random.default_rng(1)
    u_int = rng.integers(-3, 4, sh.hidden)
    u_bits = synth.bf16_bits(u_int.astype(np.float32))
    y, h = orc.expert_ffn(sh, blob, u_bits)
    g = t["gate_q"].astype(np.int64) @ u_int
    v = t["up_q"].astype(np.int64) @ u_int
    np.testing.assert_allclose(h, _silu(g.astype(np.float64)) * v, rtol=1e-13, atol=1e-9)


@pytest.mark.parametrize("bits", [4, 8])
def test_expert_ffn_matches_textbook_swiglu(orc, bits):
    """The expert MLP read through the oracle's blob reader equals a textbook SwiGLU on the
    generator's raw arrays (non-square: H=256, I=64, so a transposed operand cannot pass)."""
    sh = synth.TINY.with_bits(bits)
    t = synth.expert_tensors(sh, 7, 2, 3)
    u_bits = synth.activation_bits(sh, 7, 0)[0]
    u = synth.bf16_value(u_bits).astype(np.float64)
    y, _ = orc.expert_ffn(sh, orc.pack(sh, t), u_bits)
    np.testing.assert_allclose(y, _textbook_swiglu(t, u, sh.group), rtol=1e-11, atol=1e-11)


# ---------------------------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------------------------

def test_router_logits_and_bound(orc):
    """logits = Wr u (numpy float64 matmul on the bf16 values), and a float32 evaluation of the
    same dot products lies within the stated error bound."""
    sh = synth.TINY
    Wr = synth.router_bits(sh, 4, 0)
    u_bits = synth.activation_bits(sh, 4, 0)[0]
    lg, bd = orc.router_logits(Wr, u_bits)
    Wv = synth.bf16_value(Wr).astype(np.float64)
    uv = synth.bf16_value(u_bits).astype(np.float64)
    np.testing.assert_allclose(lg, Wv @ uv, rtol=1e-13, atol=1e-15)
    f32 = (synth.bf16_value(Wr) @ synth.bf16_value(u_bits)).astype(np.float64)
    assert np.all(np.abs(f32 - lg) <= bd)
    bias = np.linspace(-1, 1, sh.n_experts).astype(np.float32)
    lg2, _ = orc.router_logits(Wr, u_bits, bias)
    np.testing.assert_allclose(lg2, Wv @ uv + bias.astype(np.float64), rtol=1e-13, atol=1e-15)


def test_topk_bruteforce(orc):
    """Selection = sort by (binary32 value descending, index ascending), brute force; with many
    exact ties planted."""
    rng = np.random.default_rng(2)
    for trial in range(200):
        E = int(rng.integers(2, 40))
        k = int(rng.integers(1, E + 1))
        lg = rng.standard_normal(E)
        if trial % 2:
            lg = np.round(lg * 2) / 2  # many exact ties
        idx, _ = orc.topk(lg, k)
        f = lg.astype(np.float32)
        want = sorted(range(E), key=lambda e: (-float(f[e]), e))[:k]
        assert list(idx) == want


def test_topk_zero_input(orc):
    """u = 0: every logit is 0, so the k lowest indices win with weight 1/k each."""
    sh = synth.TINY
    Wr = synth.router_bits(sh, 0, 0)
    lg, _ = orc.router_logits(Wr, np.zeros(sh.hidden, np.uint16))
    idx, w = orc.topk(lg, sh.top_k)
    assert list(idx) == list(range(sh.top_k))
    np.testing.assert_allclose(w, 1.0 / sh.top_k, rtol=0, atol=1e-15)


def test_duplicated_router_rows_lower_index_wins(orc):
    sh = synth.TINY
    Wr = synth.router_bits(sh, 5, 0)
    u_bits = synth.activation_bits(sh, 5, 0)[0]
    big = synth.bf16_bits(np.float32(0.3) * np.sign(synth.bf16_value(u_bits)))
    Wr[3] = big
    Wr[11] = big
    lg, _ = orc.router_logits(Wr, u_bits)
    idx, w = orc.topk(lg, 1)
    assert list(idx) == [3]
    idx, w = orc.topk(lg, 2)
    assert list(idx) == [3, 11] and w[0] == w[1]


def test_renorm_equals_softmax_over_selected(orc):
    """With renormalisation the weights are the softmax of the k selected logits alone (the
    full denominator cancels); without it they are the full softmax at the selected experts."""
    from scipy.special import softmax
    rng = np.random.default_rng(3)
    lg = rng.standard_normal(64) * 2
    idx, w = orc.topk(lg, 6, renorm=True)
    np.testing.assert_allclose(w, softmax(lg[idx]), rtol=1e-13)
    idx2, w2 = orc.topk(lg, 6, renorm=False)
    assert list(idx2) == list(idx)
    np.testing.assert_allclose(w2, softmax(lg)[idx], rtol=1e-13)
    assert np.all(np.diff(lg[idx]) <= 0)


# ---------------------------------------------------------------------------------------------
# whole layer: special cases that reduce to textbook computations
# ---------------------------------------------------------------------------------------------

def _layer_inputs(sh, seed):
    blobs_t = [synth.expert_tensors(sh, seed, 0, e) for e in range(sh.n_experts)]
    shared_t = synth.expert_tensors(sh, seed, 0, synth.SHARED_EXPERT)
    Wr = synth.router_bits(sh, seed, 0)
    w_sg = synth.shared_gate_bits(sh, seed, 0)
    u_bits = synth.activation_bits(sh, seed, 0)[0]
    return blobs_t, shared_t, Wr, w_sg, u_bits


def test_one_hot_routing_is_dense_swiglu(orc):
    """k = 1 with renormalisation (w = 1) and the shared expert zeroed (s = b = 0) turns the
    layer into one dense SwiGLU FFN of the selected expert."""
    sh = synth.Shape(256, 16, 1, 64, 64)
    blobs_t, _, Wr, w_sg, u_bits = _layer_inputs(sh, 11)
    zero_shared = _zero_tensors(sh, shared=True)
    r = orc.moe_layer(sh, u_bits, Wr, w_sg, [orc.pack(sh, t) for t in blobs_t],
                      orc.pack(sh, zero_shared, shared=True))
    assert r["w"][0] == 1.0
    u = synth.bf16_value(u_bits).astype(np.float64)
    want = _textbook_swiglu(blobs_t[r["idx"][0]], u, sh.group)
    np.testing.assert_allclose(r["y"], want, rtol=1e-11, atol=1e-11)


def test_shared_expert_gate_is_sigmoid(orc):
    """w_sg = 0 gives gate sigmoid(0) = 1/2; with every routed expert zeroed the layer output is
    exactly half the shared SwiGLU."""
    sh = synth.TINY
    _, shared_t, Wr, _, u_bits = _layer_inputs(sh, 12)
    zero = orc.pack(sh, _zero_tensors(sh))
    r = orc.moe_layer(sh, u_bits, Wr, np.zeros(sh.hidden, np.uint16), [zero] * sh.n_experts,
                      orc.pack(sh, shared_t, shared=True))
    assert r["gamma"] == 0.5
    u = synth.bf16_value(u_bits).astype(np.float64)
    np.testing.assert_allclose(r["y"], 0.5 * _textbook_swiglu(shared_t, u, sh.group), rtol=1e-11, atol=1e-11)
    # and a nonzero gate vector gives the logistic function of the dot product
    w_sg = synth.shared_gate_bits(sh, 12, 0)
    z = float(synth.bf16_value(w_sg).astype(np.float64) @ u)
    assert abs(orc.shared_gate(w_sg, u_bits) - 1.0 / (1.0 + np.exp(-z))) < 1e-15


def test_all_experts_selected_is_soft_moe(orc):
    """k = E with renormalisation: every expert is used with its full-softmax probability."""
    from scipy.special import softmax
    sh = synth.Shape(128, 6, 6, 64, 64)
    blobs_t, shared_t, Wr, w_sg, u_bits = _layer_inputs(sh, 13)
    blobs = [orc.pack(sh, t) for t in blobs_t]
    r = orc.moe_layer(sh, u_bits, Wr, w_sg, blobs, orc.pack(sh, shared_t, shared=True))
    u = synth.bf16_value(u_bits).astype(np.float64)
    p = softmax(synth.bf16_value(Wr).astype(np.float64) @ u)
    gam = 1.0 / (1.0 + np.exp(-(synth.bf16_value(w_sg).astype(np.float64) @ u)))
    want = sum(p[e] * _textbook_swiglu(blobs_t[e], u, sh.group) for e in range(sh.n_experts))
    want = want + gam * _textbook_swiglu(shared_t, u, sh.group)
    assert sorted(r["idx"]) == list(range(sh.n_experts))
    np.testing.assert_allclose(r["y"], want, rtol=1e-10, atol=1e-11)


def test_expert_permutation_invariance(orc):
    """Relabelling the experts (router rows and blobs together) changes nothing but the labels."""
    sh = synth.TINY
    blobs_t, shared_t, Wr, w_sg, u_bits = _layer_inputs(sh, 14)
    blobs = [orc.pack(sh, t) for t in blobs_t]
    sb = orc.pack(sh, shared_t, shared=True)
    r = orc.moe_layer(sh, u_bits, Wr, w_sg, blobs, sb)
    perm = np.random.default_rng(4).permutation(sh.n_experts)   # new label e' holds old perm[e']
    r2 = orc.moe_layer(sh, u_bits, Wr[perm], w_sg, [blobs[p] for p in perm], sb)
    assert list(perm[r2["idx"]]) == list(r["idx"])
    np.testing.assert_array_equal(r2["y"], r["y"])


def test_rmsnorm_closed_forms(orc):
    H = 256
    c = 3.0
    u = orc.rmsnorm_bf16(np.full(H, c))
    assert np.all(u == orc.round_bf16(c / np.sqrt(c * c + 1e-6)))
    assert not orc.rmsnorm_bf16(np.zeros(H)).any()
    x = np.random.default_rng(5).standard_normal(H) * 100
    u1 = synth.bf16_value(orc.rmsnorm_bf16(x)).astype(np.float64)
    np.testing.assert_allclose(np.sqrt(np.mean(u1 ** 2)), 1.0, rtol=5e-3)
    np.testing.assert_allclose(u1, x / np.sqrt(np.mean(x ** 2)), rtol=2 ** -8, atol=1e-6)


def test_stack_is_residual_of_layers(orc):
    """Two layers: x2 = x1 + MoE_1(bf16(rmsnorm(x1))), x1 = x0 + MoE_0(bf16(rmsnorm(x0)))."""
    sh = synth.TINY
    layers = []
    for l in range(2):
        blobs = [orc.pack(sh, synth.expert_tensors(sh, 20, l, e)) for e in range(sh.n_experts)]
        layers.append({"Wr": synth.router_bits(sh, 20, l), "w_sg": synth.shared_gate_bits(sh, 20, l),
                       "blobs": blobs, "shared": orc.pack(sh, synth.expert_tensors(sh, 20, l, -1), shared=True)})
    x0 = synth.activation_f32(sh, 20, 0)[0].astype(np.float64)
    x2, tr = orc.stack(sh, layers, x0, record=True)
    L0 = layers[0]
    x1 = x0 + orc.moe_layer(sh, orc.rmsnorm_bf16(x0), L0["Wr"], L0["w_sg"], L0["blobs"], L0["shared"])["y"]
    np.testing.assert_array_equal(tr[1]["x_in"], x1)
    np.testing.assert_array_equal(x2, x1 + tr[1]["y"])


# ---------------------------------------------------------------------------------------------
# decision bounds, forced selection, slot policy
# ---------------------------------------------------------------------------------------------

def test_router_bound_exact_value(orc):
    """The logit error bound on a constructed row is the classical binary32 summation bound
    gamma_{H+1} * (sum |w u| + |bias|), gamma_n = n 2^-24 / (1 - n 2^-24), to the last bit of its
    double evaluation: a bound twice as wide (or half) fails."""
    H = 3
    Wr = synth.bf16_bits(np.array([[1.0, 2.0, -4.0]], np.float32))
    u = synth.bf16_bits(np.array([0.5, 0.25, 1.0], np.float32))
    bias = np.array([1.5], np.float32)
    lg, bd = orc.router_logits(Wr, u, bias)
    assert lg[0] == 0.5 + 0.5 - 4.0 + 1.5
    n = H + 1
    gam = n * 2.0 ** -24 / (1.0 - n * 2.0 ** -24)
    assert bd[0] == pytest.approx(gam * 6.5, rel=1e-15, abs=0)


def test_selection_margin_closed_form(orc):
    """Margin of a constructed selection: the smallest chosen logit less its bound, minus the
    largest unchosen one plus its bound, minus half an ulp of binary32 rounding on each (one ulp
    in total per side, as spacing at the two magnitudes)."""
    check_margin(orc.selection_margin)


def check_margin(selection_margin):
    """The closed-form margin cases (also run against planted mistakes in the mutation tests)."""
    lg = np.array([3.0, 1.0, 2.0, 0.5])
    bd = np.array([0.1, 0.2, 0.05, 0.0])
    m = selection_margin(lg, bd, np.array([0, 2]))
    slack = 2.0 ** -22 + 2.0 ** -23  # binary32 spacing at 2.0 and at 1.0
    assert m == pytest.approx((2.0 - 0.05) - (1.0 + 0.2) - slack, rel=0, abs=1e-15)
    # the sign flips where the gap meets the bounds: exactly there only the rounding slack is left
    lg2 = np.array([1.0, 0.9])
    sl2 = float(np.spacing(np.float32(1.0)) + np.spacing(np.float32(0.9)))
    assert selection_margin(lg2, np.array([0.04, 0.05]), np.array([0])) == pytest.approx(0.01 - sl2, abs=1e-15)
    assert selection_margin(lg2, np.array([0.05, 0.05]), np.array([0])) == pytest.approx(-sl2, abs=1e-15)
    assert selection_margin(lg2, np.array([0.05, 0.06]), np.array([0])) < 0
    assert selection_margin(lg, bd, np.arange(4)) == np.inf
    # the bounds decide which chosen logit is the weakest (3.0 - 1.5 below 2.0) and which unchosen
    # one the strongest (0.5 + 1.0 above 1.0)
    bd3 = np.array([1.5, 0.0, 0.0, 1.0])
    sl3 = 2.0 ** -22 + 2.0 ** -24  # binary32 spacing at 3.0 and at 0.5
    assert selection_margin(lg, bd3, np.array([0, 2])) == pytest.approx((3.0 - 1.5) - (0.5 + 1.0) - sl3, abs=1e-15)


def test_forced_selection_reproduces_own(orc):
    """The layer evaluated for a given selection equals the layer's own when given its own
    selection (bit for bit), and a selection given in another order permutes the weights and
    leaves y equal up to summation order."""
    sh = synth.TINY
    t_blobs = [orc.pack(sh, synth.expert_tensors(sh, 3, 0, e)) for e in range(sh.n_experts)]
    shared = orc.pack(sh, synth.expert_tensors(sh, 3, 0, synth.SHARED_EXPERT), shared=True)
    Wr = synth.router_bits(sh, 3, 0)
    w_sg = synth.shared_gate_bits(sh, 3, 0)
    u = synth.activation_bits(sh, 3, 0)[0]
    r = orc.moe_layer(sh, u, Wr, w_sg, t_blobs, shared)
    rf = orc.moe_layer(sh, u, Wr, w_sg, t_blobs, shared, force_idx=r["idx"])
    assert np.array_equal(rf["idx"], r["idx"]) and np.array_equal(rf["w"], r["w"]) and np.array_equal(rf["y"], r["y"])
    rev = r["idx"][::-1].copy()
    rr = orc.moe_layer(sh, u, Wr, w_sg, t_blobs, shared, force_idx=rev)
    np.testing.assert_allclose(rr["w"], r["w"][::-1], rtol=1e-15, atol=0)
    np.testing.assert_allclose(rr["y"], r["y"], rtol=1e-12, atol=1e-14)


def run_pool_trace(sim_cls, trace):
    """Replay a golden slot-policy trace on a PoolSim-like class; returns the mismatching steps."""
    sim = sim_cls(trace["n_slots"])
    bad = []
    for i, op in enumerate(trace["ops"]):
        if op["op"] == "release":
            sim.release()
            continue
        if op["op"] == "lookup":
            got = sim.lookup(op["layer"], op["experts"])
        else:
            got = sim.load(op["layer"], op["expert"])
        if got != op["expect"]:
            bad.append((i, op, got))
    return bad


def test_pool_sim_golden_trace():
    """The slot-policy simulator against a hand-derived trace (tests/golden/pool_trace.json): fills
    the lowest free slot, evicts the fewest uses, then the oldest tick, then the lowest slot, never
    a pinned slot, and refuses when every slot is pinned."""
    from oracle.pool_sim import PoolSim
    with open(os.path.join(GOLDEN, "pool_trace.json")) as f:
        trace = json.load(f)
    assert run_pool_trace(PoolSim, trace) == []


def test_threaded_oracle_is_bitwise_serial(orc):
    """The oracle's optional threaded row loops give the serial results bit for bit (rows are
    independent and keep their summation order)."""
    sh = synth.Shape(512, 64, 6, 128, 192)
    blobs = [orc.pack(sh, synth.expert_tensors(sh, 8, 0, e)) for e in range(sh.n_experts)]
    shared = orc.pack(sh, synth.expert_tensors(sh, 8, 0, synth.SHARED_EXPERT), shared=True)
    args = (sh, synth.activation_bits(sh, 8, 0)[0], synth.router_bits(sh, 8, 0), synth.shared_gate_bits(sh, 8, 0),
            blobs, shared)
    r1 = orc.moe_layer(*args)
    orc.set_threads(4)
    try:
        r4 = orc.moe_layer(*args)
    finally:
        orc.set_threads(1)
    for key in ("idx", "w", "y", "logits", "bound"):
        assert np.array_equal(r1[key], r4[key]), key
