"""GPU parity of the batched (GEMM) path against the CPU oracle, token by token.

The batched path multiplies fp16-rounded weights (w = s * q + b, one rounding of at most 2^-11
relative each) by the fp16 input (bf16 -> fp16 is exact in range), and hands h to the down GEMM
in fp16: two independent roundings of relative size <= 2^-11 feed each output, whose errors add
up like a random walk, so the expected rel-L2 is a few 1e-4. Asserted: the stated 2e-3 and a
derived 1e-3. The k + 1 expert outputs of a token are summed by fp32 reductions in whatever order
the tiles finish, so outputs agree run to run to fp32 rounding, not bit for bit."""
import json
import os

import numpy as np
import pytest
import torch

from int4_routed_expert_05_b300 import moe, synth
from int4_routed_expert_05_b300.resident import Resident

from gpu_ref import OracleLayers, check_selection, layer_reference, rel_l2

pytestmark = pytest.mark.gpu

TOL = 2e-3
# a token whose GPU selection differs from the oracle's within the binary32 error bound of the
# logits: compared with the oracle evaluated for the GPU's selection, at the stated 2e-3
NEAR_TIE_TOL = 2e-3
DERIVED = 1e-3
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_routed_expert_05_b300 import _build
    _build.build()
    assert torch.cuda.is_available()


def _bits(x_bits_np):
    return torch.from_numpy(np.ascontiguousarray(x_bits_np).view(np.int16)).cuda()


def _case(orc, sh, seed, T, sample=None, bias=None, n_unique=None):
    R = Resident(sh, 1, seed, n_unique=n_unique, bias=None if bias is None else [bias])
    O = OracleLayers(orc, sh, seed, 1, n_unique=n_unique, bias=None if bias is None else [bias])
    x = synth.activation_bits(sh, seed, 0, T)
    y, idx, w = R.layer_forward_batched(0, _bits(x))
    torch.cuda.synchronize()
    assert R.pool.device_status() == moe.OK
    y, idx, w = y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()
    toks = range(T) if sample is None else sample
    errs = []
    for t in toks:
        r, exact = layer_reference(orc, O, 0, x[t], idx[t])
        np.testing.assert_allclose(w[t], r["w"], rtol=0, atol=2e-6)
        if exact:
            errs.append(rel_l2(y[t], r["y"]))
        else:
            assert rel_l2(y[t], r["y"]) <= NEAR_TIE_TOL
    assert errs, "no token had an exactly determined selection"
    assert np.isfinite(y).all()
    return R, x, max(errs)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("renorm", [True, False])
def test_tiny_batched(orc, bits, renorm):
    sh = synth.Shape(256, 16, 2, 64, 64, bits=bits, renorm=renorm)
    _, _, err = _case(orc, sh, seed=0, T=7)
    assert err <= TOL and err <= DERIVED, err


@pytest.mark.parametrize("T", [1, 15, 17, 127, 128, 129, 300])
def test_token_counts(orc, T):
    """One token, around the 16-column MMA granule and the 128-token tile, and several tiles with
    a ragged tail."""
    _, _, err = _case(orc, synth.TINY, seed=11, T=T, sample=sorted({0, T // 2, T - 1}))
    assert err <= DERIVED, err


@pytest.mark.parametrize("dims", [
    (256, 40, 3, 64, 128, 4),     # ragged expert count, shared inter != inter
    (512, 16, 1, 128, 64, 4),     # k = 1
    (256, 16, 16, 64, 64, 4),     # k = E
    (768, 100, 7, 192, 320, 8),   # int8, inter not a multiple of the 128-row tile
    (256, 512, 16, 64, 64, 4),    # the largest expert count and top-k
])
def test_edge_shapes_batched(orc, dims):
    H, E, k, I, Is, bits = dims
    sh = synth.Shape(H, E, k, I, Is, bits=bits)
    _, _, err = _case(orc, sh, seed=5, T=37)
    assert err <= DERIVED, err


def test_logit_bias_batched(orc):
    sh = synth.TINY
    bias = np.linspace(-2, 2, sh.n_experts).astype(np.float32)
    _, _, err = _case(orc, sh, seed=6, T=9, bias=bias)
    assert err <= DERIVED, err


@pytest.mark.parametrize("T", [64, 512])
def test_s80_batched_sampled(orc, T):
    """80B-shaped layer, every expert resident; a sample of the tokens checked against the oracle."""
    seed = json.load(open(os.path.join(GOLDEN, "s80_layer_seed.json")))["seed"]
    rng = np.random.default_rng(T)
    sample = sorted(set(rng.choice(T, size=6, replace=False).tolist()) | {0, T - 1})
    _, _, err = _case(orc, synth.S80, seed=seed, T=T, sample=sample)
    assert err <= TOL and err <= DERIVED, err


def test_batched_matches_decode_path(orc):
    """Same pool, same tokens: the batched path selects the same experts with the same weights as
    the decode kernel, and the outputs agree to the batched path's rounding."""
    sh = synth.Shape(512, 64, 6, 128, 192, bits=4)
    R = Resident(sh, 1, 21)
    x = _bits(synth.activation_bits(sh, 21, 0, 40))
    yb, ib, wb = R.layer_forward_batched(0, x)
    yd, idd, wd = R.layer_forward(0, x)
    torch.cuda.synchronize()
    same = (ib == idd).all(dim=1)
    assert same.float().mean().item() >= 0.9
    assert torch.allclose(wb[same], wd[same], rtol=0, atol=2e-6)
    assert rel_l2(yb[same].cpu().numpy(), yd[same].cpu().numpy()) <= DERIVED


def test_batched_workspace_and_errors(orc):
    sh = synth.TINY
    R = Resident(sh, 1, 2)
    need = moe.batched_workspace_bytes(R.mshape, 16)
    assert need > 0 and moe.batched_workspace_bytes(R.mshape, 32) > need
    x = _bits(synth.activation_bits(sh, 2, 0, 16))
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError):
        R.layer_forward_batched(0, x, work=small)
    y1, i1, w1 = R.layer_forward_batched(0, x)
    y2, i2, w2 = R.layer_forward_batched(0, x)
    assert torch.equal(i1, i2) and torch.equal(w1, w2)
    assert rel_l2(y1.cpu().numpy(), y2.cpu().numpy()) < 1e-6


@pytest.mark.parametrize("rows,k", [((11, 3), 2), ((14, 3, 7), 2), ((5, 9, 2, 12), 3)])
def test_exact_ties_lower_index_wins_batched(orc, rows, k):
    """Planted exact logit ties (duplicated router rows) through the batched path: every token's
    selection breaks the tie by index as the oracle does (the tied rows align with token 0's signs,
    so token 0 selects them; the other tokens are compared as usual)."""
    sh = synth.Shape(256, 16, k, 64, 64)
    seed = 21
    x = synth.activation_bits(sh, seed, 0, 5)
    Wr = synth.router_bits(sh, seed, 0).copy()
    big = synth.bf16_bits(np.float32(0.3) * np.sign(synth.bf16_value(x[0])))
    for r in rows:
        Wr[r] = big
    R = Resident(sh, 1, seed, router={0: Wr})
    O = OracleLayers(orc, sh, seed, 1, router={0: Wr})
    y, idx, w = R.layer_forward_batched(0, _bits(x))
    torch.cuda.synchronize()
    assert R.pool.device_status() == moe.OK
    y, idx, w = y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()
    assert list(idx[0]) == sorted(rows)[:k]
    for t in range(x.shape[0]):
        r, exact = layer_reference(orc, O, 0, x[t], idx[t])
        np.testing.assert_allclose(w[t], r["w"], rtol=0, atol=2e-6)
        assert rel_l2(y[t], r["y"]) <= (TOL if exact else NEAR_TIE_TOL)


@pytest.mark.parametrize("bits", [4, 8])
def test_independent_bias_batched(orc, bits):
    """Bias drawn independently of the scale through the batched path."""
    sh = synth.Shape(512, 64, 6, 128, 192, bits=bits, free_bias=True)
    _, _, err = _case(orc, sh, seed=23, T=9)
    assert err <= TOL, err


def test_deterministic_combine(orc):
    """MOE_DETERMINISTIC: the batched layer is bit for bit the same on repeated calls (each token's
    contributions summed in rank order, then the shared expert's), and matches the oracle."""
    sh = synth.Shape(512, 64, 6, 128, 192)
    seed, T = 29, 37
    R = Resident(sh, 1, seed, flags=moe.RENORM | moe.DETERMINISTIC)
    x = synth.activation_bits(sh, seed, 0, T)
    outs = []
    for _ in range(3):
        y, idx, w = R.layer_forward_batched(0, _bits(x))
        torch.cuda.synchronize()
        assert R.pool.device_status() == moe.OK
        outs.append((y.clone(), idx.clone()))
    for y2, idx2 in outs[1:]:
        assert torch.equal(outs[0][0], y2) and torch.equal(outs[0][1], idx2)
    O = OracleLayers(orc, sh, seed, 1)
    y, idx = outs[0][0].cpu().numpy(), outs[0][1].cpu().numpy()
    for t in range(T):
        r, exact = layer_reference(orc, O, 0, x[t], idx[t])
        assert rel_l2(y[t], r["y"]) <= (TOL if exact else NEAR_TIE_TOL), t


@pytest.mark.parametrize("path", ["decode", "batched"])
def test_input_beyond_fp16_reports_range(path):
    """An input element above fp16's range (the kernels' fp16 operands cannot hold it) is reported
    as MOE_E_RANGE in the device status, not turned silently into inf."""
    sh = synth.Shape(256, 16, 2, 64, 64)
    R = Resident(sh, 1, 3)
    x = synth.activation_bits(sh, 3, 0, 2).copy()
    x[1, 5] = synth.bf16_bits(np.array([1.0e5], np.float32))[0]
    if path == "decode":
        R.layer_forward(0, _bits(x))
    else:
        R.layer_forward_batched(0, _bits(x))
    torch.cuda.synchronize()
    assert R.pool.device_status() == moe.E_RANGE
    # in range again: the status word was cleared by the read
    x[1, 5] = synth.bf16_bits(np.array([1.0], np.float32))[0]
    R.layer_forward_batched(0, _bits(x)) if path == "batched" else R.layer_forward(0, _bits(x))
    torch.cuda.synchronize()
    assert R.pool.device_status() == moe.OK


@pytest.mark.parametrize("flags,want", [(0, moe.E_RANGE), (moe.GEMV, moe.OK)])
def test_scale_below_fp16_normal_reports_range(flags, want):
    """A group scale below fp16's normal range (2^-14) loses its relative precision in the GEMM
    path's fp16 dequantisation: reported as MOE_E_RANGE. The matrix-vector path applies the scale in
    fp32 (codes enter the MMA exactly), so there it is exact: MOE_OK and finite outputs."""
    sh = synth.Shape(256, 16, 2, 64, 64)
    R = Resident(sh, 1, 3, flags=moe.RENORM | flags)
    # every expert's gate scales -> 1e-6 (bf16), written into the resident blobs
    for e in range(sh.n_experts):
        tt = synth.expert_tensors(sh, 3, 0, int(R.maps[0][e]))
        tt["gate_s"] = np.full_like(tt["gate_s"], synth.bf16_bits(np.float32(1e-6)))
        blob = moe.pack_expert(R.mshape, tt)
        slot = int(R.slots[0][e])
        R.arena[slot * R.stride: slot * R.stride + blob.size].copy_(torch.from_numpy(blob))
    x = synth.activation_bits(sh, 3, 0, 3)
    y, _, _ = R.layer_forward_batched(0, _bits(x))
    torch.cuda.synchronize()
    assert R.pool.device_status() == want
    if want == moe.OK:
        assert torch.isfinite(y).all()


REPEAT_SHAPES = [(256, 40, 3, 64, 128), (768, 100, 7, 192, 320), (256, 512, 16, 64, 64)]


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("dims", REPEAT_SHAPES)
@pytest.mark.parametrize("T", [37, 129, 512])
def test_batched_repeated_seeds(orc, bits, dims, T):
    """The batched kernels against the oracle over ten seeds per shape, width and token count: an
    ordering fault between the kernels' roles (mbarrier phases, proxy fences, tensor-memory waits)
    would show as an intermittent wrong output. Eight tokens per call are compared (every selected
    expert and the shared one run for all T tokens, so any tile of any expert can be wrong)."""
    H, E, k, I, Is = dims
    sh = synth.Shape(H, E, k, I, Is, bits=bits)
    rng = np.random.default_rng(T * 1000 + bits)
    for seed in range(100, 110):
        sample = sorted(rng.choice(T, size=8, replace=False).tolist())
        _, _, err = _case(orc, sh, seed=seed, T=T, sample=sample)
        assert err <= DERIVED, (seed, err)


GEMV_SHAPES = [(256, 16, 2, 64, 64, 4), (256, 16, 2, 64, 64, 8), (768, 100, 7, 192, 320, 8), (256, 512, 16, 64, 64, 4),
               (2048, 512, 10, 512, 512, 4)]


@pytest.mark.parametrize("dims", GEMV_SHAPES)
@pytest.mark.parametrize("T", [1, 8, 37, 64])
def test_gemv_small_token_path(orc, dims, T):
    """MOE_GEMV (T <= 64: the expert products as matrix-vector products, the weights exact): against
    the oracle, and against the tensor-core GEMM path (fp16-rounded weights) on the same layer and
    tokens, deterministic combine on."""
    H, E, k, I, Is, bits = dims
    sh = synth.Shape(H, E, k, I, Is, bits=bits)
    seed, nu = 31, min(64, E)
    Rg = Resident(sh, 1, seed, n_unique=nu, flags=moe.RENORM | moe.DETERMINISTIC | moe.GEMV)
    Rt = Resident(sh, 1, seed, n_unique=nu, flags=moe.RENORM | moe.DETERMINISTIC)
    x = synth.activation_bits(sh, seed, 0, T)
    yg, idxg, _ = Rg.layer_forward_batched(0, _bits(x))
    yt, idxt, _ = Rt.layer_forward_batched(0, _bits(x))
    torch.cuda.synchronize()
    assert Rg.pool.device_status() == moe.OK and Rt.pool.device_status() == moe.OK
    assert torch.equal(idxg, idxt)
    yg, yt, idx = yg.cpu().numpy(), yt.cpu().numpy(), idxg.cpu().numpy()
    # each path is held to the stated batched tolerance against the oracle; their errors are not
    # shared (measured on B300: the paths differ by 5e-5 to 2.4e-4 rel-L2 at these shapes, about
    # as much as each differs from the oracle), so the paths are compared at that tolerance too
    assert rel_l2(yg, yt) <= TOL, rel_l2(yg, yt)
    O = OracleLayers(orc, sh, seed, 1, n_unique=nu)
    for t in range(min(T, 8)):
        r, exact = layer_reference(orc, O, 0, x[t], idx[t])
        assert rel_l2(yg[t], r["y"]) <= (TOL if exact else NEAR_TIE_TOL), t
