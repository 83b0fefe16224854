"""Bounded-pool stacks on the GPU: the per-layer host loop of moe_stack_forward_streamed (route,
read back, LFU + recency lookup, miss copies from pinned host memory, experts, release) gives
bit for bit the output of the resident stack, whose layers are checked against the oracle in
test_gpu_parity (cache hit or miss gives the same answer)."""
import numpy as np
import pytest
import torch

from int4_routed_expert_05_b300 import moe, synth
from int4_routed_expert_05_b300.resident import Resident
from int4_routed_expert_05_b300.streamed import Streamed, zipf_bias

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_routed_expert_05_b300 import _build
    _build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("prefetch", [0, 4, 16])
@pytest.mark.parametrize("sh,n_slots", [(synth.Shape(2048, 512, 10, 512, 512), 24), (synth.TINY, 5)])
def test_streamed_stack_equals_resident(sh, n_slots, prefetch):
    L, seed, beta, n_unique = 4, 3, 0.7, 64
    flags = moe.RENORM | moe.PRENORM | moe.RESIDUAL
    bias = [zipf_bias(sh, seed, l, beta) for l in range(L)]
    R = Resident(sh, L, seed, n_unique=min(n_unique, sh.n_experts), flags=flags, bias=bias)
    S = Streamed(sh, L, seed, n_slots, n_unique=min(n_unique, sh.n_experts), beta=beta, prefetch=prefetch)
    out_s = torch.empty(sh.hidden, dtype=torch.float32, device="cuda")
    steps = 3
    for step in range(steps):
        x0 = torch.from_numpy(synth.activation_f32(sh, seed, step)[0]).cuda()
        out_r, _, idx_r, _ = R.stack_forward(x0)
        sel = np.zeros((L, sh.top_k), dtype=np.int32)
        S.step(x0, out_s, topk_idx=sel)
        torch.cuda.synchronize()
        assert R.pool.device_status() == moe.OK and S.pool.device_status() == moe.OK
        assert np.array_equal(sel, idx_r.cpu().numpy()), step
        assert torch.equal(out_r, out_s), step
    hits, misses, nbytes = S.pool.stats()
    assert hits + misses == steps * L * sh.top_k
    # speculative copies add bytes beyond the misses of the real selections
    assert misses > 0 and (nbytes >= misses * S.stride if prefetch else nbytes == misses * S.stride)
    if prefetch:
        with pytest.raises(moe.MoeError):
            S.pool.set_prefetch(-1)


def test_streamed_layers_against_oracle(orc):
    """The bounded pool against the oracle, teacher-forced on every layer: an 80B-shaped stack of 8
    layers (Zipf-biased routing; 96 slots for 80 selections per token out of 4096 experts, so that
    later tokens hit the experts earlier ones loaded and miss the others), three tokens; each
    layer's selection and output against the oracle evaluated on that layer's own GPU input (a
    near tie with the oracle evaluated for the GPU's selection)."""
    import sys, os
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    from gpu_ref import OracleLayers, layer_reference, rel_l2
    sh = synth.S80
    L, seed, beta, n_unique, n_slots = 8, 5, 0.7, 64, 96
    S = Streamed(sh, L, seed, n_slots, n_unique=n_unique, beta=beta)
    O = OracleLayers(orc, sh, seed, L, n_unique=n_unique, bias=[S.bias_host(l) for l in range(L)])
    x = torch.empty(sh.hidden, dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    sel = np.zeros(sh.top_k, dtype=np.int32)
    for step in range(3):
        x.copy_(torch.from_numpy(synth.activation_f32(sh, seed, step)[0]))
        for l in range(L):
            S.layer_step(l, x, y, topk_idx=sel)
            torch.cuda.synchronize()
            assert S.pool.device_status() == moe.OK
            xin, xout = x.cpu().numpy().astype(np.float64), y.cpu().numpy().astype(np.float64)
            r, _ = layer_reference(orc, O, l, orc.rmsnorm_bf16(xin), sel)
            assert rel_l2(xout - xin, r["y"]) <= 2e-3, (step, l)
            x.copy_(y)
    hits, misses, _ = S.pool.stats()
    assert hits > 0 and misses > 0, (hits, misses)


@pytest.mark.parametrize("sh,n_slots,L", [(synth.TINY, 5, 4), (synth.S80, 24, 3)])
def test_qpack_stack_equals_resident(tmp_path, sh, n_slots, L):
    """Bounded pool fed from the on-disk expert container (parallel positioned reads into a pinned
    staging ring, then copies to the pool): the output equals the resident stack's bit for bit,
    and every miss moved exactly one blob."""
    seed, beta, n_unique = 3, 0.7, 64
    flags = moe.RENORM | moe.PRENORM | moe.RESIDUAL
    bias = [zipf_bias(sh, seed, l, beta) for l in range(L)]
    R = Resident(sh, L, seed, n_unique=min(n_unique, sh.n_experts), flags=flags, bias=bias)
    S = Streamed(sh, L, seed, n_slots, n_unique=min(n_unique, sh.n_experts), beta=beta)
    path = str(tmp_path / "experts.qpack")
    S.write_qpack(path)
    q = moe.Qpack.open(path, direct=True, n_threads=4)
    n_staging = 2 * sh.top_k
    staging = S.pinned_staging(n_staging)
    out_s = torch.empty(sh.hidden, dtype=torch.float32, device="cuda")
    try:
        for step in range(3):
            x0 = torch.from_numpy(synth.activation_f32(sh, seed, step)[0]).cuda()
            out_r, _, idx_r, _ = R.stack_forward(x0)
            sel = np.zeros((L, sh.top_k), dtype=np.int32)
            S.step_qpack(x0, out_s, q, staging, n_staging, topk_idx=sel)
            torch.cuda.synchronize()
            assert R.pool.device_status() == moe.OK and S.pool.device_status() == moe.OK
            assert np.array_equal(sel, idx_r.cpu().numpy()), step
            assert torch.equal(out_r, out_s), step
        hits, misses, nbytes = S.pool.stats()
        assert misses > 0 and nbytes == misses * S.stride
        with pytest.raises(moe.MoeError):  # too few staging slots for a layer's misses
            S.step_qpack(x0, out_s, q, staging, sh.top_k - 1)
    finally:
        q.close()
