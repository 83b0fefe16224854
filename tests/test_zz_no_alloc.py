"""moe_layer_forward_static, the entry point for callers that may not allocate device memory.

Some callers cannot allocate device memory at all: a plugin inside a host application that owns
every device allocation, or a latency-critical loop that must never call cudaMalloc. They cannot
hand the library a workspace, so this entry point keeps its scratch in a fixed device array
inside the library. Its results must equal those of moe_layer_forward on the same layer.

This file is collected last on purpose: a run that stops at the first failure has run every other
test before it. It must pass on its own in a fresh process and after the rest of the suite (the
scratch array then holds an earlier call's leftovers).
"""
import numpy as np
import pytest
import torch

from int4_routed_expert_05_b300 import moe, synth
from int4_routed_expert_05_b300.resident import Resident

from gpu_ref import rel_l2

pytestmark = pytest.mark.gpu

TIGHT = 1e-4  # rel-L2 bound the GPU parity tests assert for this kernel


@pytest.fixture(scope="module", autouse=True)
def _built():
    from int4_routed_expert_05_b300 import _build
    _build.build()
    assert torch.cuda.is_available()


def test_static_scratch_matches_workspace_path():
    # 80B-shaped layer (hidden 2048, top-10, inter 512, shared 512) over 64 experts
    sh = synth.Shape(2048, 64, 10, 512, 512)
    seed, T = 21, 2
    R = Resident(sh, 1, seed)
    # the arena holds expert e at slot e: exactly the fixed-stride container layout
    assert np.array_equal(R.slots[0], np.arange(sh.n_experts))
    k, H = sh.top_k, sh.hidden
    for call in range(2):  # two calls in a row share (and must reset) the scratch array
        x = torch.from_numpy(synth.activation_bits(sh, seed, call, T).view(np.int16)).cuda()
        y_ref, idx_ref, w_ref = R.layer_forward(0, x)
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        moe.layer_forward_static(R.mshape, R.arena, R.router[0], R.shared[0], R.gate[0], x, T, y, idx, w, status)
        torch.cuda.synchronize()
        assert R.pool.device_status() == moe.OK
        assert int(status.item()) == moe.OK
        assert torch.equal(idx, idx_ref), (call, idx, idx_ref)
        assert torch.allclose(w, w_ref, rtol=0, atol=1e-6)
        err = rel_l2(y.cpu().numpy(), y_ref.cpu().numpy())
        assert err <= TIGHT, (call, err)


def _static_vs_workspace(R, sh, x_np, T):
    k, H = sh.top_k, sh.hidden
    x = torch.from_numpy(x_np.view(np.int16)).cuda()
    y_ref, idx_ref, w_ref = R.layer_forward(0, x)
    y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    moe.layer_forward_static(R.mshape, R.arena, R.router[0], R.shared[0], R.gate[0], x, T, y, idx, w, status)
    torch.cuda.synchronize()
    assert R.pool.device_status() == moe.OK and int(status.item()) == moe.OK
    assert torch.equal(idx, idx_ref), (idx, idx_ref)
    assert torch.allclose(w, w_ref, rtol=0, atol=1e-6)
    return rel_l2(y.cpu().numpy(), y_ref.cpu().numpy())


def test_static_scratch_alternating_shapes():
    """Calls with different shapes in turn (the scratch layout moves with the expert count, top-k
    and intermediate sizes): each call must match the workspace path, so no exchange word of one
    shape is taken for another's."""
    shapes = [synth.Shape(2048, 512, 10, 512, 512), synth.Shape(512, 64, 2, 128, 128)]
    Rs = [Resident(sh, 1, 31 + i, n_unique=64) for i, sh in enumerate(shapes)]
    for call, i in enumerate([0, 1, 0, 1, 1, 0]):
        sh, R = shapes[i], Rs[i]
        assert np.array_equal(R.slots[0], np.arange(sh.n_experts))
        err = _static_vs_workspace(R, sh, synth.activation_bits(sh, 40 + call, 0, 2), 2)
        assert err <= TIGHT, (call, i, err)


def test_static_scratch_rejects_oversized_shape():
    # (top_k + 1) x max(inter, shared_inter) fp32 activations alone exceed the fixed array
    big = moe.make_shape(2048, 64, 16, 4096, 4096)
    with pytest.raises(moe.MoeError) as ei:
        moe.layer_forward_static(big, 256, 256, 256, 256, 256, 1, 256)
    assert ei.value.status == moe.E_NOMEM
    assert "MOE_STATIC_SCRATCH_BYTES" in moe.load().moe_last_error().decode()
