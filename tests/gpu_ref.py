"""Helpers of the GPU parity tests: the selection check and the choice of the oracle result to
compare with (OracleLayers, the oracle's view of a resident layer, lives in oracle/layers.py)."""
import numpy as np

from int4_routed_expert_05_b300 import synth  # noqa: F401  (re-exported for the tests)
from oracle.layers import OracleLayers  # noqa: F401


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_selection(orc, r, gpu_idx):
    """Selection parity. The GPU's k indices must be distinct experts in rank order (fp32 logits
    non-increasing, equal logits by increasing index). They must equal the oracle's where the
    oracle's decision margin is positive; otherwise (a near tie within the binary32 error bound)
    they must still be a valid top-k under the bound. Returns True when the selections are
    identical (the caller then compares with the oracle's result, else with the oracle evaluated for
    the GPU's selection: see layer_reference)."""
    gpu_idx = np.asarray(gpu_idx).astype(np.int64)
    lg, bd = np.asarray(r["logits"]), np.asarray(r["bound"])
    k = len(r["idx"])
    assert gpu_idx.shape == (k,), gpu_idx
    assert np.all((gpu_idx >= 0) & (gpu_idx < lg.shape[0])), f"index out of range: {gpu_idx}"
    assert len(set(gpu_idx.tolist())) == k, f"repeated expert in the GPU selection {gpu_idx}"
    f = lg[gpu_idx].astype(np.float32)
    for j in range(k - 1):
        assert f[j] > f[j + 1] or (f[j] == f[j + 1] and gpu_idx[j] < gpu_idx[j + 1]), \
            f"GPU selection not in rank order at {j}: {gpu_idx} logits {f}"
    if np.array_equal(gpu_idx, r["idx"]):
        return True
    margin = orc.selection_margin(lg, bd, r["idx"])
    assert margin <= 0, f"selection differs with positive margin {margin}: gpu {gpu_idx} oracle {r['idx']}"
    kth = np.sort(lg)[::-1][k - 1]
    slack = np.spacing(np.float32(abs(kth))) * 2
    assert np.all(lg[gpu_idx] + bd[gpu_idx] + slack >= kth - bd.max()), "GPU selection is not a valid near-tie top-k"
    return False


def layer_reference(orc, O, l, u_bits, gpu_idx):
    """The oracle's result to compare one GPU layer output with: the oracle's own layer when the
    selections agree, else the oracle evaluated for the GPU's (valid, near-tie) selection. Returns
    (result, exact) with exact False in the second case."""
    r = O.layer(l, u_bits)
    if check_selection(orc, r, gpu_idx):
        return r, True
    rf = O.layer(l, u_bits, force_idx=np.asarray(gpu_idx))
    return rf, False
