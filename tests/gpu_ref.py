"""Helpers of the GPU parity tests: the oracle's view of a resident layer, built only from the
input generator's recipe (seed, shapes, expert maps) and never from device data."""
import numpy as np

from int4_routed_expert_05_b300 import synth


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


class OracleLayers:
    """The oracle evaluated on the same generated inputs as a ``Resident`` (same seed, maps, bias)."""

    def __init__(self, orc, sh, seed, n_layers, n_unique=None, bias=None, router=None):
        self.orc, self.sh, self.seed, self.L = orc, sh, seed, n_layers
        self.router = router or {}
        self.n_unique = n_unique or sh.n_experts
        self.maps = [synth.expert_map(sh, seed, l, self.n_unique) for l in range(n_layers)]
        self.bias = bias
        self._blobs = {}
        self._dense = {}
        self._dummy = np.zeros(orc.blob_stride(sh), np.uint8)

    def dense(self, l):
        if l not in self._dense:
            sh = self.sh
            rt = self.router[l] if l in self.router else synth.router_bits(sh, self.seed, l)
            self._dense[l] = (rt, synth.shared_gate_bits(sh, self.seed, l),
                              self.orc.pack(sh, synth.expert_tensors(sh, self.seed, l, synth.SHARED_EXPERT), shared=True))
        return self._dense[l]

    def blob(self, l, e):
        u = int(self.maps[l][e])
        if u not in self._blobs:
            self._blobs[u] = self.orc.pack(self.sh, synth.expert_tensors(self.sh, self.seed, 0, u))
        return self._blobs[u]

    def layer(self, l, u_bits, force_idx=None):
        """One layer for bf16 input u_bits: the oracle's own selection, or (``force_idx``, k indices
        in rank order) the layer evaluated for that selection."""
        orc, sh = self.orc, self.sh
        Wr, w_sg, shared = self.dense(l)
        bias = None if self.bias is None else self.bias[l]
        if force_idx is None:
            lg, bd = orc.router_logits(Wr, u_bits, bias)
            idx, _ = orc.topk(lg, sh.top_k, sh.renorm)
        else:
            idx = np.asarray(force_idx)
        blobs = [self._dummy] * sh.n_experts
        for e in idx:
            blobs[int(e)] = self.blob(l, int(e))
        return orc.moe_layer(sh, u_bits, Wr, w_sg, blobs, shared, bias, force_idx=force_idx)

    def expert_y(self, l, e, u_bits):
        y, _ = self.orc.expert_ffn(self.sh, self.blob(l, e), u_bits)
        return y


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
