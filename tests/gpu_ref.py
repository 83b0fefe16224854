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

    def __init__(self, orc, sh, seed, n_layers, n_unique=None, bias=None):
        self.orc, self.sh, self.seed, self.L = orc, sh, seed, n_layers
        self.n_unique = n_unique or sh.n_experts
        self.maps = [synth.expert_map(sh, seed, l, self.n_unique) for l in range(n_layers)]
        self.bias = bias
        self._blobs = {}
        self._dense = {}
        self._dummy = np.zeros(orc.blob_stride(sh), np.uint8)

    def dense(self, l):
        if l not in self._dense:
            sh = self.sh
            self._dense[l] = (synth.router_bits(sh, self.seed, l), synth.shared_gate_bits(sh, self.seed, l),
                              self.orc.pack(sh, synth.expert_tensors(sh, self.seed, l, synth.SHARED_EXPERT), shared=True))
        return self._dense[l]

    def blob(self, l, e):
        u = int(self.maps[l][e])
        if u not in self._blobs:
            self._blobs[u] = self.orc.pack(self.sh, synth.expert_tensors(self.sh, self.seed, 0, u))
        return self._blobs[u]

    def layer(self, l, u_bits, force_idx=None):
        """One layer for bf16 input u_bits. ``force_idx`` only chooses which expert blobs are built
        (an optimisation: unselected experts are never read by the oracle)."""
        orc, sh = self.orc, self.sh
        Wr, w_sg, shared = self.dense(l)
        bias = None if self.bias is None else self.bias[l]
        lg, bd = orc.router_logits(Wr, u_bits, bias)
        idx, _ = orc.topk(lg, sh.top_k, sh.renorm)
        blobs = [self._dummy] * sh.n_experts
        for e in idx:
            blobs[e] = self.blob(l, e)
        r = orc.moe_layer(sh, u_bits, Wr, w_sg, blobs, shared, bias)
        return r

    def expert_y(self, l, e, u_bits):
        y, _ = self.orc.expert_ffn(self.sh, self.blob(l, e), u_bits)
        return y


def check_selection(orc, r, gpu_idx):
    """Selection parity: exact where the oracle's decision margin is positive; otherwise (a near tie
    within the binary32 error bound) the GPU's set must still be a valid top-k under the bound.
    Returns True when the selections are identical."""
    gpu_idx = np.asarray(gpu_idx)
    margin = orc.selection_margin(r["logits"], r["bound"], r["idx"])
    if np.array_equal(gpu_idx, r["idx"]):
        return True
    assert margin <= 0, f"selection differs with positive margin {margin}: gpu {gpu_idx} oracle {r['idx']}"
    lg, bd = r["logits"], r["bound"]
    kth = np.sort(lg)[::-1][len(gpu_idx) - 1]
    slack = np.spacing(np.float32(abs(kth))) * 2
    assert np.all(lg[gpu_idx] + bd[gpu_idx] + slack >= kth - bd.max()), "GPU selection is not a valid near-tie top-k"
    return False
