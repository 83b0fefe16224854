"""The oracle's view of a stack of generated layers (TEST INFRASTRUCTURE, like the rest of oracle/).

OracleLayers evaluates the oracle on exactly the inputs the seeded generator (the package's synth
module, which draws numbers only) gives a resident GPU stack: the same seed, expert maps, router
override and logit bias. It is built from the generator's recipe alone, never from device data.
Only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
"""
import numpy as np

from int4_routed_expert_05_b300 import synth


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
