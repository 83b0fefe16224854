"""Bounded-pool stacks: dense weights resident on the GPU, routed experts streamed on demand from a
pinned host store into a fixed number of HBM slots (LFU + recency eviction in the library).

torch supplies device memory, pinned host memory and streams; the per-layer host loop (route,
read back the selection, look up, copy misses, run the experts, release) runs in libmoe
(``moe_stack_forward_streamed``).

The host store holds ``n_unique`` generated blobs; expert e of layer l is blob ``maps[l][e]`` (the
same maps as ``Resident``), so a miss always copies one full blob of pinned memory whatever the
store size. Routing popularity for the workload follows a per-layer Zipf law (see
:func:`zipf_bias`); it enters the router as the library's ``logit_bias`` hook.
"""
from __future__ import annotations

import time

import numpy as np
import torch

from . import moe, synth
from .resident import dense_layer, moe_shape

ZIPF_S = 1.1


def zipf_bias(sh: synth.Shape, seed: int, layer: int, beta: float, s: float = ZIPF_S) -> np.ndarray:
    """logit_bias[e] = beta * ln p_e with p_e proportional to (rank_e + 1)^-s, rank a seeded
    per-layer permutation of the experts. A synthetic routing-popularity hook, not part of the method."""
    rank = synth.expert_map(sh, seed ^ 0x5A5A, layer, sh.n_experts)  # a permutation of 0..E-1
    p = (rank.astype(np.float64) + 1.0) ** (-s)
    p /= p.sum()
    return (beta * np.log(p)).astype(np.float32)


def simulated_hit_rate(sh: synth.Shape, n_layers: int, n_slots: int, beta: float, tokens: int = 96,
                       warm: int = 32, seed: int = 0, logit_std: float | None = None) -> float:
    """Hit rate of the library's slot policy (a host-only pool, no device) on a synthetic selection
    trace: router logits taken as independent N(0, std^2) (std = 0.02 * sqrt(H) for the generator's
    N(0, 0.02) router rows against an RMS-normalised input) plus the Zipf bias, top-k per layer."""
    std = 0.02 * np.sqrt(sh.hidden) if logit_std is None else logit_std
    ms = moe_shape(sh)
    pool = moe.Pool(ms, n_layers, n_slots)
    pool.set_copy_hook(lambda slot, blob, n: 0)
    bias = [zipf_bias(sh, seed, l, beta) for l in range(n_layers)]
    rng = np.random.default_rng(seed + 7)
    hits = lookups = 0
    for t in range(warm + tokens):
        for l in range(n_layers):
            lg = rng.standard_normal(sh.n_experts) * std + bias[l]
            sel = np.argpartition(-lg, sh.top_k)[: sh.top_k].astype(np.int32)
            slots = pool.lookup(l, sel)
            for j, e in enumerate(sel):
                if slots[j] < 0:
                    pool.load_slot(l, int(e), 1)
            pool.release()
            if t >= warm:
                hits += int((slots >= 0).sum())
                lookups += sh.top_k
    pool.close()
    return hits / lookups


def calibrate_beta(sh: synth.Shape, n_layers: int, n_slots: int, target: float = 0.55, seed: int = 0) -> float:
    """Zipf bias strength whose simulated hit rate is closest to ``target`` (bisection)."""
    lo, hi = 0.0, 4.0
    for _ in range(12):
        mid = 0.5 * (lo + hi)
        if simulated_hit_rate(sh, n_layers, n_slots, mid, tokens=64, warm=16, seed=seed) < target:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


class Streamed:
    """n_layers pre-norm residual MoE layers in bounded mode (n_slots expert slots in HBM)."""

    def __init__(self, sh: synth.Shape, n_layers: int, seed: int, n_slots: int, *, n_unique: int | None = None,
                 beta: float = 0.0, prefetch: int = 0, device: str = "cuda", verbose: bool = False):
        self.prefetch = prefetch
        t0 = time.time()
        self.sh, self.L, self.seed, self.n_slots = sh, n_layers, seed, n_slots
        E = sh.n_experts
        self.n_unique = n_unique or E
        self.mshape = moe_shape(sh, moe.RENORM | moe.PRENORM | moe.RESIDUAL)
        self.stride = moe.expert_stride(self.mshape)
        self.maps = [synth.expert_map(sh, seed, l, self.n_unique) for l in range(n_layers)]
        self.store = torch.empty((self.n_unique, self.stride), dtype=torch.uint8, pin_memory=True)
        for u in range(self.n_unique):
            moe.pack_expert(self.mshape, synth.expert_tensors(sh, seed, 0, u), out=self.store[u].numpy())
        base = self.store.data_ptr()
        self.h_blobs = np.array([[base + int(self.maps[l][e]) * self.stride for e in range(E)]
                                 for l in range(n_layers)], dtype=np.uint64)
        self.beta = beta
        self.bias = [torch.from_numpy(zipf_bias(sh, seed, l, beta)).to(device) if beta else None for l in range(n_layers)]
        self.router, self.shared, self.gate = [], [], []
        for l in range(n_layers):
            rt, sb, g = dense_layer(sh, self.mshape, seed, l, device)
            self.router.append(rt)
            self.shared.append(sb)
            self.gate.append(g)
        self.arena = torch.empty(n_slots * self.stride, dtype=torch.uint8, device=device)
        self.ws = torch.zeros(moe.workspace_bytes(self.mshape, n_layers), dtype=torch.uint8, device=device)
        self.pool = None
        self.reset_pool()
        self.copy_stream = torch.cuda.Stream()
        torch.cuda.synchronize()
        if verbose:
            print(f"[streamed] {n_layers} layers x {E} experts, {n_slots} slots ({self.arena.numel() / 2**30:.2f} GiB), "
                  f"store {self.store.numel() / 1e9:.2f} GB pinned, beta {beta:.3f}, set-up {time.time() - t0:.1f} s",
                  flush=True)

    def set_beta(self, beta: float):
        """Change the Zipf routing bias strength (re-registers the layers' bias vectors)."""
        self.beta = beta
        self.bias = [torch.from_numpy(zipf_bias(self.sh, self.seed, l, beta)).to(self.arena.device) if beta else None
                     for l in range(self.L)]
        for l in range(self.L):
            self.pool.set_layer(l, self.router[l], self.shared[l], self.gate[l], self.bias[l])
        self.pool.sync()
        torch.cuda.synchronize()

    def reset_pool(self):
        """A fresh, empty pool over the same arena and workspace (counters and slot table cleared)."""
        if self.pool is not None:
            torch.cuda.synchronize()
            self.pool.close()
        self.ws.zero_()
        self.pool = moe.Pool(self.mshape, self.L, self.n_slots, self.arena, self.arena.numel(), self.ws, self.ws.numel())
        self.pool.set_prefetch(self.prefetch)
        for l in range(self.L):
            self.pool.set_layer(l, self.router[l], self.shared[l], self.gate[l], self.bias[l])
        self.pool.sync()
        torch.cuda.synchronize()

    def measure_hit_rate(self, xs: torch.Tensor, warm: int = 16, tokens: int = 24) -> float:
        """Hit rate of a fresh pool over `tokens` decode steps after `warm` steps (inputs xs[i % len])."""
        self.reset_pool()
        out = torch.empty(self.sh.hidden, dtype=torch.float32, device=xs.device)
        for i in range(warm):
            self.step(xs[i % xs.shape[0]], out)
        torch.cuda.synchronize()
        h0, m0, _ = self.pool.stats()
        for i in range(tokens):
            self.step(xs[(warm + i) % xs.shape[0]], out)
        torch.cuda.synchronize()
        h1, m1, _ = self.pool.stats()
        return (h1 - h0) / max(1, (h1 - h0) + (m1 - m0))

    def calibrate_beta(self, xs: torch.Tensor, target: float = 0.55, iters: int = 6, lo: float = 0.0,
                       hi: float = 1.5, warm: int = 16, tokens: int = 24) -> tuple[float, float]:
        """Bisect the Zipf strength on the real routing of this stack until the measured hit rate
        is near `target`; returns (beta, hit rate)."""
        best = (self.beta, None)
        for _ in range(iters):
            mid = 0.5 * (lo + hi)
            self.set_beta(mid)
            hr = self.measure_hit_rate(xs, warm=warm, tokens=tokens)
            best = (mid, hr)
            if hr < target:
                lo = mid
            else:
                hi = mid
        return best

    def bias_host(self, layer: int):
        return None if not self.beta else zipf_bias(self.sh, self.seed, layer, self.beta)

    def write_qpack(self, path: str) -> None:
        """Write every (layer, expert) blob of this stack into an on-disk container at `path`."""
        q = moe.Qpack.create(path, self.mshape, self.L)
        try:
            for l in range(self.L):
                for e in range(self.sh.n_experts):
                    q.write(l, e, self.store[int(self.maps[l][e])].numpy())
        finally:
            q.close()

    def pinned_staging(self, n: int) -> torch.Tensor:
        """Pinned host buffer of n blobs at a 4096-byte aligned address (direct reads need it; the
        caching pinned allocator does not promise that alignment), as a view of a larger buffer."""
        raw = torch.empty(n * self.stride + 4096, dtype=torch.uint8, pin_memory=True)
        off = (-raw.data_ptr()) % 4096
        return raw[off:off + n * self.stride]

    def step_qpack(self, x: torch.Tensor, out: torch.Tensor, qpack, staging: torch.Tensor, n_staging: int,
                   stream=None, topk_idx: np.ndarray | None = None):
        """One token through all layers, the misses read from the container `qpack` through the
        pinned buffer `staging` (n_staging blobs)."""
        s = torch.cuda.current_stream() if stream is None else stream
        self.pool.stack_forward_qpack(0, self.L, x, out, qpack, staging, n_staging, s, self.copy_stream, topk_idx)

    def layer_step(self, layer: int, x: torch.Tensor, out: torch.Tensor, stream=None,
                   topk_idx: np.ndarray | None = None):
        """Layer ``layer`` alone through the bounded pool (the pool's state carries over between
        calls): x, out fp32 device tensors [H]; topk_idx int32 [top_k] receives its selection."""
        s = torch.cuda.current_stream() if stream is None else stream
        self.pool.stack_forward_streamed(layer, 1, x, out, self.h_blobs, s, self.copy_stream, topk_idx)

    def step(self, x: torch.Tensor, out: torch.Tensor, stream=None, topk_idx: np.ndarray | None = None):
        """One token through all layers: x, out fp32 device tensors [H]."""
        s = torch.cuda.current_stream() if stream is None else stream
        self.pool.stack_forward_streamed(0, self.L, x, out, self.h_blobs, s, self.copy_stream, topk_idx)
