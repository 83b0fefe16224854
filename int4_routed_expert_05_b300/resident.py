"""Synthetic MoE layers made resident on one GPU (set-up for the tests, the smoke check and the
benchmark).

torch supplies device memory and copies only; every step of the layer runs in libmoe. Expert
tensors come from ``synth``: expert e of layer l holds generator tensor ``maps[l][e]`` (drawn as
``synth.expert_tensors(shape, seed, 0, maps[l][e])``), the shared expert, router and shared gate
of layer l are drawn per layer. Each (layer, expert) has its own pool slot, so a stack streams
distinct bytes from HBM even when it reuses generator tensors.
"""
from __future__ import annotations

import time

import numpy as np
import torch

from . import moe, synth


def moe_shape(sh: synth.Shape, flags: int | None = None) -> moe.Shape:
    if flags is None:
        flags = moe.RENORM if sh.renorm else 0
    return moe.make_shape(sh.hidden, sh.n_experts, sh.top_k, sh.inter, sh.shared_inter, sh.bits, sh.group, flags)


def dense_layer(sh: synth.Shape, mshape: moe.Shape, seed: int, layer: int, device: str = "cuda", router_bits=None):
    """Layer ``layer``'s resident weights on the device: router bf16 [E][H], shared-expert blob,
    shared gate bf16 [H] (all drawn by ``synth``, the router unless given; the blob packed by the
    library)."""
    if router_bits is None:
        router_bits = synth.router_bits(sh, seed, layer)
    router = torch.from_numpy(np.ascontiguousarray(router_bits).view(np.int16)).to(device)
    sb = moe.pack_expert(mshape, synth.expert_tensors(sh, seed, layer, synth.SHARED_EXPERT), shared=True)
    shared = torch.from_numpy(sb).to(device)
    gate = torch.from_numpy(synth.shared_gate_bits(sh, seed, layer).view(np.int16)).to(device)
    return router, shared, gate


class Resident:
    """n_layers layers of shape ``sh`` with every expert placed in the pool."""

    def __init__(self, sh: synth.Shape, n_layers: int, seed: int, *, n_unique: int | None = None,
                 flags: int | None = None, slot_perm_seed: int | None = None, bias: list | None = None,
                 router: dict | None = None, device: str = "cuda", verbose: bool = False):
        t0 = time.time()
        self.sh, self.L, self.seed = sh, n_layers, seed
        E = sh.n_experts
        self.n_unique = n_unique or E
        self.mshape = moe_shape(sh, flags)
        self.stride = moe.expert_stride(self.mshape)
        self.stride_s = moe.expert_stride(self.mshape, shared=True)
        self.n_slots = n_layers * E
        self.device = device
        self.maps = [synth.expert_map(sh, seed, l, self.n_unique) for l in range(n_layers)]

        # unique expert blobs: drawn and packed on the host, uploaded once
        uniq = torch.empty((self.n_unique, self.stride), dtype=torch.uint8, pin_memory=True)
        for u in range(self.n_unique):
            moe.pack_expert(self.mshape, synth.expert_tensors(sh, seed, 0, u), out=uniq[u].numpy())
        uniq_d = uniq.to(device, non_blocking=True)

        slots = np.arange(self.n_slots, dtype=np.int64).reshape(n_layers, E)
        if slot_perm_seed is not None:
            slots = np.random.default_rng(slot_perm_seed).permutation(self.n_slots).reshape(n_layers, E)
        self.slots = slots
        self.arena = torch.empty(self.n_slots * self.stride, dtype=torch.uint8, device=device)
        arena_v = self.arena.view(self.n_slots, self.stride)
        for l in range(n_layers):
            arena_v[torch.from_numpy(slots[l]).to(device)] = uniq_d[torch.from_numpy(self.maps[l]).to(device)]
        del uniq_d

        # resident dense weights of every layer
        self.router, self.shared, self.gate, self.bias = [], [], [], []
        for l in range(n_layers):
            rt, sb, g = dense_layer(sh, self.mshape, seed, l, device, None if router is None else router.get(l))
            self.router.append(rt)
            self.shared.append(sb)
            self.gate.append(g)
            b = None if bias is None or bias[l] is None else torch.as_tensor(bias[l], dtype=torch.float32).to(device)
            self.bias.append(b)

        self.ws_bytes = moe.workspace_bytes(self.mshape, n_layers)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        self.pool = moe.Pool(self.mshape, n_layers, self.n_slots, self.arena, self.arena.numel(), self.ws, self.ws_bytes)
        for l in range(n_layers):
            self.pool.set_layer(l, self.router[l], self.shared[l], self.gate[l], self.bias[l])
            for e in range(E):
                self.pool.place(l, e, int(slots[l, e]))
        self.pool.sync()
        torch.cuda.synchronize()
        if verbose:
            print(f"[resident] {n_layers} layers x {E} experts, {self.arena.numel() / 1e9:.2f} GB arena, "
                  f"{self.n_unique} unique blobs, set-up {time.time() - t0:.1f} s", flush=True)

    # -- generator tensors behind the layers (for a CPU reference of the same inputs) --
    def expert_tensors(self, layer: int, expert: int) -> dict:
        return synth.expert_tensors(self.sh, self.seed, 0, int(self.maps[layer][expert]))

    def shared_tensors(self, layer: int) -> dict:
        return synth.expert_tensors(self.sh, self.seed, layer, synth.SHARED_EXPERT)

    # -- calls --
    def layer_forward(self, layer: int, x_bits: torch.Tensor, stream=None):
        """x_bits: int16 device tensor [T][H] of bf16 bit patterns -> (y fp32 [T][H], idx, w)."""
        T = x_bits.shape[0]
        y = torch.empty((T, self.sh.hidden), dtype=torch.float32, device=self.device)
        idx = torch.empty((T, self.sh.top_k), dtype=torch.int32, device=self.device)
        w = torch.empty((T, self.sh.top_k), dtype=torch.float32, device=self.device)
        self.pool.layer_forward(layer, x_bits, T, y, idx, w, stream)
        return y, idx, w

    def layer_forward_batched(self, layer: int, x_bits: torch.Tensor, stream=None, work: torch.Tensor | None = None):
        """The batched (GEMM) path: x_bits int16 [T][H] bf16 patterns -> (y fp32 [T][H], idx, w)."""
        T = x_bits.shape[0]
        y = torch.empty((T, self.sh.hidden), dtype=torch.float32, device=self.device)
        idx = torch.empty((T, self.sh.top_k), dtype=torch.int32, device=self.device)
        w = torch.empty((T, self.sh.top_k), dtype=torch.float32, device=self.device)
        if work is None:
            work = torch.empty(moe.batched_workspace_bytes(self.mshape, T), dtype=torch.uint8, device=self.device)
        self.pool.layer_forward_batched(layer, x_bits, T, y, work, idx, w, stream)
        return y, idx, w

    def stack_forward(self, x: torch.Tensor, layer0: int = 0, n_layers: int | None = None, trace: bool = False,
                      stream=None):
        """x: fp32 device tensor [H] -> (x_out, trace [n+1][H] or None, idx [n][k], w [n][k])."""
        n = self.L - layer0 if n_layers is None else n_layers
        H, k = self.sh.hidden, self.sh.top_k
        out = torch.empty(H, dtype=torch.float32, device=self.device)
        tr = torch.empty((n + 1, H), dtype=torch.float32, device=self.device) if trace else None
        idx = torch.empty((n, k), dtype=torch.int32, device=self.device)
        w = torch.empty((n, k), dtype=torch.float32, device=self.device)
        self.pool.stack_forward(layer0, n, x, out, tr, idx, w, stream)
        return out, tr, idx, w

    def layer_forward_scalar(self, layer: int, x_bits: torch.Tensor, stream=None):
        y = torch.empty((1, self.sh.hidden), dtype=torch.float32, device=self.device)
        idx = torch.empty((1, self.sh.top_k), dtype=torch.int32, device=self.device)
        w = torch.empty((1, self.sh.top_k), dtype=torch.float32, device=self.device)
        self.pool.layer_forward_scalar(layer, x_bits, y, idx, w, stream)
        return y, idx, w
