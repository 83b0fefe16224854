"""ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every computation runs in the CUDA library. Pointers are plain integers (``tensor.data_ptr()``
for torch tensors), streams are ``torch.cuda.Stream.cuda_stream`` integers (0 = default stream).
Loading fails loudly when libmoe.so has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

OK, E_INVALID, E_SHAPE, E_NOT_RESIDENT, E_POOL_FULL, E_CUDA, E_TIMEOUT, E_NOMEM, E_RANGE = range(9)
RENORM, PRENORM, RESIDUAL, DETERMINISTIC, GEMV = 1, 2, 4, 8, 16
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_E_INVALID", 2: "MOE_E_SHAPE", 3: "MOE_E_NOT_RESIDENT",
                4: "MOE_E_POOL_FULL", 5: "MOE_E_CUDA", 6: "MOE_E_TIMEOUT", 7: "MOE_E_NOMEM", 8: "MOE_E_RANGE"}

ENTRY_POINTS = [
    "moe_expert_bytes", "moe_expert_stride", "moe_pack_expert", "moe_workspace_bytes",
    "moe_pool_create", "moe_pool_destroy", "moe_pool_slot_ptr", "moe_pool_set_layer", "moe_pool_place",
    "moe_pool_sync", "moe_pool_lookup", "moe_pool_load_slot", "moe_pool_wait_loads", "moe_pool_release",
    "moe_pool_stats", "moe_layer_forward", "moe_stack_forward", "moe_route", "moe_experts",
    "moe_layer_forward_scalar", "moe_device_status", "moe_pool_set_timeout", "moe_pool_grid",
    "moe_last_error", "moe_pool_slot_of", "moe_pool_set_copy_hook", "moe_layer_forward_static",
    "moe_pool_set_prefetch",
    "moe_stack_forward_streamed", "moe_batched_workspace_bytes", "moe_layer_forward_batched",
    "moe_pool_time_batched", "moe_pool_batched_gemm_ms",
    "moe_qpack_create", "moe_qpack_open", "moe_qpack_info", "moe_qpack_write", "moe_qpack_read",
    "moe_qpack_close", "moe_stack_forward_qpack",
]
# include/hybrid.h
HYBRID_ENTRY_POINTS = ["moe_gdn_step", "moe_gqa_workspace_bytes", "moe_gqa_decode"]
QPACK_DIRECT = 1


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("hidden", "n_experts", "top_k", "inter", "shared_inter", "bits", "group", "flags")]


class LayerWeights(ctypes.Structure):
    _fields_ = [("router", ctypes.c_void_p), ("shared_blob", ctypes.c_void_p),
                ("shared_gate", ctypes.c_void_p), ("logit_bias", ctypes.c_void_p)]


class GdnShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_key_heads", "n_value_heads", "key_dim", "value_dim")]


class GqaShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_q_heads", "n_kv_heads", "head_dim", "max_len")]


COPY_HOOK = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t)

_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ, ST = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_int
    PS = ctypes.POINTER(Shape)
    sig = {
        "moe_expert_bytes": (SZ, [PS, ctypes.c_int]),
        "moe_expert_stride": (SZ, [PS, ctypes.c_int]),
        "moe_pack_expert": (ST, [PS, ctypes.c_int, P, P, P, P]),
        "moe_workspace_bytes": (SZ, [PS, I32]),
        "moe_pool_create": (ST, [PS, I32, I32, P, SZ, P, SZ, ctypes.POINTER(P)]),
        "moe_pool_destroy": (None, [P]),
        "moe_pool_slot_ptr": (P, [P, I32]),
        "moe_pool_set_layer": (ST, [P, I32, ctypes.POINTER(LayerWeights)]),
        "moe_pool_place": (ST, [P, I32, I32, I32]),
        "moe_pool_sync": (ST, [P, P]),
        "moe_pool_lookup": (ST, [P, I32, P, I32, P]),
        "moe_pool_load_slot": (ST, [P, I32, I32, P, P, ctypes.POINTER(I32)]),
        "moe_pool_wait_loads": (ST, [P, P]),
        "moe_pool_release": (ST, [P, P]),
        "moe_pool_stats": (ST, [P, P, P, P]),
        "moe_layer_forward": (ST, [P, I32, P, I32, P, P, P, P]),
        "moe_stack_forward": (ST, [P, I32, I32, P, P, P, P, P, P]),
        "moe_route": (ST, [P, I32, P, P, P, P]),
        "moe_experts": (ST, [P, I32, P, P, P, P, P]),
        "moe_layer_forward_scalar": (ST, [P, I32, P, P, P, P, P]),
        "moe_device_status": (ST, [P, P, ctypes.POINTER(I32)]),
        "moe_pool_set_timeout": (ST, [P, ctypes.c_uint64]),
        "moe_pool_set_prefetch": (ST, [P, I32]),
        "moe_pool_grid": (I32, [P]),
        "moe_last_error": (ctypes.c_char_p, []),
        "moe_pool_slot_of": (ST, [P, I32, I32, ctypes.POINTER(I32)]),
        "moe_pool_set_copy_hook": (ST, [P, COPY_HOOK, P]),
        "moe_layer_forward_static": (ST, [PS, P, ctypes.POINTER(LayerWeights), P, I32, P, P, P, P, P]),
        "moe_stack_forward_streamed": (ST, [P, I32, I32, P, P, P, P, P, P]),
        "moe_qpack_create": (ST, [ctypes.c_char_p, PS, I32, ctypes.POINTER(P)]),
        "moe_qpack_open": (ST, [ctypes.c_char_p, I32, I32, ctypes.POINTER(P)]),
        "moe_qpack_info": (ST, [P, PS, ctypes.POINTER(I32), ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(I32)]),
        "moe_qpack_write": (ST, [P, I32, I32, P]),
        "moe_qpack_read": (ST, [P, I32, I32, P]),
        "moe_qpack_close": (ST, [P]),
        "moe_stack_forward_qpack": (ST, [P, I32, I32, P, P, P, P, I32, P, P, P]),
        "moe_batched_workspace_bytes": (SZ, [PS, I32]),
        "moe_layer_forward_batched": (ST, [P, I32, P, I32, P, P, P, P, SZ, P]),
        "moe_pool_time_batched": (ST, [P, I32]),
        "moe_pool_batched_gemm_ms": (ST, [P, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(I32)]),
        "moe_gdn_step": (ST, [ctypes.POINTER(GdnShape), I32] + [P] * 10 + [ctypes.c_float, P, P, P]),
        "moe_gqa_workspace_bytes": (SZ, [ctypes.POINTER(GqaShape), I32, I32]),
        "moe_gqa_decode": (ST, [ctypes.POINTER(GqaShape), I32, I32] + [P] * 7 + [ctypes.c_float, P, SZ, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != OK:
        raise MoeError(status, load().moe_last_error().decode())


def _p(x) -> int | None:
    """Pointer of a torch tensor / numpy array / int (None stays NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(type(x))


def _s(stream) -> int | None:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def layer_forward_static(shape: Shape, experts, router, shared_blob, shared_gate, x, n_tokens, y,
                         topk_idx=None, topk_w=None, status=None, logit_bias=None, stream=None):
    """moe_layer_forward_static: one layer with the library's fixed scratch array (no device
    allocation by the library or the caller); experts = the fixed-stride blobs, expert e at
    experts + e * stride."""
    w = LayerWeights(_p(router), _p(shared_blob), _p(shared_gate), _p(logit_bias))
    _check(load().moe_layer_forward_static(ctypes.byref(shape), _p(experts), ctypes.byref(w), _p(x), n_tokens, _p(y),
                                           _p(topk_idx), _p(topk_w), _p(status), _s(stream)))


def gdn_step(shape: GdnShape, batch: int, state, q, k, v, z, a, b, A_log, dt_bias, norm_w, scale: float, y,
             o=None, stream=None):
    """moe_gdn_step: one Gated DeltaNet decode step of ``batch`` sequences; the state is updated in
    place (layouts in include/hybrid.h)."""
    _check(load().moe_gdn_step(ctypes.byref(shape), batch, _p(state), _p(q), _p(k), _p(v), _p(z), _p(a), _p(b),
                               _p(A_log), _p(dt_bias), _p(norm_w), float(scale), _p(o), _p(y), _s(stream)))


def gqa_workspace_bytes(shape: GqaShape, batch: int, max_pos: int) -> int:
    return int(load().moe_gqa_workspace_bytes(ctypes.byref(shape), batch, max_pos))


def gqa_decode(shape: GqaShape, batch: int, max_pos: int, k_cache, v_cache, pos, q, k, v, gate, scale: float,
               work, work_bytes: int, y, status, o=None, stream=None):
    """moe_gqa_decode: one gated GQA decode step of ``batch`` sequences; row pos[b] of each cache is
    written in place, pos itself is left for the caller to advance."""
    _check(load().moe_gqa_decode(ctypes.byref(shape), batch, max_pos, _p(k_cache), _p(v_cache), _p(pos), _p(q),
                                 _p(k), _p(v), _p(gate), float(scale), _p(work), work_bytes, _p(o), _p(y),
                                 _p(status), _s(stream)))


def batched_workspace_bytes(shape: Shape, n_tokens: int) -> int:
    return int(load().moe_batched_workspace_bytes(ctypes.byref(shape), n_tokens))


def make_shape(hidden, n_experts, top_k, inter, shared_inter, bits=4, group=64, flags=RENORM) -> Shape:
    return Shape(hidden, n_experts, top_k, inter, shared_inter, bits, group, flags)


def expert_bytes(shape: Shape, shared: bool = False) -> int:
    return int(load().moe_expert_bytes(ctypes.byref(shape), int(shared)))


def expert_stride(shape: Shape, shared: bool = False) -> int:
    return int(load().moe_expert_stride(ctypes.byref(shape), int(shared)))


def workspace_bytes(shape: Shape, n_layers: int) -> int:
    return int(load().moe_workspace_bytes(ctypes.byref(shape), n_layers))


def pack_expert(shape: Shape, t: dict, shared: bool = False, out: np.ndarray | None = None) -> np.ndarray:
    """moe_pack_expert: one blob (expert_stride bytes) from code/scale/bias arrays."""
    q = [np.ascontiguousarray(t[m + "_q"], dtype=np.uint8) for m in ("gate", "up", "down")]
    s = [np.ascontiguousarray(t[m + "_s"], dtype=np.uint16) for m in ("gate", "up", "down")]
    b = [np.ascontiguousarray(t[m + "_b"], dtype=np.uint16) for m in ("gate", "up", "down")]
    arr = [(ctypes.c_void_p * 3)(*[x.ctypes.data for x in v]) for v in (q, s, b)]
    if out is None:
        out = np.empty(expert_stride(shape, shared), dtype=np.uint8)
    _check(load().moe_pack_expert(ctypes.byref(shape), int(shared), ctypes.cast(arr[0], ctypes.c_void_p),
                                  ctypes.cast(arr[1], ctypes.c_void_p), ctypes.cast(arr[2], ctypes.c_void_p),
                                  out.ctypes.data))
    return out


class Qpack:
    """The on-disk expert container (moe_qpack_*): create() to write one, open() to read one."""

    def __init__(self, handle, lib):
        self.h, self.lib = handle, lib

    @classmethod
    def create(cls, path: str, shape: Shape, n_layers: int) -> "Qpack":
        lib, h = load(), ctypes.c_void_p()
        _check(lib.moe_qpack_create(path.encode(), ctypes.byref(shape), n_layers, ctypes.byref(h)))
        return cls(h, lib)

    @classmethod
    def open(cls, path: str, direct: bool = True, n_threads: int = 8) -> "Qpack":
        lib, h = load(), ctypes.c_void_p()
        _check(lib.moe_qpack_open(path.encode(), QPACK_DIRECT if direct else 0, n_threads, ctypes.byref(h)))
        return cls(h, lib)

    def info(self) -> tuple[Shape, int, int, bool]:
        sh, nl, st, d = Shape(), ctypes.c_int32(), ctypes.c_uint64(), ctypes.c_int32()
        _check(self.lib.moe_qpack_info(self.h, ctypes.byref(sh), ctypes.byref(nl), ctypes.byref(st), ctypes.byref(d)))
        return sh, nl.value, st.value, bool(d.value)

    def write(self, layer: int, expert: int, blob: np.ndarray):
        _check(self.lib.moe_qpack_write(self.h, layer, expert, np.ascontiguousarray(blob, dtype=np.uint8).ctypes.data))

    def read(self, layer: int, expert: int, dst):
        """dst: host buffer of stride bytes (4096-byte aligned for direct reads): numpy array or
        pointer."""
        _check(self.lib.moe_qpack_read(self.h, layer, expert, dst.ctypes.data if hasattr(dst, "ctypes") else _p(dst)))

    def close(self):
        if self.h:
            _check(self.lib.moe_qpack_close(self.h))
            self.h = None


class Pool:
    """A moe_pool over a caller-owned arena and workspace (device pointers, or workspace=None for
    a host-only pool that runs the slot policy alone)."""

    def __init__(self, shape: Shape, n_layers: int, n_slots: int, arena=None, arena_bytes: int = 0,
                 workspace=None, workspace_bytes_: int = 0):
        self.shape = shape
        self.lib = load()
        h = ctypes.c_void_p()
        _check(self.lib.moe_pool_create(ctypes.byref(shape), n_layers, n_slots, _p(arena), arena_bytes,
                                        _p(workspace), workspace_bytes_, ctypes.byref(h)))
        self.h = h
        self._keep = []

    def close(self):
        if self.h:
            self.lib.moe_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def slot_ptr(self, slot: int) -> int:
        return self.lib.moe_pool_slot_ptr(self.h, slot) or 0

    def grid(self) -> int:
        return int(self.lib.moe_pool_grid(self.h))

    def set_timeout(self, ns: int):
        _check(self.lib.moe_pool_set_timeout(self.h, ns))

    def set_prefetch(self, n: int):
        """Speculative copies of the next layer's n best predicted experts in stack_forward_streamed
        (0: off)."""
        _check(self.lib.moe_pool_set_prefetch(self.h, int(n)))

    def set_layer(self, layer: int, router, shared_blob, shared_gate, logit_bias=None):
        w = LayerWeights(_p(router), _p(shared_blob), _p(shared_gate), _p(logit_bias))
        _check(self.lib.moe_pool_set_layer(self.h, layer, ctypes.byref(w)))

    def place(self, layer: int, expert: int, slot: int):
        _check(self.lib.moe_pool_place(self.h, layer, expert, slot))

    def sync(self, stream=None):
        _check(self.lib.moe_pool_sync(self.h, _s(stream)))

    def lookup(self, layer: int, experts) -> np.ndarray:
        e = np.ascontiguousarray(experts, dtype=np.int32)
        out = np.empty(e.shape[0], dtype=np.int32)
        _check(self.lib.moe_pool_lookup(self.h, layer, e.ctypes.data, e.shape[0], out.ctypes.data))
        return out

    def load_slot(self, layer: int, expert: int, h_blob, copy_stream=None) -> int:
        s = ctypes.c_int32()
        _check(self.lib.moe_pool_load_slot(self.h, layer, expert, _p(h_blob), _s(copy_stream), ctypes.byref(s)))
        return s.value

    def wait_loads(self, compute_stream=None):
        _check(self.lib.moe_pool_wait_loads(self.h, _s(compute_stream)))

    def release(self, compute_stream=None):
        _check(self.lib.moe_pool_release(self.h, _s(compute_stream)))

    def stats(self):
        v = [ctypes.c_int64() for _ in range(3)]
        _check(self.lib.moe_pool_stats(self.h, *[ctypes.addressof(x) for x in v]))
        return tuple(x.value for x in v)

    def slot_of(self, layer: int, expert: int) -> int:
        s = ctypes.c_int32()
        _check(self.lib.moe_pool_slot_of(self.h, layer, expert, ctypes.byref(s)))
        return s.value

    def set_copy_hook(self, fn):
        """fn(slot, h_blob_ptr, nbytes) -> int (0 = success); None restores the device copy."""
        if fn is None:
            cb = ctypes.cast(None, COPY_HOOK)
        else:
            cb = COPY_HOOK(lambda user, slot, blob, n: int(fn(slot, blob, n)))
        self._keep.append(cb)
        _check(self.lib.moe_pool_set_copy_hook(self.h, cb, None))

    def layer_forward(self, layer, x, n_tokens, y, topk_idx=None, topk_w=None, stream=None):
        _check(self.lib.moe_layer_forward(self.h, layer, _p(x), n_tokens, _p(y), _p(topk_idx), _p(topk_w), _s(stream)))

    def stack_forward(self, layer0, n_layers, x, x_out, trace=None, topk_idx=None, topk_w=None, stream=None):
        _check(self.lib.moe_stack_forward(self.h, layer0, n_layers, _p(x), _p(x_out), _p(trace), _p(topk_idx),
                                          _p(topk_w), _s(stream)))

    def stack_forward_qpack(self, layer0, n_layers, x, x_out, qpack: "Qpack", staging, n_staging: int,
                            compute_stream=None, copy_stream=None, topk_idx: np.ndarray | None = None):
        """Bounded-mode stack with the misses read from an on-disk container through `staging`
        (pinned host buffer of n_staging blobs)."""
        _check(self.lib.moe_stack_forward_qpack(self.h, layer0, n_layers, _p(x), _p(x_out), qpack.h, _p(staging),
                                                n_staging, _s(compute_stream), _s(copy_stream),
                                                None if topk_idx is None else topk_idx.ctypes.data))

    def stack_forward_streamed(self, layer0, n_layers, x, x_out, h_blobs: np.ndarray, compute_stream=None,
                               copy_stream=None, topk_idx: np.ndarray | None = None):
        """Bounded-mode stack for one token; h_blobs: uint64 array [n_layers][E] of pinned host
        blob addresses. topk_idx (optional): int32 array [n_layers][k] filled with the selections."""
        hb = np.ascontiguousarray(h_blobs, dtype=np.uint64)
        _check(self.lib.moe_stack_forward_streamed(self.h, layer0, n_layers, _p(x), _p(x_out), hb.ctypes.data,
                                                   _s(compute_stream), _s(copy_stream),
                                                   None if topk_idx is None else topk_idx.ctypes.data))

    def layer_forward_batched(self, layer, x, n_tokens, y, work, topk_idx=None, topk_w=None, stream=None):
        """moe_layer_forward_batched: x bf16 [T][H] -> y fp32 [T][H]; work: device buffer of
        batched_workspace_bytes(shape, T) bytes."""
        _check(self.lib.moe_layer_forward_batched(self.h, layer, _p(x), n_tokens, _p(y), _p(topk_idx), _p(topk_w),
                                                  _p(work), work.numel() if hasattr(work, "numel") else 0, _s(stream)))

    def time_batched(self, n_calls: int):
        """Record CUDA events around the expert GEMMs of the next batched calls (ring of n)."""
        _check(self.lib.moe_pool_time_batched(self.h, n_calls))

    def batched_gemm_ms(self) -> tuple[float, int]:
        """(total ms, calls) of the recorded expert-GEMM intervals; waits for them, then clears."""
        ms, n = ctypes.c_float(0.0), ctypes.c_int32(0)
        _check(self.lib.moe_pool_batched_gemm_ms(self.h, ctypes.byref(ms), ctypes.byref(n)))
        return float(ms.value), int(n.value)

    def route(self, layer, x, topk_idx, topk_w, stream=None):
        _check(self.lib.moe_route(self.h, layer, _p(x), _p(topk_idx), _p(topk_w), _s(stream)))

    def experts(self, layer, x, topk_w, slots, y, stream=None):
        sl = np.ascontiguousarray(slots, dtype=np.int32)
        _check(self.lib.moe_experts(self.h, layer, _p(x), _p(topk_w), sl.ctypes.data, _p(y), _s(stream)))

    def layer_forward_scalar(self, layer, x, y, topk_idx=None, topk_w=None, stream=None):
        _check(self.lib.moe_layer_forward_scalar(self.h, layer, _p(x), _p(y), _p(topk_idx), _p(topk_w), _s(stream)))

    def device_status(self, stream=None) -> int:
        v = ctypes.c_int32()
        _check(self.lib.moe_device_status(self.h, _s(stream), ctypes.byref(v)))
        return v.value
