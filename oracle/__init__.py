"""CPU oracle of the routed-expert MoE FFN layer (double precision).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The product library (``int4_routed_expert_05_b300``) never
imports it, and the two share no code: the arithmetic lives in ``moe_oracle.c`` (plain C, built
with gcc by :func:`build`), this module only marshals numpy arrays through ctypes and strings the
per-layer calls into a stack. Each function names the page passage it follows in moe_oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_DEFAULT_LIB = os.path.join(_HERE, "liboracle.so")
# a test may point the wrapper at a deliberately broken build of the oracle (mutation tests)
_LIB_PATH = os.environ.get("MOE_ORACLE_LIB", _DEFAULT_LIB)
_lib = None

RMS_EPS = 1e-6


def compile_c(src: str, out: str) -> str:
    """gcc -O2, no fast-math, no floating-point contraction; OpenMP for the optional threaded row
    loops (serial unless set_threads asks for more)."""
    tmp = f"{out}.tmp{os.getpid()}"  # written aside and renamed: concurrent builders never see half a file
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC",
           "-o", tmp, src, "-lm"]
    try:
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.remove(tmp)
    return out


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so next to it."""
    if _LIB_PATH != _DEFAULT_LIB:
        return _LIB_PATH
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_c(_SRC, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.orc_bf16.restype = ctypes.c_double
    lib.orc_bf16.argtypes = [ctypes.c_uint16]
    lib.orc_round_bf16.restype = ctypes.c_uint16
    lib.orc_round_bf16.argtypes = [ctypes.c_double]
    lib.orc_blob_bytes.restype = ctypes.c_size_t
    lib.orc_blob_bytes.argtypes = [I, I, I, I]
    lib.orc_blob_stride.restype = ctypes.c_size_t
    lib.orc_blob_stride.argtypes = [I, I, I, I]
    lib.orc_blob_pack.restype = None
    lib.orc_blob_pack.argtypes = [I, I, I, I, P, P, P, P]
    lib.orc_blob_unpack.restype = None
    lib.orc_blob_unpack.argtypes = [I, I, I, I, P, P, P, P]
    lib.orc_dequant.restype = None
    lib.orc_dequant.argtypes = [P, I, I, I, I, I, P]
    lib.orc_router_logits.restype = None
    lib.orc_router_logits.argtypes = [P, P, P, I, I, P, P]
    lib.orc_topk.restype = None
    lib.orc_topk.argtypes = [P, I, I, I, P, P]
    lib.orc_expert_ffn.restype = None
    lib.orc_expert_ffn.argtypes = [P, I, I, I, I, P, P, P]
    lib.orc_shared_gate.restype = ctypes.c_double
    lib.orc_shared_gate.argtypes = [P, P, I]
    lib.orc_moe_layer.restype = None
    lib.orc_moe_layer.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.orc_moe_layer_sel.restype = None
    lib.orc_moe_layer_sel.argtypes = [I, I, I, I, I, I, I, I, P, P, P, P, P, P, I, P, P, P, P, P, P]
    lib.orc_route_weights.restype = None
    lib.orc_route_weights.argtypes = [P, I, I, I, P, P]
    lib.orc_set_threads.restype = None
    lib.orc_set_threads.argtypes = [I]
    lib.orc_get_threads.restype = I
    lib.orc_get_threads.argtypes = []
    lib.orc_rmsnorm_bf16.restype = None
    lib.orc_rmsnorm_bf16.argtypes = [P, I, ctypes.c_double, P]
    _lib = lib
    return lib


def set_threads(n: int) -> None:
    """Threads of the oracle's row loops (1: serial, the default). Results do not depend on it."""
    _load().orc_set_threads(int(n))


def get_threads() -> int:
    return int(_load().orc_get_threads())


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _inter(shape, shared: bool) -> int:
    return shape.shared_inter if shared else shape.inter


# ---------------------------------------------------------------------------------------------
# values
# ---------------------------------------------------------------------------------------------

def bf16(bits) -> np.ndarray:
    lib = _load()
    return np.array([lib.orc_bf16(int(b)) for b in np.ravel(bits)]).reshape(np.shape(bits))


def round_bf16(values) -> np.ndarray:
    lib = _load()
    v = np.ravel(np.asarray(values, dtype=np.float64))
    return np.array([lib.orc_round_bf16(float(x)) for x in v], dtype=np.uint16).reshape(np.shape(values))


# ---------------------------------------------------------------------------------------------
# blob format
# ---------------------------------------------------------------------------------------------

def blob_bytes(shape, shared: bool = False) -> int:
    return int(_load().orc_blob_bytes(shape.hidden, _inter(shape, shared), shape.bits, shape.group))


def blob_stride(shape, shared: bool = False) -> int:
    return int(_load().orc_blob_stride(shape.hidden, _inter(shape, shared), shape.bits, shape.group))


def pack(shape, t: dict, shared: bool = False) -> np.ndarray:
    """The oracle's own writer of one blob (``stride`` bytes, zero padded) from code/scale arrays."""
    lib = _load()
    q = [_c(t[m + "_q"], np.uint8) for m in ("gate", "up", "down")]
    s = [_c(t[m + "_s"], np.uint16) for m in ("gate", "up", "down")]
    b = [_c(t[m + "_b"], np.uint16) for m in ("gate", "up", "down")]
    qa = (ctypes.c_void_p * 3)(*[x.ctypes.data for x in q])
    sa = (ctypes.c_void_p * 3)(*[x.ctypes.data for x in s])
    ba = (ctypes.c_void_p * 3)(*[x.ctypes.data for x in b])
    out = np.zeros(blob_stride(shape, shared), dtype=np.uint8)
    lib.orc_blob_pack(shape.hidden, _inter(shape, shared), shape.bits, shape.group,
                      ctypes.cast(qa, ctypes.c_void_p), ctypes.cast(sa, ctypes.c_void_p),
                      ctypes.cast(ba, ctypes.c_void_p), _ptr(out))
    return out


def unpack(shape, blob: np.ndarray, shared: bool = False) -> dict:
    """The oracle's own reader: codes and scale/bias bit patterns of one blob."""
    lib = _load()
    H, I, g = shape.hidden, _inter(shape, shared), shape.group
    dims = [(I, H), (I, H), (H, I)]
    q = [np.zeros(d, dtype=np.uint8) for d in dims]
    s = [np.zeros((d[0], d[1] // g), dtype=np.uint16) for d in dims]
    b = [np.zeros((d[0], d[1] // g), dtype=np.uint16) for d in dims]
    qa = (ctypes.c_void_p * 3)(*[x.ctypes.data for x in q])
    sa = (ctypes.c_void_p * 3)(*[x.ctypes.data for x in s])
    ba = (ctypes.c_void_p * 3)(*[x.ctypes.data for x in b])
    blob = _c(blob, np.uint8)
    lib.orc_blob_unpack(H, I, shape.bits, g, _ptr(blob), ctypes.cast(qa, ctypes.c_void_p),
                        ctypes.cast(sa, ctypes.c_void_p), ctypes.cast(ba, ctypes.c_void_p))
    out = {}
    for i, m in enumerate(("gate", "up", "down")):
        out[m + "_q"], out[m + "_s"], out[m + "_b"] = q[i], s[i], b[i]
    return out


def dequant(shape, blob: np.ndarray, which: int, shared: bool = False) -> np.ndarray:
    """Matrix ``which`` (0 gate, 1 up, 2 down) of a blob as float64 (w = s*q + b)."""
    H, I = shape.hidden, _inter(shape, shared)
    rows, cols = (H, I) if which == 2 else (I, H)
    W = np.zeros((rows, cols), dtype=np.float64)
    blob = _c(blob, np.uint8)
    _load().orc_dequant(_ptr(blob), H, I, shape.bits, shape.group, which, _ptr(W))
    return W


# ---------------------------------------------------------------------------------------------
# layer pieces
# ---------------------------------------------------------------------------------------------

def router_logits(Wr_bits, u_bits, bias=None):
    Wr = _c(Wr_bits, np.uint16)
    u = _c(u_bits, np.uint16)
    E, H = Wr.shape
    bias_a = None if bias is None else _c(bias, np.float32)
    lg = np.zeros(E)
    bd = np.zeros(E)
    _load().orc_router_logits(_ptr(Wr), _ptr(u), _ptr(bias_a), E, H, _ptr(lg), _ptr(bd))
    return lg, bd


def topk(logits, k: int, renorm: bool = True):
    lg = _c(logits, np.float64)
    idx = np.zeros(k, dtype=np.int32)
    w = np.zeros(k)
    _load().orc_topk(_ptr(lg), lg.shape[0], k, int(renorm), _ptr(idx), _ptr(w))
    return idx, w


def expert_ffn(shape, blob, u_bits, shared: bool = False):
    H, I = shape.hidden, _inter(shape, shared)
    y = np.zeros(H)
    h = np.zeros(I)
    blob = _c(blob, np.uint8)
    u = _c(u_bits, np.uint16)
    _load().orc_expert_ffn(_ptr(blob), H, I, shape.bits, shape.group, _ptr(u), _ptr(y), _ptr(h))
    return y, h


def shared_gate(w_sg_bits, u_bits) -> float:
    w = _c(w_sg_bits, np.uint16)
    u = _c(u_bits, np.uint16)
    return float(_load().orc_shared_gate(_ptr(w), _ptr(u), w.shape[0]))


def moe_layer(shape, u_bits, Wr_bits, w_sg_bits, expert_blobs, shared_blob, bias=None, force_idx=None) -> dict:
    """One layer for one token (see orc_moe_layer). ``expert_blobs``: sequence of E blob arrays.
    With ``force_idx`` (k indices in rank order) the layer is evaluated for that selection instead
    of the top-k's (orc_moe_layer_sel): the routing weights and y of the given experts."""
    E, k = shape.n_experts, shape.top_k
    u = _c(u_bits, np.uint16)
    Wr = _c(Wr_bits, np.uint16)
    w_sg = _c(w_sg_bits, np.uint16)
    blobs = [_c(b, np.uint8) for b in expert_blobs]
    assert len(blobs) == E
    arr = (ctypes.c_void_p * E)(*[b.ctypes.data for b in blobs])
    sb = _c(shared_blob, np.uint8)
    bias_a = None if bias is None else _c(bias, np.float32)
    if force_idx is None:
        idx = np.zeros(k, dtype=np.int32)
    else:
        idx = _c(force_idx, np.int32).copy()
        assert idx.shape == (k,) and len(set(idx.tolist())) == k and idx.min() >= 0 and idx.max() < E
    w = np.zeros(k)
    y = np.zeros(shape.hidden)
    lg = np.zeros(E)
    bd = np.zeros(E)
    gam = np.zeros(1)
    _load().orc_moe_layer_sel(shape.hidden, E, k, shape.inter, shape.shared_inter, shape.bits, shape.group,
                              int(shape.renorm), _ptr(u), _ptr(Wr), _ptr(bias_a), _ptr(w_sg),
                              ctypes.cast(arr, ctypes.c_void_p), _ptr(sb), int(force_idx is not None), _ptr(idx),
                              _ptr(w), _ptr(y), _ptr(lg), _ptr(bd), _ptr(gam))
    return {"idx": idx, "w": w, "y": y, "logits": lg, "bound": bd, "gamma": float(gam[0])}


def route_weights(logits, idx, renorm: bool = True):
    """Routing weights of a given selection (see orc_route_weights)."""
    lg = _c(logits, np.float64)
    ix = _c(idx, np.int32)
    w = np.zeros(ix.shape[0])
    _load().orc_route_weights(_ptr(lg), lg.shape[0], ix.shape[0], int(renorm), _ptr(ix), _ptr(w))
    return w


def rmsnorm_bf16(x, eps: float = RMS_EPS) -> np.ndarray:
    xa = _c(x, np.float64)
    u = np.zeros(xa.shape[0], dtype=np.uint16)
    _load().orc_rmsnorm_bf16(_ptr(xa), xa.shape[0], eps, _ptr(u))
    return u


def selection_margin(logits, bound, idx) -> float:
    """How far the k-th chosen logit clears the best unchosen one, after subtracting both
    logits' binary32 error bounds and half an ulp of rounding each. Positive means every binary32
    evaluation of these logits selects exactly ``idx``."""
    lg = np.asarray(logits, dtype=np.float64)
    bd = np.asarray(bound, dtype=np.float64)
    chosen = np.zeros(lg.shape[0], dtype=bool)
    chosen[np.asarray(idx)] = True
    if chosen.all():
        return np.inf
    lo = np.argmin(np.where(chosen, lg - bd, np.inf))
    hi = np.argmax(np.where(chosen, -np.inf, lg + bd))
    slack = np.spacing(np.float32(abs(lg[lo]))) + np.spacing(np.float32(abs(lg[hi])))
    return float((lg[lo] - bd[lo]) - (lg[hi] + bd[hi]) - slack)


def stack(shape, layers, x0, record: bool = False):
    """A residual stack, reading R9: x <- x + MoE_l(bf16(rmsnorm(x))) for each layer in order.

    ``layers``: sequence of dicts with keys Wr, w_sg, blobs (sequence of E blobs), shared,
    and optionally bias. Returns the final residual (float64) and, with ``record``, the per-layer
    results (input x, u, idx, w, y, logits, bound).
    """
    x = np.asarray(x0, dtype=np.float64).copy()
    trace = []
    for L in layers:
        u = rmsnorm_bf16(x)
        r = moe_layer(shape, u, L["Wr"], L["w_sg"], L["blobs"], L["shared"], L.get("bias"))
        if record:
            r = dict(r, x_in=x.copy(), u=u)
            trace.append(r)
        x = x + r["y"]
    return (x, trace) if record else x
