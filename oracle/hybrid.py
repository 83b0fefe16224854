"""CPU oracle of the Gated DeltaNet decode step and of gated GQA decode attention (double precision).

TEST INFRASTRUCTURE, like the rest of this package: the arithmetic lives in ``hybrid_oracle.c``
(plain C, built by :func:`build`); this module only converts numpy arrays and loops over the
sequences of a batch. The C file names the page passages and the published definitions it follows.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import compile_c

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hybrid_oracle.c")
_DEFAULT_LIB = os.path.join(_HERE, "libhybrid_oracle.so")
# a test may point the wrapper at a deliberately broken build (mutation tests)
_LIB_PATH = os.environ.get("MOE_HYBRID_ORACLE_LIB", _DEFAULT_LIB)
_lib = None

L2_EPS = 1e-6   # inside the square root of the q/k L2 normalisation
RMS_EPS = 1e-6  # inside the square root of the head-output RMS norm


def build(force: bool = False) -> str:
    if _LIB_PATH != _DEFAULT_LIB:
        return _LIB_PATH
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_c(_SRC, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.orc_gdn_gates.restype = None
        lib.orc_gdn_gates.argtypes = [I, P, P, P, P, P, P]
        lib.orc_gdn_step.restype = None
        lib.orc_gdn_step.argtypes = [I, I, I, I] + [P] * 10 + [D, D, D, P, P]
        lib.orc_gqa_step.restype = None
        lib.orc_gqa_step.argtypes = [I, I, I, I, I, P, P, P, P, P, P, D, P, P]
        _lib = lib
    return _lib


def _d(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def gdn_gates(a, b, A_log, dt_bias):
    """(alpha, beta) per value head."""
    a, b, A_log, dt_bias = _d(a), _d(b), _d(A_log), _d(dt_bias)
    n = a.size
    alpha, beta = np.empty(n), np.empty(n)
    _load().orc_gdn_gates(n, _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(alpha), _ptr(beta))
    return alpha, beta


def gdn_step(S, q, k, v, z, a, b, A_log, dt_bias, norm_w, scale, eps_l2=L2_EPS, eps=RMS_EPS):
    """One Gated DeltaNet decode step of one sequence.

    S [Hv, dv, dk]; q, k [Hk, dk]; v, z [Hv, dv]; a, b, A_log, dt_bias [Hv]; norm_w [dv].
    Returns (S_new, o, y): the new state and the head outputs before and after the gated norm.
    """
    S = _d(S).copy()
    Hv, dv, dk = S.shape
    q, k = _d(q).reshape(-1, dk), _d(k).reshape(-1, dk)
    Hk = q.shape[0]
    v, z = _d(v).reshape(Hv, dv), _d(z).reshape(Hv, dv)
    a, b, A_log, dt_bias, norm_w = _d(a), _d(b), _d(A_log), _d(dt_bias), _d(norm_w)
    o, y = np.empty((Hv, dv)), np.empty((Hv, dv))
    _load().orc_gdn_step(Hk, Hv, dk, dv, _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(a), _ptr(b),
                         _ptr(A_log), _ptr(dt_bias), _ptr(norm_w), float(scale), float(eps_l2), float(eps),
                         _ptr(o), _ptr(y))
    return S, o, y


def gqa_step(Kc, Vc, pos, q, k, v, gate, scale):
    """One gated GQA decode step of one sequence.

    Kc, Vc [Hkv, Lmax, D] (copied, then the new k, v written at ``pos``); q, gate [Hq, D];
    k, v [Hkv, D]. Returns (Kc_new, Vc_new, o, y) with o, y [Hq, D].
    """
    Kc, Vc = _d(Kc).copy(), _d(Vc).copy()
    Hkv, Lmax, D = Kc.shape
    assert 0 <= pos < Lmax
    q, gate = _d(q).reshape(-1, D), _d(gate).reshape(-1, D)
    Hq = q.shape[0]
    k, v = _d(k).reshape(Hkv, D), _d(v).reshape(Hkv, D)
    o, y = np.empty((Hq, D)), np.empty((Hq, D))
    _load().orc_gqa_step(Hq, Hkv, D, Lmax, int(pos), _ptr(Kc), _ptr(Vc), _ptr(q), _ptr(k), _ptr(v), _ptr(gate),
                         float(scale), _ptr(o), _ptr(y))
    return Kc, Vc, o, y
