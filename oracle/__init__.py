"""ctypes front end of the plain C oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only users.  The CUDA library never
imports, links or runs anything in this folder, and this folder never imports
the CUDA library.  Inputs come from the seeded generators as numpy arrays.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with plain IEEE double semantics.

    ``-ffp-contract=off`` keeps gcc from fusing a*b+c into one rounding on
    targets where it would (e.g. aarch64), so the oracle rounds identically on
    every host.
    """
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "oracle.h"))):
        return _SO
    tmp = _SO + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


class Cfg(C.Structure):
    _fields_ = [("hidden", C.c_int64), ("expert_hidden", C.c_int64), ("n_experts", C.c_int32),
                ("top_k", C.c_int32), ("n_shared", C.c_int32), ("swiglu_alpha", C.c_double),
                ("swiglu_limit", C.c_double), ("weight_scale", C.c_double), ("rms_eps", C.c_double),
                ("act_fp4", C.c_int32)]


class Expert(C.Structure):
    _fields_ = [("codes", C.c_void_p * 3), ("scales", C.c_void_p * 3), ("bias", C.c_void_p * 3)]


class Weights(C.Structure):
    _fields_ = [("gamma", C.c_void_p), ("router_w", C.c_void_p), ("router_b", C.c_void_p),
                ("codes", C.c_void_p * 3), ("scales", C.c_void_p * 3), ("bias", C.c_void_p * 3),
                ("sh_codes", C.c_void_p * 3), ("sh_scales", C.c_void_p * 3),
                ("sh_bias", C.c_void_p * 3)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_SO)
        P = C.c_void_p
        L.oracle_e2m1_value.restype = C.c_double
        L.oracle_e2m1_value.argtypes = [C.c_int]
        L.oracle_e8m0_value.restype = C.c_double
        L.oracle_e8m0_value.argtypes = [C.c_int]
        L.oracle_mxfp4_dequant.argtypes = [P, P, C.c_int64, C.c_int64, P]
        L.oracle_bf16_rne.restype = C.c_uint16
        L.oracle_bf16_rne.argtypes = [C.c_double]
        L.oracle_bf16_to_double.restype = C.c_double
        L.oracle_bf16_to_double.argtypes = [C.c_uint16]
        L.oracle_rmsnorm.argtypes = [P, C.c_int64, P, C.c_double, P, P]
        L.oracle_router_logits.argtypes = [P, P, P, C.c_int32, C.c_int64, P]
        L.oracle_topk.argtypes = [P, C.c_int32, C.c_int32, P, P]
        L.oracle_route_weights.argtypes = [P, C.c_int32, C.c_double, P]
        L.oracle_swiglu.restype = C.c_double
        L.oracle_swiglu.argtypes = [C.c_double, C.c_double, C.c_double, C.c_double]
        L.oracle_expert_ffn.argtypes = [C.POINTER(Expert), C.c_int64, C.c_int64, P, C.c_double,
                                        C.c_double, P, P, P]
        L.oracle_permutation.argtypes = [P, C.c_int64, C.c_int32, C.c_int32, P, P, P, P, P]
        L.oracle_mx_fp4_quantize.restype = C.c_int
        L.oracle_mx_fp4_quantize.argtypes = [P, C.c_int64, C.c_int64, P, P]
        L.oracle_moe_forward.restype = C.c_int
        L.oracle_moe_forward.argtypes = [C.POINTER(Cfg), C.POINTER(Weights), P, C.c_int64, P, P,
                                         P, P, P, C.c_int]
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


# ---------------------------------------------------------------- elementwise
def e2m1_value(nibble: int) -> float:
    return lib().oracle_e2m1_value(nibble)


def e8m0_value(e: int) -> float:
    return lib().oracle_e8m0_value(e)


def bf16_rne(v: float) -> int:
    return int(lib().oracle_bf16_rne(float(v)))


def bf16_to_double(b: int) -> float:
    return lib().oracle_bf16_to_double(int(b))


def swiglu(g: float, u: float, alpha: float, limit: float) -> float:
    return lib().oracle_swiglu(float(g), float(u), float(alpha), float(limit))


# -------------------------------------------------------------------- arrays
def mxfp4_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """[rows][cols/2] codes + [rows][cols/32] scales -> float64 [rows][cols]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, half = codes.shape
    cols = 2 * half
    assert scales.shape == (rows, cols // 32)
    out = np.empty((rows, cols), np.float64)
    lib().oracle_mxfp4_dequant(_p(codes), _p(scales), rows, cols, _p(out))
    return out


def mx_fp4_quantize(x: np.ndarray):
    """float32 [rows][cols] (cols % 32 == 0) -> (codes uint8 [rows][cols/2],
    E8M0 scales uint8 [rows][cols/32]): the FP4 activation encoding."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 32), np.uint8)
    if lib().oracle_mx_fp4_quantize(_p(x), rows, cols, _p(codes), _p(scales)) != 0:
        raise ValueError("oracle_mx_fp4_quantize: bad arguments")
    return codes, scales


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float):
    """x bf16 bits [H] -> (x_hat bf16 bits [H], unrounded float64 [H])."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    H = x.shape[0]
    xh = np.empty(H, np.uint16)
    pre = np.empty(H, np.float64)
    lib().oracle_rmsnorm(_p(x), H, _p(gamma), float(eps), _p(xh), _p(pre))
    return xh, pre


def router_logits(xhat: np.ndarray, router_w: np.ndarray, router_b: np.ndarray) -> np.ndarray:
    xhat = np.ascontiguousarray(xhat, np.uint16)
    router_w = np.ascontiguousarray(router_w, np.uint16)
    router_b = np.ascontiguousarray(router_b, np.float32)
    E, H = router_w.shape
    out = np.empty(E, np.float64)
    lib().oracle_router_logits(_p(xhat), _p(router_w), _p(router_b), E, H, _p(out))
    return out


def topk(logits: np.ndarray, k: int):
    logits = np.ascontiguousarray(logits, np.float64)
    ids = np.empty(k, np.int32)
    vals = np.empty(k, np.float64)
    lib().oracle_topk(_p(logits), logits.shape[0], k, _p(ids), _p(vals))
    return ids, vals


def route_weights(vals: np.ndarray, scale: float) -> np.ndarray:
    vals = np.ascontiguousarray(vals, np.float64)
    w = np.empty_like(vals)
    lib().oracle_route_weights(_p(vals), vals.shape[0], float(scale), _p(w))
    return w


def expert_ffn(codes: dict, scales: dict, bias: dict, e: int, xhat: np.ndarray, alpha: float,
               limit: float):
    """Expert ``e`` of the stacked canonical tensors on one token.

    Returns (y float64 [H], h bf16 bits [F], g/u float64 [2F])."""
    from_mats = ("gate", "up", "down")
    ex = Expert()
    keep = []
    for i, m in enumerate(from_mats):
        c = np.ascontiguousarray(codes[m][e])
        s = np.ascontiguousarray(scales[m][e])
        b = np.ascontiguousarray(bias[m][e], dtype=np.float32)
        keep += [c, s, b]
        ex.codes[i], ex.scales[i], ex.bias[i] = _p(c), _p(s), _p(b)
    F, H = codes["gate"].shape[1], codes["gate"].shape[2] * 2
    xhat = np.ascontiguousarray(xhat, np.uint16)
    y = np.empty(H, np.float64)
    h = np.empty(F, np.uint16)
    gu = np.empty(2 * F, np.float64)
    lib().oracle_expert_ffn(C.byref(ex), H, F, _p(xhat), float(alpha), float(limit), _p(y), _p(h),
                            _p(gu))
    return y, h, gu


def permutation(ids: np.ndarray, n_experts: int):
    ids = np.ascontiguousarray(ids, np.int32)
    T, K = ids.shape
    counts = np.empty(n_experts, np.int32)
    offsets = np.empty(n_experts + 1, np.int32)
    pt = np.empty(T * K, np.int32)
    ps = np.empty(T * K, np.int32)
    loc = np.empty(T * K, np.int32)
    lib().oracle_permutation(_p(ids), T, K, n_experts, _p(counts), _p(offsets), _p(pt), _p(ps),
                             _p(loc))
    return dict(counts=counts, offsets=offsets, perm_token=pt, perm_slot=ps, loc=loc)


def _cfg(shape, act_fp4: bool = False) -> Cfg:
    return Cfg(shape.hidden, shape.expert_hidden, shape.n_experts, shape.top_k, shape.n_shared,
               shape.swiglu_alpha, shape.swiglu_limit, shape.weight_scale, shape.rms_eps,
               1 if act_fp4 else 0)


def moe_forward(blk: dict, x: np.ndarray, nthreads: int = 1, shape=None, act_fp4: bool = False):
    """Whole block on tokens ``x`` (bf16 bits [T][H]) with the weights of ``blk``.
    act_fp4: every expert's inputs (x_hat, and h after its bf16 rounding) pass
    through the FP4 activation encoding and back before their projections.

    Returns dict(out float64 [T][H], ids int32 [T][K], route_w float64 [T][K],
    xhat uint16 [T][H], logits float64 [T][E])."""
    shape = shape or blk["shape"]
    cfg = _cfg(shape, act_fp4)
    w = Weights()
    keep = []

    def P(a, dt):
        a = np.ascontiguousarray(a, dtype=dt)
        keep.append(a)
        return _p(a)

    w.gamma = P(blk["gamma"], np.float32)
    w.router_w = P(blk["router_w"], np.uint16)
    w.router_b = P(blk["router_b"], np.float32)
    for i, m in enumerate(("gate", "up", "down")):
        w.codes[i] = P(blk["codes"][m], np.uint8)
        w.scales[i] = P(blk["scales"][m], np.uint8)
        w.bias[i] = P(blk["bias"][m], np.float32)
        if shape.n_shared:
            sh = blk["shared"]
            w.sh_codes[i] = P(sh["codes"][m], np.uint8)
            w.sh_scales[i] = P(sh["scales"][m], np.uint8)
            w.sh_bias[i] = P(sh["bias"][m], np.float32)
    x = np.ascontiguousarray(x, np.uint16)
    T, H = x.shape
    assert H == shape.hidden
    K, E = shape.top_k, shape.n_experts
    out = np.empty((T, H), np.float64)
    ids = np.empty((T, K), np.int32)
    rw = np.empty((T, K), np.float64)
    xh = np.empty((T, H), np.uint16)
    lg = np.empty((T, E), np.float64)
    rc = lib().oracle_moe_forward(C.byref(cfg), C.byref(w), _p(x), T, _p(out), _p(ids), _p(rw),
                                  _p(xh), _p(lg), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_moe_forward rejected its arguments")
    return dict(out=out, ids=ids, route_w=rw, xhat=xh, logits=lg)

