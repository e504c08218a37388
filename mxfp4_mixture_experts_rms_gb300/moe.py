"""Thin ctypes binding of ``include/moe.h`` (argument marshalling only).

Every step of the block runs in the CUDA kernels of ``lib/libmoe.so``; this
module only passes device pointers and sizes.  PyTorch provides device memory
and streams.  There is no fallback: if the library is missing or fails to
load, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

MOE_OK, MOE_EINVAL, MOE_ESHAPE, MOE_ENOTREADY, MOE_ECUDA, MOE_ENOMEM, MOE_EDEVICE = 0, -1, -2, -3, -4, -5, -6
_STATUS_NAMES = {0: "MOE_OK", -1: "MOE_EINVAL", -2: "MOE_ESHAPE", -3: "MOE_ENOTREADY", -4: "MOE_ECUDA",
                 -5: "MOE_ENOMEM", -6: "MOE_EDEVICE"}

_lib = None

EXPORTS = ["moe_plan_create", "moe_plan_destroy", "moe_plan_set_i", "moe_plan_set_f", "moe_plan_path_for",
           "moe_workspace_bytes",
           "moe_set_workspace", "moe_load_weights", "moe_forward", "moe_forward_ex", "moe_get_expert_counts",
           "moe_get_permutation", "moe_debug_dequant", "moe_profile_read", "moe_get_device_status",
           "moe_get_cache_state",
           "moe_forward_noalloc", "moe_cast_f32_to_bf16", "moe_mx_quantize_fp4", "moe_locality_create",
           "moe_locality_record", "moe_locality_attach", "moe_locality_read", "moe_locality_reset",
           "moe_locality_destroy", "moe_attn_create", "moe_attn_set_i", "moe_attn_set_f", "moe_attn_workspace_bytes",
           "moe_attn_set_workspace", "moe_attn_set_cache", "moe_attn_load_weights", "moe_attn_decode", "moe_attn_prefill",
           "moe_attn_destroy", "moe_attn_get_device_status", "moe_last_error"]


class LocalityStats(C.Structure):
    _fields_ = [("hist", C.c_void_p), ("weight_hist", C.c_void_p), ("layer_records", C.c_void_p),
                ("adjacent_pairs", C.c_void_p), ("overlap_sum", C.c_void_p), ("jaccard_sum", C.c_void_p),
                ("cache_hits", C.c_void_p), ("cache_weight_hits", C.c_void_p), ("caps", C.c_void_p),
                ("n_caps", C.c_int)]


class AttnWeights(C.Structure):
    _fields_ = [("gamma", C.c_void_p), ("wq", C.c_void_p), ("wk", C.c_void_p), ("wv", C.c_void_p),
                ("wo", C.c_void_p), ("bq", C.c_void_p), ("bk", C.c_void_p), ("bv", C.c_void_p),
                ("bo", C.c_void_p), ("sinks", C.c_void_p)]


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class Mat(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("bias", C.c_void_p)]


class Weights(C.Structure):
    _fields_ = [("gamma", C.c_void_p), ("router_w", C.c_void_p), ("router_b", C.c_void_p),
                ("gate", Mat), ("up", Mat), ("down", Mat),
                ("sh_gate", Mat), ("sh_up", Mat), ("sh_down", Mat)]


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load ``libmoe.so`` (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise MoeError(MOE_ENOTREADY, f"CUDA library not built: {_build.LIB}")
    L = C.CDLL(_build.LIB)
    P, I, LL, D, SZ = C.c_void_p, C.c_int, C.c_longlong, C.c_double, C.c_size_t
    L.moe_plan_create.restype = P
    L.moe_plan_create.argtypes = [I, I, I, I, C.c_float, C.c_float, C.c_float]
    L.moe_plan_destroy.restype = None
    L.moe_plan_destroy.argtypes = [P]
    L.moe_plan_set_i.argtypes = [P, C.c_char_p, LL]
    L.moe_plan_set_f.argtypes = [P, C.c_char_p, D]
    L.moe_plan_path_for.argtypes = [P, I]
    L.moe_workspace_bytes.restype = SZ
    L.moe_workspace_bytes.argtypes = [P, I]
    L.moe_set_workspace.argtypes = [P, P, SZ]
    L.moe_load_weights.argtypes = [P, C.POINTER(Weights)]
    L.moe_forward.argtypes = [P, P, I, P, P, P]
    L.moe_forward_ex.argtypes = [P, P, I, P, P, P, P, P]
    L.moe_get_expert_counts.argtypes = [P, P, P]
    L.moe_get_permutation.argtypes = [P, P, P, P, P]
    L.moe_debug_dequant.argtypes = [P, I, I, P, P]
    L.moe_get_device_status.argtypes = [P, C.POINTER(I), P]
    L.moe_get_cache_state.argtypes = [P, P, P, P]
    L.moe_profile_read.argtypes = [P, C.POINTER(C.c_double), C.POINTER(I), I]
    L.moe_forward_noalloc.argtypes = [P, P, I, P, P, P]
    L.moe_cast_f32_to_bf16.argtypes = [P, P, SZ, P]
    L.moe_mx_quantize_fp4.argtypes = [P, SZ, SZ, P, P, P]
    L.moe_locality_create.restype = P
    L.moe_locality_create.argtypes = [I, I, I, P, I]
    L.moe_locality_record.argtypes = [P, I, P, P, I, LL, P]
    L.moe_locality_attach.argtypes = [P, P, I]
    L.moe_locality_read.argtypes = [P, C.POINTER(LocalityStats)]
    L.moe_locality_reset.argtypes = [P, P]
    L.moe_locality_destroy.restype = None
    L.moe_locality_destroy.argtypes = [P]
    L.moe_attn_create.restype = P
    L.moe_attn_create.argtypes = [I, I, I, I, I, I]
    L.moe_attn_set_i.argtypes = [P, C.c_char_p, LL]
    L.moe_attn_set_f.argtypes = [P, C.c_char_p, D]
    L.moe_attn_workspace_bytes.restype = SZ
    L.moe_attn_workspace_bytes.argtypes = [P]
    L.moe_attn_set_workspace.argtypes = [P, P, SZ]
    L.moe_attn_set_cache.argtypes = [P, P, P]
    L.moe_attn_load_weights.argtypes = [P, C.POINTER(AttnWeights)]
    L.moe_attn_decode.argtypes = [P, P, I, P, P, P]
    L.moe_attn_prefill.argtypes = [P, P, I, I, I, P, P]
    L.moe_attn_get_device_status.argtypes = [P, C.POINTER(I), P]
    L.moe_attn_destroy.restype = None
    L.moe_attn_destroy.argtypes = [P]
    L.moe_last_error.restype = C.c_char_p
    L.moe_last_error.argtypes = []
    for name in EXPORTS:
        if name not in ("moe_plan_create", "moe_plan_destroy", "moe_workspace_bytes", "moe_last_error",
                        "moe_locality_create", "moe_locality_destroy", "moe_attn_create", "moe_attn_destroy",
                        "moe_attn_workspace_bytes"):
            getattr(L, name).restype = C.c_int
    _lib = L
    return L


def _check(rc: int):
    if rc != MOE_OK:
        raise MoeError(rc, load().moe_last_error().decode())


def _ptr(t):
    """Device address of a tensor the library reads or writes as one dense
    row-major array; a strided view would be misread, so it is refused."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise MoeError(MOE_EINVAL, "tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream_ptr(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def cast_f32_to_bf16(src, dst, stream=None):
    """dst (int16/uint16 bits, device) = bf16_rne(src (float32, device)); enqueued on `stream`."""
    assert src.numel() == dst.numel()
    _check(load().moe_cast_f32_to_bf16(C.c_void_p(_ptr(src)), C.c_void_p(_ptr(dst)), int(src.numel()),
                                       _stream_ptr(stream)))


def mx_quantize_fp4(x, codes, scales, stream=None):
    """FP4 activation encoding of x (bf16 bits as int16/uint16, device, [rows][cols])
    into codes (uint8 [rows][cols/2]) and E8M0 scales (uint8 [rows][cols/32]),
    both device tensors; enqueued on `stream`."""
    rows, cols = x.shape
    assert codes.numel() == rows * cols // 2 and scales.numel() == rows * cols // 32
    _check(load().moe_mx_quantize_fp4(C.c_void_p(_ptr(x)), rows, cols, C.c_void_p(_ptr(codes)),
                                      C.c_void_p(_ptr(scales)), _stream_ptr(stream)))


class DeviceBlock:
    """Device copies (torch tensors) of one block's weights, in the canonical layout."""

    def __init__(self, blk: dict, device="cuda"):
        import torch
        shape = blk["shape"]
        self.shape = shape

        def up(a, dt=None):
            if isinstance(a, torch.Tensor):   # already a tensor (e.g. drawn on the device)
                return a.to(device).contiguous()
            a = np.ascontiguousarray(a)
            t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
            return t.to(device)

        self.gamma = up(blk["gamma"])
        self.router_w = up(blk["router_w"])
        self.router_b = up(blk["router_b"])
        self.mats = {m: (up(blk["codes"][m]), up(blk["scales"][m]), up(blk["bias"][m])) for m in ("gate", "up", "down")}
        self.shared = None
        if shape.n_shared:
            sh = blk["shared"]
            self.shared = {m: (up(sh["codes"][m]), up(sh["scales"][m]), up(sh["bias"][m])) for m in ("gate", "up", "down")}

    def cstruct(self) -> Weights:
        w = Weights()
        w.gamma, w.router_w, w.router_b = _ptr(self.gamma), _ptr(self.router_w), _ptr(self.router_b)
        for m in ("gate", "up", "down"):
            c, s, b = self.mats[m]
            setattr(w, m, Mat(_ptr(c), _ptr(s), _ptr(b)))
            if self.shared is not None:
                c, s, b = self.shared[m]
                setattr(w, "sh_" + m, Mat(_ptr(c), _ptr(s), _ptr(b)))
        return w


class HostStoreBlock(DeviceBlock):
    """A block's weights for a plan with an expert cache: the routed experts'
    matrices in pinned host memory (the store the cache copies from), the
    router, the norm weight and the shared expert on the device."""

    def __init__(self, blk: dict, device="cuda"):
        super().__init__(blk, device)
        self.mats = {m: tuple(t.cpu().pin_memory() for t in v) for m, v in self.mats.items()}


class Plan:
    """One block shape: owns the plan handle and a torch-allocated workspace."""

    def __init__(self, shape, max_tokens: int = 4096, device="cuda", **opts):
        self.L = load()
        self.shape = shape
        h = self.L.moe_plan_create(shape.hidden, shape.expert_hidden, shape.n_experts, shape.top_k,
                                   shape.swiglu_alpha, shape.swiglu_limit, shape.weight_scale)
        if not h:
            raise MoeError(MOE_ESHAPE, self.L.moe_last_error().decode())
        self.h = C.c_void_p(h)
        self.set_i("n_shared_experts", shape.n_shared)
        self.set_f("rms_eps", shape.rms_eps)
        self.set_i("max_tokens", max_tokens)
        for k, v in opts.items():
            self.set_i(k, int(v))
        self.max_tokens = max_tokens
        self.device = device
        self.ws = None
        self.weights = None

    def set_i(self, key: str, v: int):
        _check(self.L.moe_plan_set_i(self.h, key.encode(), int(v)))

    def set_f(self, key: str, v: float):
        _check(self.L.moe_plan_set_f(self.h, key.encode(), float(v)))

    def path_for(self, tokens: int) -> int:
        """1 if a forward of `tokens` tokens runs the GEMV decode path, 2 the
        grouped GEMM, 3 the block-scaled FP4 grouped GEMM (act_fp4 plans)."""
        rc = int(self.L.moe_plan_path_for(self.h, int(tokens)))
        _check(min(rc, 0))
        return rc

    def workspace_bytes(self, max_tokens: int = 0) -> int:
        return int(self.L.moe_workspace_bytes(self.h, max_tokens))

    def alloc_workspace(self):
        import torch
        n = self.workspace_bytes()
        self.ws = torch.empty(n + 256, dtype=torch.uint8, device=self.device)
        p = self.ws.data_ptr()
        off = (-p) % 256
        _check(self.L.moe_set_workspace(self.h, C.c_void_p(p + off), n))
        return self

    def load_weights(self, dev: DeviceBlock):
        self.weights = dev  # keep alive
        self._wstruct = dev.cstruct()
        _check(self.L.moe_load_weights(self.h, C.byref(self._wstruct)))
        return self

    def forward(self, x, out, ids=None, stream=None):
        _check(self.L.moe_forward(self.h, C.c_void_p(_ptr(x)), int(x.shape[0]), C.c_void_p(_ptr(out)),
                                  C.c_void_p(_ptr(ids)), _stream_ptr(stream)))

    def forward_ex(self, x, out, ids=None, route_w=None, xhat=None, stream=None):
        _check(self.L.moe_forward_ex(self.h, C.c_void_p(_ptr(x)), int(x.shape[0]), C.c_void_p(_ptr(out)),
                                     C.c_void_p(_ptr(ids)), C.c_void_p(_ptr(route_w)), C.c_void_p(_ptr(xhat)),
                                     _stream_ptr(stream)))

    def expert_counts(self, out, stream=None):
        _check(self.L.moe_get_expert_counts(self.h, C.c_void_p(_ptr(out)), _stream_ptr(stream)))

    def permutation(self, offsets, perm_token, perm_slot, stream=None):
        """offsets [E + n_shared + 1]; perm_token / perm_slot of at least
        max_tokens * (top_k + n_shared) entries (the extent the library copies)."""
        R = self.max_tokens * (self.shape.top_k + self.shape.n_shared)
        if perm_token.numel() < R or perm_slot.numel() < R:
            raise MoeError(MOE_EINVAL, f"perm_token / perm_slot need {R} entries")
        if offsets.numel() < self.shape.n_experts + self.shape.n_shared + 1:
            raise MoeError(MOE_EINVAL, "offsets needs n_experts + n_shared + 1 entries")
        _check(self.L.moe_get_permutation(self.h, C.c_void_p(_ptr(offsets)), C.c_void_p(_ptr(perm_token)),
                                          C.c_void_p(_ptr(perm_slot)), _stream_ptr(stream)))

    def debug_dequant(self, expert: int, which: int, out, stream=None):
        _check(self.L.moe_debug_dequant(self.h, int(expert), int(which), C.c_void_p(_ptr(out)), _stream_ptr(stream)))

    def profile_read(self, n_slots: int = 4):
        """(total ms, launches) per kernel slot since the last read (profile option)."""
        ms = (C.c_double * n_slots)()
        cnt = (C.c_int * n_slots)()
        _check(self.L.moe_profile_read(self.h, ms, cnt, n_slots))
        return list(ms), list(cnt)

    def device_status(self, stream=None) -> int:
        s = C.c_int(0)
        rc = self.L.moe_get_device_status(self.h, C.byref(s), _stream_ptr(stream))
        if rc not in (MOE_OK, MOE_EDEVICE):
            _check(rc)
        return s.value

    def cache_state(self, stream=None):
        """Expert cache of a plan made with expert_cache_slots: (slot of each
        expert, -1 when not resident; cumulative hits; misses; forwards)."""
        slots = np.empty(self.shape.n_experts, np.int32)
        stats = np.zeros(3, np.int64)
        _check(self.L.moe_get_cache_state(self.h, slots.ctypes.data_as(C.c_void_p),
                                          stats.ctypes.data_as(C.c_void_p), _stream_ptr(stream)))
        return slots, int(stats[0]), int(stats[1]), int(stats[2])

    def close(self):
        if getattr(self, "h", None):
            self.L.moe_plan_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Locality:
    """Expert-locality statistics of the routing (ds4.c expert locality
    profiler; goosedump gpt_oss.rs ExpertRouteProfile), kept on the device."""

    def __init__(self, n_layers: int, n_experts: int, top_k: int, caps=()):
        import numpy as np
        self.L = load()
        self.n_layers, self.n_experts, self.top_k = n_layers, n_experts, top_k
        arr = (C.c_int * max(len(caps), 1))(*[int(c) for c in caps])
        h = self.L.moe_locality_create(n_layers, n_experts, top_k, arr, len(caps))
        if not h:
            raise MoeError(MOE_EINVAL, self.L.moe_last_error().decode())
        self.h = C.c_void_p(h)
        self._np = np

    def record(self, layer: int, ids, route_w, first_pos: int, stream=None):
        _check(self.L.moe_locality_record(self.h, int(layer), C.c_void_p(_ptr(ids)), C.c_void_p(_ptr(route_w)),
                                          int(ids.shape[0]), int(first_pos), _stream_ptr(stream)))

    def attach(self, plan, layer: int):
        _check(self.L.moe_locality_attach(plan.h, self.h, int(layer)))

    def reset(self, stream=None):
        _check(self.L.moe_locality_reset(self.h, _stream_ptr(stream)))

    def read(self) -> dict:
        np = self._np
        L, E = self.n_layers, self.n_experts
        out = dict(hist=np.zeros((L, E), np.uint64), weight_hist=np.zeros((L, E), np.float64),
                   layer_records=np.zeros(L, np.uint64), adjacent_pairs=np.zeros(L, np.uint64),
                   overlap_sum=np.zeros(L, np.float64), jaccard_sum=np.zeros(L, np.float64),
                   cache_hits=np.zeros((16, L), np.uint64), cache_weight_hits=np.zeros((16, L), np.float64),
                   caps=np.zeros(16, np.int32))
        st = LocalityStats(*[out[k].ctypes.data for k in ("hist", "weight_hist", "layer_records", "adjacent_pairs",
                                                          "overlap_sum", "jaccard_sum", "cache_hits",
                                                          "cache_weight_hits", "caps")], 0)
        _check(self.L.moe_locality_read(self.h, C.byref(st)))
        n = st.n_caps
        out["caps"] = out["caps"][:n].copy()
        out["cache_hits"] = out["cache_hits"][:n].copy()
        out["cache_weight_hits"] = out["cache_weight_hits"][:n].copy()
        return out

    def close(self):
        if getattr(self, "h", None):
            self.L.moe_locality_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class AttnPlan:
    """One layer's attention decode step (moe_attn_*): the plan, a torch-allocated
    workspace and fp16 key/value caches [max_seqs][max_ctx][kv_heads][64]."""

    def __init__(self, hidden: int, q_heads: int, kv_heads: int, max_seqs: int, max_ctx: int, head_dim: int = 64,
                 sliding_window: int = 0, out_bf16: bool = False, prefill_rows: int = 0, device="cuda"):
        import torch
        self.L = load()
        h = self.L.moe_attn_create(hidden, q_heads, kv_heads, head_dim, max_seqs, max_ctx)
        if not h:
            raise MoeError(MOE_EINVAL, self.L.moe_last_error().decode())
        self.h = C.c_void_p(h)
        self.hidden, self.q_heads, self.kv_heads, self.max_seqs, self.max_ctx = hidden, q_heads, kv_heads, max_seqs, max_ctx
        _check(self.L.moe_attn_set_i(self.h, b"sliding_window", int(sliding_window)))
        _check(self.L.moe_attn_set_i(self.h, b"out_bf16", int(out_bf16)))
        if prefill_rows:
            _check(self.L.moe_attn_set_i(self.h, b"prefill_rows", int(prefill_rows)))
        n = int(self.L.moe_attn_workspace_bytes(self.h))
        self.ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
        off = (-self.ws.data_ptr()) % 256
        _check(self.L.moe_attn_set_workspace(self.h, C.c_void_p(self.ws.data_ptr() + off), n))
        self.k_cache = torch.zeros((max_seqs, max_ctx, kv_heads, head_dim), dtype=torch.float16, device=device)
        self.v_cache = torch.zeros_like(self.k_cache)
        _check(self.L.moe_attn_set_cache(self.h, C.c_void_p(self.k_cache.data_ptr()),
                                         C.c_void_p(self.v_cache.data_ptr())))
        self.weights = None

    def load_weights(self, wts: dict):
        """wts: device tensors gamma, wq, wk, wv, wo (bf16 bits as int16), bq, bk, bv, bo, sinks (float32)."""
        self.weights = wts
        self._w = AttnWeights(*[_ptr(wts[k]) for k in ("gamma", "wq", "wk", "wv", "wo", "bq", "bk", "bv", "bo",
                                                        "sinks")])
        _check(self.L.moe_attn_load_weights(self.h, C.byref(self._w)))
        return self

    def decode(self, x, positions, out, stream=None):
        _check(self.L.moe_attn_decode(self.h, C.c_void_p(_ptr(x)), int(x.shape[0]), C.c_void_p(_ptr(positions)),
                                      C.c_void_p(_ptr(out)), _stream_ptr(stream)))

    def prefill(self, x, seq: int, pos0: int, out, stream=None):
        """x: bf16 bits [n][hidden] (n new tokens of cache sequence seq at positions pos0 ..)."""
        _check(self.L.moe_attn_prefill(self.h, C.c_void_p(_ptr(x)), int(x.shape[0]), int(seq), int(pos0),
                                       C.c_void_p(_ptr(out)), _stream_ptr(stream)))

    def set_i(self, key: str, value: int):
        _check(self.L.moe_attn_set_i(self.h, key.encode(), int(value)))

    def device_status(self, stream=None) -> int:
        s = C.c_int(0)
        rc = self.L.moe_attn_get_device_status(self.h, C.byref(s), _stream_ptr(stream))
        if rc not in (MOE_OK, MOE_EDEVICE):
            _check(rc)
        return s.value

    def close(self):
        if getattr(self, "h", None):
            self.L.moe_attn_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
