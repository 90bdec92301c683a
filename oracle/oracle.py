"""ctypes wrapper of the C oracle (oracle.c).  Test infrastructure only.

Argument marshalling only: every computation happens in oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(HERE, "liboracle.so")
SRC = os.path.join(HERE, "oracle.c")
HDR = os.path.join(HERE, "oracle.h")

c_i32, c_i64, c_f64, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p


def build(force: bool = False) -> str:
    stale = not os.path.exists(SO) or max(os.path.getmtime(SRC), os.path.getmtime(HDR)) > os.path.getmtime(SO)
    if force or stale:
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", SO, SRC, "-lm"])
    return SO


class OrcMat(ctypes.Structure):
    _fields_ = [("fmt", c_i32), ("rows", c_i64), ("cols", c_i64), ("bf16", c_vp), ("qs", c_vp), ("scales", c_vp)]


class OrcConfig(ctypes.Structure):
    _fields_ = [(n, c_i32) for n in ("n_layers", "hidden", "vocab", "ffn", "gdn_heads", "gdn_dk", "gdn_dv", "conv_k",
                                     "attn_q_heads", "attn_kv_heads", "head_dim", "n_experts", "top_k",
                                     "expert_ffn", "shared_ffn")] + [
        ("rms_eps", c_f64), ("rope_theta", c_f64), ("is_attn", c_vp), ("kv_format", c_i32)]


class OrcLayer(ctypes.Structure):
    _fields_ = [("norm1", c_vp), ("w_in", OrcMat), ("conv_w", c_vp), ("w_o", OrcMat), ("norm2", c_vp),
                ("w_gate", OrcMat), ("w_up", OrcMat), ("w_down", OrcMat), ("router", OrcMat),
                ("exp_gate", OrcMat), ("exp_up", OrcMat), ("exp_down", OrcMat),
                ("sh_gate", OrcMat), ("sh_up", OrcMat), ("sh_down", OrcMat)]


class OrcWeights(ctypes.Structure):
    _fields_ = [("embed", c_vp), ("final_norm", c_vp), ("lm_head", OrcMat), ("layers", c_vp)]


class OrcCache(ctypes.Structure):
    _fields_ = [("len", c_i32), ("capacity", c_i32), ("gdn_state", c_vp), ("conv_state", c_vp),
                ("k_cache", c_vp), ("v_cache", c_vp), ("k_q", c_vp), ("v_q", c_vp), ("k_s", c_vp), ("v_s", c_vp)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        L = _lib
        P = ctypes.POINTER
        L.orc_bf16_to_double.argtypes, L.orc_bf16_to_double.restype = [ctypes.c_uint16], c_f64
        L.orc_to_bf16.argtypes, L.orc_to_bf16.restype = [c_f64], ctypes.c_uint16
        L.orc_fp16_to_double.argtypes, L.orc_fp16_to_double.restype = [ctypes.c_uint16], c_f64
        L.orc_q4_value.argtypes, L.orc_q4_value.restype = [P(OrcMat), c_i64, c_i64], c_f64
        L.orc_mat_row.argtypes = [P(OrcMat), c_i64, c_vp]
        L.orc_gemv.argtypes = [P(OrcMat), c_vp, c_vp]
        L.orc_rmsnorm.argtypes = [c_vp, c_vp, c_i32, c_f64, c_vp]
        L.orc_l2norm.argtypes = [c_vp, c_i32, c_f64]
        L.orc_sigmoid.argtypes, L.orc_sigmoid.restype = [c_f64], c_f64
        L.orc_silu.argtypes, L.orc_silu.restype = [c_f64], c_f64
        L.orc_rope.argtypes = [c_vp, c_i32, c_i32, c_f64]
        L.orc_conv_step.argtypes = [c_vp, c_vp, c_vp, c_i32, c_i32, c_vp]
        L.orc_gdn_step.argtypes = [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_f64, c_f64, c_vp]
        L.orc_attention.argtypes = [c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp]
        L.orc_attention_split.argtypes = [c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp]
        L.orc_quant_i8.argtypes = [c_vp, c_i32, c_vp, c_vp]
        L.orc_attention_i8.argtypes = [c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp]
        L.orc_argmax.argtypes, L.orc_argmax.restype = [c_vp, c_i64], c_i32
        L.orc_topk.argtypes = [c_vp, c_i32, c_i32, c_vp]
        L.orc_softmax.argtypes = [c_vp, c_i32, c_vp]
        L.orc_cache_create.argtypes, L.orc_cache_create.restype = [P(OrcConfig), c_i32, P(OrcCache)], ctypes.c_int
        L.orc_cache_destroy.argtypes = [P(OrcCache)]
        L.orc_cache_reset.argtypes = [P(OrcConfig), P(OrcCache)]
        L.orc_forward_token.argtypes = [P(OrcConfig), P(OrcWeights), P(OrcCache), c_i32, c_vp, c_vp, c_vp, c_vp]
        L.orc_forward_token.restype = ctypes.c_int
        L.orc_threads.restype = ctypes.c_int
        L.orc_set_threads.argtypes = [ctypes.c_int]
        for f in (L.orc_mat_row, L.orc_gemv, L.orc_rmsnorm, L.orc_l2norm, L.orc_rope, L.orc_conv_step,
                  L.orc_gdn_step, L.orc_attention, L.orc_attention_split, L.orc_topk, L.orc_softmax,
                  L.orc_quant_i8, L.orc_attention_i8,
                  L.orc_cache_destroy, L.orc_cache_reset, L.orc_set_threads):
            f.restype = None
    return _lib


# ---------------------------------------------------------------- helpers

def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def mat(w, keep: list) -> OrcMat:
    """OrcMat over a bf16 uint16 array [.., cols] or a 4-bit (qs, scales) pair."""
    m = OrcMat()
    if isinstance(w, tuple):
        qs, sc = (np.ascontiguousarray(w[0], dtype=np.uint8), np.ascontiguousarray(w[1]).view(np.uint16))
        keep += [qs, sc]
        m.fmt, m.cols = 1, qs.shape[-1] * 2
        m.rows = qs.size // qs.shape[-1]
        m.qs, m.scales = _p(qs), _p(sc)
    else:
        a = np.ascontiguousarray(w).view(np.uint16)
        keep.append(a)
        m.fmt, m.cols = 0, a.shape[-1]
        m.rows = a.size // a.shape[-1]
        m.bf16 = _p(a)
    return m


# ------------------------------------------------------- primitive wrappers

def gemv(w, x) -> np.ndarray:
    keep: list = []
    m = mat(w, keep)
    x = f64(x)
    y = np.zeros(m.rows, dtype=np.float64)
    lib().orc_gemv(ctypes.byref(m), _p(x), _p(y))
    return y


def mat_row(w, r: int) -> np.ndarray:
    keep: list = []
    m = mat(w, keep)
    out = np.zeros(m.cols, dtype=np.float64)
    lib().orc_mat_row(ctypes.byref(m), r, _p(out))
    return out


def rmsnorm(x, g, eps: float) -> np.ndarray:
    x = f64(x)
    g = np.ascontiguousarray(g, dtype=np.float32)
    y = np.zeros_like(x)
    lib().orc_rmsnorm(_p(x), _p(g), x.size, eps, _p(y))
    return y


def l2norm(v, eps: float = 1e-6) -> np.ndarray:
    v = f64(v).copy()
    lib().orc_l2norm(_p(v), v.size, eps)
    return v


def rope(v, pos: int, theta: float = 1e4) -> np.ndarray:
    v = f64(v).copy()
    lib().orc_rope(_p(v), v.size, pos, theta)
    return v


def conv_step(u, state, w_bf16, k: int):
    """Returns (out, new_state); state is [k-1][channels] float64."""
    u = f64(u)
    st = f64(state).copy()
    w = np.ascontiguousarray(w_bf16).view(np.uint16)
    out = np.zeros_like(u)
    lib().orc_conv_step(_p(u), _p(st), _p(w), u.size, k, _p(out))
    return out, st


def gdn_step(S, q, k, v, alpha: float, beta: float):
    """S: float32 [dv][dk] (copied).  Returns (o, S_new)."""
    S = np.ascontiguousarray(S, dtype=np.float32).copy()
    dv, dk = S.shape
    q, k, v = f64(q), f64(k), f64(v)
    o = np.zeros(dv, dtype=np.float64)
    lib().orc_gdn_step(_p(S), dk, dv, _p(q), _p(k), _p(v), alpha, beta, _p(o))
    return o, S


def attention(q, K, V, npos: int, nsplit: int = 0) -> np.ndarray:
    """q: [nq][hd]; K, V: bf16 bits [nkv][cap][hd]."""
    q = f64(q)
    nq, hd = q.shape
    K = np.ascontiguousarray(K).view(np.uint16)
    V = np.ascontiguousarray(V).view(np.uint16)
    nkv, cap, _ = K.shape
    o = np.zeros_like(q)
    if nsplit:
        lib().orc_attention_split(_p(q), _p(K), _p(V), nq, nkv, hd, cap, npos, nsplit, _p(o))
    else:
        lib().orc_attention(_p(q), _p(K), _p(V), nq, nkv, hd, cap, npos, _p(o))
    return o


def quant_i8(x):
    """(int8 codes, FP32 scale) of one cached vector."""
    x = f64(x)
    q = np.zeros(x.size, dtype=np.int8)
    sc = np.zeros(1, dtype=np.float32)
    lib().orc_quant_i8(_p(x), x.size, _p(q), _p(sc))
    return q, float(sc[0])


def attention_i8(q, Kq, Ks, Vq, Vs, npos: int) -> np.ndarray:
    """q: [nq][hd]; Kq, Vq: int8 codes [nkv][cap][hd]; Ks, Vs: FP32 scales [nkv][cap]."""
    q = f64(q)
    nq, hd = q.shape
    Kq, Vq = np.ascontiguousarray(Kq, dtype=np.int8), np.ascontiguousarray(Vq, dtype=np.int8)
    Ks, Vs = np.ascontiguousarray(Ks, dtype=np.float32), np.ascontiguousarray(Vs, dtype=np.float32)
    nkv, cap, _ = Kq.shape
    o = np.zeros_like(q)
    lib().orc_attention_i8(_p(q), _p(Kq), _p(Ks), _p(Vq), _p(Vs), nq, nkv, hd, cap, npos, _p(o))
    return o


def argmax(v) -> int:
    v = f64(v)
    return int(lib().orc_argmax(_p(v), v.size))


def topk(r, k: int) -> np.ndarray:
    r = f64(r)
    ids = np.zeros(k, dtype=np.int32)
    lib().orc_topk(_p(r), r.size, k, _p(ids))
    return ids


def softmax(x) -> np.ndarray:
    x = f64(x)
    p = np.zeros_like(x)
    lib().orc_softmax(_p(x), x.size, _p(p))
    return p


def to_bf16(x: float) -> int:
    return int(lib().orc_to_bf16(float(x)))


def bf16_to_double(b: int) -> float:
    return float(lib().orc_bf16_to_double(int(b)))


def fp16_to_double(h: int) -> float:
    return float(lib().orc_fp16_to_double(int(h)))


def set_threads(n: int) -> None:
    lib().orc_set_threads(n)


def threads() -> int:
    return int(lib().orc_threads())


# --------------------------------------------------------------- the model

class Oracle:
    """The whole-model oracle for one sequence.

    ``shape`` is any object with the model-shape attributes (n_layers, hidden,
    vocab, ffn, gdn_heads, gdn_dk, gdn_dv, conv_k, attn_q_heads, attn_kv_heads,
    head_dim, n_experts, top_k, expert_ffn, shared_ffn, rms_eps, rope_theta and
    is_attn(layer)).  ``weights`` maps tensor names (``l{i}.w_in``, ...,
    ``embed``, ``final_norm``, ``lm_head``) to numpy arrays (bf16 as uint16
    bits, float32, or (qs, scales) for 4-bit).
    """

    def __init__(self, shape, weights: dict, capacity: int):
        self.shape = shape
        self._keep: list = []
        s = shape
        cfg = OrcConfig()
        for n in ("n_layers", "hidden", "vocab", "ffn", "gdn_heads", "gdn_dk", "gdn_dv", "conv_k", "attn_q_heads",
                  "attn_kv_heads", "head_dim", "n_experts", "top_k", "expert_ffn", "shared_ffn"):
            setattr(cfg, n, int(getattr(s, n)))
        cfg.rms_eps, cfg.rope_theta = float(s.rms_eps), float(s.rope_theta)
        cfg.kv_format = int(getattr(s, "kv_format", 0))
        self._is_attn = np.array([1 if s.is_attn(l) else 0 for l in range(s.n_layers)], dtype=np.uint8)
        cfg.is_attn = _p(self._is_attn)
        self.cfg = cfg

        def arr(name, dtype):
            a = np.ascontiguousarray(weights[name])
            a = a.view(dtype) if a.dtype != dtype and a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
            self._keep.append(a)
            return _p(a)

        layers = (OrcLayer * s.n_layers)()
        for l in range(s.n_layers):
            L = layers[l]
            L.norm1 = arr(f"l{l}.norm1", np.float32)
            L.norm2 = arr(f"l{l}.norm2", np.float32)
            L.w_in = mat(weights[f"l{l}.w_in"], self._keep)
            L.w_o = mat(weights[f"l{l}.w_o"], self._keep)
            if not s.is_attn(l):
                L.conv_w = arr(f"l{l}.conv_w", np.uint16)
            if s.ffn > 0:
                for n in ("w_gate", "w_up", "w_down"):
                    setattr(L, n, mat(weights[f"l{l}.{n}"], self._keep))
            else:
                for n in ("router", "exp_gate", "exp_up", "exp_down", "sh_gate", "sh_up", "sh_down"):
                    setattr(L, n, mat(weights[f"l{l}.{n}"], self._keep))
        self._layers = layers
        w = OrcWeights()
        w.embed = arr("embed", np.uint16)
        w.final_norm = arr("final_norm", np.float32)
        w.lm_head = mat(weights["lm_head"], self._keep)
        w.layers = ctypes.addressof(layers)
        self.w = w
        self.cache = OrcCache()
        if lib().orc_cache_create(ctypes.byref(cfg), capacity, ctypes.byref(self.cache)) != 0:
            raise MemoryError("oracle cache allocation failed")

    def __del__(self):
        try:
            lib().orc_cache_destroy(ctypes.byref(self.cache))
        except Exception:
            pass

    @property
    def len(self) -> int:
        return int(self.cache.len)

    def reset(self) -> None:
        lib().orc_cache_reset(ctypes.byref(self.cfg), ctypes.byref(self.cache))

    def forward(self, token: int, want_hidden: bool = True, want_router: bool = False) -> dict:
        s = self.shape
        logits = np.zeros(s.vocab, dtype=np.float64)
        hidden = np.zeros((s.n_layers, s.hidden), dtype=np.float64) if want_hidden else None
        moe = want_router and s.ffn == 0
        rids = np.zeros((s.n_layers, max(s.top_k, 1)), dtype=np.int32) if moe else None
        rlog = np.zeros((s.n_layers, s.n_experts + 1), dtype=np.float64) if moe else None
        rc = lib().orc_forward_token(ctypes.byref(self.cfg), ctypes.byref(self.w), ctypes.byref(self.cache), int(token),
                                     _p(logits), _p(hidden) if hidden is not None else None,
                                     _p(rids) if rids is not None else None, _p(rlog) if rlog is not None else None)
        if rc != 0:
            raise RuntimeError("oracle cache is full")
        return {"logits": logits, "hidden": hidden, "router_ids": rids, "router_logits": rlog}

    # raw views of the cache, for tests that inspect the stored state
    def kv_cache(self, attn_index: int):
        s, cap = self.shape, self.cache.capacity
        n = s.attn_kv_heads * cap * s.head_dim
        base = ctypes.cast(self.cache.k_cache, ctypes.POINTER(ctypes.c_uint16))
        vbase = ctypes.cast(self.cache.v_cache, ctypes.POINTER(ctypes.c_uint16))
        k = np.ctypeslib.as_array(base, shape=(n * (attn_index + 1),))[n * attn_index:]
        v = np.ctypeslib.as_array(vbase, shape=(n * (attn_index + 1),))[n * attn_index:]
        return k.reshape(s.attn_kv_heads, cap, s.head_dim), v.reshape(s.attn_kv_heads, cap, s.head_dim)

    def kv_cache_i8(self, attn_index: int):
        """(K codes, K scales, V codes, V scales) of an int8 cache layer."""
        s, cap = self.shape, self.cache.capacity
        n, ns = s.attn_kv_heads * cap * s.head_dim, s.attn_kv_heads * cap
        out = []
        for ptr, cnt, ty, shp in ((self.cache.k_q, n, ctypes.c_int8, (s.attn_kv_heads, cap, s.head_dim)),
                                  (self.cache.k_s, ns, ctypes.c_float, (s.attn_kv_heads, cap)),
                                  (self.cache.v_q, n, ctypes.c_int8, (s.attn_kv_heads, cap, s.head_dim)),
                                  (self.cache.v_s, ns, ctypes.c_float, (s.attn_kv_heads, cap))):
            base = ctypes.cast(ptr, ctypes.POINTER(ty))
            out.append(np.ctypeslib.as_array(base, shape=(cnt * (attn_index + 1),))[cnt * attn_index:].reshape(shp))
        return tuple(out)

    def gdn_state(self, gdn_index: int) -> np.ndarray:
        s = self.shape
        n = s.gdn_heads * s.gdn_dv * s.gdn_dk
        base = ctypes.cast(self.cache.gdn_state, ctypes.POINTER(ctypes.c_float))
        a = np.ctypeslib.as_array(base, shape=(n * (gdn_index + 1),))[n * gdn_index:]
        return a.reshape(s.gdn_heads, s.gdn_dv, s.gdn_dk)
