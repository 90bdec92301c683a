"""Thin object wrapper over the C ABI: builds hy_config / hy_weights from torch
CUDA tensors and forwards every call to libhybrid.so (marshalling only)."""
from __future__ import annotations

import ctypes

from . import capi
from .capi import check, hy_config, hy_layer_weights, hy_tensor, hy_weights


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _tensor(t) -> hy_tensor:
    """hy_tensor of a bf16 matrix, or of a 4-bit (packed nibbles, fp16 scales) pair."""
    if t is None:
        return hy_tensor(None, None)
    if isinstance(t, tuple):
        return hy_tensor(t[0].data_ptr(), t[1].data_ptr())
    return hy_tensor(t.data_ptr(), None)


def _stream(stream=None) -> int | None:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def make_config(shape, splits: int = 0, flags: int = 0) -> hy_config:
    """hy_config from any object with the model-shape attributes."""
    c = hy_config()
    for n in ("n_layers", "hidden", "vocab", "ffn", "gdn_heads", "gdn_dk", "gdn_dv", "conv_k", "attn_q_heads",
              "attn_kv_heads", "head_dim", "n_experts", "top_k", "expert_ffn", "shared_ffn"):
        setattr(c, n, int(getattr(shape, n)))
    mask = 0
    for l in range(shape.n_layers):
        if shape.is_attn(l):
            mask |= 1 << l
    c.attn_layer_mask = mask
    c.rms_eps = float(shape.rms_eps)
    c.rope_theta = float(shape.rope_theta)
    c.weight_format = int(getattr(shape, "weight_format", 0))
    c.kv_format = int(getattr(shape, "kv_format", 0))
    c.attn_splits = int(splits)
    c.flags = int(flags)
    return c


class HybridModel:
    """One model plus its cache of ``len(capacities)`` sequences.

    ``weights`` maps the tensor names of include/hybrid.h (``l{i}.w_in``,
    ``l{i}.norm1``, ..., ``embed``, ``final_norm``, ``lm_head``) to CUDA
    tensors (bf16 matrices, float32 gains).  The tensors are borrowed and kept
    referenced by this object.
    """

    def __init__(self, shape, weights: dict, capacities, splits: int = 0, flags: int = 0, pages=None):
        """pages: (page_tokens, pool_pages) for a paged KV cache (hy_cache_alloc_paged)."""
        L = capi.lib()
        self.shape = shape
        self._weights = weights
        self.cfg = make_config(shape, splits, flags)
        layers = (hy_layer_weights * shape.n_layers)()
        for l in range(shape.n_layers):
            w = layers[l]
            g = lambda n: weights.get(f"l{l}.{n}")  # noqa: E731
            w.norm1, w.norm2 = _ptr(g("norm1")), _ptr(g("norm2"))
            w.w_in = _tensor(g("w_in"))
            w.w_o = _tensor(g("w_o"))
            w.conv_w = _ptr(g("conv_w"))
            for n in ("w_gate", "w_up", "w_down", "exp_gate", "exp_up", "exp_down", "sh_gate", "sh_up", "sh_down"):
                setattr(w, n, _tensor(g(n)))
            w.router = _ptr(g("router"))
        self._layers = layers
        hw = hy_weights()
        hw.embed = _ptr(weights["embed"])
        hw.final_norm = _ptr(weights["final_norm"])
        hw.lm_head = _tensor(weights["lm_head"])
        hw.layers = layers
        self._hw = hw
        m = ctypes.c_void_p()
        check(L.hy_model_create(ctypes.byref(self.cfg), ctypes.byref(hw), ctypes.byref(m)), "hy_model_create")
        self.m = m
        caps = (ctypes.c_int32 * len(capacities))(*[int(x) for x in capacities])
        c = ctypes.c_void_p()
        if pages:
            rc = L.hy_cache_alloc_paged(m, len(capacities), caps, int(pages[0]), int(pages[1]), ctypes.byref(c))
        else:
            rc = L.hy_cache_alloc(m, len(capacities), caps, ctypes.byref(c))
        if rc != capi.HY_OK:
            L.hy_model_free(m)
            self.m = None
            check(rc, "hy_cache_alloc")
        self.c = c

    # --------------------------------------------------------------- calls
    def prefill(self, seq: int, tokens, logits=None, stream=None) -> None:
        check(capi.lib().hy_prefill(self.m, self.c, seq, _ptr(tokens), int(tokens.numel()), _ptr(logits),
                                    _stream(stream)), "hy_prefill")

    def decode_step(self, seq: int, token, ids, logits=None, stream=None) -> None:
        seqs = (ctypes.c_int32 * 1)(seq)
        check(capi.lib().hy_decode_step(self.m, self.c, seqs, 1, _ptr(token), _ptr(logits), _ptr(ids),
                                        _stream(stream)), "hy_decode_step")

    def decode_batch(self, seqs, tokens, ids, logits=None, stream=None) -> None:
        """One step for the distinct sequences `seqs` (tokens, ids: int32 CUDA
        tensors [len(seqs)]; logits: FP32 [len(seqs)][V] or None)."""
        arr = (ctypes.c_int32 * len(seqs))(*[int(s) for s in seqs])
        check(capi.lib().hy_decode_step(self.m, self.c, arr, len(seqs), _ptr(tokens), _ptr(logits), _ptr(ids),
                                        _stream(stream)), "hy_decode_step")

    def decode_step_host(self, seq: int, token_host, ids_host, logits_host=None, stream=None) -> None:
        """token_host / ids_host / logits_host: CPU tensors (pinned or not)."""
        seqs = (ctypes.c_int32 * 1)(seq)
        check(capi.lib().hy_decode_step_host(self.m, self.c, seqs, 1, token_host.data_ptr(),
                                             None if logits_host is None else logits_host.data_ptr(),
                                             ids_host.data_ptr(), _stream(stream)), "hy_decode_step_host")

    def decode_batch_host(self, seqs, tokens_host, ids_host, logits_host=None, stream=None) -> None:
        """decode_batch with CPU tensors (int32 [len(seqs)]; logits FP32 [len(seqs)][V])."""
        arr = (ctypes.c_int32 * len(seqs))(*[int(s) for s in seqs])
        check(capi.lib().hy_decode_step_host(self.m, self.c, arr, len(seqs), tokens_host.data_ptr(),
                                             None if logits_host is None else logits_host.data_ptr(),
                                             ids_host.data_ptr(), _stream(stream)), "hy_decode_step_host")

    def experts_read(self, stream=None) -> int:
        """Distinct routed experts the batched steps read since the last call
        (summed over layers and steps); resets the count."""
        v = ctypes.c_uint64(0)
        check(capi.lib().hy_experts_read(self.c, _stream(stream), ctypes.byref(v)), "hy_experts_read")
        return int(v.value)

    def fill_synthetic(self, seq: int, length: int, seed: int = 0, stream=None) -> None:
        """Give sequence `seq` `length` positions of seeded synthetic cache
        contents (KV rows and recurrent state) without running a prompt."""
        check(capi.lib().hy_seq_fill_synthetic(self.c, seq, int(length), int(seed), _stream(stream)),
              "hy_seq_fill_synthetic")

    def seq_len(self, seq: int) -> int:
        return int(capi.lib().hy_seq_len(self.c, seq))

    def seq_capacity(self, seq: int) -> int:
        return int(capi.lib().hy_seq_capacity(self.c, seq))

    def step_kernels(self) -> int:
        """Kernels the last recorded decode step launches (one per operation)."""
        return int(capi.lib().hy_step_kernels(self.c))

    def step_splits(self, seq: int = 0) -> int:
        """Split-KV chunks per kv head of sequence `seq`'s batch-1 step."""
        return int(capi.lib().hy_step_splits(self.c, seq))

    def free_pages(self) -> int:
        """Pages left in the pool of a paged cache (-1 without pages)."""
        return int(capi.lib().hy_cache_free_pages(self.c))

    def reset(self, seq: int, stream=None) -> None:
        check(capi.lib().hy_seq_reset(self.c, seq, _stream(stream)), "hy_seq_reset")

    def check_device(self, stream=None) -> int:
        bits = ctypes.c_uint32(0)
        rc = capi.lib().hy_check_device(self.c, _stream(stream), ctypes.byref(bits))
        if rc not in (capi.HY_OK, capi.HY_ERR_DEVICE_GUARD):
            check(rc, "hy_check_device")
        return int(bits.value)

    def debug_hidden(self, layer: int, stream=None):
        import torch
        out = torch.empty(self.shape.hidden, dtype=torch.float32, device="cuda")
        check(capi.lib().hy_debug_hidden(self.c, layer, out.data_ptr(), _stream(stream)), "hy_debug_hidden")
        return out

    def debug_router(self, layer: int, stream=None):
        import torch
        lg = torch.empty(self.shape.n_experts + 1, dtype=torch.float32, device="cuda")
        ids = torch.empty(self.shape.top_k, dtype=torch.int32, device="cuda")
        check(capi.lib().hy_debug_router(self.c, layer, lg.data_ptr(), ids.data_ptr(), _stream(stream)),
              "hy_debug_router")
        return lg, ids

    def close(self) -> None:
        L = capi.lib()
        if getattr(self, "c", None):
            L.hy_cache_free(self.c)
            self.c = None
        if getattr(self, "m", None):
            L.hy_model_free(self.m)
            self.m = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
