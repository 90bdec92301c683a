"""Shapes, seeds and tensor tables of the synthetic workloads.

Each workload mirrors a model the pages measure (a dense Qwen-3.5-4B-shaped
Gated-DeltaNet / GQA hybrid and a 35B-A3B-shaped MoE hybrid) with seeded
synthetic weights ~N(0, 0.02) and uniform random prompts; throughput does not
depend on weight values at a fixed shape.  No decode arithmetic lives here.

Weight tensors (all row-major; ``H`` = hidden):

per layer ``l``
  ``norm1`` / ``norm2``  float32 [H]           RMSNorm gains (1.0)
  GDN layer:
    ``w_in``    [2*nh*dk + nh*dv + 2*nh, H]  rows: q | k | v | a | b
    ``conv_w``  bf16 [2*nh*dk + nh*dv, conv_k]  depthwise causal conv taps
    ``w_o``     [H, nh*dv]
  attention layer:
    ``w_in``    [(nq + 2*nkv)*hd, H]         rows: q | k | v
    ``w_o``     [H, nq*hd]
  dense FFN: ``w_gate`` [F, H], ``w_up`` [F, H], ``w_down`` [H, F]
  MoE FFN:   ``router`` [E + 1, H] (row E gates the shared expert),
             ``exp_gate`` / ``exp_up`` [E, Fe, H], ``exp_down`` [E, H, Fe],
             ``sh_gate`` / ``sh_up`` [Fs, H], ``sh_down`` [H, Fs]
global: ``embed`` bf16 [V, H], ``final_norm`` float32 [H], ``lm_head`` [V, H]

Linear weights are bf16, or, for 4-bit workloads, blocks of 32 along the
input dimension: ``qs`` uint8 [rows, cols/2] (byte b of a block holds element
b in its low nibble and element b+16 in its high nibble, each stored as
value+8) and ``scales`` fp16 [rows, cols/32].  The router, the conv taps and
the embedding stay bf16 in 4-bit workloads.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np

from . import gen, host

KIND = {
    "norm1": 0, "w_in": 1, "conv_w": 2, "w_o": 3, "norm2": 4,
    "w_gate": 5, "router": 5, "w_up": 6, "w_down": 7,
    "exp_gate": 8, "exp_up": 9, "exp_down": 10,
    "sh_gate": 11, "sh_up": 12, "sh_down": 13,
}
GLOBAL_TID = {"embed": 1_000_000, "final_norm": 1_000_001, "lm_head": 1_000_002}
PROMPT_TID = 2_000_000
CONTEXT_TID = 2_100_000

BF16, F32, Q4 = "bf16", "f32", "q4"


@dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    hidden: int
    vocab: int
    ffn: int                      # dense SwiGLU width; 0 means MoE
    gdn_heads: int
    gdn_dk: int
    gdn_dv: int
    attn_q_heads: int
    attn_kv_heads: int
    head_dim: int
    attn_layers: tuple
    conv_k: int = 4
    n_experts: int = 0
    top_k: int = 0
    expert_ffn: int = 0
    shared_ffn: int = 0
    rms_eps: float = 1e-6
    rope_theta: float = 1e4
    weight_format: int = 0        # 0 bf16, 1 4-bit blocks of 32
    kv_format: int = 0            # 0 bf16 KV cache, 1 int8 codes with one FP32 scale per cached vector
    seed: int = 0

    @property
    def is_moe(self) -> bool:
        return self.ffn == 0

    def is_attn(self, layer: int) -> bool:
        return layer in self.attn_layers

    @property
    def conv_channels(self) -> int:
        return 2 * self.gdn_heads * self.gdn_dk + self.gdn_heads * self.gdn_dv

    @property
    def gdn_in_rows(self) -> int:
        return self.conv_channels + 2 * self.gdn_heads

    @property
    def attn_in_rows(self) -> int:
        return (self.attn_q_heads + 2 * self.attn_kv_heads) * self.head_dim

    def attn_mask(self) -> int:
        m = 0
        for l in self.attn_layers:
            m |= 1 << l
        return m


def every_fourth(n_layers: int) -> tuple:
    """3:1 DeltaNet:attention pattern, attention at layers 3, 7, 11, ..."""
    return tuple(l for l in range(n_layers) if l % 4 == 3)


TINY = ModelShape("tiny", n_layers=2, hidden=256, vocab=1024, ffn=512, gdn_heads=4, gdn_dk=64, gdn_dv=64,
                  attn_q_heads=4, attn_kv_heads=2, head_dim=64, attn_layers=(1,), seed=0)
DENSE4B = ModelShape("dense-4b", n_layers=32, hidden=2560, vocab=151936, ffn=9216, gdn_heads=16, gdn_dk=128,
                     gdn_dv=128, attn_q_heads=16, attn_kv_heads=4, head_dim=128, attn_layers=every_fourth(32),
                     seed=0)
MOE35B = ModelShape("moe-35b-a3b", n_layers=40, hidden=2048, vocab=151936, ffn=0, gdn_heads=16, gdn_dk=128,
                    gdn_dv=128, attn_q_heads=16, attn_kv_heads=2, head_dim=256, attn_layers=every_fourth(40),
                    n_experts=256, top_k=8, expert_ffn=512, shared_ffn=512, seed=0)
MOE35B_Q4 = dataclasses.replace(MOE35B, name="moe-35b-a3b-q4", weight_format=1)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    prompt_len: int
    decode_steps: int
    batch: int = 1
    splits: tuple = ()
    ragged_context: tuple = ()    # (lo, hi) for per-sequence contexts
    prompt_seed: int = 1
    context_seed: int = 2


WORKLOADS = {
    "tiny": Workload("tiny hybrid, 2 layers, prompt 128 + 16 decode", TINY, 128, 16),
    "dense4b": Workload("dense 4B-shaped hybrid, prompt 4096 + 256 decode", DENSE4B, 4096, 256),
    "dense4b-32k": Workload("dense 4B-shaped hybrid, prompt 32768 + 128 decode", DENSE4B, 32768, 128,
                            splits=(1, 2, 4, 8, 16)),
    "dense4b-32k-kv8": Workload("dense 4B-shaped hybrid, int8 KV cache, prompt 32768 + 128 decode",
                                dataclasses.replace(DENSE4B, name="dense-4b-kv8", kv_format=1), 32768, 128),
    "moe35b": Workload("MoE 35B-A3B-shaped hybrid, prompt 2048 + 256 decode", MOE35B, 2048, 256),
    "moe35b-q4-b8": Workload("MoE 35B-A3B-shaped hybrid, 4-bit, batch 8, ragged context 1024..16384, 128 decode",
                             MOE35B_Q4, 0, 128, batch=8, ragged_context=(1024, 16384)),
}


@dataclass(frozen=True)
class TensorSpec:
    name: str
    tid: int
    dims: tuple
    fmt: str          # bf16 | f32 | q4

    @property
    def rows(self) -> int:
        r = 1
        for d in self.dims[:-1]:
            r *= d
        return r

    @property
    def cols(self) -> int:
        return self.dims[-1]

    def nbytes(self) -> int:
        n = self.rows * self.cols
        if self.fmt == F32:
            return 4 * n
        if self.fmt == BF16:
            return 2 * n
        return n // 2 + 2 * (n // 32)


def tensor_specs(s: ModelShape) -> list[TensorSpec]:
    lin = Q4 if s.weight_format == 1 else BF16
    H = s.hidden
    out: list[TensorSpec] = []
    for l in range(s.n_layers):
        t = lambda k: l * 32 + KIND[k]  # noqa: E731
        out.append(TensorSpec(f"l{l}.norm1", t("norm1"), (H,), F32))
        if s.is_attn(l):
            out.append(TensorSpec(f"l{l}.w_in", t("w_in"), (s.attn_in_rows, H), lin))
            out.append(TensorSpec(f"l{l}.w_o", t("w_o"), (H, s.attn_q_heads * s.head_dim), lin))
        else:
            out.append(TensorSpec(f"l{l}.w_in", t("w_in"), (s.gdn_in_rows, H), lin))
            out.append(TensorSpec(f"l{l}.conv_w", t("conv_w"), (s.conv_channels, s.conv_k), BF16))
            out.append(TensorSpec(f"l{l}.w_o", t("w_o"), (H, s.gdn_heads * s.gdn_dv), lin))
        out.append(TensorSpec(f"l{l}.norm2", t("norm2"), (H,), F32))
        if s.is_moe:
            E, Fe, Fs = s.n_experts, s.expert_ffn, s.shared_ffn
            out.append(TensorSpec(f"l{l}.router", t("router"), (E + 1, H), BF16))
            out.append(TensorSpec(f"l{l}.exp_gate", t("exp_gate"), (E, Fe, H), lin))
            out.append(TensorSpec(f"l{l}.exp_up", t("exp_up"), (E, Fe, H), lin))
            out.append(TensorSpec(f"l{l}.exp_down", t("exp_down"), (E, H, Fe), lin))
            out.append(TensorSpec(f"l{l}.sh_gate", t("sh_gate"), (Fs, H), lin))
            out.append(TensorSpec(f"l{l}.sh_up", t("sh_up"), (Fs, H), lin))
            out.append(TensorSpec(f"l{l}.sh_down", t("sh_down"), (H, Fs), lin))
        else:
            out.append(TensorSpec(f"l{l}.w_gate", t("w_gate"), (s.ffn, H), lin))
            out.append(TensorSpec(f"l{l}.w_up", t("w_up"), (s.ffn, H), lin))
            out.append(TensorSpec(f"l{l}.w_down", t("w_down"), (H, s.ffn), lin))
    out.append(TensorSpec("embed", GLOBAL_TID["embed"], (s.vocab, H), BF16))
    out.append(TensorSpec("final_norm", GLOBAL_TID["final_norm"], (H,), F32))
    out.append(TensorSpec("lm_head", GLOBAL_TID["lm_head"], (s.vocab, H), lin))
    return out


def host_tensor(s: ModelShape, spec: TensorSpec, std: float = 0.02):
    """numpy copy of one tensor: uint16 bf16 bits, float32, or (qs, scales)."""
    if spec.fmt == F32:
        return np.ones(spec.dims, dtype=np.float32)
    if spec.fmt == BF16:
        return host.normal_bf16(s.seed, spec.tid, spec.rows * spec.cols, std).reshape(spec.dims)
    n = spec.rows * spec.cols
    qs = host.q4_packed(s.seed, spec.tid, n // 2).reshape(*spec.dims[:-1], spec.cols // 2)
    sc = host.q4_scales(s.seed, spec.tid, n // 32).reshape(*spec.dims[:-1], spec.cols // 32)
    return (qs, sc)


def host_weights(s: ModelShape, names=None) -> dict:
    out = {}
    for spec in tensor_specs(s):
        if names is None or spec.name in names:
            out[spec.name] = host_tensor(s, spec)
    return out


def device_weights(s: ModelShape, names=None) -> dict:
    """torch CUDA tensors filled on the device by the CUDA generator copy."""
    import torch

    from . import device
    out = {}
    for spec in tensor_specs(s):
        if names is not None and spec.name not in names:
            continue
        if spec.fmt == F32:
            t = torch.empty(spec.dims, dtype=torch.float32, device="cuda")
            device.fill_f32(t, 1.0)
            out[spec.name] = t
        elif spec.fmt == BF16:
            t = torch.empty(spec.dims, dtype=torch.bfloat16, device="cuda")
            device.fill_normal_bf16(t, s.seed, spec.tid)
            out[spec.name] = t
        else:
            qs = torch.empty((*spec.dims[:-1], spec.cols // 2), dtype=torch.uint8, device="cuda")
            sc = torch.empty((*spec.dims[:-1], spec.cols // 32), dtype=torch.float16, device="cuda")
            device.fill_q4_packed(qs, s.seed, spec.tid)
            device.fill_q4_scales(sc, s.seed, spec.tid)
            out[spec.name] = (qs, sc)
    return out


def prompt_ids(w: Workload, seq: int = 0, n: int | None = None) -> np.ndarray:
    n = w.prompt_len if n is None else n
    return host.uniform_ids(w.prompt_seed + seq, PROMPT_TID, n, w.shape.vocab)


def ragged_contexts(w: Workload) -> np.ndarray:
    lo, hi = w.ragged_context
    return lo + host.uniform_ids(w.context_seed, CONTEXT_TID, w.batch, hi - lo + 1)


# Keys of hy_seq_fill_synthetic's streams: K (w = 0) or V (w = 1) of
# attention layer a, kv head g, rows [0, length) row-major over [length, hd];
# the DeltaNet states of all layers as one stream [n_gdn][nh][dv][dk] at scale
# 0.01; conv rings zero.
FILL_SEED_MULT = 1000003
FILL_STATE_KEY = 977
FILL_STATE_SCALE = 0.01


def synthetic_cache(s: ModelShape, length: int, seed: int) -> dict:
    """Host copy of the cache contents hy_seq_fill_synthetic writes: ``k`` and
    ``v``, one uint16 (bf16 bits) array [nkv, length, hd] per attention layer,
    and ``state``, float32 [n_gdn, nh, dv, dk]."""
    n_attn = sum(1 for l in range(s.n_layers) if s.is_attn(l))
    n_gdn = s.n_layers - n_attn
    base = seed * FILL_SEED_MULT
    out = {"k": [], "v": []}
    for a in range(n_attn):
        for w, name in ((0, "k"), (1, "v")):
            heads = [gen.f32_to_bf16_bits(gen.fill_values(base + (a * 2 + w) * 64 + g, length * s.head_dim))
                     .reshape(length, s.head_dim) for g in range(s.attn_kv_heads)]
            out[name].append(np.stack(heads) if heads else np.zeros((0, length, s.head_dim), np.uint16))
    out["state"] = gen.fill_values(base + FILL_STATE_KEY, n_gdn * s.gdn_heads * s.gdn_dv * s.gdn_dk,
                                   FILL_STATE_SCALE).reshape(n_gdn, s.gdn_heads, s.gdn_dv, s.gdn_dk)
    return out


def param_count(s: ModelShape) -> int:
    return sum(sp.rows * sp.cols for sp in tensor_specs(s))
