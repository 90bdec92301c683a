"""Algorithmic bytes of one decode step: what the method must move per token.

A batch-1 decode step streams every weight it uses once, reads and writes the
recurrent state once, and reads the KV cache once, so its roofline is
tokens/s = bandwidth / bytes per token ("Beating llama.cpp from Scratch on
Consumer AMD", Act 6: theoretical max tok/s = memory bandwidth / model size).
MoE counts only the experts a token selects; the embedding counts one row.
"""
from __future__ import annotations

from dataclasses import dataclass

BF16 = 2
F32 = 4


@dataclass
class StepBytes:
    weights: int
    state: int
    kv_read: int
    kv_write: int
    activations: int

    @property
    def total(self) -> int:
        return self.weights + self.state + self.kv_read + self.kv_write + self.activations


def gdn_state_bytes_per_layer(nh: int, dk: int, dv: int) -> int:
    """FP32 recurrent state of one Gated DeltaNet layer."""
    return nh * dv * dk * F32


def kv_bytes_per_token(n_attn: int, nkv: int, hd: int, elem: int = BF16, kv_format: int = 0) -> int:
    """K and V of one position over all attention layers: bf16 elements, or
    int8 codes plus one FP32 scale per cached vector (kv_format 1)."""
    if kv_format == 1:
        return n_attn * 2 * nkv * (hd + F32)
    return n_attn * 2 * nkv * hd * elem


def roofline_tokens_per_s(bandwidth_gbs: float, bytes_per_token: float) -> float:
    return bandwidth_gbs * 1e9 / bytes_per_token


def linear_bytes(rows: int, cols: int, weight_format: int) -> int:
    if weight_format == 1:  # 4-bit blocks of 32: 16 bytes of nibbles + a 2-byte scale per block
        return rows * cols // 2 + rows * (cols // 32) * 2
    return rows * cols * BF16


def step_bytes(shape, context: int, experts_touched: int | None = None, logits: bool = False) -> StepBytes:
    """Bytes one decode step at position ``context`` must move.

    ``shape`` has the model-shape attributes; ``experts_touched`` (MoE) is
    the number of distinct routed experts read per layer (top_k at batch 1).
    """
    s = shape
    H = s.hidden
    fmt = getattr(s, "weight_format", 0)
    n_attn = sum(1 for l in range(s.n_layers) if s.is_attn(l))
    n_gdn = s.n_layers - n_attn
    CC = 2 * s.gdn_heads * s.gdn_dk + s.gdn_heads * s.gdn_dv
    w = 0
    w += n_gdn * (linear_bytes(CC + 2 * s.gdn_heads, H, fmt) + linear_bytes(H, s.gdn_heads * s.gdn_dv, fmt)
                  + CC * s.conv_k * BF16)
    w += n_attn * (linear_bytes((s.attn_q_heads + 2 * s.attn_kv_heads) * s.head_dim, H, fmt)
                   + linear_bytes(H, s.attn_q_heads * s.head_dim, fmt))
    w += s.n_layers * 2 * H * F32  # norm gains
    if s.ffn > 0:
        w += s.n_layers * (2 * linear_bytes(s.ffn, H, fmt) + linear_bytes(H, s.ffn, fmt))
    else:
        e = s.top_k if experts_touched is None else experts_touched
        w += s.n_layers * ((s.n_experts + 1) * H * BF16
                           + e * (2 * linear_bytes(s.expert_ffn, H, fmt) + linear_bytes(H, s.expert_ffn, fmt))
                           + 2 * linear_bytes(s.shared_ffn, H, fmt) + linear_bytes(H, s.shared_ffn, fmt))
    w += H * BF16 + H * F32 + linear_bytes(s.vocab, H, fmt)  # embedding row, final norm, LM head
    state = n_gdn * (2 * gdn_state_bytes_per_layer(s.gdn_heads, s.gdn_dk, s.gdn_dv) + s.conv_k * CC * F32)
    kvf = getattr(s, "kv_format", 0)
    kv_read = kv_bytes_per_token(n_attn, s.attn_kv_heads, s.head_dim, kv_format=kvf) * context
    kv_write = kv_bytes_per_token(n_attn, s.attn_kv_heads, s.head_dim, kv_format=kvf)
    return StepBytes(weights=w, state=state, kv_read=kv_read, kv_write=kv_write,
                     activations=s.vocab * F32 if logits else 0)


def prefill_flops(shape, n: int, t0: int = 0) -> dict:
    """FLOPs of a prompt chunk of n tokens at positions t0 .. t0+n-1: the
    linear projections (2 per weight and token; the LM head for the last token
    only), the causal attention (scores and P V: 4 nq hd per (query, key)
    pair), the DeltaNet recurrence (about 6 dk dv per head and token), and the
    tensor-core share (the projections; they run as two bf16 parts of the
    activations, so the tensor pipe executes twice their FLOPs)."""
    H = shape.hidden
    n_attn = sum(1 for l in range(shape.n_layers) if shape.is_attn(l))
    n_gdn = shape.n_layers - n_attn
    lin = n_gdn * (shape.gdn_in_rows * H + H * shape.gdn_heads * shape.gdn_dv)
    lin += n_attn * ((shape.attn_q_heads + 2 * shape.attn_kv_heads) * shape.head_dim * H +
                     H * shape.attn_q_heads * shape.head_dim)
    if shape.ffn > 0:
        lin += shape.n_layers * 3 * shape.ffn * H
    else:
        lin += shape.n_layers * ((shape.n_experts + 1) * H + (shape.top_k + 1) * 3 * shape.expert_ffn * H)
    gemm = 2.0 * lin * n
    pairs = n * t0 + n * (n + 1) / 2.0
    attn = 4.0 * n_attn * shape.attn_q_heads * shape.head_dim * pairs
    gdn = 6.0 * n_gdn * shape.gdn_heads * shape.gdn_dk * shape.gdn_dv * n
    head = 2.0 * shape.vocab * H
    return {"gemm": gemm, "attention": attn, "deltanet": gdn, "lm_head": head, "total": gemm + attn + gdn + head,
            "tensor_executed": 2 * gemm}


def expected_union(n_experts: int, top_k: int, batch: int) -> float:
    """Expected number of distinct experts `batch` tokens select when each
    picks top_k of n_experts uniformly without replacement, independently."""
    return n_experts * (1.0 - (1.0 - top_k / n_experts) ** batch)


def batch_step_bytes(shape, contexts, experts_touched: float | None = None) -> StepBytes:
    """Bytes one step over a batch of sequences at positions `contexts` must
    move: the weights once (MoE: the union of the experts the batch selects,
    by default its expectation under uniform routing), and per sequence its
    recurrent state and KV cache."""
    B = len(contexts)
    if shape.ffn == 0 and experts_touched is None:
        experts_touched = expected_union(shape.n_experts, shape.top_k, B)
    one = step_bytes(shape, 0, None if shape.ffn > 0 else int(round(experts_touched)))
    w = one.weights + (B - 1) * (shape.hidden * BF16)  # an embedding row per token
    if shape.ffn == 0:  # fractional expected union
        fmt = getattr(shape, "weight_format", 0)
        per_exp = 2 * linear_bytes(shape.expert_ffn, shape.hidden, fmt) + linear_bytes(shape.hidden, shape.expert_ffn, fmt)
        w += int(round(shape.n_layers * per_exp * (experts_touched - round(experts_touched))))
    n_attn = sum(1 for l in range(shape.n_layers) if shape.is_attn(l))
    kv1 = kv_bytes_per_token(n_attn, shape.attn_kv_heads, shape.head_dim, kv_format=getattr(shape, "kv_format", 0))
    return StepBytes(weights=w, state=B * one.state, kv_read=kv1 * int(sum(contexts)), kv_write=B * kv1,
                     activations=0)


def gemv_batch_bytes(rows: int, cols: int, batch: int, weight_format: int) -> int:
    """One batched GEMV launch: the matrix once, `batch` FP32 input vectors and
    `batch` FP32 output vectors."""
    return linear_bytes(rows, cols, weight_format) + batch * (cols + rows) * F32


def gemv_swiglu_bytes(rows: int, cols: int) -> int:
    """One gate/up SwiGLU GEMV launch: two bf16 [rows][cols] matrices, the FP32
    input vector and the FP32 output."""
    return 2 * rows * cols * BF16 + cols * F32 + rows * F32


def kernels_per_step(shape, debug: bool = False) -> int:
    """Kernel launches of one batch-1 decode step (each layer: input
    projection, mixer, output projection, 2 dense or 3 MoE FFN kernels; then
    the LM head)."""
    per = 3 + (2 if shape.ffn > 0 else 3) + (1 if debug else 0)
    return shape.n_layers * per + 1
