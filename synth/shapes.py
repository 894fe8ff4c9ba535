"""Tensor shape lists of the model families the optimizer state is sized for.

Each function returns a list of ``(name, shape, layer)`` tuples: ``shape`` is the
parameter tensor's shape (a Linear layer's weight is ``(out_features,
in_features)``), ``layer`` is the index of the packed state block the tensor
belongs to. Shapes only; no values and no optimizer arithmetic.

Sources of the shapes:
  * TinyLlama-1.1B: "Fine-tuning memory" article (community.cloudera.com profile
    page, worked configuration): 22 layers, hidden 2,048, 32 heads, 4 key-value
    heads, feed-forward 5,632, vocabulary 32,000, untied head, RMSNorm.
  * LLaMA-7B: "Transformer Training 09 - Memory" deck (calculator section):
    32 layers, h 4,096, 32 heads, SwiGLU FFN 11,008, vocabulary 32,000, untied
    head, RMSNorm; 6,738,415,616 parameters.
  * Llama-70B depth slice: h 8,192, 64 heads / 8 key-value heads, SwiGLU FFN
    28,672 (855,654,400 parameters per decoder layer).
  * LoRA rank r on Q, K, V, O, gate, up, down: same fine-tuning article (LoRA
    rank 8 on all seven projection targets, 6.3 million trainable parameters).
"""

from __future__ import annotations

from typing import List, Tuple

Shape = Tuple[int, ...]
TensorSpec = Tuple[str, Shape, int]


def decoder_layer(layer: int, hidden: int, n_heads: int, n_kv_heads: int, ffn: int,
                  prefix: str = "") -> List[TensorSpec]:
    """One pre-norm SwiGLU decoder layer: Q, K, V, O, gate, up, down, two RMSNorms."""
    head_dim = hidden // n_heads
    kv = n_kv_heads * head_dim
    p = prefix or f"layers.{layer}."
    return [
        (p + "q_proj", (hidden, hidden), layer),
        (p + "k_proj", (kv, hidden), layer),
        (p + "v_proj", (kv, hidden), layer),
        (p + "o_proj", (hidden, hidden), layer),
        (p + "gate_proj", (ffn, hidden), layer),
        (p + "up_proj", (ffn, hidden), layer),
        (p + "down_proj", (hidden, ffn), layer),
        (p + "input_norm", (hidden,), layer),
        (p + "post_attn_norm", (hidden,), layer),
    ]


TINYLLAMA = dict(hidden=2048, n_heads=32, n_kv_heads=4, ffn=5632, vocab=32000, n_layers=22)
LLAMA7B = dict(hidden=4096, n_heads=32, n_kv_heads=32, ffn=11008, vocab=32000, n_layers=32)
LLAMA70B = dict(hidden=8192, n_heads=64, n_kv_heads=8, ffn=28672, vocab=32000, n_layers=80)


def _dec(cfg: dict, layer: int) -> List[TensorSpec]:
    return decoder_layer(layer, cfg["hidden"], cfg["n_heads"], cfg["n_kv_heads"], cfg["ffn"],
                         prefix=f"layers.{layer}.")


def tinyllama_layer() -> List[TensorSpec]:
    """A single TinyLlama-1.1B decoder layer as one block (44,044,288 parameters)."""
    return _dec(TINYLLAMA, 0)


def full_model(cfg: dict, n_layers: int | None = None) -> List[TensorSpec]:
    """Embedding block, one block per decoder layer, then final norm + untied head."""
    L = cfg["n_layers"] if n_layers is None else n_layers
    h, V = cfg["hidden"], cfg["vocab"]
    out: List[TensorSpec] = [("embed_tokens", (V, h), 0)]
    for i in range(L):
        out += [(n, s, i + 1) for (n, s, _) in _dec(cfg, i)]
    out += [("final_norm", (h,), L + 1), ("lm_head", (V, h), L + 1)]
    return out


def tinyllama_full() -> List[TensorSpec]:
    """TinyLlama-1.1B: 24 blocks, 1,100,048,384 parameters."""
    return full_model(TINYLLAMA)


def llama7b() -> List[TensorSpec]:
    """LLaMA-7B: 34 blocks, 6,738,415,616 parameters."""
    return full_model(LLAMA7B)


def llama70b_slice(n_layers: int = 8) -> List[TensorSpec]:
    """A depth slice of Llama-70B: n_layers decoder layers, one block each."""
    return [s for i in range(n_layers) for s in _dec(LLAMA70B, i)]


LORA_TARGETS = ("q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj")


def lora(cfg: dict, rank: int = 8) -> List[TensorSpec]:
    """LoRA adapters on the seven projections of every layer, one block per layer.

    Each target weight (out, in) gets A of shape (rank, in) and B of shape
    (out, rank); the frozen base weights are not part of the optimizer state.
    """
    out: List[TensorSpec] = []
    for i in range(cfg["n_layers"]):
        for (n, s, _) in _dec(cfg, i):
            base = n.rsplit(".", 1)[1]
            if base not in LORA_TARGETS:
                continue
            o, k = s
            out.append((n + ".lora_A", (rank, k), i))
            out.append((n + ".lora_B", (o, rank), i))
    return out


def tinyllama_lora(rank: int = 8) -> List[TensorSpec]:
    """TinyLlama-1.1B LoRA r=8: 22 blocks x 14 tensors, 6,307,840 parameters."""
    return lora(TINYLLAMA, rank)


def numel(shape: Shape) -> int:
    n = 1
    for d in shape:
        n *= int(d)
    return n


def total_params(specs: List[TensorSpec]) -> int:
    return sum(numel(s) for (_, s, _) in specs)


def n_blocks(specs: List[TensorSpec]) -> int:
    return 1 + max(l for (_, _, l) in specs) if specs else 0


WORKLOADS = {
    # name: (shape function, format name)
    "tinyllama_layer_l12": (tinyllama_layer, "L12"),
    "tinyllama_full_l16m": (tinyllama_full, "L16M"),
    "tinyllama_lora_l16f": (tinyllama_lora, "L16F"),
    "llama7b_l12": (llama7b, "L12"),
    "llama70b_slice8_l12": (llama70b_slice, "L12"),
}
