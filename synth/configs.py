"""Model shapes and workloads of the decode benchmarks (inputs only).

Each entry is a Llama-style decoder shape plus the synthetic workload run on
it.  The shapes are the ones the megakernel pages talk about: an ~8B model
with 16 GB of bf16 weights decoding a 39-token prompt for 512 tokens (MPK's
single-A100 measurement, "Compilar LLM en un MegaKernel…", section "Valor
central de MPK"), a Llama-1B-shaped low-latency model and a Llama-70B-shaped
large-batch model (the Hazy megakernels, "Llama-70B 向け…megakernel",
sections 概要 and 低レイテンシMegakernelの振り返り), plus a tiny decoder for
exhaustive parity.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class ModelCfg:
    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 5e5
    tied_embeddings: bool = False
    weight_std: float = 0.02
    random_gains: bool = False  # norm gains 1 + N(0, 0.1) instead of 1


@dataclass(frozen=True)
class Workload:
    model: ModelCfg
    batch: int
    prompt_len: int  # tokens before the first decode step
    decode_steps: int
    page_size: int = 64
    seed: int = 0
    # extra positions kept in the cache beyond prompt + decode steps
    max_seq: int = 0
    batch_sweep: tuple = field(default_factory=tuple)

    @property
    def seq_capacity(self) -> int:
        need = self.prompt_len + self.decode_steps + 8
        cap = max(self.max_seq, need)
        return (cap + self.page_size - 1) // self.page_size * self.page_size


TINY = ModelCfg("tiny", 2, 256, 4, 2, 64, 688, 1024, rope_theta=1e4)
# tiny variants covering the other GQA group sizes (8 q heads per kv head as
# in the 70B shape, and plain multi-head attention) and head_dim 128
TINY_G8 = ModelCfg("tiny-g8", 2, 256, 16, 2, 64, 688, 1024, rope_theta=1e4)
TINY_MHA = ModelCfg("tiny-mha", 2, 256, 4, 4, 64, 688, 1024, rope_theta=1e4)
TINY_D128 = ModelCfg("tiny-d128", 2, 512, 8, 2, 128, 1376, 1024, rope_theta=1e4)
# tiny variants whose batch-1 matvec inputs are longer than the 4096 columns
# kept in registers: a wide hidden size (QKV, gate/up and LM-head inputs of
# 4608 columns, the last 2048-column piece ragged) and a wide feed-forward
# (down-projection input of 5000 columns)
# (weights N(0, 0.01): with 0.02 the wide q and k make the softmax sharp
# enough that rounding the cache to bf16 alone moves the logits by up to
# 2.9e-2 against the fp64 oracle, at the edge of the tolerance)
TINY_WIDE = ModelCfg("tiny-wide", 2, 4608, 4, 2, 128, 688, 1024, rope_theta=1e4, weight_std=0.01)
TINY_LONGFF = ModelCfg("tiny-longff", 2, 256, 4, 2, 64, 5000, 1024, rope_theta=1e4)
# a feed-forward width that is a multiple of 2048: the batch-1 down projection
# then fills each ring slot with one 3-D TMA copy instead of one copy per row
TINY_FFN6K = ModelCfg("tiny-ffn6144", 2, 256, 4, 2, 64, 6144, 1024, rope_theta=1e4)
LLAMA_1B = ModelCfg("llama-3.2-1b-shaped", 16, 2048, 32, 8, 64, 8192, 128256, rope_theta=5e5, tied_embeddings=True)
LLAMA_8B = ModelCfg("llama-3-8b-shaped", 32, 4096, 32, 8, 128, 14336, 128256, rope_theta=5e5)
LLAMA_70B = ModelCfg("llama-70b-shaped", 80, 8192, 64, 8, 128, 28672, 128256, rope_theta=5e5)

WORKLOADS = {
    "tiny": Workload(TINY, batch=1, prompt_len=32, decode_steps=16),
    "1b": Workload(LLAMA_1B, batch=1, prompt_len=512, decode_steps=128),
    "8b": Workload(LLAMA_8B, batch=1, prompt_len=39, decode_steps=512),
    "8b-batch": Workload(LLAMA_8B, batch=1, prompt_len=4096, decode_steps=64, batch_sweep=(1, 8, 32, 64)),
    "70b": Workload(LLAMA_70B, batch=16, prompt_len=2048, decode_steps=32),
}


def with_random_gains(m: ModelCfg) -> ModelCfg:
    return replace(m, random_gains=True, name=m.name + "+gains")


# Tensor ids of the seeded generator (any distinct 64-bit values would do).
TID_EMBED = 1
TID_LM_HEAD = 2
TID_FINAL_NORM = 3
LAYER_TIDS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down")


def layer_tid(layer: int, name: str) -> int:
    return 16 + layer * 16 + LAYER_TIDS.index(name)


def kv_tid(layer: int, which: str) -> int:
    return (1 << 20) + layer * 2 + (0 if which == "k" else 1)


def token_tid(seq: int) -> int:
    return (1 << 24) + seq


def layer_shapes(m: ModelCfg) -> dict:
    H, d, I = m.hidden, m.head_dim, m.ffn_dim
    return {
        "attn_norm": (H,),
        "wq": (m.n_q_heads * d, H),
        "wk": (m.n_kv_heads * d, H),
        "wv": (m.n_kv_heads * d, H),
        "wo": (H, m.n_q_heads * d),
        "mlp_norm": (H,),
        "w_gate": (I, H),
        "w_up": (I, H),
        "w_down": (H, I),
    }


def weight_bytes(m: ModelCfg) -> int:
    """bf16 bytes of every weight tensor (embedding counted once when tied)."""
    per_layer = sum(_numel(s) for s in layer_shapes(m).values())
    emb = m.vocab * m.hidden
    total = m.n_layers * per_layer + emb + m.hidden + (0 if m.tied_embeddings else emb)
    return 2 * total


def _numel(shape) -> int:
    n = 1
    for s in shape:
        n *= s
    return n
