"""Seeded synthetic inputs for the k-quant decode GEMV workloads.

This module is the one thing the oracle side (tests, oracle/) and the library
side (bench.py, smoke) share: it only draws random bytes and floats and lays
them out as GGUF blocks.  It holds none of the method's arithmetic (no
dequantisation, no quantisation, no dot products).

Distributions (the synthetic stand-in for real Qwen2.5 GGUF weights):
  q6_K: ql, qh uniform bytes; the 16 int8 sub-block scales uniform in
        [-32, 31]; d = fp16(uniform[1e-4, 1e-3]).
  q4_K: d, dmin = fp16(uniform[1e-4, 1e-3]); the 12 packed scale bytes and
        the 128 nibble bytes uniform.
  activations: f32 N(0, 1); rms gain N(1, 0.1); eps 1e-6.
Every tensor has its own numpy PCG64 stream seeded from (workload, tensor
name), so both sides see identical bytes on any machine.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import numpy as np

Q6K_BYTES = 210
Q4K_BYTES = 144
Q5K_BYTES = 176
QK = 256


def rng(*key) -> np.random.Generator:
    h = hashlib.sha256("/".join(str(k) for k in key).encode()).digest()
    return np.random.Generator(np.random.PCG64(int.from_bytes(h[:8], "little")))


def _f16_bits(vals: np.ndarray) -> np.ndarray:
    return vals.astype(np.float16).view(np.uint16)


def q6k_blocks(g: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """GGUF q6_K rows: (rows, cols/256*210) uint8, blocks [ql 128|qh 64|sc 16|d 2]."""
    assert cols % QK == 0
    nblk = rows * (cols // QK)
    out = np.empty((nblk, Q6K_BYTES), np.uint8)
    out[:, :192] = g.integers(0, 256, size=(nblk, 192), dtype=np.uint8)
    out[:, 192:208] = g.integers(-32, 32, size=(nblk, 16), dtype=np.int8).view(np.uint8)
    d = _f16_bits(g.uniform(1e-4, 1e-3, size=nblk))
    out[:, 208] = d & 0xFF
    out[:, 209] = d >> 8
    return out.reshape(rows, -1)


def q4k_blocks(g: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """GGUF q4_K rows: (rows, cols/256*144) uint8, blocks [d 2|dmin 2|scales 12|qs 128]."""
    assert cols % QK == 0
    nblk = rows * (cols // QK)
    out = np.empty((nblk, Q4K_BYTES), np.uint8)
    d = _f16_bits(g.uniform(1e-4, 1e-3, size=nblk))
    dm = _f16_bits(g.uniform(1e-4, 1e-3, size=nblk))
    out[:, 0] = d & 0xFF
    out[:, 1] = d >> 8
    out[:, 2] = dm & 0xFF
    out[:, 3] = dm >> 8
    out[:, 4:] = g.integers(0, 256, size=(nblk, 140), dtype=np.uint8)
    return out.reshape(rows, -1)


def q5k_blocks(g: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    """GGUF q5_K rows: (rows, cols/256*176) uint8, blocks
    [d 2|dmin 2|scales 12|qh 32|qs 128]; d, dmin uniform in [1e-4, 1e-3],
    every other byte uniform."""
    assert cols % QK == 0
    nblk = rows * (cols // QK)
    out = np.empty((nblk, Q5K_BYTES), np.uint8)
    d = _f16_bits(g.uniform(1e-4, 1e-3, size=nblk))
    dm = _f16_bits(g.uniform(1e-4, 1e-3, size=nblk))
    out[:, 0] = d & 0xFF
    out[:, 1] = d >> 8
    out[:, 2] = dm & 0xFF
    out[:, 3] = dm >> 8
    out[:, 4:] = g.integers(0, 256, size=(nblk, Q5K_BYTES - 4), dtype=np.uint8)
    return out.reshape(rows, -1)


def blocks(fmt: str, g: np.random.Generator, rows: int, cols: int) -> np.ndarray:
    return {"q6k": q6k_blocks, "q4k": q4k_blocks, "q5k": q5k_blocks}[fmt](g, rows, cols)


def normal(g: np.random.Generator, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    return (g.standard_normal(n) * std + mean).astype(np.float32)


# --------------------------------------------------------------------------
# The named workloads.  A GEMV entry is (name, fmt, rows, cols, producer),
# producer in {"quantize", "rms", "swiglu"}: the op that makes its q8 input.
# --------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    gemvs: list = field(default_factory=list)

    def weight_bytes(self) -> int:
        return sum(rows * (cols // QK) * {"q6k": Q6K_BYTES, "q4k": Q4K_BYTES, "q5k": Q5K_BYTES}[fmt]
                   for _, fmt, rows, cols, _ in self.gemvs)


HIDDEN_14B, INTER_14B, KV_14B, VOCAB = 5120, 13824, 1024, 152064


def _sweep_14b(layers: int = 48) -> list:
    g = []
    for i in range(layers):
        g += [(f"blk{i}.attn_q", "q4k", HIDDEN_14B, HIDDEN_14B, "rms"),
              (f"blk{i}.attn_k", "q4k", KV_14B, HIDDEN_14B, "rms"),
              (f"blk{i}.attn_v", "q6k", KV_14B, HIDDEN_14B, "rms"),
              (f"blk{i}.attn_output", "q4k", HIDDEN_14B, HIDDEN_14B, "quantize"),
              (f"blk{i}.ffn_gate", "q4k", INTER_14B, HIDDEN_14B, "rms"),
              (f"blk{i}.ffn_up", "q4k", INTER_14B, HIDDEN_14B, "rms"),
              (f"blk{i}.ffn_down", "q6k", HIDDEN_14B, INTER_14B, "swiglu")]
    g.append(("output", "q6k", VOCAB, HIDDEN_14B, "rms"))
    return g


WORKLOADS = {
    # one q6_K x q8 GEMV, x -> standalone quantize
    "q6k_512x2048": Workload("q6k_512x2048", [("w", "q6k", 512, 2048, "quantize")]),
    # Qwen2.5-7B ffn_down: tall rows (74 super-blocks), fed by swiglu -> q8
    "ffn_down_7b": Workload("ffn_down_7b", [("ffn_down", "q6k", 3584, 18944, "swiglu")]),
    # Qwen2.5-14B attn_v and ffn_down, each fed by rms_norm -> q8
    "layer_14b": Workload("layer_14b", [("attn_v", "q6k", KV_14B, HIDDEN_14B, "rms"),
                                        ("ffn_down", "q6k", HIDDEN_14B, INTER_14B, "rms")]),
    # the shapes of the pages' MMVQ-vs-f32 crossover (the D3 page, §2.3):
    # 14B attn_v alone, and 2048 x 4864
    "attn_v_14b": Workload("attn_v_14b", [("attn_v", "q6k", KV_14B, HIDDEN_14B, "rms")]),
    "q6k_2048x4864": Workload("q6k_2048x4864", [("w", "q6k", 2048, 4864, "quantize")]),
    # the q5_K sibling class on the 14B ffn_down shape
    "ffn_down_14b_q5k": Workload("ffn_down_14b_q5k", [("ffn_down", "q5k", HIDDEN_14B, INTER_14B, "rms")]),
    # the 152064 x 5120 q6_K output head, fed by rms_norm -> q8
    "lm_head_14b": Workload("lm_head_14b", [("output", "q6k", VOCAB, HIDDEN_14B, "rms")]),
    # the FFN half of a Qwen2.5-14B layer: rms_norm -> q8 -> gate, up (q4_K)
    # -> SwiGLU -> q8 -> down (q6_K)
    "ffn_14b": Workload("ffn_14b", [("ffn_gate", "q4k", INTER_14B, HIDDEN_14B, "rms"),
                                    ("ffn_up", "q4k", INTER_14B, HIDDEN_14B, "rms"),
                                    ("ffn_down", "q6k", HIDDEN_14B, INTER_14B, "swiglu")]),
    # single launches of the sweep's q4_K shapes: attn_q (and attn_output)
    # 5120 x 5120, ffn_gate (and ffn_up) 13824 x 5120, and the q, k, v
    # matrices of a layer grouped in one launch over one rms_norm -> q8 plane
    "attn_q_14b": Workload("attn_q_14b", [("attn_q", "q4k", HIDDEN_14B, HIDDEN_14B, "rms")]),
    "ffn_gate_14b": Workload("ffn_gate_14b", [("ffn_gate", "q4k", INTER_14B, HIDDEN_14B, "rms")]),
    "attn_qkv_14b": Workload("attn_qkv_14b", [("attn_q", "q4k", HIDDEN_14B, HIDDEN_14B, "rms"),
                                              ("attn_k", "q4k", KV_14B, HIDDEN_14B, "rms"),
                                              ("attn_v", "q6k", KV_14B, HIDDEN_14B, "rms")]),
    # full 48-layer 14B decode weight sweep plus the head
    "sweep_14b": Workload("sweep_14b", _sweep_14b()),
}
