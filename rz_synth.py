"""Seeded synthetic inputs for the Q4_K x Q8_1 decode path.

This module generates bytes and floats only.  It holds none of the method's
arithmetic: no dequantisation, no quantisation, no scale/min packing.  A Q4_K
super-block is 144 bytes whose first two fp16 fields (d, dmin) are drawn from
U[1e-3, 1e-2] and whose remaining 140 bytes are uniform random.  Uniform random
bytes in the 12-byte scale area give every packed 6-bit scale and min the
distribution U{0..63} (the 96 bits hold exactly eight 6-bit scales and eight
6-bit mins), and uniform random bytes in the 128-byte quant area give every
4-bit quant U{0..15}.  Q4_0 blocks likewise: fp16 d ~ U[1e-3, 1e-2] and 16
uniform random bytes (nibbles U{0..15}).

Both the oracle side and the GPU side of every test and benchmark draw their
inputs from here, so the two see identical bytes.

Workload shapes (one decode token unless stated):
  GEMV_SMALL     Q4_K x Q8_1 GEMV 256 x 1024 (4 super-blocks per row).
  QWEN2_LAYER    Qwen2-0.5B-shaped layer: hidden 896 (padded to 1024 for the
                 GEMVs), intermediate 4864, 14 heads / 2 KV heads, head_dim 64,
                 RoPE theta 1e6 (half-split pairs), eps 1e-6, position 127.
  LLAMA_SWEEP    (out, in) = (4096,4096) (11008,4096) (4096,11008)
                 (14336,4096) (4096,14336).
  LM_HEADS       Q4_0 LM heads 151936 x 896 and 32000 x 4096.
  LLAMA_STACK    32 Llama-7B-shaped layers: hidden 4096, intermediate 11008,
                 32 / 32 heads, head_dim 128, RoPE theta 1e4 (adjacent pairs),
                 Q4_0 LM head 32000 x 4096, batches M in {1,4,8,16},
                 positions in {1,128,512,1024,2048}, KV cache prefilled N(0,1).
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass, field

import numpy as np

Q4K_BYTES = 144   # bytes of one 256-weight super-block
Q4_0_BYTES = 18   # bytes of one 32-weight block
SEED = 0x5EED


def rng(name: str, seed: int = SEED) -> np.random.Generator:
    """Independent stream per named tensor."""
    return np.random.default_rng([seed, zlib.crc32(name.encode())])


def pad256(n: int) -> int:
    return (n + 255) // 256 * 256


def _fp16_uniform(g: np.random.Generator, n: int, lo=1e-3, hi=1e-2) -> np.ndarray:
    return g.uniform(lo, hi, size=n).astype(np.float16).view(np.uint16)


def q4k_weight(name: str, out_dim: int, in_dim: int, seed: int = SEED) -> np.ndarray:
    """uint8 [out_dim, in_dim/256*144]: random Q4_K super-blocks, row-major."""
    assert in_dim % 256 == 0
    g = rng(name, seed)
    nsb = out_dim * (in_dim // 256)
    blk = np.frombuffer(g.bytes(nsb * Q4K_BYTES), np.uint8).reshape(nsb, Q4K_BYTES).copy()
    d = _fp16_uniform(g, nsb)
    dmin = _fp16_uniform(g, nsb)
    blk[:, 0:2] = d.view(np.uint8).reshape(nsb, 2)
    blk[:, 2:4] = dmin.view(np.uint8).reshape(nsb, 2)
    return blk.reshape(out_dim, (in_dim // 256) * Q4K_BYTES)


def q4_0_weight(name: str, out_dim: int, in_dim: int, seed: int = SEED) -> np.ndarray:
    """uint8 [out_dim, in_dim/32*18]: random Q4_0 blocks, row-major."""
    assert in_dim % 32 == 0
    g = rng(name, seed)
    nb = out_dim * (in_dim // 32)
    blk = np.frombuffer(g.bytes(nb * Q4_0_BYTES), np.uint8).reshape(nb, Q4_0_BYTES).copy()
    blk[:, 0:2] = _fp16_uniform(g, nb).view(np.uint8).reshape(nb, 2)
    return blk.reshape(out_dim, (in_dim // 32) * Q4_0_BYTES)


def normal(name: str, shape, seed: int = SEED) -> np.ndarray:
    return rng(name, seed).standard_normal(size=shape, dtype=np.float32)


def uniform(name: str, shape, lo: float, hi: float, seed: int = SEED) -> np.ndarray:
    return rng(name, seed).uniform(lo, hi, size=shape).astype(np.float32)


def hidden_input(name: str, m: int, hidden: int, hidden_pad: int, seed: int = SEED) -> np.ndarray:
    """float32 [m, hidden_pad]: N(0,1) in the first `hidden` columns, zeros after."""
    x = np.zeros((m, hidden_pad), np.float32)
    x[:, :hidden] = normal(name, (m, hidden), seed)
    return x


@dataclass(frozen=True)
class LayerShape:
    hidden: int
    inter: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    rope_theta: float
    rope_mode: int          # 0 adjacent pairs, 1 half-split pairs
    eps: float = 1e-6

    @property
    def hidden_pad(self) -> int:
        return pad256(self.hidden)

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def q_pad(self) -> int:
        return pad256(self.q_dim)

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def weight_shapes(self):
        """name -> (out_dim, in_dim) of the seven Q4_K matrices."""
        hp = self.hidden_pad
        return {
            "wq": (self.q_dim, hp), "wk": (self.kv_dim, hp), "wv": (self.kv_dim, hp),
            "wo": (self.hidden, self.q_pad),
            "wgate": (self.inter, hp), "wup": (self.inter, hp),
            "wdown": (self.hidden, self.inter),
        }

    def weight_bytes(self) -> int:
        return sum(o * (i // 256) * Q4K_BYTES for o, i in self.weight_shapes().values())


QWEN2 = LayerShape(hidden=896, inter=4864, n_heads=14, n_kv_heads=2, head_dim=64,
                   rope_theta=1e6, rope_mode=1)
LLAMA7B = LayerShape(hidden=4096, inter=11008, n_heads=32, n_kv_heads=32, head_dim=128,
                     rope_theta=1e4, rope_mode=0)

GEMV_SMALL = (256, 1024)
LLAMA_SWEEP = [(4096, 4096), (11008, 4096), (4096, 11008), (14336, 4096), (4096, 14336)]
LM_HEADS = [(151936, 896), (32000, 4096)]
LLAMA_VOCAB = 32000
LLAMA_LAYERS = 32
STACK_BATCHES = (1, 4, 8, 16)
STACK_POSITIONS = (1, 128, 512, 1024, 2048)
LLAMA_MAX_SEQ = 2056


@dataclass
class HostLayer:
    """Host (numpy) tensors of one layer."""
    shape: LayerShape
    w: dict = field(default_factory=dict)   # name -> uint8 Q4_K blocks
    attn_gamma: np.ndarray = None
    ffn_gamma: np.ndarray = None


def layer(shape: LayerShape, tag: str, seed: int = SEED) -> HostLayer:
    """Random layer: Q4_K matrices as above, gammas ~ U[0.5, 1.5]."""
    L = HostLayer(shape)
    for nm, (o, i) in shape.weight_shapes().items():
        L.w[nm] = q4k_weight(f"{tag}.{nm}", o, i, seed)
    L.attn_gamma = uniform(f"{tag}.attn_gamma", shape.hidden, 0.5, 1.5, seed)
    L.ffn_gamma = uniform(f"{tag}.ffn_gamma", shape.hidden, 0.5, 1.5, seed)
    return L


def kv_prefill(shape: LayerShape, tag: str, max_seq: int, filled: int, m: int = 1,
               seed: int = SEED):
    """float32 K and V caches [m, max_seq, kv_dim]; rows < filled ~ N(0,1), rest 0.
    The filled rows stand in for earlier tokens' post-RoPE keys and values."""
    k = np.zeros((m, max_seq, shape.kv_dim), np.float32)
    v = np.zeros((m, max_seq, shape.kv_dim), np.float32)
    if filled > 0:
        k[:, :filled] = normal(f"{tag}.k", (m, filled, shape.kv_dim), seed)
        v[:, :filled] = normal(f"{tag}.v", (m, filled, shape.kv_dim), seed)
    return k, v


# ----------------------------------------------------------------------------- device-side
# The same distributions drawn with torch's generator directly in device memory,
# for workloads too large to generate on the host (the 32-layer stack and its KV
# caches).  Used by the benchmark; the parity tests use the host generators above.
def torch_gen(name: str, device, seed: int = SEED):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((seed << 32) ^ zlib.crc32(name.encode()))
    return g


def q4k_weight_device(name: str, out_dim: int, in_dim: int, device, seed: int = SEED):
    import torch
    g = torch_gen(name, device, seed)
    nsb = out_dim * (in_dim // 256)
    blk = torch.randint(0, 256, (nsb, Q4K_BYTES), dtype=torch.uint8, device=device, generator=g)
    dd = (torch.rand((nsb, 2), device=device, generator=g) * 9e-3 + 1e-3).to(torch.float16)
    blk[:, 0:4] = dd.view(torch.uint8).view(nsb, 4)
    return blk.view(out_dim, (in_dim // 256) * Q4K_BYTES)


def q4_0_weight_device(name: str, out_dim: int, in_dim: int, device, seed: int = SEED):
    import torch
    g = torch_gen(name, device, seed)
    nb = out_dim * (in_dim // 32)
    blk = torch.randint(0, 256, (nb, Q4_0_BYTES), dtype=torch.uint8, device=device, generator=g)
    d = (torch.rand((nb, 1), device=device, generator=g) * 9e-3 + 1e-3).to(torch.float16)
    blk[:, 0:2] = d.view(torch.uint8).view(nb, 2)
    return blk.view(out_dim, (in_dim // 32) * Q4_0_BYTES)


def layer_device(shape: LayerShape, tag: str, device, seed: int = SEED) -> dict:
    import torch
    out = {nm: q4k_weight_device(f"{tag}.{nm}", o, i, device, seed)
           for nm, (o, i) in shape.weight_shapes().items()}
    for nm in ("attn_gamma", "ffn_gamma"):
        g = torch_gen(f"{tag}.{nm}", device, seed)
        out[nm] = torch.rand(shape.hidden, device=device, generator=g) + 0.5
    return out


def kv_prefill_device(shape: LayerShape, tag: str, max_seq: int, filled: int, m: int, device,
                      seed: int = SEED):
    import torch
    k = torch.zeros((m, max_seq, shape.kv_dim), dtype=torch.float32, device=device)
    v = torch.zeros_like(k)
    if filled > 0:
        k[:, :filled] = torch.randn((m, filled, shape.kv_dim), device=device,
                                    generator=torch_gen(f"{tag}.k", device, seed))
        v[:, :filled] = torch.randn((m, filled, shape.kv_dim), device=device,
                                    generator=torch_gen(f"{tag}.v", device, seed))
    return k, v


# ----------------------------------------------------------------------------- Q4_0 whole-model layer
@dataclass(frozen=True)
class Q40Shape:
    """A layer whose projections are all Q4_0 (f32 activations): fused QKV, O,
    gate (SwiGLU) or none (GELU FFN), up, down."""
    hidden: int
    inter: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    rope_theta: float
    rope_mode: int
    gated: bool
    eps: float = 1e-6

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def weight_shapes(self):
        s = {"wqkv": (self.q_dim + 2 * self.kv_dim, self.hidden), "wo": (self.hidden, self.q_dim),
             "wup": (self.inter, self.hidden), "wdown": (self.hidden, self.inter)}
        if self.gated:
            s["wgate"] = (self.inter, self.hidden)
        return s


# a phi-2-sized GELU layer (hidden 2560, intermediate 10240; 40 heads of 64, the
# attention kernels taking head dimensions that are multiples of 32) and a
# TinyLlama-sized SwiGLU layer with grouped KV heads
Q40_GELU = Q40Shape(hidden=2560, inter=10240, n_heads=40, n_kv_heads=40, head_dim=64,
                    rope_theta=1e4, rope_mode=1, gated=False)
Q40_SWIGLU = Q40Shape(hidden=2048, inter=5632, n_heads=32, n_kv_heads=4, head_dim=64,
                      rope_theta=1e4, rope_mode=0, gated=True)


def layer_q4_0(shape: Q40Shape, tag: str, seed: int = SEED) -> dict:
    """Random Q4_0 layer: matrices as q4_0_weight, gammas ~ U[0.5, 1.5]."""
    out = {nm: q4_0_weight(f"{tag}.{nm}", o, i, seed) for nm, (o, i) in shape.weight_shapes().items()}
    out["attn_gamma"] = uniform(f"{tag}.attn_gamma", shape.hidden, 0.5, 1.5, seed)
    out["ffn_gamma"] = uniform(f"{tag}.ffn_gamma", shape.hidden, 0.5, 1.5, seed)
    return out
