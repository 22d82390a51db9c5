"""Seeded synthetic inputs for frozen-prefix chunk attention.

This module only draws random numbers and lays them out in memory.  It holds
none of the attention arithmetic, so both the CUDA path and the fp64 oracle can
take their inputs from it without sharing any of the method.

Workloads (shapes from the pages' windows):

* ``tiny``   -- batch 1, Hq=2, Hkv=1, d=64, Lp=256, Lc=64, dO ~ N(0,1).
* ``qwen3_1p7b`` -- one Qwen3-1.7B-shaped layer: Hq=16, Hkv=8, d=128,
  Lp=1536, Lc=512 (the 2048-token microbench length of the prime-rl
  stop-gradient POC, "Measured").
* ``qwen3_8b`` -- one Qwen3-8B-shaped layer: Hq=32, Hkv=8, d=128,
  Lp=16128, Lc=256 (a 16k window, as on the "Training Large Context Models On
  Low VRAM" summary, trained in one 256-row chunk).
* ``window_63k_q8`` -- the 63k-token window of the llama.cpp walk ("train: walk
  the window"): Lp=62976, Lc=512, prefix K/V stored as q8_0.
* ``varlen8`` -- eight windows packed through ``cu_seqlens``; each prefix
  length is drawn uniformly from [1024, 32768], every chunk has 256 rows.

Draw order (all from one ``torch.Generator`` seeded with ``seed``): for the
varlen workload the eight prefix lengths first, then q, k_prefix, v_prefix,
k_chunk, v_chunk, dO.  Values are drawn in fp32 and rounded to bf16 (RNE).
q8_0 prefixes are drawn as fp32 N(0,1) values and then encoded.

q8_0 encoding (the llama.cpp cache type the walk trains against): a block is
32 consecutive values along head_dim stored as 34 bytes -- a little-endian
fp16 scale ``d`` followed by 32 int8 codes.  The encoder takes
``d32 = absmax / 127`` in fp32, ``q = round_half_away(x / d32)`` clamped to
[-127, 127], and stores ``fp16(d32)`` (RNE).  An all-zero block gets d=0, q=0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

Q8_0_BLOCK = 32          # values per q8_0 block
Q8_0_BYTES = 34          # fp16 scale + 32 int8 codes

PREFIX_BF16 = 0
PREFIX_Q8_0 = 1
PREFIX_F16 = 2


@dataclass
class Workload:
    name: str
    hq: int
    hkv: int
    head_dim: int
    lp: list            # prefix length per window
    lc: list            # chunk length per window
    prefix_dtype: int = PREFIX_BF16
    dout_std: float = 0.1
    seed: int = 0
    softmax_scale: float = field(default=0.0)
    shape_seed: int = None   # seed the varlen window lengths were drawn with (default: seed)

    def __post_init__(self):
        if not self.softmax_scale:
            self.softmax_scale = 1.0 / math.sqrt(self.head_dim)

    @property
    def batch(self) -> int:
        return len(self.lc)


def _varlen_lp(seed: int, n: int = 8) -> list:
    g = torch.Generator().manual_seed(seed)
    return torch.randint(1024, 32769, (n,), generator=g).tolist()


def workload(name: str, seed: int = 0, shape_seed: int = None) -> Workload:
    """The named workload, with its shapes and input distributions.  ``seed``
    seeds the values; ``shape_seed`` (default ``seed``) the varlen window
    lengths, so replicas with different values can share one shape."""
    ss = seed if shape_seed is None else shape_seed
    if name == "tiny":
        return Workload(name, 2, 1, 64, [256], [64], dout_std=1.0, seed=seed)
    if name == "qwen3_1p7b":
        return Workload(name, 16, 8, 128, [1536], [512], seed=seed)
    if name == "qwen3_8b":
        return Workload(name, 32, 8, 128, [16128], [256], seed=seed)
    if name == "window_63k_q8":
        return Workload(name, 32, 8, 128, [62976], [512], prefix_dtype=PREFIX_Q8_0, seed=seed)
    if name == "varlen8":
        return Workload(name, 32, 8, 128, _varlen_lp(ss), [256] * 8, seed=seed, shape_seed=ss)
    raise KeyError(name)


WORKLOADS = ("tiny", "qwen3_1p7b", "qwen3_8b", "window_63k_q8", "varlen8")


def custom(hq, hkv, head_dim, lp, lc, prefix_dtype=PREFIX_BF16, dout_std=1.0,
           seed=0, softmax_scale=0.0, name="custom") -> Workload:
    """A workload with explicit per-window lengths (edge and ragged cases)."""
    return Workload(name, hq, hkv, head_dim, list(lp), list(lc), prefix_dtype,
                    dout_std, seed, softmax_scale)


def cu_seqlens(lengths) -> torch.Tensor:
    out = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    out[1:] = torch.tensor(lengths, dtype=torch.int64).cumsum(0).to(torch.int32)
    return out


def encode_q8_0(x: torch.Tensor) -> torch.Tensor:
    """Encode fp32 values ``[..., d]`` (d a multiple of 32) as q8_0 bytes
    ``[..., d/32 * 34]`` (uint8)."""
    assert x.dtype == torch.float32 and x.shape[-1] % Q8_0_BLOCK == 0
    lead = x.shape[:-1]
    nb = x.shape[-1] // Q8_0_BLOCK
    v = x.reshape(-1, Q8_0_BLOCK).numpy()
    absmax = np.abs(v).max(axis=1).astype(np.float32)
    d32 = (absmax / np.float32(127.0)).astype(np.float32)
    safe = np.where(d32 == 0, np.float32(1.0), d32).astype(np.float32)
    r = (v / safe[:, None]).astype(np.float32)
    # round half away from zero, exactly (|r| + 0.5 in float64 cannot round)
    ra = np.abs(r).astype(np.float64)
    q = np.sign(r) * np.floor(ra + 0.5)
    q = np.clip(q, -127, 127)
    q = np.where(d32[:, None] == 0, 0, q).astype(np.int8)
    d16 = d32.astype(np.float16)                      # RNE
    blocks = np.empty((v.shape[0], Q8_0_BYTES), dtype=np.uint8)
    blocks[:, 0:2] = d16.view(np.uint8).reshape(-1, 2)  # little-endian fp16
    blocks[:, 2:] = q.view(np.uint8)
    return torch.from_numpy(blocks.reshape(*lead, nb * Q8_0_BYTES))


def make_inputs(w: Workload) -> dict:
    """Draw every input of one fwd+bwd step on the host (CPU tensors).

    Returns a dict with q, k_prefix, v_prefix, k_chunk, v_chunk, dout,
    cu_seqlens_prefix, cu_seqlens_chunk and the workload itself.
    """
    g = torch.Generator().manual_seed(w.seed)
    if w.name == "varlen8":
        # the eight prefix lengths are the first draw from the stream (drawn
        # even when the lengths come from another seed, so the values of a
        # seed are the same whatever the shape)
        lp = torch.randint(1024, 32769, (8,), generator=g).tolist()
        if w.shape_seed is None or w.shape_seed == w.seed:
            assert lp == w.lp, (lp, w.lp)
    tp, tc = sum(w.lp), sum(w.lc)
    d = w.head_dim

    def normal(shape, std=1.0):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        return x * std if std != 1.0 else x

    q = normal((tc, w.hq, d)).to(torch.bfloat16)
    if w.prefix_dtype == PREFIX_Q8_0:
        kp = encode_q8_0(normal((tp, w.hkv, d)))
        vp = encode_q8_0(normal((tp, w.hkv, d)))
    elif w.prefix_dtype == PREFIX_F16:
        kp = normal((tp, w.hkv, d)).to(torch.float16)
        vp = normal((tp, w.hkv, d)).to(torch.float16)
    else:
        kp = normal((tp, w.hkv, d)).to(torch.bfloat16)
        vp = normal((tp, w.hkv, d)).to(torch.bfloat16)
    kc = normal((tc, w.hkv, d)).to(torch.bfloat16)
    vc = normal((tc, w.hkv, d)).to(torch.bfloat16)
    dout = normal((tc, w.hq, d), w.dout_std).to(torch.bfloat16)
    return dict(q=q, k_prefix=kp, v_prefix=vp, k_chunk=kc, v_chunk=vc, dout=dout,
                cu_seqlens_prefix=cu_seqlens(w.lp), cu_seqlens_chunk=cu_seqlens(w.lc),
                workload=w)
