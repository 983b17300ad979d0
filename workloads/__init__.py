"""Seeded synthetic workloads for LSH-sampled decode attention.

This module only draws inputs. It holds none of the method's arithmetic (no
hashing, no centering, no attention): it is shared by the CPU oracle tests, the
GPU parity tests and the benchmark so that both sides see identical bytes.

Every random number comes from a stateless counter-based generator: a 32-bit
murmur3-style finaliser applied to (stream key, element counter). A block of any
tensor can therefore be regenerated on its own, on any device, without drawing the
rest. Gaussians use the Box-Muller transform in float64. Integer arithmetic is kept
inside int64 without overflow so that CPU and CUDA tensors give the same integers.

Geometry of the synthetic data follows the attention geometry described in
"MagicPIG: LSH Sampling for Efficient LLM Generation" (arXiv 2410.16179v2), §3.1 and
Figure 2c: keys in a cone around a direction mu (k = a·mu + N(0, I), a = ``cone``,
3 by default), the sink key opposite (k_0 = -sink_scale·a·mu, -6·mu by default) and
queries on the sink's side (q = -2·mu + N(0, I)); values N(0, 1). How narrow the cone
is, the pages leave open beyond "almost identical" key directions (§3.1, Figure 5a:
cosine above 0.99 between keys); a = 40 to 80 at d = 128 gives cos(k, mu) of 0.96 to
0.99 (the tight-cone recipe). ``constant_keys`` draws every key but the sink as a·mu
exactly (no noise), the degenerate head in which every centered key is zero. The
projection matrix W has the shape d x (K·L) given in Algorithm 1 of the same page,
drawn N(0, 1).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = [
    "Workload", "WORKLOADS", "stream_key", "uniform", "gaussian",
    "head_mu", "keys_block", "values_block", "query_block", "projection",
    "generate", "round_to", "uniform_streams", "gaussian_streams",
]

_M32 = 0xFFFFFFFF

# purposes (mixed into the stream key)
P_MU, P_KEY, P_VALUE, P_QUERY, P_PROJ, P_MIX = 1, 2, 3, 4, 5, 6


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and recipe of one synthetic decode-attention workload.

    The sequence holds ``n_prefill`` tokens when the hash tables are built; each of
    the ``steps`` decode steps then (if ``append``) appends one token and attends
    over all tokens so far.  ``capacity`` = n_prefill + steps when appending.
    """
    name: str
    layers: int
    batch: int
    kv_heads: int
    q_heads: int
    head_dim: int
    n_prefill: int
    steps: int
    append: bool
    K: int
    L: int
    dtype: str            # "f32" or "bf16": keys, values and queries
    seed: int
    n_sink: int = 4
    window: int = 64
    iso_fraction: float = 0.0   # share of keys drawn isotropic N(0, I) instead of from the cone
    cone: float = 3.0           # a in k = a·mu + N(0, I)
    sink_scale: float = 2.0     # the sink key is -sink_scale·a·mu
    constant_keys: bool = False  # every key but the sink is a·mu exactly (no noise)
    w_per_layer: bool = False
    w_bf16: bool = True         # W rounded to bf16-representable values

    @property
    def capacity(self) -> int:
        return self.n_prefill + (self.steps if self.append else 0)

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def seq_len(self, step: int) -> int:
        """Tokens visible to the query of decode step ``step``."""
        return self.n_prefill + (step + 1 if self.append else 0)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # tiny single head, fp32
    0: Workload("tiny-1h-d64-n2048-fp32", layers=1, batch=1, kv_heads=1, q_heads=1,
                head_dim=64, n_prefill=2048, steps=1, append=False, K=8, L=75,
                dtype="f32", seed=0, w_bf16=False),
    # Llama-3.1-8B-shaped decode attention layer at 16K
    1: Workload("llama8b-layer-gqa32x8-d128-n16k-bf16", layers=1, batch=1, kv_heads=8,
                q_heads=32, head_dim=128, n_prefill=16384, steps=1, append=False, K=8,
                L=75, dtype="bf16", seed=1),
    # Llama-3.1-8B-shaped long-context decode: 32 layers, 96K, 64 appending steps
    2: Workload("llama8b-32L-gqa32x8-d128-n96k-64steps-bf16", layers=32, batch=1,
                kv_heads=8, q_heads=32, head_dim=128, n_prefill=98304, steps=64,
                append=True, K=10, L=150, dtype="bf16", seed=2, w_per_layer=True),
    # CodeLlama-13B-shaped batched decode: MHA 40 heads, batch 16, 16K, build + 32 steps
    3: Workload("codellama13b-b16-mha40-d128-n16k-32steps-bf16", layers=1, batch=16,
                kv_heads=40, q_heads=40, head_dim=128, n_prefill=16384, steps=32,
                append=True, K=9, L=120, dtype="bf16", seed=3),
    # Llama-3.1-70B-shaped decode: GQA 64/8, batch 4, 128K, 64 appending steps, 10% isotropic keys
    4: Workload("llama70b-b4-gqa64x8-d128-n128k-64steps-bf16", layers=1, batch=4,
                kv_heads=8, q_heads=64, head_dim=128, n_prefill=131072, steps=64,
                append=True, K=10, L=150, dtype="bf16", seed=4, iso_fraction=0.1),
}
# profiling case: the long-context workload cut to 4 layers (K/V 1.6 GB, still larger
# than L2) so that a multi-pass kernel capture holds a few GB of device memory only
WORKLOADS[5] = WORKLOADS[2].replace(name="llama8b-4L-gqa32x8-d128-n96k-64steps-bf16", layers=4)
# profiling case for the sampled-set kernel: the 4-layer job with 256 query heads per layer
# (group 32), so that one decode step has the 32-layer job's 1024 query heads while the
# device holds the 4-layer job's few GB
WORKLOADS[6] = WORKLOADS[5].replace(name="llama8b-4L-gqa256x8-d128-n96k-64steps-bf16", q_heads=256)


# ----------------------------------------------------------------------------------
# counter-based generator
# ----------------------------------------------------------------------------------

def _mul32(h: torch.Tensor, c: int) -> torch.Tensor:
    """(h * c) mod 2^32 for 0 <= h < 2^32 without leaving the int64 range."""
    lo = h & 0xFFFF
    hi = h >> 16
    return (lo * c + (((hi * c) & 0xFFFF) << 16)) & _M32


def _fmix32(h: torch.Tensor) -> torch.Tensor:
    h = h ^ (h >> 16)
    h = _mul32(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32(h, 0xC2B2AE35)
    h = h ^ (h >> 16)
    return h


def _fmix32_int(h: int) -> int:
    h &= _M32
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & _M32
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & _M32
    h ^= h >> 16
    return h


def stream_key(*parts: int) -> tuple[int, int]:
    """Two 32-bit keys for one stream, from any number of small integers."""
    a, b = 0x243F6A88, 0x85A308D3
    for p in parts:
        p = int(p) & _M32
        a = _fmix32_int(a ^ _fmix32_int(p + 0x9E3779B9))
        b = _fmix32_int(b + _fmix32_int(p ^ 0x7F4A7C15) + a)
    return a, b


def _bits(key: tuple[int, int], counter: torch.Tensor) -> torch.Tensor:
    a, b = key
    return _fmix32(_fmix32((counter + a) & _M32) ^ b)


def uniform(key: tuple[int, int], count: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """``count`` float64 uniforms in (0, 1) for counters offset .. offset+count-1."""
    ctr = torch.arange(offset, offset + count, dtype=torch.int64, device=device)
    h = _bits(key, ctr)
    return ((h >> 8).to(torch.float64) + 0.5) * (1.0 / 16777216.0)


def gaussian(key: tuple[int, int], count: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """``count`` float64 standard normals (Box-Muller, cosine branch) for element
    counters offset .. offset+count-1; element i uses counters 2i and 2i+1."""
    ctr = torch.arange(offset, offset + count, dtype=torch.int64, device=device) * 2
    u1 = ((_bits(key, ctr) >> 8).to(torch.float64) + 0.5) * (1.0 / 16777216.0)
    u2 = ((_bits(key, ctr + 1) >> 8).to(torch.float64) + 0.5) * (1.0 / 16777216.0)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def _bits_streams(keys: list[tuple[int, int]], counter: torch.Tensor) -> torch.Tensor:
    """``_bits`` for several streams at once: [len(keys), len(counter)], row s equal to
    ``_bits(keys[s], counter)`` element by element."""
    a = torch.tensor([k[0] for k in keys], dtype=torch.int64, device=counter.device)[:, None]
    b = torch.tensor([k[1] for k in keys], dtype=torch.int64, device=counter.device)[:, None]
    return _fmix32(_fmix32((counter[None, :] + a) & _M32) ^ b)


def uniform_streams(keys: list[tuple[int, int]], count: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """Row s equals ``uniform(keys[s], count, device, offset)``."""
    ctr = torch.arange(offset, offset + count, dtype=torch.int64, device=device)
    h = _bits_streams(keys, ctr)
    return ((h >> 8).to(torch.float64) + 0.5) * (1.0 / 16777216.0)


def gaussian_streams(keys: list[tuple[int, int]], count: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """Row s equals ``gaussian(keys[s], count, device, offset)``: one set of kernel
    launches for many streams instead of one per stream."""
    ctr = torch.arange(offset, offset + count, dtype=torch.int64, device=device) * 2
    u1 = ((_bits_streams(keys, ctr) >> 8).to(torch.float64) + 0.5) * (1.0 / 16777216.0)
    u2 = ((_bits_streams(keys, ctr + 1) >> 8).to(torch.float64) + 0.5) * (1.0 / 16777216.0)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def round_to(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if dtype == "bf16" else x.to(torch.float32)


# ----------------------------------------------------------------------------------
# tensors of a workload
# ----------------------------------------------------------------------------------

def head_mu(wl: Workload, layer: int, b: int, h: int, device="cpu") -> torch.Tensor:
    """Unit cone direction of KV head ``h`` of sequence ``b`` in ``layer`` (float64 [d])."""
    g = gaussian(stream_key(wl.seed, P_MU, layer, b, h), wl.head_dim, device)
    return g / torch.linalg.vector_norm(g)


def keys_block(wl: Workload, layer: int, b: int, h: int, t0: int, t1: int,
               device="cpu") -> torch.Tensor:
    """Keys of tokens [t0, t1) of one KV head, float64 [t1-t0, d] (not yet rounded)."""
    d = wl.head_dim
    n = t1 - t0
    mu = head_mu(wl, layer, b, h, device)
    noise = gaussian(stream_key(wl.seed, P_KEY, layer, b, h), n * d, device,
                     offset=t0 * d).view(n, d)
    k = wl.cone * mu + (0.0 * noise if wl.constant_keys else noise)
    if wl.iso_fraction > 0.0:
        pick = uniform(stream_key(wl.seed, P_MIX, layer, b, h), n, device, offset=t0)
        k = torch.where((pick < wl.iso_fraction)[:, None], noise, k)
    if t0 == 0 and n > 0:
        k[0] = -(wl.sink_scale * wl.cone) * mu
    return k


def values_block(wl: Workload, layer: int, b: int, h: int, t0: int, t1: int,
                 device="cpu") -> torch.Tensor:
    d = wl.head_dim
    n = t1 - t0
    return gaussian(stream_key(wl.seed, P_VALUE, layer, b, h), n * d, device,
                    offset=t0 * d).view(n, d)


def query_block(wl: Workload, step: int, layer: int, b: int, device="cpu") -> torch.Tensor:
    """Queries of all query heads of sequence ``b`` in ``layer`` at decode step
    ``step``, float64 [q_heads, d]; head j belongs to KV head j // group."""
    d = wl.head_dim
    mus = torch.stack([head_mu(wl, layer, b, h, device) for h in range(wl.kv_heads)])
    noise = gaussian(stream_key(wl.seed, P_QUERY, step, layer, b), wl.q_heads * d, device).view(wl.q_heads, d)
    idx = torch.arange(wl.q_heads, device=device) // wl.group
    return noise - 2.0 * mus[idx]


def projection(wl: Workload, layer: int, device="cpu") -> torch.Tensor:
    """Projection matrix W of ``layer`` (shape d x K·L, float32 holding the drawn
    values, rounded to bf16-representable values when ``w_bf16``)."""
    d, kl = wl.head_dim, wl.K * wl.L
    lay = layer if wl.w_per_layer else 0
    w = gaussian(stream_key(wl.seed, P_PROJ, lay), d * kl, device).view(d, kl)
    w = w.to(torch.bfloat16) if wl.w_bf16 else w
    return w.to(torch.float32)


def generate(wl: Workload, device="cpu", layers: Optional[list[int]] = None,
             with_values: bool = True) -> dict:
    """All tensors of a workload in the library's layout.

    keys, values : [layers, batch, kv_heads, capacity, d] in the workload dtype
    W            : [layers if w_per_layer else 1, d, K·L] float32
    queries      : [steps, layers, batch, q_heads, d] in the workload dtype
    ``layers`` restricts generation to a subset of layers (others left zero).
    """
    lay = list(range(wl.layers)) if layers is None else list(layers)
    cap, d = wl.capacity, wl.head_dim
    dt = wl.torch_dtype
    shape = (wl.layers, wl.batch, wl.kv_heads, cap, d)
    keys = torch.zeros(shape, dtype=dt, device=device)
    values = torch.zeros(shape, dtype=dt, device=device) if with_values else None
    queries = torch.zeros(wl.steps, wl.layers, wl.batch, wl.q_heads, d, dtype=dt, device=device)
    # the same values as keys_block / values_block / query_block, drawn for all KV heads
    # (and all decode steps) of a sequence at once to keep the number of launches small
    H = wl.kv_heads
    q_head_kv = torch.arange(wl.q_heads, device=device) // wl.group
    for l in lay:
        for b in range(wl.batch):
            mus = torch.stack([head_mu(wl, l, b, h, device) for h in range(H)])
            noise = gaussian_streams([stream_key(wl.seed, P_KEY, l, b, h) for h in range(H)], cap * d,
                                     device).view(H, cap, d)
            k = wl.cone * mus[:, None, :] + (0.0 * noise if wl.constant_keys else noise)
            if wl.iso_fraction > 0.0:
                pick = uniform_streams([stream_key(wl.seed, P_MIX, l, b, h) for h in range(H)], cap, device)
                k = torch.where((pick < wl.iso_fraction)[:, :, None], noise, k)
            if cap > 0:
                k[:, 0] = -(wl.sink_scale * wl.cone) * mus
            keys[l, b] = round_to(k, wl.dtype)
            del noise, k
            if with_values:
                values[l, b] = round_to(gaussian_streams([stream_key(wl.seed, P_VALUE, l, b, h) for h in range(H)],
                                                         cap * d, device).view(H, cap, d), wl.dtype)
            if wl.steps > 0:
                qn = gaussian_streams([stream_key(wl.seed, P_QUERY, s, l, b) for s in range(wl.steps)],
                                      wl.q_heads * d, device).view(wl.steps, wl.q_heads, d)
                queries[:, l, b] = round_to(qn - 2.0 * mus[q_head_kv][None], wl.dtype)
    nw = wl.layers if wl.w_per_layer else 1
    W = torch.stack([projection(wl, l, device) for l in range(nw)])
    return {"keys": keys, "values": values, "W": W, "queries": queries}
