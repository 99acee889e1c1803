"""Seeded synthetic workloads for the data-parallel ZeRO-2 gradient step.

This module only draws random numbers and lays them out; it holds none of the
step's arithmetic (no reduction, normalisation, optimizer or rounding rule of
the method).  Both the CUDA path's tests/benchmark and the CPU oracle receive
exactly the buffers produced here (the oracle gets host copies).

Parameter lists follow the shapes of the named model families, in module
registration order (embedding first, head last); the bucket planner reverses
that order itself.  Values:
  * gradients: bf16( N(0, grad_std) ) per replica (and per microbatch), zero in
    every padding slot of the flat layout;
  * fp32 master weights: N(0, 0.02);  Adam moments: m = v = 0 (first step) or,
    for "warm" cases, m ~ N(0, grad_std/10) and v = N(0, grad_std)^2;
  * valid-token counts: fixed for the tiny case, otherwise uniform integers in
    [3000, 4096] per (replica, microbatch).
Random numbers come from torch's seeded generators (CPU or CUDA); the seed of
config i is 0xD960000 + i, and each buffer derives its own stream from
(kind, replica, microbatch) so buffers are independent of generation order.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

MiB = 1 << 20
SEED_BASE = 0xD960000

KIND_GRAD, KIND_MASTER, KIND_M, KIND_V, KIND_TOKENS = 1, 2, 3, 4, 5


# --------------------------------------------------------------------------
# parameter lists (registration order)
# --------------------------------------------------------------------------

def tiny_shapes() -> List[Tuple[str, Tuple[int, ...]]]:
    return [("p0", (64, 32)), ("p1", (32,)), ("p2", (32, 10))]


def gpt2_small_shapes() -> List[Tuple[str, Tuple[int, ...]]]:
    d, vocab, ctx, L = 768, 50257, 1024, 12
    s = [("wte", (vocab, d)), ("wpe", (ctx, d))]
    for i in range(L):
        s += [(f"h{i}.ln1.w", (d,)), (f"h{i}.ln1.b", (d,)),
              (f"h{i}.attn.qkv.w", (d, 3 * d)), (f"h{i}.attn.qkv.b", (3 * d,)),
              (f"h{i}.attn.proj.w", (d, d)), (f"h{i}.attn.proj.b", (d,)),
              (f"h{i}.ln2.w", (d,)), (f"h{i}.ln2.b", (d,)),
              (f"h{i}.mlp.fc.w", (d, 4 * d)), (f"h{i}.mlp.fc.b", (4 * d,)),
              (f"h{i}.mlp.proj.w", (4 * d, d)), (f"h{i}.mlp.proj.b", (d,))]
    s += [("lnf.w", (d,)), ("lnf.b", (d,))]
    return s


def llama_shapes(d: int, ffn: int, vocab: int, layers: int, kv_dim: int
                 ) -> List[Tuple[str, Tuple[int, ...]]]:
    s = [("embed", (vocab, d))]
    for i in range(layers):
        s += [(f"l{i}.attn_norm", (d,)), (f"l{i}.q", (d, d)), (f"l{i}.k", (kv_dim, d)),
              (f"l{i}.v", (kv_dim, d)), (f"l{i}.o", (d, d)), (f"l{i}.mlp_norm", (d,)),
              (f"l{i}.gate", (ffn, d)), (f"l{i}.up", (ffn, d)), (f"l{i}.down", (d, ffn))]
    s += [("norm", (d,)), ("lm_head", (vocab, d))]
    return s


def sweep_shapes(n_tensors: int = 10_000, seed: int = SEED_BASE + 4
                 ) -> List[Tuple[str, Tuple[int, ...]]]:
    """Log-uniform sizes in [1, 4096]: n = clamp(floor(exp(u ln 4097)), 1, 4096)."""
    rng = np.random.Generator(np.random.Philox(seed))
    u = rng.random(n_tensors)
    n = np.clip(np.floor(np.exp(u * math.log(4097.0))), 1, 4096).astype(np.int64)
    return [(f"t{i}", (int(k),)) for i, k in enumerate(n)]


@dataclass(frozen=True)
class Config:
    name: str
    index: int
    shapes: Tuple[Tuple[str, Tuple[int, ...]], ...]
    R: int
    cap_bytes: int
    grad_std: float
    K: int = 1                       # microbatches per step (no_sync accumulation)
    fixed_tokens: Optional[Tuple[int, ...]] = None
    token_range: Tuple[int, int] = (3000, 4096)
    cap_sweep: Tuple[int, ...] = field(default_factory=tuple)
    master_std: float = 0.02

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def numels(self) -> np.ndarray:
        return np.array([math.prod(s) for _, s in self.shapes], dtype=np.int64)

    @property
    def psi(self) -> int:
        return int(self.numels.sum())


def _cfgs():
    return {
        "tiny": Config("tiny", 0, tuple(tiny_shapes()), R=4, cap_bytes=2048, grad_std=1e-2,
                       fixed_tokens=(100, 80, 120, 60)),
        "gpt2": Config("gpt2", 1, tuple(gpt2_small_shapes()), R=8, cap_bytes=25 * MiB,
                       grad_std=1e-3),
        "llama1b": Config("llama1b", 2, tuple(llama_shapes(2048, 8192, 32000, 16, 2048)), R=8,
                          cap_bytes=25 * MiB, grad_std=1e-3,
                          cap_sweep=(1 * MiB, 25 * MiB, 100 * MiB)),
        "llama8b16l": Config("llama8b16l", 3,
                             tuple(llama_shapes(4096, 14336, 128256, 16, 1024)), R=4,
                             cap_bytes=100 * MiB, grad_std=1e-3, K=4),
        "sweep": Config("sweep", 4, tuple(sweep_shapes()), R=8, cap_bytes=4096,
                        grad_std=1e-3,
                        cap_sweep=tuple(4096 * 2 ** i for i in range(17))),
    }


CONFIGS = _cfgs()


def stream_seed(base: int, kind: int, replica: int = 0, micro: int = 0) -> int:
    """Seed of one buffer's random stream (independent of generation order)."""
    return (base * 1_000_003 + kind * 10_007 + replica * 101 + micro) & ((1 << 63) - 1)


# --------------------------------------------------------------------------
# layouts: which slots of a flat buffer carry values (the rest are padding)
# --------------------------------------------------------------------------

def segments(param_offset: Sequence[int], numels: Sequence[int]) -> List[Tuple[int, int]]:
    """(offset, numel) of every non-empty parameter slice."""
    return [(int(o), int(n)) for o, n in zip(param_offset, numels) if int(n) > 0]


def padding_ranges(segs: List[Tuple[int, int]], total: int) -> List[Tuple[int, int]]:
    """Complement of the segments inside [0, total)."""
    out, cur = [], 0
    for o, n in sorted(segs):
        if o > cur:
            out.append((cur, o))
        cur = max(cur, o + n)
    if cur < total:
        out.append((cur, total))
    return out


# --------------------------------------------------------------------------
# torch-based generators (CPU or CUDA)
# --------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _gen(device, seed: int):
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_f32(n: int, std: float, seed: int, device="cpu"):
    """float32 tensor of n draws from N(0, std)."""
    torch = _torch()
    t = torch.empty(n, dtype=torch.float32, device=device)
    if n:
        t.normal_(0.0, std, generator=_gen(device, seed))
    return t


def flat_grads_bf16(segs, total: int, std: float, seed: int, device="cpu", chunk=1 << 28):
    """bf16 tensor [total]: N(0, std) in every segment, zero in padding."""
    torch = _torch()
    out = torch.empty(total, dtype=torch.bfloat16, device=device)
    g = _gen(device, seed)
    for lo in range(0, total, chunk):
        hi = min(total, lo + chunk)
        tmp = torch.empty(hi - lo, dtype=torch.float32, device=device)
        tmp.normal_(0.0, std, generator=g)
        out[lo:hi].copy_(tmp)
        del tmp
    for a, b in padding_ranges(segs, total):
        out[a:b].zero_()
    return out


def flat_values_f32(segs, total: int, std: float, seed: int, device="cpu"):
    """float32 tensor [total]: N(0, std) in every segment, zero in padding."""
    out = normal_f32(total, std, seed, device)
    for a, b in padding_ranges(segs, total):
        out[a:b].zero_()
    return out


def master_f32(total: int, seed: int, std: float = 0.02, device="cpu"):
    return normal_f32(total, std, seed, device)


def warm_moments(total: int, grad_std: float, seed_m: int, seed_v: int, device="cpu"):
    m = normal_f32(total, grad_std / 10.0, seed_m, device)
    v = normal_f32(total, grad_std, seed_v, device)
    v.mul_(v)
    return m, v


def token_counts(cfg: Config) -> np.ndarray:
    """int64 [R*K] valid-token counts, replica-major (index r*K + k)."""
    if cfg.fixed_tokens is not None:
        return np.array(cfg.fixed_tokens, dtype=np.int64)
    rng = np.random.Generator(np.random.Philox(stream_seed(cfg.seed, KIND_TOKENS)))
    lo, hi = cfg.token_range
    return rng.integers(lo, hi + 1, size=cfg.R * cfg.K, dtype=np.int64)


def bf16_bits(t) -> np.ndarray:
    """numpy uint16 view of a CPU bf16 tensor's bit patterns."""
    torch = _torch()
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def random_param_list(rng: np.random.Generator, n: int, max_numel: int) -> np.ndarray:
    """Ragged parameter sizes for property tests (some zero-size, some tiny)."""
    sizes = np.exp(rng.random(n) * math.log(max_numel + 1)).astype(np.int64)
    zero = rng.random(n) < 0.05
    sizes[zero] = 0
    return np.clip(sizes, 0, max_numel)
