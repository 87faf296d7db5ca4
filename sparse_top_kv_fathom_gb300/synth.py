"""Seeded synthetic workloads for the Fathom decode step.

This module only draws inputs (keys, values, queries, budgets); it holds none
of the method's arithmetic, and both the CUDA path and the CPU oracle are fed
from it.  The pages measure real models and sessions (Qwen3-8B and others at up
to 1M tokens, retrieval tasks, coding-agent traces); none of those are
available, so these generators stand in with Qwen3-8B's shapes (36 layers,
8 KV heads, 128 dims, 32 query heads; [A] "How big the cache actually gets")
and key statistics chosen to stress the allocator: per-channel scales that
span a wide range, a few outlier channels, RoPE-style rotation of channel
pairs by position, and for the session batch heavy-tailed (Student-t) keys.

Each row (layer or session, KV head) draws from its own torch.Generator seeded
from (workload seed, row), so any subset of rows can be regenerated alone, on
the device the caller chooses.  The CPU and CUDA generators give different
streams: a test draws once on one device and hands the same tensors to both
sides.
"""
from dataclasses import dataclass
import math

import torch

D = 128


@dataclass(frozen=True)
class Workload:
    name: str
    layers: int           # layers (or sessions)
    kv_heads: int
    group: int            # query heads per KV head
    n: int                # tokens per row
    k: int                # winners per row
    budgets: tuple        # candidate bits-per-token budgets
    seed: int
    k_dtype: torch.dtype
    kv_dtype: torch.dtype
    outliers: int = 0     # outlier channels per head
    outlier_scale: float = 1.0
    rope: bool = False
    rope_base: float = 1.0e6
    layer_scale: tuple = None   # (lo, hi) log-uniform per-layer std multiplier
    student_t: float = 0.0      # nu > 0: Student-t keys
    per_row_budget: bool = False
    independent_layers: bool = False  # "layers" are independent sessions (one batched step)
    description: str = ""

    @property
    def rows(self):
        return self.layers * self.kv_heads


WORKLOADS = {
    "tiny": Workload(
        "tiny", 1, 1, 1, 4096, 64, (92,), 0, torch.float32, torch.float32,
        description="1 KV head, 1 query, d=128, n=4096, fp32 keys ~N(0, s_c^2) with s_c log-uniform "
                    "in [0.1, 4], query and values ~N(0,1), B=92, k=64, seed 0"),
    "qwen_layer": Workload(
        "qwen_layer", 1, 8, 4, 32768, 512, (68, 92, 136), 1, torch.bfloat16, torch.bfloat16,
        outliers=4, outlier_scale=8.0, rope=True,
        description="one Qwen3-8B-shaped layer: 8 KV heads x 128, 32 query heads, n=32768, bf16 K/V, "
                    "4 outlier channels per head at 8x std, RoPE pair rotation, B in {68,92,136}, k=512"),
    "decode36": Workload(
        "decode36", 36, 8, 4, 262144, 2048, (92,), 2, torch.bfloat16, torch.bfloat16,
        outliers=4, outlier_scale=8.0, rope=True, layer_scale=(0.5, 2.0),
        description="36 layers x 8 KV heads, n=262144, bf16 K/V as qwen_layer with per-layer std "
                    "log-uniform [0.5, 2], B=92, k=2048, index in HBM"),
    "million": Workload(
        "million", 36, 8, 4, 1 << 20, 2048, (68, 92, 136), 3, torch.bfloat16, torch.bfloat16,
        outliers=4, outlier_scale=8.0, rope=True, layer_scale=(0.5, 2.0),
        description="36 layers x 8 KV heads, n=2^20, B in {68,92,136}, k=2048, index and K/V in "
                    "pinned host memory"),
    "sessions": Workload(
        "sessions", 16, 8, 4, 131072, 1024, (48, 68, 92, 136, 256), 4, torch.bfloat16, torch.bfloat16,
        outliers=3, outlier_scale=10.0, student_t=3.0, per_row_budget=True, independent_layers=True,
        description="16 sessions x 131072 tokens, one layer (8 KV heads, 32 query heads), Student-t "
                    "(nu=3) keys with 3 channels per head at 10x scale, per-session budgets uniform "
                    "over {48,68,92,136,256}, k=1024"),
}


def _gen(seed, row, device, salt):
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + row * 7919 + salt * 104_729) & 0x7FFF_FFFF_FFFF)
    return g


def _channel_scales(w: Workload, row: int):
    """Per-channel std of one row, drawn on the CPU (tiny, device-independent)."""
    g = _gen(w.seed, row, "cpu", 1)
    if w.student_t > 0:
        s = torch.ones(D, dtype=torch.float64)
    else:
        u = torch.rand(D, generator=g, dtype=torch.float64)
        s = torch.exp(math.log(0.1) + u * (math.log(4.0) - math.log(0.1)))
    if w.outliers:
        perm = torch.randperm(D, generator=g)[: w.outliers]
        s[perm] *= w.outlier_scale
    if w.layer_scale is not None:
        layer = row // w.kv_heads
        gl = _gen(w.seed, layer, "cpu", 2)
        lo, hi = w.layer_scale
        u = torch.rand(1, generator=gl, dtype=torch.float64)
        s *= float(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    return s


def _rope(x: torch.Tensor, pos0: int, base: float):
    """Rotate channel pairs (i, i+64) by angle pos * base^(-2i/128) (fp64 angles)."""
    n = x.shape[0]
    half = D // 2
    inv = (base ** (-torch.arange(half, dtype=torch.float64) * 2.0 / D)).to(x.device)
    pos = torch.arange(pos0, pos0 + n, dtype=torch.float64, device=x.device)
    ang = pos[:, None] * inv[None, :]
    cos = torch.cos(ang).to(torch.float32)
    sin = torch.sin(ang).to(torch.float32)
    a, b = x[:, :half], x[:, half:]
    return torch.cat([a * cos - b * sin, a * sin + b * cos], dim=1)


def keys(w: Workload, row: int, device="cpu", n: int = None, chunk: int = 1 << 18) -> torch.Tensor:
    """K of one row: [n][128] in w.k_dtype on `device`."""
    n = w.n if n is None else n
    s = _channel_scales(w, row).to(device=device, dtype=torch.float32)
    g = _gen(w.seed, row, device, 3)
    out = torch.empty((n, D), dtype=w.k_dtype, device=device)
    for t0 in range(0, n, chunk):
        m = min(chunk, n - t0)
        z = torch.randn((m, D), generator=g, device=device, dtype=torch.float32)
        if w.student_t > 0:
            chi = torch.randn((m, D, int(w.student_t)), generator=g, device=device, dtype=torch.float32)
            z = z / torch.sqrt((chi * chi).sum(-1) / w.student_t)
        x = z * s
        if w.rope:
            x = _rope(x, t0, w.rope_base)
        out[t0:t0 + m] = x.to(w.k_dtype)
    return out


def values(w: Workload, row: int, device="cpu", n: int = None, chunk: int = 1 << 18) -> torch.Tensor:
    """V of one row: [n][128] ~N(0,1) in w.kv_dtype."""
    n = w.n if n is None else n
    g = _gen(w.seed, row, device, 4)
    out = torch.empty((n, D), dtype=w.kv_dtype, device=device)
    for t0 in range(0, n, chunk):
        m = min(chunk, n - t0)
        out[t0:t0 + m] = torch.randn((m, D), generator=g, device=device, dtype=torch.float32).to(w.kv_dtype)
    return out


def queries(w: Workload, layer: int, device="cpu", n: int = None, step: int = 0) -> torch.Tensor:
    """Queries of one layer (or session): [kv_heads*group][128] ~N(0,1), rotated at position n."""
    n = w.n if n is None else n
    g = _gen(w.seed, layer, device, 5 + 17 * step)
    q = torch.randn((w.kv_heads * w.group, D), generator=g, device=device, dtype=torch.float32)
    if w.rope:
        q = _rope_at(q, n, w.rope_base)
    return q.to(w.k_dtype)


def _rope_at(q: torch.Tensor, pos: int, base: float):
    half = D // 2
    inv = base ** (-torch.arange(half, dtype=torch.float64) * 2.0 / D)
    ang = pos * inv
    cos = torch.cos(ang).to(device=q.device, dtype=torch.float32)
    sin = torch.sin(ang).to(device=q.device, dtype=torch.float32)
    a, b = q[:, :half], q[:, half:]
    return torch.cat([a * cos - b * sin, a * sin + b * cos], dim=1)


def row_budgets(w: Workload, budget: int = None) -> torch.Tensor:
    """Bits-per-token budget of every row (uint16 values as int32 CPU tensor)."""
    if not w.per_row_budget:
        b = w.budgets[len(w.budgets) // 2] if budget is None else budget
        return torch.full((w.rows,), b, dtype=torch.int32)
    g = _gen(w.seed, 0, "cpu", 6)
    pick = torch.randint(0, len(w.budgets), (w.layers,), generator=g)
    per_session = torch.tensor([w.budgets[i] for i in pick.tolist()], dtype=torch.int32)
    return per_session.repeat_interleave(w.kv_heads)


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields replaced (e.g. a smaller n for tests)."""
    d = dict(w.__dict__)
    d.update(changes)
    return Workload(**d)
