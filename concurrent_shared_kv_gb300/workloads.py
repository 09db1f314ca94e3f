"""Seeded synthetic workloads shaped like the Hogwild! Inference configurations.

This module only draws numbers and packs them into buffers.  It holds none of
the method's arithmetic (no RoPE, no softmax, no view offsets), so that both the
oracle's tests and the CUDA path can take their inputs from it.

Stored keys are drawn directly as i.i.d. N(0,1): a stored key is a raw key
rotated by RoPE at its block-local position, and since RoPE is an orthogonal
map and the isotropic Gaussian is rotation invariant, the stored keys have the
same distribution as rotated N(0,1) raw keys.  The attention-sink key (token 0
of each common block) is scaled by 8; at block-local position 0 the rotation is
the identity, so scaling the stored key is the same as scaling the raw key.

Cache pools: one K pool and one V pool per layer, each [Hkv][capacity][D].  The
blocks of problem p are laid out back to back in the pool: its common block
(with its own capacity) followed by its W worker blocks.  Block ids follow the
same order: p*(W+1) is problem p's common block, p*(W+1)+1+w is worker w's.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

try:  # torch is only needed for bf16 rounding on the host and device draws
    import torch
except Exception:  # pragma: no cover
    torch = None


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str                 # "f32" or "bf16"
    n_problems: int
    n_workers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    rope_theta: float
    layers: int
    common_len: List[int]      # per problem
    worker_len: List[List[int]]  # per problem, per worker
    common_extra: int = 0      # capacity beyond common_len (room for commits)
    sink: bool = True
    seed: int = 0
    commit_tokens: int = 0     # tokens moved by one commit in the timed step

    @property
    def n_rows(self) -> int:
        return self.n_problems * self.n_workers

    @property
    def n_blocks(self) -> int:
        return self.n_problems * (self.n_workers + 1)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def scale(self) -> float:
        return float(self.head_dim) ** -0.5

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def block_lengths(self) -> np.ndarray:
        out = []
        for p in range(self.n_problems):
            out.append(self.common_len[p])
            out.extend(self.worker_len[p])
        return np.asarray(out, np.int32)

    def block_capacities(self) -> np.ndarray:
        out = []
        for p in range(self.n_problems):
            out.append(self.common_len[p] + self.common_extra)
            out.extend(self.worker_len[p])
        return np.asarray(out, np.int32)

    def block_starts(self) -> np.ndarray:
        cap = self.block_capacities().astype(np.int64)
        return np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int32)

    @property
    def capacity(self) -> int:
        return int(self.block_capacities().astype(np.int64).sum())

    def kv_tokens(self) -> int:
        """Tokens per kv head read by one decode call (each block once)."""
        return int(self.block_lengths().astype(np.int64).sum())

    def kv_bytes_per_layer(self) -> int:
        """Algorithmic KV bytes of one decode call: every K and V row once."""
        return self.kv_tokens() * self.n_kv_heads * self.head_dim * 2 * self.elem_bytes

    def commit_bytes_per_layer(self) -> int:
        """One commit of commit_tokens: K and V read once, written once."""
        return 2 * 2 * self.commit_tokens * self.n_kv_heads * self.head_dim * self.elem_bytes


def tiny_f32() -> Workload:
    return Workload("tiny-f32 W2 Hq4/Hkv2 D64 common256 blocks32/40", "f32", 1, 2, 4, 2, 64, 1e4,
                    1, [256], [[32, 40]], common_extra=32, sink=False, seed=1001,
                    commit_tokens=32)


def qwq32b_w2() -> Workload:
    return Workload("qwq32b-shape bf16 W2 Hq40/Hkv8 D128 common8192 blocks256x2 64 layers",
                    "bf16", 1, 2, 40, 8, 128, 1e6, 64, [8192], [[256, 256]], seed=1002)


def qwq32b_w4() -> Workload:
    return Workload("qwq32b-shape bf16 W4 Hq40/Hkv8 D128 common16384 blocks512/384/256/128 64 layers",
                    "bf16", 1, 4, 40, 8, 128, 1e6, 64, [16384], [[512, 384, 256, 128]], seed=1003)


def qwq32b_w8() -> Workload:
    """Eight workers on the QwQ-32B shape: 8 view references x G = 5 put 40
    query columns on the common block and on every worker block."""
    return Workload("qwq32b-shape bf16 W8 Hq40/Hkv8 D128 common16384 blocks512/384/256/128x2"
                    " 64 layers", "bf16", 1, 8, 40, 8, 128, 1e6, 64, [16384],
                    [[512, 384, 256, 128, 512, 384, 256, 128]], seed=1006)


def qwen3_8b_w4() -> Workload:
    return Workload("qwen3-8b-shape bf16 W4 Hq32/Hkv8 D128 common32768 blocks1024x4 36 layers"
                    " + commit 1024", "bf16", 1, 4, 32, 8, 128, 1e6, 36, [32768],
                    [[1024] * 4], common_extra=1024, seed=1004, commit_tokens=1024)


def serve_ragged(n_problems: int = 16, seed: int = 1005) -> Workload:
    """16 problems x 4 workers; common ~ U[2048, 65536], blocks ~ U[64, 2048]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    common = [int(x) for x in rng.integers(2048, 65536, size=n_problems, endpoint=True)]
    blocks = [[int(x) for x in rng.integers(64, 2048, size=4, endpoint=True)]
              for _ in range(n_problems)]
    return Workload(f"serve-ragged bf16 {n_problems}x W4 Hq40/Hkv8 D128 common U[2048,65536]"
                    " blocks U[64,2048] one layer", "bf16", n_problems, 4, 40, 8, 128, 1e6, 1,
                    common, blocks, seed=seed)


ALL = {"C1": tiny_f32, "C2": qwq32b_w2, "C3": qwq32b_w4, "C4": qwen3_8b_w4, "C5": serve_ragged}
# wider than one tile's 32 query columns (column groups)
EXTRA = {"W8": qwq32b_w8}


# ---------------------------------------------------------------------------
# host draws (numpy PCG64): storage values, f32 or bf16 bit patterns (uint16)
# ---------------------------------------------------------------------------

def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> storage values: float32, or bf16 bit patterns (round to nearest even)."""
    if dtype == "f32":
        return np.asarray(x, np.float32)
    assert torch is not None, "bf16 storage needs torch for the rounding"
    t = torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def storage_to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(x, np.float64)
    return (np.asarray(x, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def draw_host(w: Workload, layer: int = 0, poison: Optional[float] = None):
    """q [rows][Hq][D], K and V pools [Hkv][capacity][D] as storage values.

    poison: value written into pool slots beyond each block's length (default 0).
    """
    rng = np.random.Generator(np.random.PCG64(w.seed * 1000 + layer))
    D, Hkv = w.head_dim, w.n_kv_heads
    q = rng.standard_normal((w.n_rows, w.n_q_heads, D))
    k = np.full((Hkv, w.capacity, D), 0.0 if poison is None else poison)
    v = np.full((Hkv, w.capacity, D), 0.0 if poison is None else poison)
    starts, lens = w.block_starts(), w.block_lengths()
    for b in range(w.n_blocks):
        s, n = int(starts[b]), int(lens[b])
        k[:, s:s + n] = rng.standard_normal((Hkv, n, D))
        v[:, s:s + n] = rng.standard_normal((Hkv, n, D))
    if w.sink:
        for p in range(w.n_problems):
            if lens[p * (w.n_workers + 1)] > 0:
                k[:, int(starts[p * (w.n_workers + 1)])] *= 8.0
    return to_storage(q, w.dtype), to_storage(k, w.dtype), to_storage(v, w.dtype)


# ---------------------------------------------------------------------------
# device draws (torch Philox on the GPU) for the large configurations
# ---------------------------------------------------------------------------

def draw_device_layer(w: Workload, layer: int, device, poison: float = 0.0):
    """Same recipe as draw_host but drawn on the device: (q, k_pool, v_pool) tensors."""
    assert torch is not None
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    g = torch.Generator(device=device)
    g.manual_seed(w.seed * 1000 + layer)
    D, Hkv = w.head_dim, w.n_kv_heads
    q = torch.randn((w.n_rows, w.n_q_heads, D), generator=g, device=device).to(tdt)
    k = torch.full((Hkv, w.capacity, D), poison, device=device, dtype=tdt)
    v = torch.full((Hkv, w.capacity, D), poison, device=device, dtype=tdt)
    starts, lens = w.block_starts(), w.block_lengths()
    for b in range(w.n_blocks):
        s, n = int(starts[b]), int(lens[b])
        k[:, s:s + n] = torch.randn((Hkv, n, D), generator=g, device=device).to(tdt)
        v[:, s:s + n] = torch.randn((Hkv, n, D), generator=g, device=device).to(tdt)
    if w.sink:
        for p in range(w.n_problems):
            if lens[p * (w.n_workers + 1)] > 0:
                s0 = int(starts[p * (w.n_workers + 1)])
                k[:, s0] = (k[:, s0].float() * 8.0).to(tdt)
    return q, k, v


# ---------------------------------------------------------------------------
# E4M3 caches: a pool's values packed as 8-bit codes with one scale per kv head
# ---------------------------------------------------------------------------

def e4m3_pack(pool, lens=None, starts=None):
    """Pack a [Hkv][capacity][D] pool (float64 numpy or a torch tensor) as E4M3
    codes with one scale per kv head: scale_h = max |x| over the head's
    cached rows / 448 (the largest E4M3 value), code = x / scale_h rounded to
    the nearest E4M3 value by torch's float8_e4m3fn cast.  lens/starts, when
    given, restrict the maximum to the blocks' rows (slack rows are packed
    too, clipped into range).  Returns (codes uint8, scales float32 [Hkv]),
    numpy or torch like the input."""
    assert torch is not None
    is_np = isinstance(pool, np.ndarray)
    t = torch.from_numpy(np.asarray(pool, np.float64)) if is_np else pool.float()
    Hkv = t.shape[0]
    if lens is not None:
        mask = torch.zeros(t.shape[1], dtype=torch.bool, device=t.device)
        for s, n in zip(starts, lens):
            mask[int(s):int(s) + int(n)] = True
        amax = t[:, mask].abs().reshape(Hkv, -1).amax(dim=1) if mask.any() else torch.zeros(Hkv, device=t.device)
    else:
        amax = t.abs().reshape(Hkv, -1).amax(dim=1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).float()
    z = (t / scale.to(t.dtype)[:, None, None]).clamp(-448.0, 448.0)
    codes = z.float().to(torch.float8_e4m3fn).view(torch.uint8)
    if is_np:
        return codes.numpy(), scale.numpy()
    return codes, scale


def e4m3_values(codes) -> np.ndarray:
    """Decoded E4M3 codes (float64), by torch's float8_e4m3fn."""
    assert torch is not None
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)) if isinstance(codes, np.ndarray) else codes
    return t.view(torch.float8_e4m3fn).double().cpu().numpy()
