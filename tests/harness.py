"""Shared helpers of the GPU tests: put one seeded workload on the device, run
the library through its C ABI, run the oracle on the same inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from concurrent_shared_kv_gb300 import api, engine
from concurrent_shared_kv_gb300 import workloads as wl

F32_TOL = 1e-5                     # max-abs, fp32 storage
BF16_MAX, BF16_MEAN = 2e-2, 1e-2   # max-abs / mean-abs, bf16 storage, fp32 accumulation
# Long views average many V rows, so |out| ~ 1/sqrt(L) and an absolute bar
# alone is loose; the error is also bounded relative to the output's scale
# (max-abs / max|ref| and rms error / rms ref).  bf16: the output's own
# rounding is 2^-9 relative; bf16 queries and probabilities in the tensor-core
# path add a few parts in 1e3.
REL_TOL = {"f32": 1e-4, "bf16": 2e-2}
LSE_TOL = {"f32": 1e-5, "bf16": 2e-2}


def torch_dtype(w: wl.Workload):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def to_storage_np(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> host storage values (float32, or bf16 bits as uint16)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def from_storage_np(x: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)
    return torch.from_numpy(np.ascontiguousarray(x, np.uint16).view(np.int16)).view(torch.bfloat16).to(device)


def out_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class Case:
    """Inputs of one decode call, on host (storage values) and device."""

    def __init__(self, w: wl.Workload, q, k, v, block_start=None, block_len=None, views=None,
                 q_to_kv=None):
        self.w = w
        self.q, self.k, self.v = q, k, v  # device tensors
        self.block_start = w.block_starts() if block_start is None else np.asarray(block_start, np.int32)
        self.block_len = w.block_lengths() if block_len is None else np.asarray(block_len, np.int32)
        if views is None:
            views = api.views_combined(self.block_len, w.n_problems, w.n_workers)
        self.view_block, self.view_offset, self.q_pos = [np.asarray(x, np.int32) for x in views]
        self.q_to_kv = None if q_to_kv is None else np.asarray(q_to_kv, np.int32)

    @property
    def capacity(self):
        return int(self.k.shape[1])

    def session(self, view_limits: bool = False) -> engine.DecodeSession:
        w = self.w
        s = engine.DecodeSession(n_rows=self.q.shape[0], n_q_heads=w.n_q_heads,
                                 n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
                                 n_blocks=len(self.block_len), max_view_blocks=self.view_block.shape[1],
                                 capacity=self.capacity, dtype=torch_dtype(w), rope_theta=w.rope_theta,
                                 scale=w.scale, view_limits=view_limits)
        s.set_metadata(self.block_start, self.block_len, self.view_block, self.view_offset,
                       self.q_pos, self.q_to_kv)
        return s

    def run_gpu(self, session=None):
        s = session or self.session()
        out, lse = s.decode(self.q, self.k, self.v)
        torch.cuda.synchronize()
        return out, lse, s

    def run_oracle(self, rows=None, brute=False):
        w = self.w
        return oracle.get().attn_decode(
            q=to_storage_np(self.q), k_cache=to_storage_np(self.k), v_cache=to_storage_np(self.v),
            block_start=self.block_start, block_len=self.block_len, view_block=self.view_block,
            view_offset=self.view_offset, q_pos=self.q_pos, n_kv_heads=w.n_kv_heads,
            rope_theta=w.rope_theta, scale=w.scale,
            dtype=oracle.F32 if w.dtype == "f32" else oracle.BF16, q_to_kv=self.q_to_kv, rows=rows,
            brute=brute)


def host_case(w: wl.Workload, layer=0, poison=None, **kw) -> Case:
    q, k, v = wl.draw_host(w, layer, poison=poison)
    return Case(w, from_storage_np(q, w.dtype), from_storage_np(k, w.dtype),
                from_storage_np(v, w.dtype), **kw)


def device_case(w: wl.Workload, layer=0, **kw) -> Case:
    q, k, v = wl.draw_device_layer(w, layer, "cuda")
    return Case(w, q, k, v, **kw)


def compare(w_dtype: str, out_gpu, lse_gpu, out_ref, lse_ref, rows=None, what=""):
    """Assert the stated tolerance; returns (max_abs, mean_abs, max_rel_to_inf_norm)."""
    g = out_f64(out_gpu)
    r = out_ref
    lg = lse_gpu.detach().cpu().numpy().astype(np.float64) if lse_gpu is not None else None
    if rows is not None:
        g, r = g[rows], r[rows]
        lg = lg[rows] if lg is not None else None
        lr = lse_ref[rows]
    else:
        lr = lse_ref
    assert np.all(np.isfinite(g)), what
    err = np.abs(g - r)
    mx, mean = float(err.max()), float(err.mean())
    rel = float(mx / max(np.abs(r).max(), 1e-30))
    rms = float(np.sqrt(np.mean(err ** 2)) / max(np.sqrt(np.mean(r ** 2)), 1e-30))
    assert rel <= REL_TOL[w_dtype] and rms <= REL_TOL[w_dtype] / 2, \
        f"{what}: max-abs/max|ref| {rel:.3e}, rms rel {rms:.3e}"
    if w_dtype == "f32":
        assert mx <= F32_TOL, f"{what}: max-abs {mx}"
    else:
        assert mx <= BF16_MAX and mean <= BF16_MEAN, f"{what}: max-abs {mx} mean-abs {mean}"
    if lg is not None:
        fin = np.isfinite(lr)
        assert np.array_equal(np.isneginf(lg), np.isneginf(lr)), what
        if fin.any():
            le = float(np.abs(lg[fin] - lr[fin]).max())
            assert le <= LSE_TOL[w_dtype], f"{what}: lse max-abs {le}"
    return mx, mean, rel
