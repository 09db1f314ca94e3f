"""Torch-facing convenience layer over the C ABI: it owns a workspace and the
device copies of the per-step metadata.  PyTorch only allocates memory and
provides streams here; every step of the computation runs in libhogwild."""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import api

DTYPES = {torch.float32: api.HW_F32, torch.bfloat16: api.HW_BF16,
          torch.uint8: api.HW_FP8_E4M3, torch.float8_e4m3fn: api.HW_FP8_E4M3}


class DecodeSession:
    """One decode configuration: shapes, pools, workspace and metadata."""

    def __init__(self, *, n_rows: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                 n_blocks: int, max_view_blocks: int, capacity: int, dtype: torch.dtype,
                 rope_theta: float, scale: Optional[float] = None, device="cuda",
                 view_limits: bool = False, kv_fp8: bool = False):
        """view_limits: the steps are planned with per-view-entry token limits
        (plan_limited; decode_planned then applies them).  kv_fp8: the K and V
        pools hold E4M3 codes with per-kv-head scales (decode_planned_fp8);
        dtype is then that of q and out (bf16)."""
        self.device = torch.device(device)
        self.dtype = dtype
        self.desc = api.make_desc(n_rows, n_q_heads, n_kv_heads, head_dim, n_blocks,
                                  max_view_blocks, capacity,
                                  api.HW_FP8_E4M3 if kv_fp8 else DTYPES[dtype], rope_theta,
                                  head_dim ** -0.5 if scale is None else scale,
                                  flags=api.HW_DESC_VIEW_LIMITS if view_limits else 0)
        # the same description with the early-loads promise (see early= below)
        self.desc_early = api.make_desc(n_rows, n_q_heads, n_kv_heads, head_dim, n_blocks,
                                        max_view_blocks, capacity,
                                        api.HW_FP8_E4M3 if kv_fp8 else DTYPES[dtype], rope_theta,
                                        head_dim ** -0.5 if scale is None else scale,
                                        flags=self.desc.flags | api.HW_DESC_EARLY_LOADS)
        self.ws_bytes = api.attn_decode_workspace_size(self.desc)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)
        api.workspace_init(self.workspace, self.ws_bytes)
        self.meta = None

    def set_metadata(self, block_start, block_len, view_block, view_offset, q_pos, q_to_kv=None,
                     non_blocking: bool = False):
        """Upload the step's metadata (shared by every layer of the step)."""
        def dev(x):
            if x is None:
                return None
            t = torch.as_tensor(np.ascontiguousarray(x, dtype=np.int32)) if not torch.is_tensor(x) else x
            return t.to(self.device, dtype=torch.int32, non_blocking=non_blocking).contiguous()
        self.meta = dict(block_start=dev(block_start), block_len=dev(block_len),
                         view_block=dev(view_block), view_offset=dev(view_offset),
                         q_pos=dev(q_pos), q_to_kv=dev(q_to_kv))

    def decode(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
               out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               want_lse: bool = True, stream=None, early: bool = False):
        d = self.desc_early if early else self.desc
        if out is None:
            out = torch.empty((d.n_rows, d.n_q_heads, d.head_dim), dtype=self.dtype, device=self.device)
        if lse is None and want_lse:
            lse = torch.empty((d.n_rows, d.n_q_heads), dtype=torch.float32, device=self.device)
        m = self.meta
        api.attn_decode(d, q, k_cache, v_cache, m["block_start"], m["block_len"], m["view_block"],
                        m["view_offset"], m["q_pos"], out, lse, self.workspace, self.ws_bytes,
                        q_to_kv=m["q_to_kv"], stream=stream)
        return out, lse

    def plan(self, stream=None):
        """hw_attn_plan on the uploaded metadata: once per step, before the
        layers' decode_planned calls."""
        m = self.meta
        api.attn_plan(self.desc, m["block_start"], m["block_len"], m["view_block"],
                      m["view_offset"], m["q_pos"], self.workspace, self.ws_bytes,
                      q_to_kv=m["q_to_kv"], stream=stream)

    def plan_limited(self, view_limit, stream=None):
        """hw_attn_plan_limited: plan the step with a token limit per view
        entry ([rows][V]; negative = the whole block), e.g. the causal order
        of a chunk of queries within its own block."""
        m = self.meta
        t = torch.as_tensor(np.ascontiguousarray(view_limit, dtype=np.int32)) \
            if not torch.is_tensor(view_limit) else view_limit
        self.view_limit = t.to(self.device, dtype=torch.int32).contiguous()
        api.attn_plan_limited(self.desc, m["block_start"], m["block_len"], m["view_block"],
                              m["view_offset"], self.view_limit, m["q_pos"], self.workspace,
                              self.ws_bytes, q_to_kv=m["q_to_kv"], stream=stream)

    def plan_append(self, append_block, append_pos, stream=None):
        """hw_attn_plan_append: plan the step with each row's new token
        (append_block[r] = its block or -1, append_pos[r] = its block-local
        position; block_len of the uploaded metadata must count it)."""
        m = self.meta
        def dev(x):
            t = torch.as_tensor(np.ascontiguousarray(x, dtype=np.int32)) if not torch.is_tensor(x) else x
            return t.to(self.device, dtype=torch.int32).contiguous()
        self.append = (dev(append_block), dev(append_pos))
        api.attn_plan_append(self.desc, m["block_start"], m["block_len"], m["view_block"],
                             m["view_offset"], m["q_pos"], self.append[0], self.append[1],
                             self.workspace, self.ws_bytes, q_to_kv=m["q_to_kv"], stream=stream)

    def append_decode_planned(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                              k_cache: torch.Tensor, v_cache: torch.Tensor,
                              out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                              want_lse: bool = True, stream=None, early: bool = False):
        """One layer: its new tokens ([rows][Hkv][D]) written, then decoded."""
        d = self.desc_early if early else self.desc
        if out is None:
            out = torch.empty((d.n_rows, d.n_q_heads, d.head_dim), dtype=self.dtype, device=self.device)
        if lse is None and want_lse:
            lse = torch.empty((d.n_rows, d.n_q_heads), dtype=torch.float32, device=self.device)
        api.attn_append_decode_planned(d, q, k_new, v_new, k_cache, v_cache, out, lse,
                                       self.workspace, self.ws_bytes, stream=stream)
        return out, lse

    def decode_planned(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                       out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                       want_lse: bool = True, stream=None, early: bool = False):
        """One layer against the step's plan (see plan()).  early=True promises
        that the work enqueued just before this call on the stream writes
        neither this layer's K/V pools nor the plan (HW_DESC_EARLY_LOADS): true
        for every layer of a step after the first one that follows the plan."""
        d = self.desc_early if early else self.desc
        if out is None:
            out = torch.empty((d.n_rows, d.n_q_heads, d.head_dim), dtype=self.dtype, device=self.device)
        if lse is None and want_lse:
            lse = torch.empty((d.n_rows, d.n_q_heads), dtype=torch.float32, device=self.device)
        api.attn_decode_planned(d, q, k_cache, v_cache, out, lse, self.workspace, self.ws_bytes,
                                stream=stream)
        return out, lse

    def decode_planned_fp8(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           k_scale: torch.Tensor, v_scale: torch.Tensor,
                           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                           want_lse: bool = True, stream=None, early: bool = False):
        """One layer over E4M3 pools (codes, [Hkv][cap][D]) with float32 scales [Hkv]."""
        d = self.desc_early if early else self.desc
        if out is None:
            out = torch.empty((d.n_rows, d.n_q_heads, d.head_dim), dtype=self.dtype, device=self.device)
        if lse is None and want_lse:
            lse = torch.empty((d.n_rows, d.n_q_heads), dtype=torch.float32, device=self.device)
        api.attn_decode_planned_fp8(d, q, k_cache, v_cache, k_scale, v_scale, out, lse,
                                    self.workspace, self.ws_bytes, stream=stream)
        return out, lse

    def append_decode_planned_fp8(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                  k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  k_scale: torch.Tensor, v_scale: torch.Tensor,
                                  out: Optional[torch.Tensor] = None,
                                  lse: Optional[torch.Tensor] = None, want_lse: bool = True,
                                  stream=None, early: bool = False):
        """One layer over E4M3 pools: its new tokens (bf16, [rows][Hkv][D])
        written as codes with the head scales, then decoded."""
        d = self.desc_early if early else self.desc
        if out is None:
            out = torch.empty((d.n_rows, d.n_q_heads, d.head_dim), dtype=self.dtype, device=self.device)
        if lse is None and want_lse:
            lse = torch.empty((d.n_rows, d.n_q_heads), dtype=torch.float32, device=self.device)
        api.attn_append_decode_planned_fp8(d, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                                           out, lse, self.workspace, self.ws_bytes, stream=stream)
        return out, lse

    def device_flags(self) -> int:
        return api.workspace_status(self.workspace)


def block_commit(k_src: torch.Tensor, v_src: torch.Tensor, src_begin: int, n_tokens: int,
                 k_dst: torch.Tensor, v_dst: torch.Tensor, dst_offset: int, pos_delta: int,
                 rope_theta: float, stream=None):
    """Pools shaped [layers][Hkv][cap][D] or [Hkv][cap][D]."""
    def dims(t):
        return (1,) + tuple(t.shape) if t.dim() == 3 else tuple(t.shape)
    L, H, cs, D = dims(k_src)
    _, _, cd, _ = dims(k_dst)
    return api.block_commit(DTYPES[k_src.dtype], L, H, D, rope_theta, k_src, v_src, cs, src_begin,
                            n_tokens, k_dst, v_dst, cd, dst_offset, pos_delta, stream=stream)


def block_commit_many(k_src: torch.Tensor, v_src: torch.Tensor, commits, k_dst: torch.Tensor,
                      v_dst: torch.Tensor, rope_theta: float, stream=None):
    """Several finished steps in one launch.  `commits`: (src_begin, n_tokens,
    dst_offset, pos_delta) tuples; pools as in block_commit."""
    def dims(t):
        return (1,) + tuple(t.shape) if t.dim() == 3 else tuple(t.shape)
    L, H, cs, D = dims(k_src)
    _, _, cd, _ = dims(k_dst)
    cols = list(zip(*commits)) if commits else [(), (), (), ()]
    return api.block_commit_many(DTYPES[k_src.dtype], L, H, D, rope_theta, k_src, v_src, cs, k_dst,
                                 v_dst, cd, *cols, stream=stream)
