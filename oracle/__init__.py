"""Float64 CPU oracle for Hogwild! concurrent decode attention and block commit.

TEST INFRASTRUCTURE ONLY.  The product path (the ``concurrent_shared_kv_gb300``
package and its CUDA library) never imports this package; only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` do.  It shares
no code with the CUDA path: the arithmetic lives in ``hwref.c`` (plain C, double
precision) and the layout builder below is written independently of the
library's own.

Pages followed (title, section):
  * "Hogwild! Inference: Parallel LLM Generation via Concurrent Attention"
    (paper notes): key design 1 (the query-rotation equation), key design 2
    (combined cache layout; step commit), implementation notes (block-local
    positions, query rotation handles the real position).
  * omica.com.cn article on Hogwild! Inference: section 2.1 (rotate_query),
    section 3.2 (blockwise attention with one softmax across blocks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
SRC = os.path.join(HERE, "hwref.c")

F32, BF16, FP8 = 0, 1, 2  # FP8: bf16 queries, E4M3 K and V with per-kv-head scales


def lib_path(mutant: int = 0) -> str:
    name = "libhwref.so" if mutant == 0 else f"libhwref_mutant{mutant}.so"
    return os.path.join(BUILD_DIR, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile hwref.c with gcc (IEEE double, no fast-math)."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC",
           "-pthread", f"-DHWREF_MUTANT={mutant}", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class HwrefDesc(ctypes.Structure):
    _fields_ = [
        ("n_rows", ctypes.c_int32),
        ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("n_blocks", ctypes.c_int32),
        ("max_view_blocks", ctypes.c_int32),
        ("cache_capacity", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("rope_theta", ctypes.c_double),
        ("scale", ctypes.c_double),
    ]


_P = ctypes.c_void_p


class Oracle:
    """ctypes handle on one build of hwref.c (the default, or a planted mutant)."""

    def __init__(self, mutant: int = 0):
        self.mutant = mutant
        self.lib = ctypes.CDLL(build(mutant))
        L = self.lib
        L.hwref_rope.argtypes = [_P, ctypes.c_int, ctypes.c_double, ctypes.c_double, _P]
        L.hwref_rope.restype = None
        L.hwref_rope_freqs.argtypes = [ctypes.c_int, ctypes.c_double, _P]
        L.hwref_rope_freqs.restype = None
        L.hwref_attn_decode.argtypes = [ctypes.POINTER(HwrefDesc), _P, _P, _P, _P, _P, _P, _P, _P,
                                        _P, _P, ctypes.c_int32, ctypes.c_int, _P, _P, ctypes.c_int]
        L.hwref_attn_decode.restype = ctypes.c_int
        L.hwref_attn_decode_limited.argtypes = [ctypes.POINTER(HwrefDesc), _P, _P, _P, _P, _P, _P, _P,
                                                _P, _P, _P, _P, ctypes.c_int32, ctypes.c_int, _P, _P,
                                                ctypes.c_int]
        L.hwref_attn_decode_limited.restype = ctypes.c_int
        L.hwref_attn_decode_scaled.argtypes = [ctypes.POINTER(HwrefDesc)] + [_P] * 13 + [
            ctypes.c_int32, ctypes.c_int, _P, _P, ctypes.c_int]
        L.hwref_attn_decode_scaled.restype = ctypes.c_int
        L.hwref_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.hwref_e4m3_to_double.restype = ctypes.c_double
        L.hwref_e4m3_from_double.argtypes = [ctypes.c_double]
        L.hwref_e4m3_from_double.restype = ctypes.c_uint8
        L.hwref_block_commit.argtypes = [ctypes.c_int, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_double, _P, _P, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.c_int32, _P, _P, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.c_int32, _P]
        L.hwref_block_commit.restype = ctypes.c_int
        L.hwref_bf16_from_double.argtypes = [ctypes.c_double]
        L.hwref_bf16_from_double.restype = ctypes.c_uint16

    # -- RoPE ---------------------------------------------------------------
    def rope(self, x, theta: float, pos: float) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float64)
        y = np.empty_like(x)
        self.lib.hwref_rope(x.ctypes.data, x.shape[-1], float(theta), float(pos), y.ctypes.data)
        return y

    def freqs(self, D: int, theta: float) -> np.ndarray:
        w = np.empty(D // 2, np.float64)
        self.lib.hwref_rope_freqs(D, float(theta), w.ctypes.data)
        return w

    def bf16_from_double(self, x: float) -> int:
        return int(self.lib.hwref_bf16_from_double(float(x)))

    def e4m3_to_double(self, code: int) -> float:
        return float(self.lib.hwref_e4m3_to_double(int(code)))

    def e4m3_from_double(self, x: float) -> int:
        return int(self.lib.hwref_e4m3_from_double(float(x)))

    # -- decode -------------------------------------------------------------
    def attn_decode(self, *, q, k_cache, v_cache, block_start, block_len, view_block, view_offset,
                    q_pos, n_kv_heads: int, rope_theta: float, scale: float, dtype: int,
                    q_to_kv=None, rows: Optional[Sequence[int]] = None, brute: bool = False,
                    n_threads: Optional[int] = None, view_limit=None, k_scale=None,
                    v_scale=None):
        """Returns (out [rows][Hq][D] float64, lse [rows][Hq] float64).

        view_limit [rows][V] (optional): an entry with a limit >= 0 attends
        only the first min(limit, len) tokens of its block.

        q, k_cache, v_cache hold storage values: float32 arrays for ``dtype=F32``,
        uint16 bf16 bit patterns for ``dtype=BF16``; for ``dtype=FP8`` q is bf16
        and the caches hold uint8 E4M3 codes, a cached element being its value
        times its kv head's k_scale / v_scale (float32 [Hkv]).  k_cache/v_cache
        are [Hkv][capacity][D].  Unselected rows of the outputs are NaN.
        """
        sd = np.float32 if dtype == F32 else np.uint16
        cd = np.uint8 if dtype == FP8 else sd
        q = np.ascontiguousarray(q, dtype=sd)
        k_cache = np.ascontiguousarray(k_cache, dtype=cd)
        v_cache = np.ascontiguousarray(v_cache, dtype=cd)
        if dtype == FP8:
            k_scale = np.ascontiguousarray(k_scale, dtype=np.float32)
            v_scale = np.ascontiguousarray(v_scale, dtype=np.float32)
            assert k_scale.shape == (n_kv_heads,) and v_scale.shape == (n_kv_heads,)
        n_rows, Hq, D = q.shape
        assert k_cache.shape[0] == n_kv_heads and k_cache.shape[2] == D
        assert v_cache.shape == k_cache.shape
        i32 = lambda a: np.ascontiguousarray(a, dtype=np.int32)
        block_start, block_len = i32(block_start), i32(block_len)
        view_block, view_offset, q_pos = i32(view_block), i32(view_offset), i32(q_pos)
        assert view_block.shape == view_offset.shape and view_block.shape[0] == n_rows
        qmap = None if q_to_kv is None else i32(q_to_kv)
        sel = None if rows is None else i32(rows)
        desc = HwrefDesc(n_rows, Hq, n_kv_heads, D, int(block_len.shape[0]),
                         int(view_block.shape[1]), int(k_cache.shape[1]), dtype,
                         float(rope_theta), float(scale))
        out = np.full((n_rows, Hq, D), np.nan)
        lse = np.full((n_rows, Hq), np.nan)
        nt = n_threads or len(os.sched_getaffinity(0))
        vlim = None if view_limit is None else i32(view_limit)
        if vlim is not None:
            assert vlim.shape == view_block.shape
        rc = self.lib.hwref_attn_decode_scaled(
            ctypes.byref(desc), q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
            k_scale.ctypes.data if dtype == FP8 else None,
            v_scale.ctypes.data if dtype == FP8 else None,
            block_start.ctypes.data, block_len.ctypes.data, view_block.ctypes.data,
            view_offset.ctypes.data, q_pos.ctypes.data,
            None if qmap is None else qmap.ctypes.data,
            None if vlim is None else vlim.ctypes.data,
            None if sel is None else sel.ctypes.data, 0 if sel is None else len(sel),
            1 if brute else 0, out.ctypes.data, lse.ctypes.data, int(nt))
        if rc != 0:
            raise ValueError(f"hwref_attn_decode rejected its inputs (status {rc})")
        return out, lse

    # -- commit -------------------------------------------------------------
    def block_commit(self, *, dtype: int, rope_theta: float, k_src, v_src, src_begin: int,
                     n_tokens: int, k_dst, v_dst, dst_offset: int, pos_delta: int,
                     want_exact: bool = False):
        """In-place on copies of k_dst/v_dst ([Hkv][cap][D] storage values).

        Returns (k_dst_new, v_dst_new[, k_exact [Hkv][n][D] float64]).
        FP8: uint8 E4M3 codes, no scale (a rotation carries a head's scale over).
        """
        sd = np.float32 if dtype == F32 else np.uint8 if dtype == FP8 else np.uint16
        k_src = np.ascontiguousarray(k_src, dtype=sd)
        v_src = np.ascontiguousarray(v_src, dtype=sd)
        kd = np.array(k_dst, dtype=sd, copy=True, order="C")
        vd = np.array(v_dst, dtype=sd, copy=True, order="C")
        Hkv, _, D = k_src.shape
        exact = np.zeros((Hkv, n_tokens, D)) if want_exact else None
        rc = self.lib.hwref_block_commit(
            dtype, Hkv, D, float(rope_theta), k_src.ctypes.data, v_src.ctypes.data,
            int(k_src.shape[1]) * D, int(src_begin), int(n_tokens), kd.ctypes.data,
            vd.ctypes.data, int(kd.shape[1]) * D, int(dst_offset), int(pos_delta),
            None if exact is None else exact.ctypes.data)
        if rc != 0:
            raise ValueError(f"hwref_block_commit rejected its inputs (status {rc})")
        return (kd, vd, exact) if want_exact else (kd, vd)


    def append_tokens(self, *, dtype: int, rope_theta: float, k_cache, v_cache, k_new, v_new,
                      block_start, append_block, append_pos, want_exact: bool = False):
        """Each row's new token into its block, the step before every layer's
        attention: the key is stored like every key of the cache, rotated at
        its block-local position p (keys sit at 0..len-1 of their block), the
        value as it is.  For row r with b = append_block[r] >= 0 and
        p = append_pos[r], every kv head h:
            K[h][block_start[b] + p] = rho(k_new[r][h], p),  V[...] = v_new[r][h]
        which is the block commit of a one-token source by delta = p.
        k_new, v_new: [rows][Hkv][D] storage values; caches [Hkv][cap][D].
        Returns (k, v[, exact keys {row: [Hkv][D] float64}]) on copies.
        """
        sd = np.float32 if dtype == F32 else np.uint16
        kd = np.array(k_cache, dtype=sd, copy=True, order="C")
        vd = np.array(v_cache, dtype=sd, copy=True, order="C")
        exact = {}
        for r in range(len(append_block)):
            b = int(append_block[r])
            if b < 0:
                continue
            p = int(append_pos[r])
            ks = np.ascontiguousarray(np.asarray(k_new[r], dtype=sd)[:, None, :])
            vs = np.ascontiguousarray(np.asarray(v_new[r], dtype=sd)[:, None, :])
            kd, vd, ex = self.block_commit(dtype=dtype, rope_theta=rope_theta, k_src=ks, v_src=vs,
                                           src_begin=0, n_tokens=1, k_dst=kd, v_dst=vd,
                                           dst_offset=int(block_start[b]) + p, pos_delta=p,
                                           want_exact=True)
            exact[r] = ex[:, 0, :]
        return (kd, vd, exact) if want_exact else (kd, vd)


def append_tokens_e4m3(o: "Oracle", *, rope_theta: float, k_cache, v_cache, k_new, v_new,
                       k_scale, v_scale, block_start, append_block, append_pos):
    """The append into E4M3 caches: row r's new key (bf16 storage, rotated at
    its block-local position p, in double) divided by its kv head's k_scale and
    rounded to the nearest E4M3 code (ties to even, saturating at 448); its
    value divided by v_scale and rounded likewise.  k_new, v_new: [rows][Hkv][D]
    bf16 storage; caches [Hkv][cap][D] uint8 codes.  Returns (k, v, exact) on
    copies, exact = {row: ([Hkv][D] key / k_scale, [Hkv][D] value / v_scale)}
    before rounding."""
    kd = np.array(k_cache, dtype=np.uint8, copy=True, order="C")
    vd = np.array(v_cache, dtype=np.uint8, copy=True, order="C")
    Hkv, _, D = kd.shape
    bf = lambda a: (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    exact = {}
    for r in range(len(append_block)):
        b = int(append_block[r])
        if b < 0:
            continue
        p, row = int(append_pos[r]), int(block_start[b]) + int(append_pos[r])
        ek = np.stack([o.rope(bf(k_new[r][h]), rope_theta, float(p)) / float(k_scale[h])
                       for h in range(Hkv)])
        ev = np.stack([bf(v_new[r][h]) / float(v_scale[h]) for h in range(Hkv)])
        for h in range(Hkv):
            kd[h, row] = [o.e4m3_from_double(x) for x in ek[h]]
            vd[h, row] = [o.e4m3_from_double(x) for x in ev[h]]
        exact[r] = (ek, ev)
    return kd, vd, exact


_default: Optional[Oracle] = None


def get(mutant: int = 0) -> Oracle:
    global _default
    if mutant:
        return Oracle(mutant)
    if _default is None:
        _default = Oracle(0)
    return _default


# ---------------------------------------------------------------------------
# Views: the combined layout, written out independently of the library.
# ---------------------------------------------------------------------------

def combined_views(block_len: Sequence[int], n_problems: int, n_workers: int):
    """The combined cache layout of key design 2: each worker sees the common
    block, then the other workers' in-progress blocks in worker order, then its
    own block.  Problem p owns blocks p*(W+1) (common) and p*(W+1)+1+w (worker w).

    Returns (view_block [rows][W+1], view_offset [rows][W+1], q_pos [rows]); the
    offset of a block is the number of tokens before it in that worker's view and
    the query sits right after the whole view (i_q = view length).
    """
    W = n_workers
    rows = n_problems * W
    vb = np.full((rows, W + 1), -1, np.int32)
    vo = np.zeros((rows, W + 1), np.int32)
    qp = np.zeros(rows, np.int32)
    for p in range(n_problems):
        base = p * (W + 1)
        for w in range(W):
            order = [base] + [base + 1 + o for o in range(W) if o != w] + [base + 1 + w]
            pos = 0
            for v, b in enumerate(order):
                vb[p * W + w, v] = b
                vo[p * W + w, v] = pos
                pos += int(block_len[b])
            qp[p * W + w] = pos
    return vb, vo, qp


def interleaved_views(block_len: Sequence[int], n_problems: int, n_workers: int):
    """The interleaved cache layout of the notes' layout ablation (step-level
    synchronisation only): a worker sees the common history - the prompt and
    every finished step committed into it - then its own unfinished step; the
    other workers' unfinished steps stay invisible until they are committed.
    Same block ids and return values as combined_views; unused view entries
    are -1 with offset 0.
    """
    W = n_workers
    rows = n_problems * W
    vb = np.full((rows, W + 1), -1, np.int32)
    vo = np.zeros((rows, W + 1), np.int32)
    qp = np.zeros(rows, np.int32)
    for p in range(n_problems):
        common = p * (W + 1)
        for w in range(W):
            own = common + 1 + w
            r = p * W + w
            vb[r, 0], vo[r, 0] = common, 0
            vb[r, 1], vo[r, 1] = own, int(block_len[common])
            qp[r] = int(block_len[common]) + int(block_len[own])
    return vb, vo, qp


def contiguous_views(block_len: Sequence[int], n_problems: int, n_workers: int):
    """The contiguous cache layout of the notes' layout ablation (token-level
    synchronisation only): every worker's whole generation is one growing
    block that is never committed, so the common block holds only the prompt;
    a worker sees the prompt, the other workers' generations in worker order,
    then its own - the combined order, over blocks that are never moved.
    """
    return combined_views(block_len, n_problems, n_workers)


def layout_views(layout: str, block_len: Sequence[int], n_problems: int, n_workers: int):
    """Views of a layout by name: "combined", "interleaved" or "contiguous"."""
    return {"combined": combined_views, "interleaved": interleaved_views,
            "contiguous": contiguous_views}[layout](block_len, n_problems, n_workers)


def chunk_views(layout: str, block_len: Sequence[int], n_problems: int, n_workers: int,
                chunk: int):
    """Views of T-token query chunks (T = chunk): each worker's last T tokens,
    already in its own block, are queried at once, one row per token.  Row
    (p, w, t), index (p*W + w)*T + t, sees the blocks of worker w's view in
    the layout's order; every other block whole, its own block only up to its
    own token (causal order inside the chunk): own block position
    len - T + t, so the first len - T + t + 1 tokens, and q_pos is that
    token's position in the view.  Returns (view_block, view_offset,
    view_limit, q_pos); view_limit is -1 (whole block) except on the own
    entry."""
    vb1, vo1, _ = layout_views(layout, block_len, n_problems, n_workers)
    W, T = n_workers, chunk
    rows = n_problems * W * T
    vb = np.repeat(vb1, T, axis=0)
    vo = np.repeat(vo1, T, axis=0)
    lim = np.full(vb.shape, -1, np.int32)
    qp = np.zeros(rows, np.int32)
    for p in range(n_problems):
        for w in range(W):
            own = p * (W + 1) + 1 + w
            n = int(block_len[own])
            assert n >= T, "each own block holds its chunk"
            for t in range(T):
                r = (p * W + w) * T + t
                v = int(np.where(vb[r] == own)[0][0])
                lim[r, v] = n - T + t + 1
                qp[r] = vo[r, v] + n - T + t
    return vb, vo, lim, qp



# ---------------------------------------------------------------------------
# The tensor-core kernel's work split, written out from its definition (for
# the bit-exact check of the plan the library exports; not the method's
# arithmetic, its scheduling).
# ---------------------------------------------------------------------------

def stream_k_split(block_start, block_len, view_block, n_q_heads: int, n_kv_heads: int,
                   grid: int, seg_weight: int = 2, tile: int = 128, max_cols: int = 32):
    """The work split of the KV cache over the SMs (omica.com.cn article, §3.2:
    the cache is divided evenly over the SMs, partial results merged).

    A segment is one column group of one (block, kv head): a block's query
    columns are its view references x the group size G, and a tile serves at
    most max_cols of them, so the references of block b, in view-entry order,
    form ng[b] = ceil(refs[b] / rpg) groups of rpg = max_cols // G (the last
    one shorter); reference k is in group k // rpg.  A block takes part when
    some view references it and it has tokens.  Units are 128-token tiles of
    one segment, ordered kv-head-major, then block, then group, then tile, so
    every group reads the block's tiles once.  Every unit weighs 1 and every
    segment start seg_weight more: unit (h, b, g, t) starts at weight
    h*WH + ubase[b] + g*tiles[b] + t + seg_weight*(sord[b] + g + 1), with
    ubase/sord the units/segments of the head before block b and
    WH = UH + seg_weight*NSH (units and segments per head).
    C = min(grid, W // (seg_weight + 1)) CTAs; CTA c < C takes the units whose
    weight lies in [floor(c W / C), floor((c+1) W / C)).

    Returns per CTA c < grid: (u0, u1, n_first, rows[3], heads[3], flags[3],
    groups[3]) as an int64 array [grid][15], the layout of hw_plan_export.
    """
    vb = np.asarray(view_block).ravel()
    G = n_q_heads // n_kv_heads
    assert 1 <= G <= max_cols
    rpg = max_cols // G
    nb = len(block_len)
    refs = np.array([(vb == b).sum() for b in range(nb)])
    taking = [refs[b] > 0 and block_len[b] > 0 for b in range(nb)]
    tiles = np.array([(int(block_len[b]) + tile - 1) // tile if taking[b] else 0
                      for b in range(nb)], np.int64)
    ng = np.array([-(-int(refs[b]) // rpg) if taking[b] else 0 for b in range(nb)], np.int64)
    UH = int((tiles * ng).sum())
    NSH = int(ng.sum())
    WH = UH + seg_weight * NSH
    W = WH * n_kv_heads
    C = min(grid, W // (seg_weight + 1))
    # every unit, brute force: (h, b, g, t) and its weight
    units = [(h, b, g, t) for h in range(n_kv_heads) for b in range(nb) for g in range(int(ng[b]))
             for t in range(int(tiles[b]))]
    ubase = np.concatenate([[0], np.cumsum(tiles * ng)])
    sord = np.concatenate([[0], np.cumsum(ng)])
    weight = np.array([h * WH + ubase[b] + g * tiles[b] + t + seg_weight * (sord[b] + g + 1)
                       for (h, b, g, t) in units], np.int64)
    assert np.all(np.diff(weight) > 0)
    out = np.zeros((grid, 15), np.int64)
    for c in range(grid):
        if c < C:
            u0 = int(np.searchsorted(weight, (W * c) // C, side="left"))
            u1 = int(np.searchsorted(weight, (W * (c + 1)) // C, side="left"))
        else:
            u0 = u1 = len(units)
        nf = min(3, u1 - u0)
        out[c, 0], out[c, 1], out[c, 2] = u0, u1, nf
        for i in range(nf):
            u = u0 + i
            h, b, g, t = units[u]
            first = u == u0 or t == 0
            last = u + 1 == u1 or t == tiles[b] - 1
            out[c, 3 + i] = int(block_start[b]) + t * tile
            out[c, 6 + i] = h
            out[c, 9 + i] = (1 if first else 0) | (2 if last else 0)
            out[c, 12 + i] = g
    return out
