"""Pins for the float64 oracle: checks against things other than the oracle itself.

Each pin takes an ``oracle.Oracle`` handle and raises AssertionError when the
oracle disagrees with what the pages or the mathematics fix:

* golden frequencies worked out by hand from the rotate_query rule
  (omica.com.cn article, section 2.1) and the combined layout worked out by hand
  from key designs 1 and 2 of the Hogwild! notes;
* RoPE written as complex multiplication (pair (x_i, x_{i+D/2}) as
  x_i + 1j*x_{i+D/2}, rotated by exp(1j*pos*w_i)) - a different formulation of
  rotate_half that catches a wrong sign, pairing or direction;
* the query-rotation equation of key design 1: the block form (query rotated
  once per block) against brute force (every key re-encoded at its absolute
  position in the worker's view);
* textbook single-block decode attention through scipy's softmax/logsumexp;
* closed forms and invariants: q = 0 gives the mean of V, permuting blocks with
  their offsets fixed changes nothing, a saturating one-hot score returns one V
  row exactly, grouped-query head mapping, empty views;
* commit: delta 0 is a bit copy, V is a bit copy, nothing outside the target
  range moves, and rotating a stored key by delta equals encoding its raw key
  at the shifted position; a single worker's output does not change when its
  block is committed into the common history.

``tests/test_oracle_mutants.py`` builds the oracle with planted mistakes and
checks that every one of them fails at least one pin.
"""
from __future__ import annotations

import os

import numpy as np
from scipy.special import logsumexp, softmax

import oracle as O
from concurrent_shared_kv_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# independent helpers (not the oracle)
# ---------------------------------------------------------------------------

def golden_freqs():
    rows = []
    for line in open(os.path.join(GOLDEN, "rope_freqs.txt")):
        line = line.split("#")[0].split()
        if line:
            rows.append((int(line[0]), float(line[1]), int(line[2]), float(line[3])))
    return rows


def golden_tiny_layout():
    out = {}
    for line in open(os.path.join(GOLDEN, "combined_layout_tiny.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        a, b, c = line.split("|")
        a = a.split()
        out[int(a[0])] = ([int(x) for x in a[1:]], [int(x) for x in b.split()], int(c))
    return out


def complex_rope(x, w, pos):
    """RoPE as complex multiplication; w are the per-pair frequencies."""
    x = np.asarray(x, np.float64)
    h = x.shape[-1] // 2
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * pos * np.asarray(w))
    return np.concatenate([z.real, z.imag], axis=-1)


def case_tiny(dtype=O.F32, seed=7, D=16, Hq=4, Hkv=2, lens=(23, 5, 9), layout="combined"):
    """A small random problem: block 0 common, blocks 1.. workers."""
    rng = np.random.default_rng(seed)
    W = len(lens) - 1
    cap = [l + 3 for l in lens]  # slack slots filled with noise that must not be read
    starts = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int32)
    C = int(sum(cap))
    sd = "f32" if dtype == O.F32 else "bf16"
    k = wl.to_storage(rng.standard_normal((Hkv, C, D)) * 50, sd)
    v = wl.to_storage(rng.standard_normal((Hkv, C, D)) * 50, sd)
    kk = wl.to_storage(rng.standard_normal((Hkv, C, D)), sd)
    vv = wl.to_storage(rng.standard_normal((Hkv, C, D)), sd)
    for b in range(len(lens)):
        s = starts[b]
        k[:, s:s + lens[b]] = kk[:, s:s + lens[b]]
        v[:, s:s + lens[b]] = vv[:, s:s + lens[b]]
    q = wl.to_storage(rng.standard_normal((W, Hq, D)), sd)
    if layout == "combined":
        vb, vo, qp = O.combined_views(lens, 1, W)
    else:  # arbitrary offsets and orders: the equation holds for any of them
        vb = np.stack([rng.permutation(len(lens)) for _ in range(W)]).astype(np.int32)
        vo = rng.integers(0, 500, size=vb.shape).astype(np.int32)
        qp = rng.integers(0, 700, size=W).astype(np.int32)
    return dict(q=q, k_cache=k, v_cache=v, block_start=starts, block_len=np.asarray(lens, np.int32),
                view_block=vb, view_offset=vo, q_pos=qp, n_kv_heads=Hkv, rope_theta=1e4,
                scale=D ** -0.5, dtype=dtype)


def f64(x, dtype):
    return wl.storage_to_f64(x, "f32" if dtype == O.F32 else "bf16")


# ---------------------------------------------------------------------------
# RoPE pins
# ---------------------------------------------------------------------------

def pin_rope_golden_freqs(o: O.Oracle):
    for D, theta, i, w in golden_freqs():
        # rotate the unit vector e_i by one position: it lands on
        # (cos w_i, sin w_i) in the pair (i, i + D/2); w_i <= 1 < pi, so atan2
        # recovers w_i without ambiguity
        e = np.zeros(D)
        e[i] = 1.0
        y = o.rope(e, theta, 1.0)
        got = np.arctan2(y[i + D // 2], y[i])
        assert abs(got - w) <= 1e-12 * max(1.0, w), (D, theta, i, got, w)
        assert abs(o.freqs(D, theta)[i] - w) <= 1e-15 * max(w, 1e-300) * 8, (D, theta, i)


def pin_rope_complex(o: O.Oracle):
    rng = np.random.default_rng(1)
    for D, theta in [(2, 1e4), (8, 1e4), (64, 1e4), (128, 1e6)]:
        w = o.freqs(D, theta)
        for pos in [0.0, 1.0, -3.0, 17.0, 328.0, 70000.0]:
            x = rng.standard_normal(D)
            want = complex_rope(x, w, pos)
            got = o.rope(x, theta, pos)
            assert np.max(np.abs(got - want)) < 1e-12 * (1 + abs(pos)), (D, pos)


def pin_rope_group(o: O.Oracle):
    rng = np.random.default_rng(2)
    for D, theta in [(8, 1e4), (128, 1e6)]:
        x = rng.standard_normal(D)
        assert np.array_equal(o.rope(x, theta, 0.0), x)
        for a, b in [(3.0, 5.0), (-7.0, 7.0), (1000.0, -250.0)]:
            ab = o.rope(o.rope(x, theta, a), theta, b)
            assert np.max(np.abs(ab - o.rope(x, theta, a + b))) < 1e-12 * (1 + abs(a) + abs(b))
            assert abs(np.linalg.norm(o.rope(x, theta, a)) - np.linalg.norm(x)) < 1e-12


# ---------------------------------------------------------------------------
# attention pins
# ---------------------------------------------------------------------------

def pin_textbook_single_block(o: O.Oracle):
    """One worker, one block at offset 0: ordinary RoPE decode attention."""
    rng = np.random.default_rng(3)
    for D, n, Hq, Hkv in [(8, 1, 2, 1), (16, 37, 4, 2), (64, 200, 4, 2)]:
        theta = 1e4
        q = rng.standard_normal((1, Hq, D)).astype(np.float32)
        k = rng.standard_normal((Hkv, n, D)).astype(np.float32)
        v = rng.standard_normal((Hkv, n, D)).astype(np.float32)
        iq = n  # the query follows the block
        out, lse = o.attn_decode(q=q, k_cache=k, v_cache=v, block_start=[0], block_len=[n],
                                 view_block=[[0]], view_offset=[[0]], q_pos=[iq], n_kv_heads=Hkv,
                                 rope_theta=theta, scale=D ** -0.5, dtype=O.F32)
        w = o.freqs(D, theta)  # pinned on their own by pin_rope_golden_freqs
        for h in range(Hq):
            g = h // (Hq // Hkv)
            qa = complex_rope(q[0, h].astype(np.float64), w, iq)
            s = (k[g].astype(np.float64) @ qa) * D ** -0.5
            want = softmax(s) @ v[g].astype(np.float64)
            assert np.max(np.abs(out[0, h] - want)) < 1e-12, (D, n, h)
            assert abs(lse[0, h] - logsumexp(s)) < 1e-12, (D, n, h)


def pin_identity_block_vs_brute(o: O.Oracle):
    """Key design 1's equation: rotating the query by i_q - i_k^block against the
    stored keys equals re-encoding every key at its absolute view position."""
    for dtype in (O.F32, O.BF16):
        for seed, layout, D in [(11, "combined", 16), (12, "random", 16), (13, "combined", 64),
                                (14, "random", 8)]:
            c = case_tiny(dtype=dtype, seed=seed, D=D, layout=layout)
            a, la = o.attn_decode(**c)
            b, lb = o.attn_decode(**c, brute=True)
            scale = np.max(np.abs(b))
            assert np.max(np.abs(a - b)) <= 1e-12 * scale, (dtype, seed, layout)
            assert np.max(np.abs(la - lb)) <= 1e-12 * np.max(np.abs(lb)), (dtype, seed, layout)


def pin_q_zero_mean(o: O.Oracle):
    c = case_tiny(seed=21)
    c["q"] = np.zeros_like(c["q"])
    out, lse = o.attn_decode(**c)
    vv = f64(c["v_cache"], c["dtype"])
    Hq = c["q"].shape[1]
    G = Hq // c["n_kv_heads"]
    for r in range(c["q"].shape[0]):
        toks = [(c["block_start"][b], c["block_len"][b]) for b in c["view_block"][r] if b >= 0]
        N = sum(int(n) for _, n in toks)
        for h in range(Hq):
            rows = np.concatenate([vv[h // G, s:s + n] for s, n in toks])
            assert np.max(np.abs(out[r, h] - rows.mean(0))) < 1e-13
            assert abs(lse[r, h] - np.log(N)) < 1e-13


def pin_permutation_invariance(o: O.Oracle):
    c = case_tiny(seed=31, layout="random")
    a, la = o.attn_decode(**c)
    rng = np.random.default_rng(5)
    perm = np.stack([rng.permutation(c["view_block"].shape[1]) for _ in range(len(c["q"]))])
    c2 = dict(c)
    c2["view_block"] = np.take_along_axis(c["view_block"], perm, 1)
    c2["view_offset"] = np.take_along_axis(c["view_offset"], perm, 1)
    b, lb = o.attn_decode(**c2)
    assert np.max(np.abs(a - b)) < 1e-12 and np.max(np.abs(la - lb)) < 1e-12


def one_hot_case(o_freqs, D=16, seed=41, block=2, t=3, row=0, head=1, dtype=O.F32):
    """All keys zero except token t of `block`, and q chosen so that its score is
    >= 200 nats: the output must be that token's V row exactly."""
    c = case_tiny(dtype=dtype, seed=seed, D=D, layout="random")
    sd = "f32" if dtype == O.F32 else "bf16"
    k = np.zeros_like(c["k_cache"])
    Hq = c["q"].shape[1]
    g = head // (Hq // c["n_kv_heads"])
    s0 = c["block_start"][block]
    kt = wl.to_storage(np.random.default_rng(seed).standard_normal(D), sd)
    k[g, s0 + t] = kt
    c["k_cache"] = k
    v = np.where(c["view_block"][row] == block)[0]
    assert len(v) == 1
    off = c["view_offset"][row][v[0]]
    rel = int(c["q_pos"][row]) - int(off)
    ktd = f64(kt, dtype)
    # choose q with rho(q, rel) = lam * k_t  =>  score = lam*|k_t|^2*scale
    lam = 300.0 / (np.dot(ktd, ktd) * c["scale"])
    qv = complex_rope(lam * ktd, o_freqs(D), -rel)
    q = c["q"].copy()
    q[row, head] = wl.to_storage(qv, sd) if dtype == O.BF16 else qv.astype(np.float32)
    c["q"] = q
    return c, g, s0 + t


def pin_one_hot_exact(o: O.Oracle):
    for block, t, head in [(0, 0, 0), (0, 22, 1), (1, 4, 2), (2, 0, 3), (2, 8, 1)]:
        c, g, tok = one_hot_case(lambda D: o.freqs(D, 1e4), block=block, t=t, head=head)
        out, _ = o.attn_decode(**c)
        want = f64(c["v_cache"][g, tok], c["dtype"])
        assert np.array_equal(out[0, head], want), (block, t, head)


def pin_gqa_mapping(o: O.Oracle):
    c = case_tiny(seed=51)
    Hkv, C, D = c["k_cache"].shape
    v = np.zeros((Hkv, C, D), np.float32)
    for g in range(Hkv):
        v[g] = g + 1
    c["v_cache"] = v
    out, _ = o.attn_decode(**c)
    Hq = c["q"].shape[1]
    for h in range(Hq):
        assert np.max(np.abs(out[:, h] - (h // (Hq // Hkv) + 1))) < 1e-13, h
    qmap = np.array([1, 0, 1, 0], np.int32)
    out, _ = o.attn_decode(**c, q_to_kv=qmap)
    for h in range(Hq):
        assert np.max(np.abs(out[:, h] - (qmap[h] + 1))) < 1e-13, h


def pin_empty_view(o: O.Oracle):
    c = case_tiny(seed=61)
    c["block_len"] = np.array([0, 0, 0], np.int32)
    out, lse = o.attn_decode(**c)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    c = case_tiny(seed=61)
    c["view_block"] = np.full_like(c["view_block"], -1)
    out, lse = o.attn_decode(**c)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def pin_combined_layout(o: O.Oracle):
    vb, vo, qp = O.combined_views([256, 32, 40], 1, 2)
    for w, (blocks, offs, iq) in golden_tiny_layout().items():
        assert list(vb[w]) == blocks and list(vo[w]) == offs and qp[w] == iq, w


# ---------------------------------------------------------------------------
# commit pins
# ---------------------------------------------------------------------------

def commit_case(dtype, seed=71, D=16, Hkv=2, n=7):
    rng = np.random.default_rng(seed)
    sd = "f32" if dtype == O.F32 else "bf16"
    raw = rng.standard_normal((Hkv, n, D))
    return rng, sd, raw


def pin_commit_placement_and_copy(o: O.Oracle):
    for dtype in (O.F32, O.BF16):
        rng, sd, raw = commit_case(dtype)
        Hkv, n, D = raw.shape
        src_cap, dst_cap, s0, o0 = n + 5, 40, 3, 11
        ks = wl.to_storage(rng.standard_normal((Hkv, src_cap, D)), sd)
        vs = wl.to_storage(rng.standard_normal((Hkv, src_cap, D)), sd)
        sentinel = wl.to_storage(np.full((Hkv, dst_cap, D), -7.25), sd)
        kd, vd = o.block_commit(dtype=dtype, rope_theta=1e4, k_src=ks, v_src=vs, src_begin=s0,
                                n_tokens=n, k_dst=sentinel, v_dst=sentinel, dst_offset=o0,
                                pos_delta=0)
        assert np.array_equal(kd[:, o0:o0 + n], ks[:, s0:s0 + n])  # delta 0: bit copy
        assert np.array_equal(vd[:, o0:o0 + n], vs[:, s0:s0 + n])
        kd, vd = o.block_commit(dtype=dtype, rope_theta=1e4, k_src=ks, v_src=vs, src_begin=s0,
                                n_tokens=n, k_dst=sentinel, v_dst=sentinel, dst_offset=o0,
                                pos_delta=1234)
        assert np.array_equal(vd[:, o0:o0 + n], vs[:, s0:s0 + n])  # V never rotates
        for arr in (kd, vd):
            assert np.array_equal(arr[:, :o0], sentinel[:, :o0])
            assert np.array_equal(arr[:, o0 + n:], sentinel[:, o0 + n:])


def pin_commit_rotation(o: O.Oracle):
    """Stored key = raw key encoded at block-local j; after a commit by delta it
    must equal the raw key encoded at j + delta (complex formulation)."""
    for dtype, tol in ((O.F32, 1e-6), (O.BF16, None)):
        rng, sd, raw = commit_case(dtype, D=64, n=9)
        Hkv, n, D = raw.shape
        theta = 1e4
        w = o.freqs(D, theta)
        stored = np.stack([np.stack([complex_rope(raw[h, j], w, j) for j in range(n)])
                           for h in range(Hkv)])
        ks = wl.to_storage(stored, sd)
        vs = wl.to_storage(rng.standard_normal((Hkv, n, D)), sd)
        stored_q = f64(ks, dtype)
        for delta in (256, -5, 32768):
            kd, vd, exact = o.block_commit(dtype=dtype, rope_theta=theta, k_src=ks, v_src=vs,
                                           src_begin=0, n_tokens=n, k_dst=np.zeros_like(ks),
                                           v_dst=np.zeros_like(vs), dst_offset=0,
                                           pos_delta=delta, want_exact=True)
            want = np.stack([np.stack([complex_rope(stored_q[h, j], w, delta) for j in range(n)])
                             for h in range(Hkv)])
            assert np.max(np.abs(exact - want)) < 1e-10, (dtype, delta)
            # and through the raw key directly (storage rounding of the input aside)
            if dtype == O.F32:
                direct = np.stack([np.stack([complex_rope(raw[h, j], w, j + delta)
                                             for j in range(n)]) for h in range(Hkv)])
                assert np.max(np.abs(f64(kd, dtype) - direct)) < tol, delta
            else:
                # stored result is the exact value rounded once to bf16
                got = f64(kd, dtype)
                ulp = np.abs(want) * 2.0 ** -8
                assert np.all(np.abs(got - want) <= ulp + 1e-30), delta


def pin_commit_single_worker_invariance(o: O.Oracle):
    """W = 1: committing the worker's block into the common block at its own
    offset (delta = that offset) leaves the worker's attention output unchanged."""
    rng = np.random.default_rng(81)
    D, Hq, Hkv, C, n = 16, 2, 1, 20, 6
    cap_common = C + n
    k = np.zeros((Hkv, cap_common + n, D), np.float32)
    v = np.zeros_like(k)
    k[:, :C] = rng.standard_normal((Hkv, C, D))
    v[:, :C] = rng.standard_normal((Hkv, C, D))
    k[:, cap_common:] = rng.standard_normal((Hkv, n, D))
    v[:, cap_common:] = rng.standard_normal((Hkv, n, D))
    q = rng.standard_normal((1, Hq, D)).astype(np.float32)
    starts = [0, cap_common]
    before, lb = o.attn_decode(q=q, k_cache=k, v_cache=v, block_start=starts, block_len=[C, n],
                               view_block=[[0, 1]], view_offset=[[0, C]], q_pos=[C + n],
                               n_kv_heads=Hkv, rope_theta=1e4, scale=D ** -0.5, dtype=O.F32)
    kd, vd = o.block_commit(dtype=O.F32, rope_theta=1e4, k_src=k, v_src=v, src_begin=cap_common,
                            n_tokens=n, k_dst=k, v_dst=v, dst_offset=C, pos_delta=C)
    after, la = o.attn_decode(q=q, k_cache=kd, v_cache=vd, block_start=starts,
                              block_len=[C + n, 0], view_block=[[0, 1]], view_offset=[[0, C + n]],
                              q_pos=[C + n], n_kv_heads=Hkv, rope_theta=1e4, scale=D ** -0.5,
                              dtype=O.F32)
    assert np.max(np.abs(before - after)) < 1e-5 and np.max(np.abs(lb - la)) < 1e-5


def pin_bf16_rounding(o: O.Oracle):
    """The oracle's own double -> bf16 rounding against torch's float -> bf16 on
    values exact in float (so only one rounding happens on either side)."""
    rng = np.random.default_rng(91)
    xs = np.concatenate([rng.standard_normal(2000).astype(np.float32),
                         np.float32(1.0) + np.float32(2.0 ** -8) * np.arange(8, dtype=np.float32),
                         np.array([0.0, -0.0, 1e-40, -3e38, 3.3e38], np.float32)])
    want = wl.to_storage(xs.astype(np.float64), "bf16")
    got = np.array([o.bf16_from_double(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, want)


def pin_view_limits(o: O.Oracle):
    """Per-entry limits (a chunk's causal order within its block): limits at or
    past the block's length change nothing; a limit of 0 is the entry dropped;
    T query rows of one worker over one block at offset 0, row t at position
    P + t seeing the block's first P + t + 1 tokens, are textbook causal
    attention (scipy), row by row."""
    c = case_tiny()
    base_out, base_lse = o.attn_decode(**c)
    vb = c["view_block"]
    none = np.full(vb.shape, -1, np.int32)
    past = np.array([[c["block_len"][b] + 5 for b in row] for row in vb], np.int32)
    for lim in (none, past):
        out, lse = o.attn_decode(**c, view_limit=lim)
        assert np.array_equal(out, base_out) and np.array_equal(lse, base_lse)
    lim = none.copy()
    lim[0, 1] = 0
    out1, lse1 = o.attn_decode(**c, view_limit=lim)
    dropped = dict(c)
    dropped["view_block"] = vb.copy()
    dropped["view_block"][0, 1] = -1
    out2, lse2 = o.attn_decode(**dropped)
    assert np.array_equal(out1[0], out2[0]) and np.array_equal(lse1[0], lse2[0])
    assert not np.allclose(out1[0], base_out[0])  # the limit did hide tokens
    rng = np.random.default_rng(13)
    D, P, T, Hq, Hkv, theta = 16, 37, 3, 4, 2, 1e4
    n = P + T
    q = rng.standard_normal((T, Hq, D)).astype(np.float32)
    k = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    v = rng.standard_normal((Hkv, n, D)).astype(np.float32)
    out, lse = o.attn_decode(q=q, k_cache=k, v_cache=v, block_start=[0], block_len=[n],
                             view_block=[[0]] * T, view_offset=[[0]] * T,
                             q_pos=[P + t for t in range(T)], n_kv_heads=Hkv, rope_theta=theta,
                             scale=D ** -0.5, dtype=O.F32, view_limit=[[P + t + 1] for t in range(T)])
    w = o.freqs(D, theta)
    for t in range(T):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            qa = complex_rope(q[t, h].astype(np.float64), w, P + t)
            s_ = (k[g, :P + t + 1].astype(np.float64) @ qa) * D ** -0.5
            want = softmax(s_) @ v[g, :P + t + 1].astype(np.float64)
            assert np.max(np.abs(out[t, h] - want)) < 1e-12, (t, h)
            assert abs(lse[t, h] - logsumexp(s_)) < 1e-12, (t, h)


def pin_e4m3_codes(o: O.Oracle):
    """E4M3 decoding against torch's float8_e4m3fn for all 256 codes (the two
    NaN codes included), and rounding: values exactly representable in
    float32 against torch's cast, hand-worked ties and saturation, and every
    finite code back to itself."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    mine = np.array([o.e4m3_to_double(c) for c in codes])
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(mine[fin], ref[fin])
    for c in codes[fin]:
        got = o.e4m3_from_double(o.e4m3_to_double(c))
        assert got == c or (mine[c] == 0 and got & 0x7f == 0), c
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(4000) * np.exp2(rng.integers(-12, 9, 4000))).astype(np.float32)
    x = x[np.abs(x) < 440]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([o.e4m3_from_double(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, want)
    # ties to even: 17 between 16 and 18, 2^-10 between 0 and 2^-9, 3 * 2^-10
    # between 2^-9 and 2^-8; beyond 448 everything saturates
    for v, c in ((17.0, 0x58), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (448.0, 0x7E),
                 (465.0, 0x7E), (1e9, 0x7E), (-500.0, 0xFE), (0.0, 0x00)):
        assert o.e4m3_from_double(v) == c, (v, c)


def fp8_case(seed=3, D=16, Hq=4, Hkv=2, lens=(23, 5, 9)):
    """case_tiny with E4M3 caches (random codes, NaN codes avoided) and
    power-of-two head scales, different per head."""
    c = case_tiny(dtype=O.BF16, seed=seed, D=D, Hq=Hq, Hkv=Hkv, lens=lens)
    rng = np.random.default_rng(seed + 100)
    shape = c["k_cache"].shape
    k = rng.integers(0, 256, size=shape).astype(np.uint8)
    v = rng.integers(0, 256, size=shape).astype(np.uint8)
    for a in (k, v):
        a[(a & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    c.update(k_cache=k, v_cache=v, dtype=O.FP8)
    c["k_scale"] = np.exp2(rng.integers(-6, 3, Hkv)).astype(np.float32)
    c["v_scale"] = np.exp2(rng.integers(-6, 3, Hkv)).astype(np.float32)
    return c


def pin_fp8_decode_is_the_decode_of_the_scaled_values(o: O.Oracle):
    """A cache of E4M3 codes with power-of-two head scales is the fp32 cache
    of the decoded values times the scales (exact in fp32): the same outputs
    bit for bit; a head scale doubled doubles that head's outputs (V) or
    equals a query doubled (K)."""
    import torch
    c = fp8_case()
    out, lse = o.attn_decode(**c)
    dec = lambda a: torch.from_numpy(a).view(torch.float8_e4m3fn).float().numpy()
    f = dict(c)
    f.pop("k_scale"), f.pop("v_scale")
    f.update(dtype=O.F32, q=wl.storage_to_f64(c["q"], "bf16").astype(np.float32),
             k_cache=dec(c["k_cache"]) * c["k_scale"][:, None, None],
             v_cache=dec(c["v_cache"]) * c["v_scale"][:, None, None])
    out32, lse32 = o.attn_decode(**f)
    assert np.array_equal(out, out32) and np.array_equal(lse, lse32)
    g = dict(c, v_scale=c["v_scale"] * 2)
    out2, lse2 = o.attn_decode(**g)
    assert np.array_equal(out2, 2 * out) and np.array_equal(lse2, lse)


def pin_fp8_commit(o: O.Oracle):
    """E4M3 commit: delta 0 keeps every key value, values are copied as codes, and
    a rotated key is the E4M3 neighbour of the exact rotation (of the decoded
    key) nearest to it."""
    c = fp8_case(D=16)
    k, v = c["k_cache"], c["v_cache"]
    for delta in (0, 37):
        kd, vd, ex = o.block_commit(dtype=O.FP8, rope_theta=1e4, k_src=k, v_src=v, src_begin=0,
                                    n_tokens=5, k_dst=k, v_dst=v, dst_offset=40, pos_delta=delta,
                                    want_exact=True)
        assert np.array_equal(vd[:, 40:45], v[:, 0:5])
        dec = np.vectorize(o.e4m3_to_double)
        if delta == 0:  # the same values (a zero may change its sign: -0 - -0 = +0)
            assert np.array_equal(dec(kd[:, 40:45]), dec(k[:, 0:5]))
            nz = dec(k[:, 0:5]) != 0
            assert np.array_equal(kd[:, 40:45][nz], k[:, 0:5][nz])
        x = np.stack([np.stack([o.rope(dec(k[h, j]), 1e4, float(delta)) for j in range(5)])
                      for h in range(k.shape[0])])
        assert np.array_equal(x, ex)
        got = dec(kd[:, 40:45])
        # the nearest code: no finite code is closer to the exact value
        grid = np.array(sorted({o.e4m3_to_double(b) for b in range(256)
                                if not np.isnan(o.e4m3_to_double(b))}))
        xs = np.clip(x, -448, 448)
        best = np.min(np.abs(grid[None, :] - xs.reshape(-1, 1)), axis=1).reshape(xs.shape)
        assert np.all(np.abs(got - xs) <= best + 0.0)


ALL_PINS = [
    pin_rope_golden_freqs, pin_rope_complex, pin_rope_group, pin_textbook_single_block,
    pin_identity_block_vs_brute, pin_q_zero_mean, pin_permutation_invariance, pin_one_hot_exact,
    pin_gqa_mapping, pin_empty_view, pin_combined_layout, pin_commit_placement_and_copy,
    pin_commit_rotation, pin_commit_single_worker_invariance, pin_bf16_rounding, pin_view_limits,
    pin_e4m3_codes, pin_fp8_decode_is_the_decode_of_the_scaled_values, pin_fp8_commit,
]
