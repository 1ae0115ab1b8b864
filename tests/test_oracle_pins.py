"""Pins for the float64 oracle (CPU only).

Each test checks the oracle against something other than itself: numpy's or
a brute-force IEEE rounding, mpmath, a pure-Python restatement, the pages'
online-softmax recurrence, closed forms and invariants.  Source: pages
"Building Kshipra" part 3 (kshipra-3), sections 1 (block arena, KV bytes per
token) and 4 (chunked prefill: online softmax over in-place blocks equals
dense masking; RoPE at absolute positions; causal mask over the chunk).
"""

import math
import os

import numpy as np
import pytest

from oracle import brute
from workloads import build_workload, make_config

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(seed, Hq, Hkv, d, bs, dtype, prefix, qlen, spare=0, shared_len=0, shared=(), theta=1.0e4):
    rng = np.random.Generator(np.random.PCG64(seed))
    return build_workload("t", rng, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=bs, dtype=dtype,
                          theta=theta, prefix_lens=prefix, query_lens=qlen, spare_blocks=spare,
                          shared_prefix_len=shared_len, shared_seqs=shared)


MICRO = [
    lambda: make_config("tiny"),
    lambda: small(11, 2, 2, 8, 4, "f16", [5, 0], [3, 2], spare=3),
    lambda: small(12, 8, 1, 16, 2, "bf16", [7], [4], spare=1, theta=5.0e5),
    lambda: small(13, 4, 2, 8, 4, "f16", [8, 9, 3], [2, 1, 4], spare=2, shared_len=8, shared=(0, 1)),
]


# ---------------------------------------------------------------- IEEE bits

def test_decode_f16_exhaustive(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.bits_to_f64(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_decode_bf16_exhaustive(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32)
    got = oracle_mod.bits_to_f64(bits.astype(np.uint16), "bf16")
    ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def _probe_doubles(rng, lo_exp, hi_exp, n=200000):
    mant = rng.uniform(1.0, 2.0, n)
    ex = rng.integers(lo_exp, hi_exp, n)
    sign = rng.choice([-1.0, 1.0], n)
    return sign * np.ldexp(mant, ex)


def _midpoints(finite_vals):
    v = np.sort(finite_vals[finite_vals >= 0])
    v = np.unique(v)
    return (v[:-1] + v[1:]) / 2.0  # exact in float64 for these small floats


def test_round_to_f16_matches_numpy(oracle_mod):
    rng = np.random.default_rng(0)
    all_h = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    fin = all_h[np.isfinite(all_h)]
    mids = _midpoints(fin)
    x = np.concatenate([_probe_doubles(rng, -30, 18), mids, -mids, fin,
                        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, np.inf, -np.inf, 2.0 ** -25,
                         2.0 ** -24, 3 * 2.0 ** -26, 1e-300]])
    got = oracle_mod.f64_to_bits(x, "f16")
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_round_to_bf16_bruteforce(oracle_mod):
    rng = np.random.default_rng(1)
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    pos = np.isfinite(vals) & (vals >= 0) & ~np.signbit(vals)
    table_v = vals[pos]
    table_b = bits[pos]
    order = np.argsort(table_v, kind="stable")
    table_v, table_b = table_v[order], table_b[order]
    mids = _midpoints(table_v)
    x = np.concatenate([_probe_doubles(rng, -140, 130, 100000), mids, -mids,
                        [0.0, 3.3895313892515355e38, 3.4e38, 1e39, 2.0 ** -133, 2.0 ** -134]])
    got = oracle_mod.f64_to_bits(x, "bf16").astype(np.uint32)
    ax = np.abs(x)
    hi = np.searchsorted(table_v, ax, side="left")
    exp = np.empty(len(x), dtype=np.uint32)
    maxv = table_v[-1]
    ulp_top = maxv - table_v[-2]
    for n in range(len(x)):
        a = ax[n]
        if a >= maxv + ulp_top / 2:  # rounds past the largest finite value
            e = 0x7F80
        elif hi[n] < len(table_v) and table_v[hi[n]] == a:
            e = table_b[hi[n]]
        else:
            lo_v, lo_b = table_v[hi[n] - 1], table_b[hi[n] - 1]
            if hi[n] >= len(table_v):
                e = 0x7F80 if a - lo_v >= ulp_top / 2 else lo_b
            else:
                up_v, up_b = table_v[hi[n]], table_b[hi[n]]
                dl, du = a - lo_v, up_v - a
                if dl < du:
                    e = lo_b
                elif du < dl:
                    e = up_b
                else:
                    e = lo_b if (lo_b & 1) == 0 else up_b
        if x[n] < 0 or (x[n] == 0 and np.signbit(x[n])):
            e |= 0x8000
        exp[n] = e
    assert np.array_equal(got, exp)


# ---------------------------------------------------------------- RoPE

def test_rope_table_against_mpmath(oracle_mod):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    for d, theta, max_pos in [(64, 1.0e4, 64), (128, 5.0e5, 40000)]:
        tab = oracle_mod.rope_table(max_pos, d, theta) if max_pos <= 64 else None
        rng = np.random.default_rng(d)
        for _ in range(60):
            p = int(rng.integers(0, max_pos))
            i = int(rng.integers(0, d // 2))
            if tab is None:
                tab_p = oracle_mod.rope_table(p + 1, d, theta)[p]
            else:
                tab_p = tab[p]
            ang = mpmath.mpf(p) * mpmath.power(mpmath.mpf(theta), mpmath.mpf(-2 * i) / d)
            # the float64 angle is rounded once: allow its half-ulp (<= 2^-37 here)
            assert abs(tab_p[i, 0] - float(mpmath.cos(ang))) < 1e-11
            assert abs(tab_p[i, 1] - float(mpmath.sin(ang))) < 1e-11


def test_rope_position_zero_is_identity(oracle_mod):
    w = make_config("tiny")
    out = oracle_mod.rope_rows(w.q, np.zeros(len(w.q), np.int32), w.theta, "f16")
    assert np.array_equal(out, w.q)


def test_rope_one_hot_rows_give_table_entries(oracle_mod):
    d, theta = 8, 1.0e4
    one = np.float16(1.0).view(np.uint16)
    rows = np.zeros((d // 2, 1, d), dtype=np.uint16)
    for i in range(d // 2):
        rows[i, 0, i] = one  # e_i
    pos = np.full(d // 2, 7, np.int32)
    out = oracle_mod.bits_to_f64(oracle_mod.rope_rows(rows, pos, theta, "f16"), "f16")
    tab = oracle_mod.rope_table(8, d, theta)[7].astype(np.float32)  # stored rotations use float32 cos/sin
    for i in range(d // 2):
        # rotating e_i gives (cos) at i and (+sin) at i + d/2, nothing else
        assert out[i, 0, i] == np.float16(tab[i, 0])
        assert out[i, 0, i + d // 2] == np.float16(tab[i, 1])
        rest = np.delete(out[i, 0], [i, i + d // 2])
        assert np.all(rest == 0)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_stored_rotation_is_one_rounding_from_exact(oracle_mod, dtype):
    # the stored (float32-computed) rotation differs from the exact rotation by
    # at most half a storage ulp plus the float32 error (a few 2^-24 relative)
    rng = np.random.default_rng(8)
    d, theta = 64, 1.0e4
    conv = {"f16": lambda a: a.astype(np.float16).view(np.uint16),
            "bf16": lambda a: ((a.astype(np.float32).view(np.uint32) + 0x8000) >> 16).astype(np.uint16)}[dtype]
    rows = conv(rng.standard_normal((200, 1, d)))
    pos = rng.integers(0, 5000, 200).astype(np.int32)
    got = oracle_mod.bits_to_f64(oracle_mod.rope_rows(rows, pos, theta, dtype), dtype)[:, 0]
    x = oracle_mod.bits_to_f64(rows, dtype)[:, 0]
    unit = 2.0 ** -11 if dtype == "f16" else 2.0 ** -8
    for t in range(200):
        exact = brute.rotate(list(x[t]), int(pos[t]), theta)
        for i in range(d):
            e = abs(got[t, i] - exact[i])
            assert e <= unit * abs(exact[i]) + 4 * 2.0 ** -24 * (abs(x[t, i]) + abs(x[t, (i + d // 2) % d])) + 1e-30


def _f32_rotation_restated(rows, pos, theta, dtype, mutate=None):
    """The stored rotation written out again with numpy float32 scalars in
    arrays (no code shared with the oracle): cos and sin of the float64
    angle position * theta^(-2i/d) from Python's math module, each rounded
    once to float32; y_i = x_i c - x_{i+d/2} s and y_{i+d/2} = x_{i+d/2} c +
    x_i s with every product and the add/subtract rounded to float32 (numpy
    never fuses them); then one rounding, nearest with ties to even, to the
    storage type.  ``mutate`` plants one plausible mistake: "fma" (the
    subtract/add fused with its first product, one rounding), "cos32" (the
    angle and its cos/sin evaluated in float32), "f64" (the whole rotation
    in float64, rounded once to storage)."""
    import math
    n, H, d = rows.shape
    h = d // 2
    if dtype == "f16":
        x = rows.view(np.float16).astype(np.float32)
    else:
        x = (rows.astype(np.uint32) << 16).view(np.float32)
    cs = {}
    for p in np.unique(pos):
        c = np.empty(h, np.float64)
        s = np.empty(h, np.float64)
        for i in range(h):
            ang = float(p) * theta ** (-2.0 * i / d)
            c[i], s[i] = math.cos(ang), math.sin(ang)
        if mutate == "cos32":
            ang32 = (np.float32(p) * (np.float32(theta) ** (np.float32(-2.0) * np.arange(h, dtype=np.float32)
                                                            / np.float32(d)))).astype(np.float32)
            cs[int(p)] = (np.cos(ang32).astype(np.float32), np.sin(ang32).astype(np.float32))
        elif mutate == "f64":
            cs[int(p)] = (c, s)
        else:
            cs[int(p)] = (c.astype(np.float32), s.astype(np.float32))
    C = np.stack([cs[int(p)][0] for p in pos])[:, None, :]
    S = np.stack([cs[int(p)][1] for p in pos])[:, None, :]
    a, b = x[..., :h], x[..., h:]
    if mutate == "f64":
        a, b = a.astype(np.float64), b.astype(np.float64)
        y = np.concatenate([a * C - b * S, b * C + a * S], axis=-1)
    elif mutate == "fma":
        a64, b64, C64, S64 = (v.astype(np.float64) for v in (a, b, C, S))
        lo = (a64 * C64 - (b * S).astype(np.float64)).astype(np.float32)  # a*c exact in float64
        hi = (b64 * C64 + (a * S).astype(np.float64)).astype(np.float32)
        y = np.concatenate([lo, hi], axis=-1)
    else:
        y = np.concatenate([a * C - b * S, b * C + a * S], axis=-1)
        assert y.dtype == np.float32
    if dtype == "f16":
        return y.astype(np.float16).view(np.uint16)
    u = y.astype(np.float32).view(np.uint32) if mutate != "f64" else None
    if mutate == "f64":  # one rounding of the float64 value straight to bfloat16
        from oracle import f64_to_bits
        return f64_to_bits(y, "bf16")
    return ((u + (((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF))) >> np.uint32(16)).astype(np.uint16)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d,theta", [(64, 1.0e4), (128, 5.0e5)])
def test_stored_rotation_bit_for_bit(oracle_mod, dtype, d, theta):
    # 100,000 rows at positions up to 32767 (4000 distinct, the ends included)
    rng = np.random.default_rng(17 + d)
    n = 100000
    draw = rng.standard_normal((n, 1, d)).astype(np.float32) * np.float32(3.0)
    if dtype == "f16":
        rows = draw.astype(np.float16).view(np.uint16)
    else:
        u = draw.view(np.uint32)
        rows = ((u + (((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF))) >> np.uint32(16)).astype(np.uint16)
    distinct = np.concatenate([[0, 1, 32766, 32767], rng.integers(0, 32768, 3996)])
    pos = distinct[rng.integers(0, len(distinct), n)].astype(np.int32)
    got = oracle_mod.rope_rows(rows, pos, theta, dtype)
    want = _f32_rotation_restated(rows, pos, theta, dtype)
    assert np.array_equal(got, want)
    # the pin is sharp: each planted mistake changes some of these rows
    for mutate in ("fma", "cos32", "f64"):
        assert not np.array_equal(got, _f32_rotation_restated(rows, pos, theta, dtype, mutate)), mutate


def _rot_f64(x, p, tab_row):
    h = len(x) // 2
    c, s = tab_row[:, 0], tab_row[:, 1]
    return np.concatenate([x[:h] * c - x[h:] * s, x[h:] * c + x[:h] * s])


def test_rope_relative_position_and_norm(oracle_mod):
    d, theta = 128, 5.0e5
    tab = oracle_mod.rope_table(5000, d, theta)
    rng = np.random.default_rng(3)
    for _ in range(20):
        x, y = rng.standard_normal(d), rng.standard_normal(d)
        p, p2, c = (int(v) for v in rng.integers(0, 2000, 3))
        a = _rot_f64(x, p, tab[p]) @ _rot_f64(y, p2, tab[p2])
        b = _rot_f64(x, p + c, tab[p + c]) @ _rot_f64(y, p2 + c, tab[p2 + c])
        assert abs(a - b) < 1e-9 * (1 + abs(a))
        assert abs(np.linalg.norm(_rot_f64(x, p, tab[p])) - np.linalg.norm(x)) < 1e-12 * np.linalg.norm(x)


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("make", MICRO)
def test_bruteforce_matches_oracle(oracle_mod, make):
    w = make()
    got = oracle_mod.workload_attention(w)
    ref = brute.attention(w.q.tolist(), w.k_all.tolist(), w.v_all.tolist(), w.prefix_lens.tolist(),
                          w.query_lens.tolist(), w.block_tables.tolist(), w.block_size, w.num_kv_heads, w.theta,
                          w.scale, w.dtype)
    assert np.max(np.abs(got - np.array(ref))) < 1e-12


def _random_micro(seed):
    """A random micro batch: group size, head_dim, block size, dtype, prefix
    and chunk lengths, shared prefix blocks and spare blocks drawn from a
    seeded generator."""
    rng = np.random.default_rng(500 + seed)
    Hkv = int(rng.integers(1, 3))
    G = int(rng.choice([1, 2, 4]))
    d = int(rng.choice([4, 8, 16]))
    bs = int(rng.choice([2, 4, 8]))
    S = int(rng.integers(1, 4))
    prefix = [int(rng.integers(0, 14)) for _ in range(S)]
    qlen = [int(rng.integers(1, 6)) for _ in range(S)]
    shared_len, shared = 0, ()
    members = [i for i in range(S) if prefix[i] >= bs]
    if len(members) >= 2 and rng.random() < 0.5:
        shared_len, shared = bs, tuple(members)
    theta = float(rng.choice([1.0e4, 5.0e5]))
    return small(600 + seed, G * Hkv, Hkv, d, bs, str(rng.choice(["f16", "bf16"])), prefix, qlen,
                 spare=int(rng.integers(0, 4)), shared_len=shared_len, shared=shared, theta=theta)


@pytest.mark.parametrize("seed", range(12))
def test_bruteforce_matches_oracle_random(oracle_mod, seed):
    w = _random_micro(seed)
    got = oracle_mod.workload_attention(w)
    ref = brute.attention(w.q.tolist(), w.k_all.tolist(), w.v_all.tolist(), w.prefix_lens.tolist(),
                          w.query_lens.tolist(), w.block_tables.tolist(), w.block_size, w.num_kv_heads, w.theta,
                          w.scale, w.dtype)
    assert np.max(np.abs(got - np.array(ref))) < 1e-12


def _rotated_f64(oracle_mod, w):
    """q and k rotated in float64 through the oracle's table (test restatement)."""
    tab = oracle_mod.rope_table(w.max_context_len + 1, w.head_dim, w.theta)
    q = oracle_mod.bits_to_f64(w.q, w.dtype)
    k = oracle_mod.bits_to_f64(w.k_all, w.dtype)
    v = oracle_mod.bits_to_f64(w.v_all, w.dtype)
    pos = w.positions
    qr = np.stack([np.stack([_rot_f64(q[t, h], pos[t], tab[pos[t]]) for h in range(q.shape[1])])
                   for t in range(len(q))])
    ks = w.kv_start
    kr = np.empty_like(k)
    for s in range(w.num_seqs):
        for j in range(int(w.context_lens[s])):
            for h in range(w.num_kv_heads):
                kr[ks[s] + j, h] = _rot_f64(k[ks[s] + j, h], j, tab[j])
    return qr, kr, v


def _online(qrow, K, V, scale, bs, upto):
    """The pages' per-row loop: running max m, sum l, rescaled accumulator o,
    one KV block at a time (kshipra-3 section 4)."""
    m, l, o = -np.inf, 0.0, np.zeros(K.shape[1])
    for b0 in range(0, upto, bs):
        kb, vb = K[b0:min(b0 + bs, upto)], V[b0:min(b0 + bs, upto)]
        s = kb @ qrow * scale
        m_new = max(m, s.max())
        p = np.exp(s - m_new)
        l = l * np.exp(m - m_new) + p.sum()
        o = o * np.exp(m - m_new) + p @ vb
        m = m_new
    return o / l


@pytest.mark.parametrize("make", MICRO)
def test_online_softmax_equals_dense(oracle_mod, make):
    w = make()
    qr, kr, v = _rotated_f64(oracle_mod, w)
    dense = oracle_mod.workload_attention(w)
    G = w.num_q_heads // w.num_kv_heads
    qsl, ks, pos = w.query_start_loc, w.kv_start, w.positions
    for s in range(w.num_seqs):
        for t in range(qsl[s], qsl[s + 1]):
            for h in range(w.num_q_heads):
                g = h // G
                K = kr[ks[s]:ks[s + 1], g]
                V = v[ks[s]:ks[s + 1], g]
                o = _online(qr[t, h], K, V, w.scale, w.block_size, int(pos[t]) + 1)
                assert np.max(np.abs(o - dense[t, h])) < 1e-12


def _merge(parts):
    """Combine (m, l, o) partials of disjoint key ranges (log-sum-exp rule)."""
    M = max(p[0] for p in parts)
    L = sum(p[1] * np.exp(p[0] - M) for p in parts)
    O = sum(p[2] * np.exp(p[0] - M) for p in parts)
    return O / L


def _partial(qrow, K, V, scale):
    s = K @ qrow * scale
    m = s.max()
    p = np.exp(s - m)
    return m, p.sum(), p @ V


def test_split_combine_equals_dense(oracle_mod):
    w = small(21, 4, 1, 16, 4, "f16", [60, 33], [1, 3])
    qr, kr, v = _rotated_f64(oracle_mod, w)
    dense = oracle_mod.workload_attention(w)
    qsl, ks, pos = w.query_start_loc, w.kv_start, w.positions
    rng = np.random.default_rng(5)
    for s in range(w.num_seqs):
        for t in range(qsl[s], qsl[s + 1]):
            n = int(pos[t]) + 1
            for h in range(w.num_q_heads):
                K, V = kr[ks[s]:ks[s] + n, 0], v[ks[s]:ks[s] + n, 0]
                cuts = sorted(set(int(c) for c in rng.integers(1, n, 3))) if n > 1 else []
                edges = [0] + cuts + [n]
                parts = [_partial(qr[t, h], K[a:b], V[a:b], w.scale) for a, b in zip(edges[:-1], edges[1:])]
                assert np.max(np.abs(_merge(parts) - dense[t, h])) < 1e-12


def test_decode_equals_last_row_of_prefill(oracle_mod):
    # the oracle's decode of each sequence's last token equals the last row of
    # the brute-force prefill over the same sequence (kshipra-3 section 4:
    # a query at position p sees keys 0..p whichever call it comes in)
    w = small(31, 8, 2, 32, 4, "f16", [19, 4], [9, 6], spare=2)
    full = brute.attention(w.q.tolist(), w.k_all.tolist(), w.v_all.tolist(), w.prefix_lens.tolist(),
                           w.query_lens.tolist(), w.block_tables.tolist(), w.block_size, w.num_kv_heads, w.theta,
                           w.scale, w.dtype)
    w1 = small(31, 8, 2, 32, 4, "f16", [19, 4], [9, 6], spare=2)
    w1.prefix_lens = w.prefix_lens + w.query_lens - 1
    w1.query_lens = np.ones_like(w.query_lens)
    last = w.query_start_loc[1:] - 1
    w1.q = w.q[last]
    dec = oracle_mod.workload_attention(w1)
    assert np.max(np.abs(dec - np.array(full)[last])) < 1e-12


def test_first_token_attends_only_to_itself(oracle_mod):
    # a chunk with no cached prefix: its first query sees one key, so out = v_0
    w = small(41, 4, 2, 16, 4, "f16", [0], [5])
    out = oracle_mod.workload_attention(w)
    v0 = oracle_mod.bits_to_f64(w.v_all[0], "f16")
    G = 2
    for h in range(4):
        assert np.array_equal(out[0, h], v0[h // G])


def test_zero_query_averages_visible_values(oracle_mod):
    w = small(42, 4, 2, 16, 4, "f16", [10, 3], [3, 1])
    w.q = np.zeros_like(w.q)
    out = oracle_mod.workload_attention(w)
    v = oracle_mod.bits_to_f64(w.v_all, "f16")
    qsl, ks, pos = w.query_start_loc, w.kv_start, w.positions
    for s in range(w.num_seqs):
        for t in range(qsl[s], qsl[s + 1]):
            for h in range(4):
                mean = v[ks[s]:ks[s] + pos[t] + 1, h // 2].mean(axis=0)
                assert np.max(np.abs(out[t, h] - mean)) < 1e-14


def test_dominant_key_selects_its_value(oracle_mod):
    # with a huge scale the softmax puts all weight on the best-scoring key
    w = small(43, 2, 1, 16, 4, "f16", [12], [1])
    qr, kr, v = _rotated_f64(oracle_mod, w)
    w.scale = 1.0e4
    out = oracle_mod.workload_attention(w)
    for h in range(2):
        best = int(np.argmax(kr[:13, 0] @ qr[0, h]))
        assert np.max(np.abs(out[0, h] - v[best, 0])) < 1e-9


@pytest.mark.parametrize("make", MICRO)
def test_arena_route_equals_logical_route(oracle_mod, make):
    # keys and values written into the oracle's arena and gathered back
    # through the block tables are the rows read in logical order (kshipra-3
    # section 1), shared prefix blocks included
    w = make()
    assert np.array_equal(oracle_mod.workload_attention(w), oracle_mod.workload_attention(w, gather=False))


def test_arena_route_rejects_aliased_blocks(oracle_mod):
    # two sequences whose tables name one physical block for different rows
    w = small(61, 4, 2, 8, 4, "f16", [9, 14], [3, 1], spare=3)
    w.block_tables[1, 0] = w.block_tables[0, 0]
    with pytest.raises(ValueError, match="two different rows"):
        oracle_mod.workload_attention(w)
    # the same aliasing inside one sequence
    w = small(62, 4, 2, 8, 4, "f16", [9], [3], spare=3)
    w.block_tables[0, 1] = w.block_tables[0, 0]
    with pytest.raises(ValueError, match="two different rows"):
        oracle_mod.workload_attention(w)


def test_arena_route_rejects_ids_outside_the_arena(oracle_mod):
    w = small(63, 4, 2, 8, 4, "f16", [9, 14], [3, 1], spare=3)
    w.block_tables[0, 2] = w.num_blocks
    with pytest.raises(ValueError, match="outside the arena"):
        oracle_mod.workload_attention(w)


def test_arena_route_reports_a_gathered_nan(oracle_mod):
    w = small(64, 4, 2, 8, 4, "f16", [9, 14], [3, 1], spare=3)
    w.k_all[5, 1, 3] = 0x7E00  # a NaN row in the arena
    with pytest.raises(ValueError, match="NaN"):
        oracle_mod.workload_attention(w)


# ---------------------------------------------------------------- arena

def _gather(arena, table, s, ctx, bs):
    return np.stack([arena[table[s, j // bs], :, j % bs] for j in range(ctx)])


@pytest.mark.parametrize("make", MICRO)
def test_arena_image_placement(oracle_mod, make):
    w = make()
    sentinel = 0x7E01  # a NaN pattern in both binary16 and bfloat16
    ka, va = oracle_mod.workload_arena(w, sentinel)
    ks = w.kv_start
    used = np.zeros(ka.shape[:3], dtype=bool)
    krot_all = oracle_mod.rope_rows(w.k_all, np.concatenate([np.arange(c) for c in w.context_lens]).astype(np.int32),
                                    w.theta, w.dtype)
    for s in range(w.num_seqs):
        ctx = int(w.context_lens[s])
        # values are stored bit for bit, keys as their rotation at the row's position
        assert np.array_equal(_gather(va, w.block_tables, s, ctx, w.block_size), w.v_all[ks[s]:ks[s + 1]])
        assert np.array_equal(_gather(ka, w.block_tables, s, ctx, w.block_size), krot_all[ks[s]:ks[s + 1]])
        for j in range(ctx):
            used[w.block_tables[s, j // w.block_size], :, j % w.block_size] = True
    # slots that no row maps to keep the sentinel
    assert np.all(ka[~used] == sentinel) and np.all(va[~used] == sentinel)
    # position 0 is not rotated
    for s in range(w.num_seqs):
        assert np.array_equal(ka[w.block_tables[s, 0], :, 0], w.k_all[ks[s]])


def test_arena_image_follows_block_permutation(oracle_mod):
    w = small(51, 4, 2, 8, 4, "f16", [9, 14], [3, 1], spare=3)
    ka, va = oracle_mod.workload_arena(w, 0)
    perm = np.random.default_rng(2).permutation(w.num_blocks).astype(np.int32)
    w2 = small(51, 4, 2, 8, 4, "f16", [9, 14], [3, 1], spare=3)
    w2.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    ka2, va2 = oracle_mod.workload_arena(w2, 0)
    assert np.array_equal(ka2[perm], ka) and np.array_equal(va2[perm], va)


def test_shared_prefix_blocks_written_consistently(oracle_mod):
    w = small(52, 4, 2, 8, 4, "f16", [8, 9, 12], [2, 1, 3], spare=1, shared_len=8, shared=(0, 2))
    ka, va = oracle_mod.workload_arena(w, 0)
    # the two sharing sequences read identical rows for the shared positions
    g0 = _gather(ka, w.block_tables, 0, 8, 4)
    g2 = _gather(ka, w.block_tables, 2, 8, 4)
    assert np.array_equal(g0, g2)
    assert np.array_equal(w.block_tables[0, :2], w.block_tables[2, :2])


# ---------------------------------------------------------------- sizing

def test_kv_bytes_formula_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "kv_bytes.txt")) if l.strip() and not l.startswith("#")]
    for layers, heads, hd, be, tokens, expected in (map(int, r) for r in rows):
        assert 2 * layers * heads * hd * be * tokens == expected
    # the printed round numbers
    assert 131072 == 128 * 1024 and 536870912 == 512 * 1024 ** 2 and 2147483648 == 2 * 1024 ** 3
