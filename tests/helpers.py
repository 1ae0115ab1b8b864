"""Shared helpers for the GPU parity tests."""

import numpy as np

from workloads import build_workload

# Tolerance on attention outputs against the float64 oracle, per output
# tensor: max |got - ref| and max |got - ref| / max |ref|.  binary16: as
# specified for fp16 I/O with fp32 accumulation.  bfloat16 keeps 8 fraction
# bits instead of 11, so every rounding in the chain (stored q_rot and K, the
# fp16/bf16 probabilities fed to the tensor cores, the output) is 8x coarser:
# both bounds scale by 8.
TOL = {"f16": (2e-3, 1e-2), "bf16": (1.6e-2, 8e-2)}


def errors(got: np.ndarray, ref: np.ndarray):
    diff = np.abs(got - ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    denom = float(np.abs(ref).max()) if ref.size else 1.0
    return max_abs, max_abs / max(denom, 1e-30)


# (what, dtype, max abs, max rel, rows compared) of every check, printed at the
# end of the session by conftest.py
RECORDED = []


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "attention"):
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    max_abs, max_rel = errors(got, ref)
    RECORDED.append((what, dtype, max_abs, max_rel, int(got.shape[0]) if got.ndim else 1))
    atol, rtol = TOL[dtype]
    assert max_abs <= atol and max_rel <= rtol, "%s: max abs %.3g (tol %g), max rel %.3g (tol %g)" % (
        what, max_abs, atol, max_rel, rtol)
    return max_abs, max_rel


def custom(seed, *, Hq=32, Hkv=8, d=128, bs=16, dtype="f16", prefix, qlen, spare=8, shared_len=0, shared=(),
           theta=5.0e5):
    rng = np.random.Generator(np.random.PCG64(seed))
    return build_workload("custom", rng, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=bs, dtype=dtype,
                          theta=theta, prefix_lens=prefix, query_lens=qlen, spare_blocks=spare,
                          shared_prefix_len=shared_len, shared_seqs=shared)


def random_decode(seed, S, lo, hi, **kw):
    """S single-token decodes with contexts drawn from [lo, hi]."""
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    ctx = rng.integers(lo, hi, size=S, endpoint=True)
    return custom(seed, prefix=ctx - 1, qlen=np.ones(S, dtype=np.int64), **kw)


def one_sequence(w, s):
    """Sequence s of workload w on its own: same arena size and block ids,
    same q, k and v rows."""
    import dataclasses
    qsl, ks = w.query_start_loc, w.kv_start
    return dataclasses.replace(
        w, name="%s[%d]" % (w.name, s), prefix_lens=w.prefix_lens[s:s + 1].copy(),
        query_lens=w.query_lens[s:s + 1].copy(), block_tables=w.block_tables[s:s + 1].copy(),
        q=w.q[qsl[s]:qsl[s + 1]].copy(), k_all=w.k_all[ks[s]:ks[s + 1]].copy(),
        v_all=w.v_all[ks[s]:ks[s + 1]].copy(), shared_prefix_len=0, shared_seqs=())
