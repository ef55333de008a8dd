"""Pins for the float64 oracle, independent of the oracle's own formulas.

Each test checks the oracle against something it cannot share a mistake
with: hand-worked fixtures in tests/golden/ (each citing the passage of the
pages it follows), explicit-loop brute force on contiguous inputs, closed
forms, invariants (page permutation, causality, poison pages) and reductions
to a library routine (complex multiplication for the rotation).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def test_bf16_rounding_golden(golden_dir):
    g = _load(golden_dir, "bf16_rounding.json")
    for c in g["cases"]:
        got = float(oracle.round_to_bf16(np.array([c["x"]]))[0])
        assert got == c["bf16"], c


def test_bf16_rounding_matches_bit_level_rounding():
    # Two independent definitions of the same rounding: the oracle's
    # significant-bit quantisation and the generator's integer bit trick.
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200_000) * np.exp(rng.uniform(-30, 30, 200_000))).astype(np.float32)
    bits = synth.bf16_bits_from_f32(x)
    via_bits = synth.f32_from_bf16_bits(bits).astype(np.float64)
    via_oracle = oracle.round_to_bf16(x.astype(np.float64))
    assert np.array_equal(via_bits, via_oracle)
    assert np.array_equal(oracle.narrow(x.astype(np.float64), "bf16"), bits)
    assert np.array_equal(oracle.widen(bits, "bf16"), via_bits)


# ---------------------------------------------------------------------------
# slot mapping and KV write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", ["decode", "prefill"])
def test_slot_mapping_golden(golden_dir, case):
    g = _load(golden_dir, "slot_mapping_worked.json")
    c = g[case]
    pos, slots = oracle.slot_mapping(np.array(g["block_tables"]), c["context_lens"],
                                     c["cu_seqlens_q"], g["page_size"])
    assert pos.tolist() == c["positions"]
    assert slots.tolist() == c["slots"]


def test_kv_write_skip_untouched_and_bitwise():
    rng = np.random.default_rng(1)
    cache_shape = (6, 4, 2, 8)
    k_cache = np.full(cache_shape, 0x7FC0, dtype=np.uint16)
    v_cache = np.full(cache_shape, 0x7FC0, dtype=np.uint16)
    k = rng.integers(0, 1 << 16, size=(5, 2, 8)).astype(np.uint16)
    v = rng.integers(0, 1 << 16, size=(5, 2, 8)).astype(np.uint16)
    slots = np.array([3, -1, 17, 0, 23], dtype=np.int64)
    before_k, before_v = k_cache.copy(), v_cache.copy()
    oracle.kv_write(k, v, slots, k_cache, v_cache)
    flat_k = k_cache.reshape(24, 16)
    flat_v = v_cache.reshape(24, 16)
    for t, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(flat_k[s], k[t].reshape(-1))
            assert np.array_equal(flat_v[s], v[t].reshape(-1))
    untouched = np.setdiff1d(np.arange(24), slots[slots >= 0])
    assert np.array_equal(flat_k[untouched], before_k.reshape(24, 16)[untouched])
    assert np.array_equal(flat_v[untouched], before_v.reshape(24, 16)[untouched])
    # row 1 (slot -1) was written nowhere
    for s in range(24):
        assert not np.array_equal(flat_k[s], k[1].reshape(-1)) or s in slots


def test_slot_mapping_and_gather_round_trip():
    # Rows written through the slot formula come back, in logical order, from
    # a gather that only walks the block table page by page.
    wl = synth.make_workload("tiny_fp32_decode")
    k_cache = wl.poison_storage(wl.cache_shape())
    v_cache = wl.poison_storage(wl.cache_shape())
    _, slots = oracle.slot_mapping(wl.block_tables, wl.hist_lens, wl.cu_hist, wl.page_size)
    oracle.kv_write(wl.hist_k, wl.hist_v, slots, k_cache, v_cache)
    for b in range(wl.batch):
        n = int(wl.hist_lens[b])
        K, V = oracle.gather_kv(k_cache, v_cache, wl.block_tables[b], n, wl.dtype)
        lo, hi = wl.cu_hist[b], wl.cu_hist[b + 1]
        assert np.array_equal(K, wl.hist_k[lo:hi].astype(np.float64))
        assert np.array_equal(V, wl.hist_v[lo:hi].astype(np.float64))
    # the slots are distinct and never land in the poison page
    assert len(set(slots.tolist())) == len(slots)
    assert not np.any(slots // wl.page_size == wl.poison_page)


# ---------------------------------------------------------------------------
# RMSNorm and RoPE
# ---------------------------------------------------------------------------

def test_rmsnorm_golden_rounding_order(golden_dir):
    g = _load(golden_dir, "rmsnorm_worked.json")
    y = oracle.rms_norm(np.array([g["x"]]), np.array(g["w"]), g["eps"], g["dtype"])
    assert y[0].tolist() == g["y"]


def test_rmsnorm_closed_form_rms():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((50, 128)) * rng.uniform(0.01, 10, (50, 1))
    eps = 1e-6
    y = oracle.rms_norm(x, np.ones(128), eps, "f64")
    rms_y = np.sqrt(np.mean(y * y, axis=-1))
    ms_x = np.mean(x * x, axis=-1)
    assert np.allclose(rms_y, 1.0 / np.sqrt(1.0 + eps / ms_x), rtol=1e-13, atol=0)
    # scale invariance with eps = 0, and the weight acts elementwise
    w = rng.standard_normal(128)
    assert np.allclose(oracle.rms_norm(3.7 * x, w, 0.0, "f64"), oracle.rms_norm(x, w, 0.0, "f64"),
                       rtol=1e-13, atol=1e-15)
    assert np.allclose(oracle.rms_norm(x, w, eps, "f64"), oracle.rms_norm(x, np.ones(128), eps, "f64") * w,
                       rtol=1e-14, atol=0)


def test_rope_golden(golden_dir):
    g = _load(golden_dir, "rope_worked.json")
    for c in g["cases"]:
        y = oracle.rope(np.array([[c["x"]]], dtype=np.float64), [c["pos"]], g["theta"], "f64")
        assert np.allclose(y[0, 0], c["y"], rtol=0, atol=1e-15), c


def test_rope_is_complex_rotation():
    # Reduction to a library routine: pair (x1_i, x2_i) as the complex number
    # x1_i + i x2_i, multiplied by exp(i * pos * theta^(-2i/hd)).
    rng = np.random.default_rng(3)
    hd, theta = 128, 1e6
    x = rng.standard_normal((7, 3, hd))
    pos = rng.integers(0, 40000, 7)
    y = oracle.rope(x, pos, theta, "f64")
    z = x[..., : hd // 2] + 1j * x[..., hd // 2:]
    freqs = np.power(theta, -np.arange(hd // 2) * 2.0 / hd)
    w = z * np.exp(1j * pos[:, None, None] * freqs[None, None, :])
    assert np.allclose(y[..., : hd // 2], w.real, atol=1e-12)
    assert np.allclose(y[..., hd // 2:], w.imag, atol=1e-12)


def test_rope_invariants():
    rng = np.random.default_rng(4)
    hd, theta = 128, 1e6
    x = rng.standard_normal((5, 2, hd))
    assert np.array_equal(oracle.rope(x, [0] * 5, theta, "f64"), x)
    y = oracle.rope(x, [3, 77, 1000, 4095, 32767], theta, "f64")
    n_x = x[..., : hd // 2] ** 2 + x[..., hd // 2:] ** 2
    n_y = y[..., : hd // 2] ** 2 + y[..., hd // 2:] ** 2
    assert np.allclose(n_x, n_y, rtol=1e-12)
    # <R(m) q, R(n) k> depends only on m - n
    q = rng.standard_normal((1, 1, hd))
    k = rng.standard_normal((1, 1, hd))
    d1 = np.sum(oracle.rope(q, [100], theta, "f64") * oracle.rope(k, [40], theta, "f64"))
    d2 = np.sum(oracle.rope(q, [1060], theta, "f64") * oracle.rope(k, [1000], theta, "f64"))
    assert abs(d1 - d2) < 1e-9


def test_qk_norm_rope_golden(golden_dir):
    # Hand-worked q and k of two tokens at positions 1 and 2 with different
    # q and k norm weights: the weights, the positions and each bf16 cast
    # (after x*r, after the weight, after the rotation) all move some output.
    g = _load(golden_dir, "qk_norm_rope_worked.json")
    bf = lambda a: oracle.narrow(np.array(a, dtype=np.float64), "bf16")
    qo, ko = oracle.qk_norm_rope(bf(g["q"]), bf(g["k"]), bf(g["q_norm_w"]), bf(g["k_norm_w"]),
                                 np.array(g["positions"]), g["eps"], g["theta"], g["dtype"])
    assert oracle.widen(qo, "bf16").tolist() == g["q_out"]
    assert oracle.widen(ko, "bf16").tolist() == g["k_out"]


def test_qk_norm_rope_rows_are_independent_tokens():
    # A token of a chunk gives the same bits as that token alone at its
    # position, and every head of a token uses the one weight vector.
    rng = np.random.default_rng(5)
    n, Hq, Hkv, hd = 6, 4, 2, 16
    q = oracle.narrow(rng.standard_normal((n, Hq, hd)), "bf16")
    k = oracle.narrow(rng.standard_normal((n, Hkv, hd)), "bf16")
    wq = oracle.narrow(1 + 0.1 * rng.standard_normal(hd), "bf16")
    wk = oracle.narrow(1 + 0.1 * rng.standard_normal(hd), "bf16")
    pos = np.array([0, 1, 2, 37, 38, 4095])
    qo, ko = oracle.qk_norm_rope(q, k, wq, wk, pos, 1e-6, 1e6, "bf16")
    for t in range(n):
        q1, k1 = oracle.qk_norm_rope(q[t:t + 1], k[t:t + 1], wq, wk, pos[t:t + 1], 1e-6, 1e6, "bf16")
        assert np.array_equal(q1[0], qo[t]) and np.array_equal(k1[0], ko[t])
        for h in range(Hq):
            qh, _ = oracle.qk_norm_rope(q[t:t + 1, h:h + 1], k[t:t + 1, :1], wq, wk, pos[t:t + 1],
                                        1e-6, 1e6, "bf16")
            assert np.array_equal(qh[0, 0], qo[t, h])


def test_reference_step_rotates_new_tokens_at_their_positions():
    # The step's new tokens sit after each request's cached prefix: token j of
    # a chunk after c cached tokens is rotated at position c + j.
    chunks, prefixes = [1, 3, 2], [0, 9, 16]
    wl = synth.make_workload("qwen3_0p6b_chunked_prefill", chunks=chunks, prefixes=prefixes, B=3)
    r = oracle.reference_step(wl, with_attention=False)
    t = 0
    for b in range(3):
        for j in range(chunks[b]):
            q1, k1 = oracle.qk_norm_rope(wl.q[t:t + 1], wl.k_new[t:t + 1], wl.q_norm_w, wl.k_norm_w,
                                         np.array([prefixes[b] + j]), wl.eps, wl.rope_theta, "bf16")
            assert np.array_equal(r["q"][t], q1[0]) and np.array_equal(r["k"][t], k1[0])
            t += 1


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def _brute_attention(q, K, V, positions, scale):
    """Explicit loops over rows, heads, keys and dims; math.exp only."""
    n, Hq, hd = q.shape
    L, Hkv, _ = K.shape
    G = Hq // Hkv
    o = [[[0.0] * hd for _ in range(Hq)] for _ in range(n)]
    for i in range(n):
        for h in range(Hq):
            g = h // G
            scores = []
            for j in range(positions[i] + 1):
                acc = 0.0
                for d in range(hd):
                    acc += float(q[i, h, d]) * float(K[j, g, d])
                scores.append(scale * acc)
            m = max(scores)
            e = [math.exp(s - m) for s in scores]
            tot = sum(e)
            for d in range(hd):
                o[i][h][d] = sum(e[j] * float(V[j, g, d]) for j in range(len(e))) / tot
    return np.array(o)


def test_attention_golden(golden_dir):
    g = _load(golden_dir, "attention_worked.json")
    o, lse = oracle.attend(np.array(g["q"]), np.array(g["K"]), np.array(g["V"]), [1], g["scale"])
    assert np.allclose(o, g["o"], rtol=0, atol=1e-14)
    assert np.allclose(lse, g["lse"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_attention_matches_brute_force(G):
    rng = np.random.default_rng(5 + G)
    Hkv, hd, L, n = 2, 8, 13, 4
    q = rng.standard_normal((n, Hkv * G, hd))
    K = rng.standard_normal((L, Hkv, hd))
    V = rng.standard_normal((L, Hkv, hd))
    positions = [3, 7, 11, 12]
    o, _ = oracle.attend(q, K, V, positions, 0.3)
    ref = _brute_attention(q, K, V, positions, 0.3)
    assert np.max(np.abs(o - ref)) <= 1e-12


def _paged(K, V, P, rng, extra_pages=3, dtype=np.float64):
    """Place contiguous K/V rows into a shuffled page pool (test helper)."""
    L = K.shape[0]
    n = (L + P - 1) // P
    Np = n + extra_pages
    pages = rng.permutation(Np)[:n]
    kc = np.full((Np, P) + K.shape[1:], np.nan, dtype=dtype)
    vc = np.full((Np, P) + K.shape[1:], np.nan, dtype=dtype)
    for i in range(L):
        kc[pages[i // P], i % P] = K[i]
        vc[pages[i // P], i % P] = V[i]
    return kc, vc, pages


def test_decode_equals_contiguous_and_poison_never_read():
    rng = np.random.default_rng(8)
    L, Hkv, G, hd, P = 37, 2, 2, 16, 8
    K = rng.standard_normal((L, Hkv, hd))
    V = rng.standard_normal((L, Hkv, hd))
    q = rng.standard_normal((1, Hkv * G, hd))
    kc, vc, pages = _paged(K, V, P, rng)
    o, lse = oracle.decode(q.astype(np.float32), kc.astype(np.float32), vc.astype(np.float32),
                           pages[None], [L], 0.25, "f32")
    assert np.all(np.isfinite(o))      # NaN poison fills every unwritten slot
    ref = _brute_attention(q.astype(np.float32).astype(np.float64),
                           K.astype(np.float32).astype(np.float64),
                           V.astype(np.float32).astype(np.float64), [L - 1], 0.25)
    assert np.max(np.abs(o - ref)) <= 1e-12


def test_page_permutation_invariance_bitwise():
    wl = synth.make_workload("tiny_fp32_decode")
    r = oracle.reference_step(wl)
    rng = np.random.default_rng(9)
    perm = rng.permutation(wl.num_pages)           # new id of old page p is perm[p]
    kc = np.empty_like(r["k_cache"])
    vc = np.empty_like(r["v_cache"])
    kc[perm] = r["k_cache"]
    vc[perm] = r["v_cache"]
    bt = perm[wl.block_tables]
    o2, _ = oracle.decode(r["q"], kc, vc, bt, wl.context_lens, wl.scale, wl.dtype)
    assert np.array_equal(o2, r["o"])


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(10)
    q = rng.standard_normal((6, 4, 16)) * 3
    K = rng.standard_normal((20, 2, 16))
    V = rng.standard_normal((20, 2, 16))
    _, _, p = oracle.attend(q, K, V, [0, 3, 8, 12, 19, 19], 0.5, return_probs=True)
    assert np.all(p >= 0)
    assert np.max(np.abs(p.sum(-1) - 1.0)) <= 1e-12


def test_closed_forms():
    rng = np.random.default_rng(12)
    hd = 16
    V = rng.standard_normal((9, 1, hd))
    K = rng.standard_normal((9, 1, hd))
    # L = 1: the output is V_0 exactly
    o, _ = oracle.attend(rng.standard_normal((1, 2, hd)), K[:1], V[:1], [0], 1.0)
    assert np.array_equal(o[0, 0], V[0, 0]) and np.array_equal(o[0, 1], V[0, 0])
    # q = 0, or all keys equal: the mean of V
    o, _ = oracle.attend(np.zeros((1, 1, hd)), K, V, [8], 1.0)
    assert np.allclose(o[0, 0], V[:, 0].mean(0), atol=1e-14)
    Ksame = np.repeat(K[:1], 9, axis=0)
    o, _ = oracle.attend(rng.standard_normal((1, 1, hd)), Ksame, V, [8], 1.0)
    assert np.allclose(o[0, 0], V[:, 0].mean(0), atol=1e-14)
    # one dominant score: the output is that key's value
    q = np.zeros((1, 1, hd))
    q[0, 0, 0] = 1.0
    Kd = np.zeros((9, 1, hd))
    Kd[4, 0, 0] = 1000.0
    o, _ = oracle.attend(q, Kd, V, [8], 1.0)
    assert np.allclose(o[0, 0], V[4, 0], atol=1e-12)


def test_causal_mask_ignores_future_keys():
    rng = np.random.default_rng(13)
    q = rng.standard_normal((5, 2, 8))
    K = rng.standard_normal((12, 1, 8))
    V = rng.standard_normal((12, 1, 8))
    pos = [2, 5, 7, 9, 11]
    o1, _ = oracle.attend(q, K, V, pos, 0.7)
    K2, V2 = K.copy(), V.copy()
    K2[8:] += 50.0
    V2[8:] -= 50.0
    o2, _ = oracle.attend(q, K2, V2, pos, 0.7)
    assert np.array_equal(o1[:3], o2[:3])       # rows at positions <= 7
    assert not np.allclose(o1[3:], o2[3:])


def test_prefill_length_one_chunks_equal_decode():
    wl = synth.make_workload("qwen3_0p6b_decode", B=6)
    r = oracle.reference_step(wl)
    o_pf, lse_pf = oracle.prefill(r["q"], wl.cu_seqlens_q, r["k_cache"], r["v_cache"],
                                  wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
    assert np.array_equal(o_pf, r["o"]) and np.array_equal(lse_pf, r["lse"])


def test_prefill_without_prefix_is_causal_attention():
    spec = dict(kind="prefill", dtype="f32", B=2, Hq=4, Hkv=2, hd=8, P=4,
                chunks=[6, 9], prefixes=[0, 0], seed=14)
    wl = synth.make_workload(spec)
    r = oracle.reference_step(wl)
    for b in range(2):
        s0, s1 = wl.cu_seqlens_q[b], wl.cu_seqlens_q[b + 1]
        q = r["q"][s0:s1].astype(np.float64)
        K = wl.k_new[s0:s1].astype(np.float64)
        V = wl.v_new[s0:s1].astype(np.float64)
        ref = _brute_attention(q, K, V, list(range(s1 - s0)), wl.scale)
        assert np.max(np.abs(r["o"][s0:s1] - ref)) <= 1e-12


def test_prefill_with_prefix_matches_brute_force():
    spec = dict(kind="prefill", dtype="f32", B=2, Hq=4, Hkv=2, hd=8, P=4,
                chunks=[3, 5], prefixes=[7, 2], seed=15)
    wl = synth.make_workload(spec)
    r = oracle.reference_step(wl)
    for b in range(2):
        s0, s1 = wl.cu_seqlens_q[b], wl.cu_seqlens_q[b + 1]
        h0, h1 = wl.cu_hist[b], wl.cu_hist[b + 1]
        K = np.concatenate([wl.hist_k[h0:h1], wl.k_new[s0:s1]]).astype(np.float64)
        V = np.concatenate([wl.hist_v[h0:h1], wl.v_new[s0:s1]]).astype(np.float64)
        prefix = h1 - h0
        ref = _brute_attention(r["q"][s0:s1].astype(np.float64), K, V,
                               [prefix + i for i in range(s1 - s0)], wl.scale)
        assert np.max(np.abs(r["o"][s0:s1] - ref)) <= 1e-12


def test_split_merge_equals_unsplit():
    rng = np.random.default_rng(16)
    q = rng.standard_normal((4, 16))
    K = rng.standard_normal((100, 2, 16))
    V = rng.standard_normal((100, 2, 16))
    o_full, lse_full = oracle.attend(q[None], K, V, [99], 0.25)
    for bounds in ([(0, 100)], [(0, 37), (37, 100)], [(0, 1), (1, 50), (50, 64), (64, 100)]):
        op, lp = oracle.decode_partials(q, K, V, bounds, 0.25)
        o, lse = oracle.merge_partials(op, lp)
        assert np.max(np.abs(o - o_full[0])) <= 1e-12
        assert np.max(np.abs(lse - lse_full[0])) <= 1e-12


def test_norm_rope_step_bf16_values_are_bf16():
    wl = synth.make_workload("qwen3_0p6b_chunked_prefill", chunks=[1, 3], prefixes=[0, 9], B=2)
    r = oracle.reference_step(wl)
    assert r["q"].dtype == np.uint16 and r["k"].dtype == np.uint16
    q64 = oracle.widen(r["q"], "bf16")
    assert np.array_equal(oracle.round_to_bf16(q64), q64)
    assert np.all(np.isfinite(r["o"]))


def test_tolerance_rule():
    ref = np.array([0.5, -1.0, 2.0])
    assert oracle.within_tolerance(ref + 1.5e-2, ref, "bf16")[0]
    assert not oracle.within_tolerance(ref + 2.5e-2, ref, "bf16")[0]
    small = ref * 0.1                    # max|ref| = 0.2 -> bound 2e-3
    assert not oracle.within_tolerance(small + 5e-3, small, "bf16")[0]
    assert oracle.within_tolerance(ref + 9e-6, ref, "f32")[0]
    assert not oracle.within_tolerance(ref + 2e-5, ref, "f32")[0]
