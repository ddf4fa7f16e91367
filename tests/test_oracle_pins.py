"""Pins of the fp64 oracle against facts fixed outside it.

Each test checks the oracle (``oracle/``) against something it does not share
code with: a pure-Python brute-force softmax written here (no block table, no
max subtraction, math.fsum), closed forms, and invariants the pages state
(paging changes layout, not the attention scores -- Triptych "Paged Attention
for Efficient Memory Management", body; aitalk "PagedAttention: Memory Like an
Operating System").  The placement of logical tokens into the pool is done
here with a separate loop, so a wrong index in the oracle's gather fails the
brute-force comparison.
"""
import math
import zlib

import numpy as np
import pytest

B = 16


# ---------------------------------------------------------------- helpers
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 -> bfloat16 bits (ties to even), from the IEEE definition."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def brute_attention(q, K, V, scale):
    """Textbook softmax attention, one query: no max subtraction, fsum sums."""
    n = len(K)
    w = [math.exp(scale * math.fsum(q[d] * K[j][d] for d in range(len(q)))) for j in range(n)]
    den = math.fsum(w)
    return [math.fsum(w[j] * V[j][d] for j in range(n)) / den for d in range(len(q))]


def place(logical, table, num_blocks, fill=np.nan):
    """Scatter logical per-sequence caches [S][L_s][Hkv][D] into a pool [NB,Hkv,B,D]."""
    hkv, d = logical[0].shape[1], logical[0].shape[2]
    pool = np.full((num_blocks, hkv, B, d), fill, dtype=logical[0].dtype)
    for s, arr in enumerate(logical):
        for j in range(arr.shape[0]):
            pool[table[s][j // B], :, j % B, :] = arr[j]
    return pool


def make_tables(lens, num_blocks, rng):
    nblk = [math.ceil(L / B) for L in lens]
    perm = rng.permutation(num_blocks)[:sum(nblk)]
    table = np.full((len(lens), max(nblk)), -1, np.int32)
    pos = 0
    for s, n in enumerate(nblk):
        table[s, :n] = perm[pos:pos + n]
        pos += n
    return table


def rand_case(rng, lens, hq, hkv, d, num_blocks, dtype="f32"):
    K = [rng.standard_normal((L, hkv, d)).astype(np.float32) for L in lens]
    V = [rng.standard_normal((L, hkv, d)).astype(np.float32) for L in lens]
    q = rng.standard_normal((len(lens), hq, d)).astype(np.float32)
    if dtype == "bf16":
        K = [bf16_bits(k) for k in K]
        V = [bf16_bits(v) for v in V]
        q = bf16_bits(q)
    table = make_tables(lens, num_blocks, rng)
    fill = np.nan if dtype == "f32" else np.uint16(0x7FC0)
    kp = place(K, table, num_blocks, fill)
    vp = place(V, table, num_blocks, fill)
    return q, K, V, kp, vp, table


def as_f64(a):
    return bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(4, 4, 64, (17, 33, 5, 64)),     # the tiny published config
                                   (8, 2, 4, (1, 16, 70, 31)),       # GQA 4, D 4
                                   (2, 1, 64, (15, 17, 48))])        # GQA 2
def test_decode_matches_brute_force(oracle_mod, dtype, shape):
    hq, hkv, d, lens = shape
    rng = np.random.default_rng(zlib.crc32(repr((dtype, shape)).encode()))
    q, K, V, kp, vp, table = rand_case(rng, lens, hq, hkv, d, 64, dtype)
    scale = 1.0 / math.sqrt(d)
    got = oracle_mod.paged_decode(q, kp, vp, table, np.array(lens, np.int32), scale)
    G = hq // hkv
    for s, L in enumerate(lens):
        Kf, Vf, qf = as_f64(K[s]), as_f64(V[s]), as_f64(q[s])
        for h in range(hq):
            ref = brute_attention(list(qf[h]), Kf[:, h // G].tolist(), Vf[:, h // G].tolist(),
                                  scale)
            np.testing.assert_allclose(got[s, h], ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("cached,new", [((0, 5), (9, 3)), ((20, 1), (1, 16)), ((33,), (31,))])
def test_prefill_matches_brute_force(oracle_mod, cached, new):
    hq, hkv, d = 4, 2, 8
    rng = np.random.default_rng(sum(cached) * 131 + sum(new))
    lens = [c + n for c, n in zip(cached, new)]
    K = [rng.standard_normal((L, hkv, d)).astype(np.float32) for L in lens]
    V = [rng.standard_normal((L, hkv, d)).astype(np.float32) for L in lens]
    table = make_tables(lens, 32, rng)
    kp, vp = place(K, table, 32), place(V, table, 32)
    N = sum(new)
    q = rng.standard_normal((N, hq, d)).astype(np.float32)
    qo = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    scale = 0.3
    got = oracle_mod.paged_prefill(q, kp, vp, table, np.array(cached, np.int32),
                                   np.array(new, np.int32), qo, scale)
    G = hq // hkv
    for r, (c, n) in enumerate(zip(cached, new)):
        for i in range(n):
            for h in range(hq):
                keys = K[r][:c + i + 1, h // G].astype(np.float64).tolist()
                vals = V[r][:c + i + 1, h // G].astype(np.float64).tolist()
                ref = brute_attention(q[qo[r] + i, h].astype(np.float64).tolist(), keys, vals,
                                      scale)
                np.testing.assert_allclose(got[qo[r] + i, h], ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- closed forms
def _single(oracle_mod, K, V, q, scale=0.125):
    L, d = K.shape
    table = make_tables([L], 8, np.random.default_rng(L))
    kp = place([K[:, None, :]], table, 8)
    vp = place([V[:, None, :]], table, 8)
    return oracle_mod.paged_decode(q[None, None, :], kp, vp, table, np.array([L], np.int32),
                                   scale)[0, 0]


def test_constant_values_give_that_constant(oracle_mod):
    rng = np.random.default_rng(1)
    K = rng.standard_normal((37, 16)).astype(np.float32)
    V = np.tile(rng.standard_normal(16).astype(np.float32), (37, 1))
    out = _single(oracle_mod, K, V, rng.standard_normal(16).astype(np.float32))
    np.testing.assert_allclose(out, V[0], rtol=1e-13)


def test_single_token_returns_its_value(oracle_mod):
    rng = np.random.default_rng(2)
    K = rng.standard_normal((1, 16)).astype(np.float32)
    V = rng.standard_normal((1, 16)).astype(np.float32)
    out = _single(oracle_mod, K, V, rng.standard_normal(16).astype(np.float32))
    np.testing.assert_array_equal(out, V[0].astype(np.float64))


def test_zero_query_gives_mean_value(oracle_mod):
    rng = np.random.default_rng(3)
    K = rng.standard_normal((50, 16)).astype(np.float32)
    V = rng.standard_normal((50, 16)).astype(np.float32)
    out = _single(oracle_mod, K, V, np.zeros(16, np.float32))
    np.testing.assert_allclose(out, V.astype(np.float64).mean(0), rtol=1e-12, atol=1e-15)


def test_identical_keys_give_mean_value(oracle_mod):
    """Every key the same: all scores equal whatever the query, so the weights are
    uniform and the output is the mean of V (a scale applied to only some scores, or a
    key index mixed up with a value index, breaks this)."""
    rng = np.random.default_rng(13)
    k = rng.standard_normal(16).astype(np.float32)
    K = np.tile(k, (37, 1))
    V = rng.standard_normal((37, 16)).astype(np.float32)
    out = _single(oracle_mod, K, V, rng.standard_normal(16).astype(np.float32) * 4, 0.7)
    np.testing.assert_allclose(out, V.astype(np.float64).mean(0), rtol=1e-12, atol=1e-15)


def test_two_tokens_sigmoid_weights(oracle_mod):
    rng = np.random.default_rng(4)
    K = rng.standard_normal((2, 16)).astype(np.float32)
    V = rng.standard_normal((2, 16)).astype(np.float32)
    q = rng.standard_normal(16).astype(np.float32)
    scale = 0.5
    x = scale * (K.astype(np.float64) @ q.astype(np.float64))
    w0 = 1.0 / (1.0 + math.exp(x[1] - x[0]))
    ref = w0 * V[0].astype(np.float64) + (1 - w0) * V[1].astype(np.float64)
    np.testing.assert_allclose(_single(oracle_mod, K, V, q, scale), ref, rtol=1e-12)


def test_dominant_score_selects_its_value(oracle_mod):
    rng = np.random.default_rng(5)
    K = rng.standard_normal((40, 16)).astype(np.float32)
    V = rng.standard_normal((40, 16)).astype(np.float32)
    q = np.zeros(16, np.float32)
    q[0] = 1.0
    K[:, 0] = 0.0
    K[23, 0] = 1.0e4  # score gap 1e4 * scale dwarfs the rest
    out = _single(oracle_mod, K, V, q, scale=1.0)
    np.testing.assert_array_equal(out, V[23].astype(np.float64))


def test_scores_are_shift_invariant_at_large_magnitude(oracle_mod):
    """Softmax is invariant to a common shift of all scores; a +1000 shift must
    neither overflow nor change the result (exp(1000) overflows double)."""
    rng = np.random.default_rng(6)
    K = rng.standard_normal((30, 8)).astype(np.float32)
    V = rng.standard_normal((30, 8)).astype(np.float32)
    q = rng.standard_normal(8).astype(np.float32)
    q[7] = 1.0
    K[:, 7] = np.round(K[:, 7] * 8) / 8          # exact in fp32 after +1000
    K2 = K.copy()
    K2[:, 7] += 1000.0                           # every score grows by exactly 1000
    out_a = _single(oracle_mod, K, V, q, 1.0)
    out_b = _single(oracle_mod, K2, V, q, 1.0)
    assert np.all(np.isfinite(out_b))
    np.testing.assert_allclose(out_b, out_a, rtol=1e-9, atol=1e-12)


# ---------------------------------------------------------------- invariants
def test_physical_placement_does_not_change_output(oracle_mod):
    rng = np.random.default_rng(7)
    lens = (17, 33, 5, 64)
    q, K, V, kp, vp, table = rand_case(rng, lens, 4, 4, 64, 64, "bf16")
    out_a = oracle_mod.paged_decode(q, kp, vp, table, np.array(lens, np.int32), 0.125)
    table2 = make_tables(lens, 64, np.random.default_rng(99))
    assert not np.array_equal(table, table2)
    kp2, vp2 = place(K, table2, 64, np.uint16(0x7FC0)), place(V, table2, 64, np.uint16(0x7FC0))
    out_b = oracle_mod.paged_decode(q, kp2, vp2, table2, np.array(lens, np.int32), 0.125)
    np.testing.assert_array_equal(out_a, out_b)


def test_gather_returns_logical_rows(oracle_mod):
    rng = np.random.default_rng(8)
    lens = (40, 3)
    q, K, V, kp, vp, table = rand_case(rng, lens, 2, 2, 8, 16)
    for s, L in enumerate(lens):
        for h in range(2):
            Kg, Vg = oracle_mod.gather(kp, vp, table[s], L, h)
            np.testing.assert_array_equal(Kg, K[s][:, h].astype(np.float64))
            np.testing.assert_array_equal(Vg, V[s][:, h].astype(np.float64))


def test_shared_prefix_equals_copied_prefix(oracle_mod):
    """Sharing is a pointer change: shared and copied prefix blocks give identical bits."""
    rng = np.random.default_rng(9)
    hkv, d, nb = 2, 16, 64
    prefix = rng.standard_normal((32, hkv, d)).astype(np.float32)       # 2 blocks
    suffixes = [rng.standard_normal((n, hkv, d)).astype(np.float32) for n in (5, 16, 21)]
    S = len(suffixes)
    lens = [32 + len(x) for x in suffixes]
    # shared: all sequences point at blocks 0 and 1
    shared = np.full((S, 4), -1, np.int32)
    copied = np.full((S, 4), -1, np.int32)
    kp = np.full((nb, hkv, B, d), np.nan, np.float32)
    vp = np.full((nb, hkv, B, d), np.nan, np.float32)
    vpre = rng.standard_normal((32, hkv, d)).astype(np.float32)
    nxt = 2
    for j in range(32):
        kp[j // B, :, j % B] = prefix[j]
        vp[j // B, :, j % B] = vpre[j]
    for s in range(S):
        shared[s, :2] = [0, 1]
        copied[s, :2] = [nxt, nxt + 1]
        kp[nxt:nxt + 2] = kp[0:2]
        vp[nxt:nxt + 2] = vp[0:2]
        nxt += 2
        for j, row in enumerate(suffixes[s]):
            blk_i = 2 + j // B
            if shared[s, blk_i] < 0:
                shared[s, blk_i] = copied[s, blk_i] = nxt
                nxt += 1
            kp[shared[s, blk_i], :, j % B] = row
            vp[shared[s, blk_i], :, j % B] = row * 0.5
    q = rng.standard_normal((S, 4, d)).astype(np.float32)
    a = oracle_mod.paged_decode(q, kp, vp, shared, np.array(lens, np.int32), 0.25)
    b = oracle_mod.paged_decode(q, kp, vp, copied, np.array(lens, np.int32), 0.25)
    np.testing.assert_array_equal(a, b)


def test_decode_equals_last_prefill_row(oracle_mod):
    rng = np.random.default_rng(10)
    L, n = 45, 7
    q, K, V, kp, vp, table = rand_case(rng, (L,), 4, 2, 8, 16)
    qp = rng.standard_normal((n, 4, 8)).astype(np.float32)
    qp[-1] = q[0]
    pre = oracle_mod.paged_prefill(qp, kp, vp, table, np.array([L - n], np.int32),
                                   np.array([n], np.int32), np.array([0, n], np.int32), 0.3)
    dec = oracle_mod.paged_decode(q, kp, vp, table, np.array([L], np.int32), 0.3)
    np.testing.assert_array_equal(pre[-1], dec[0])


def test_prefill_without_cache_is_causal_attention(oracle_mod):
    rng = np.random.default_rng(11)
    n, d = 20, 8
    q, K, V, kp, vp, table = rand_case(rng, (n,), 2, 1, d, 8)
    qp = rng.standard_normal((n, 2, d)).astype(np.float32)
    got = oracle_mod.paged_prefill(qp, kp, vp, table, np.array([0], np.int32),
                                   np.array([n], np.int32), np.array([0, n], np.int32), 0.5)
    Kf, Vf = K[0][:, 0].astype(np.float64), V[0][:, 0].astype(np.float64)
    for i in range(n):
        for h in range(2):
            x = 0.5 * (Kf[:i + 1] @ qp[i, h].astype(np.float64))
            w = np.exp(x - x.max())
            ref = (w[:, None] * Vf[:i + 1]).sum(0) / w.sum()
            np.testing.assert_allclose(got[i, h], ref, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("parts", [2, 3, 4])
def test_split_kv_lse_merge_equals_one_pass(oracle_mod, parts):
    rng = np.random.default_rng(100 + parts)
    L, d = 203, 16
    K = rng.standard_normal((L, d))
    V = rng.standard_normal((L, d))
    q = rng.standard_normal(d)
    cuts = np.sort(rng.choice(np.arange(1, L), size=parts - 1, replace=False))
    bounds = [0, *cuts.tolist(), L]
    os_, ms, ls = [], [], []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        o, m, l = oracle_mod.attend_partial(q, K, V, lo, hi, 0.4)
        os_.append(o)
        ms.append(m)
        ls.append(l)
    merged = oracle_mod.lse_merge(np.array(os_), np.array(ms), np.array(ls))
    full, _, _ = oracle_mod.attend_partial(q, K, V, 0, L, 0.4)
    x = 0.4 * (K @ q)
    w = np.exp(x - x.max())
    ref = (w[:, None] * V).sum(0) / w.sum()
    np.testing.assert_allclose(full, ref, rtol=1e-12)
    np.testing.assert_allclose(merged, ref, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- append / copy
def test_kv_append_writes_slots_and_skips_negative(oracle_mod):
    rng = np.random.default_rng(12)
    nb, hkv, d = 8, 2, 4
    kp = np.full((nb, hkv, B, d), 0x7FC0, np.uint16)
    vp = kp.copy()
    slots = np.array([5, -1, 16 * 7 + 15, 16 * 2], np.int64)
    k = rng.integers(0, 2**16, (4, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 2**16, (4, hkv, d), dtype=np.uint16)
    before = kp.copy()
    n = oracle_mod.kv_append(slots, k, v, kp, vp)
    assert n == 3 * hkv
    expect_k = before.copy()
    expect_v = before.copy()
    for t, s in enumerate(slots):
        if s >= 0:
            expect_k[s // B, :, s % B] = k[t]
            expect_v[s // B, :, s % B] = v[t]
    np.testing.assert_array_equal(kp, expect_k)
    np.testing.assert_array_equal(vp, expect_v)
    with pytest.raises(ValueError):
        oracle_mod.kv_append(np.array([nb * B], np.int64), k[:1], v[:1], kp, vp)


def test_copy_blocks_duplicates_whole_blocks(oracle_mod):
    rng = np.random.default_rng(13)
    kp = rng.standard_normal((6, 2, B, 4)).astype(np.float32)
    vp = rng.standard_normal((6, 2, B, 4)).astype(np.float32)
    k0, v0 = kp.copy(), vp.copy()
    oracle_mod.copy_blocks(np.array([[1, 4], [2, 0]], np.int32), kp, vp)
    np.testing.assert_array_equal(kp[4], k0[1])
    np.testing.assert_array_equal(kp[0], k0[2])
    np.testing.assert_array_equal(vp[4], v0[1])
    np.testing.assert_array_equal(kp[[1, 2, 3, 5]], k0[[1, 2, 3, 5]])
