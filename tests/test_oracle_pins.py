"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
closed forms, invariants, special cases that reduce to a library routine, the
pages' own worked examples (tests/golden/), and agreement between two different
algorithms for the same quantity. CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_head_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([float(x) if "." in x else int(x) for x in line.split()])
    return rows


# ---------------------------------------------------------------- bf16 storage
def test_bf16_widen_exhaustive_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours_c = oracle.bf16_to_f64(bits)
    ours_np = oracle.bf16_widen(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    both_nan = np.isnan(ours_c) & np.isnan(ref)
    assert np.array_equal(ours_c[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ours_c), np.isnan(ref))
    assert np.array_equal(ours_np[~both_nan], ref[~both_nan])


def test_round_bf16_matches_torch_rne_on_binary32_values():
    gen = np.random.default_rng(7)
    # random bit patterns cover normals, subnormals, huge values and exact ties
    u = gen.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ties = (gen.integers(0, 2**16, size=2000, dtype=np.uint32) << 16 | 0x8000).astype(np.uint32).view(np.float32)
    f = np.concatenate([f, ties[np.isfinite(ties)]])
    ours = oracle.round_bf16(f.astype(np.float64))
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_round_bf16_hand_cases():
    one = 0x3F80
    cases = [
        (1.0 + 2.0**-8, one),            # halfway, even neighbour is 1.0
        (1.0 + 3 * 2.0**-8, one + 2),    # halfway, even neighbour is 1 + 2^-6
        (1.0 + 2.0**-8 + 2.0**-30, one + 1),  # just above halfway rounds up
        (-2.0, 0xC000),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (math.ldexp(2 - 2**-7, 127), 0x7F7F),  # largest finite
        (math.ldexp(2 - 2**-8, 127), 0x7F80),  # midpoint to 2^128 -> inf
        (math.ldexp(1.0, -133), 0x0001),       # smallest subnormal
        (math.ldexp(1.0, -134), 0x0000),       # half of it, ties to even zero
    ]
    for x, want in cases:
        assert int(oracle.round_bf16(x)) == want, (x, hex(int(oracle.round_bf16(x))), hex(want))


# ---------------------------------------------------------------- A3 RMSNorm
def test_rmsnorm_constant_vector_closed_form():
    D = 128
    for c in (1e-3, 0.5, 3.0):
        out = oracle.head_rmsnorm(np.full(D, c), np.ones(D), eps=1e-6)
        np.testing.assert_allclose(out, c / math.sqrt(c * c + 1e-6), rtol=1e-14)


def test_rmsnorm_unit_rms_and_gain():
    gen = np.random.default_rng(1)
    x = gen.standard_normal(128)
    g = gen.uniform(0.5, 1.5, 128)
    plain = oracle.head_rmsnorm(x, np.ones(128), eps=0.0)
    assert abs(math.sqrt(np.mean(plain**2)) - 1.0) < 1e-13  # mean, not sum, of squares
    np.testing.assert_allclose(oracle.head_rmsnorm(x, g, eps=0.0), g * plain, rtol=1e-14)
    np.testing.assert_allclose(oracle.head_rmsnorm(7.5 * x, np.ones(128), eps=0.0), plain, rtol=1e-13)


# ---------------------------------------------------------------- A4 RoPE
THETA = 1e6


def test_rope_identity_at_position_zero():
    x = np.random.default_rng(2).standard_normal(128)
    np.testing.assert_array_equal(oracle.rope_half(x, 0, THETA), x)


def test_rope_preserves_norm():
    gen = np.random.default_rng(3)
    for pos in (1, 17, 8191, 131071):
        x = gen.standard_normal(128)
        y = oracle.rope_half(x, pos, THETA)
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12 * np.linalg.norm(x)


def test_rope_unit_vectors_pin_pairing_frequency_and_sign():
    D = 128
    e = np.eye(D)
    # dimension 0 pairs with dimension 64 and turns by pos * theta^0 = pos rad
    y = oracle.rope_half(e[0], 1, THETA)
    assert abs(y[0] - math.cos(1.0)) < 1e-15 and abs(y[64] - math.sin(1.0)) < 1e-15
    assert np.count_nonzero(np.abs(y) > 1e-15) == 2
    y = oracle.rope_half(e[64], 1, THETA)
    assert abs(y[0] + math.sin(1.0)) < 1e-15 and abs(y[64] - math.cos(1.0)) < 1e-15
    # dimension 1 turns at theta^(-2/D) rad per position
    w1 = THETA ** (-2.0 / D)
    y = oracle.rope_half(e[1], 3, THETA)
    assert abs(y[1] - math.cos(3 * w1)) < 1e-15 and abs(y[65] - math.sin(3 * w1)) < 1e-15
    # the slowest pair (i = 63)
    w63 = THETA ** (-126.0 / D)
    y = oracle.rope_half(e[63], 1000, THETA)
    assert abs(y[63] - math.cos(1000 * w63)) < 1e-15 and abs(y[127] - math.sin(1000 * w63)) < 1e-15


def test_rope_relative_position_and_inverse():
    gen = np.random.default_rng(4)
    q = gen.standard_normal(128)
    k = gen.standard_normal(128)
    for p, s in ((5, 2), (300, 299), (70000, 12)):
        lhs = oracle.rope_half(q, p, THETA) @ oracle.rope_half(k, s, THETA)
        rhs = oracle.rope_half(q, p - s, THETA) @ k
        assert abs(lhs - rhs) < 1e-9
        back = oracle.rope_half(oracle.rope_half(q, p, THETA), -p, THETA)
        np.testing.assert_allclose(back, q, atol=1e-12)


# ---------------------------------------------------------------- A5 GQA map
def test_gqa_map_matches_page_example():
    for Hq, Hkv, h, want in _golden_rows("gqa_head_map.txt"):
        assert oracle.kv_head(h, Hq, Hkv) == want


def test_gqa_map_groups_are_consecutive_and_equal():
    for Hq, Hkv in ((16, 8), (32, 8), (8, 8), (28, 4), (64, 4)):
        g = Hq // Hkv
        heads = [oracle.kv_head(h, Hq, Hkv) for h in range(Hq)]
        assert heads == sorted(heads)
        assert all(heads.count(k) == g for k in range(Hkv))


# ---------------------------------------------------------------- A7 addressing
def test_paged_offset_worked_examples():
    table = np.array([[2, 0, 1]], dtype=np.int32)
    for pos, kvh, want in _golden_rows("paged_offset.txt"):
        assert oracle.cache_offset(table, 0, kvh, pos, Hkv=2, P=4, D=8, num_pages=3) == want


def test_paged_offsets_are_a_bijection_onto_owned_slots():
    kv = inputs.paged_kv(5, [37, 16, 1, 64], Hkv=3, D=8, page_size=16, spare_pages=2)
    seen = set()
    for b, T in enumerate(kv.context_lens):
        for h in range(3):
            for pos in range(T):
                off = oracle.cache_offset(kv.block_table, b, h, pos, 3, 16, 8, kv.num_pages)
                assert 0 <= off < kv.k_cache.size and off % 8 == 0
                seen.add(off)
    assert len(seen) == 3 * int(kv.context_lens.sum())
    # a table entry outside the pool is refused
    bad = kv.block_table.copy()
    bad[0, 0] = kv.num_pages
    assert oracle.cache_offset(bad, 0, 0, 0, 3, 16, 8, kv.num_pages) == -1


def test_kv_cache_bytes_page_figure():
    for layers, B, Hkv, D, T, mib in _golden_rows("kv_cache_bytes.txt"):
        per_layer = 2 * B * Hkv * D * T * 2
        assert layers * per_layer == mib * 2**20
    # the generator's pool holds exactly that many bytes for a whole-page history
    kv = inputs.paged_kv(9, [1024], Hkv=8, D=128, page_size=16, spare_pages=0, fill_unused="normal")
    assert kv.k_cache.nbytes + kv.v_cache.nbytes == 2 * 1 * 8 * 128 * 1024 * 2


# ---------------------------------------------------------------- A6 attention
def _scatter(k_contig, v_contig, kv):
    """Write contiguous [B,T,Hkv,D] rows into kv's pool via the oracle's addressing."""
    B, T, Hkv, D = k_contig.shape
    kc = kv.k_cache.reshape(-1).copy()
    vc = kv.v_cache.reshape(-1).copy()
    for b in range(B):
        for t in range(T):
            for h in range(Hkv):
                off = oracle.cache_offset(kv.block_table, b, h, t, Hkv, kv.page_size, D, kv.num_pages)
                kc[off:off + D] = k_contig[b, t, h]
                vc[off:off + D] = v_contig[b, t, h]
    return kc.reshape(kv.k_cache.shape), vc.reshape(kv.v_cache.shape)


def test_paged_attention_equals_contiguous_attention_after_scatter():
    B, T, Hq, Hkv, D = 2, 37, 4, 2, 16
    k, v = inputs.contiguous_kv(11, B, T, Hkv, D)
    q = inputs.query(11, B, Hq, D)
    kv = inputs.paged_kv(12, [T] * B, Hkv=Hkv, D=D, page_size=8, spare_pages=3)
    kc, vc = _scatter(k, v, kv)
    paged = oracle.decode_attention(q, kc, vc, kv.block_table, kv.context_lens, 0.25)
    contig = oracle.attention_contiguous(q, k, v, 0.25)
    np.testing.assert_array_equal(paged, contig)
    assert np.isfinite(paged).all()  # NaN-filled unowned slots were never read


def test_attention_t1_returns_v_and_gqa_map():
    Hq, Hkv, D = 16, 8, 128
    kv = inputs.paged_kv(13, [1], Hkv=Hkv, D=D, page_size=16)
    q = inputs.query(13, 1, Hq, D)
    out = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, 128**-0.5)
    page = kv.block_table[0, 0]
    for h in range(Hq):
        np.testing.assert_array_equal(out[0, h], oracle.bf16_widen(kv.v_cache[page, h // 2, 0]))


def test_attention_equal_scores_is_mean_of_v():
    T, Hkv, D = 45, 2, 128
    kv = inputs.paged_kv(14, [T], Hkv=Hkv, D=D, page_size=16)
    q = np.zeros((1, 4, D), dtype=np.uint16)  # q = 0: every score is 0
    out = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, 0.1)
    for h in range(4):
        rows = [kv.v_cache[kv.block_table[0, t // 16], h // 2, t % 16] for t in range(T)]
        mean = oracle.bf16_widen(np.array(rows)).mean(axis=0)
        np.testing.assert_allclose(out[0, h], mean, rtol=1e-13, atol=1e-15)


def test_attention_t2_closed_form():
    D = 128
    scale = 1.0 / math.sqrt(D)
    q = np.zeros((1, 1, D), dtype=np.uint16)
    q[0, 0, 0] = 0x4000  # q = 2 e0
    kv = inputs.paged_kv(15, [2], Hkv=1, D=D, page_size=16)
    page = kv.block_table[0, 0]
    kv.k_cache[page, 0, 0] = 0
    kv.k_cache[page, 0, 1] = 0
    kv.k_cache[page, 0, 0, 0] = 0x3F80  # k0 = e0 -> s0 = 2 * scale
    kv.k_cache[page, 0, 1, 0] = 0xBF80  # k1 = -e0 -> s1 = -2 * scale
    out = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, scale)
    v0 = oracle.bf16_widen(kv.v_cache[page, 0, 0])
    v1 = oracle.bf16_widen(kv.v_cache[page, 0, 1])
    w0 = 1.0 / (1.0 + math.exp(-4 * scale))  # sigma(s0 - s1)
    np.testing.assert_allclose(out[0, 0], w0 * v0 + (1 - w0) * v1, rtol=1e-13, atol=1e-15)


def test_attention_ignores_history_past_context_and_page_order():
    T, Hq, Hkv, D = 33, 4, 2, 32
    k, v = inputs.contiguous_kv(16, 1, T, Hkv, D)
    q = inputs.query(16, 1, Hq, D)
    outs = []
    for seed in (20, 21):  # two different permutations of the pool
        kv = inputs.paged_kv(seed, [T], Hkv=Hkv, D=D, page_size=8, spare_pages=2)
        kc, vc = _scatter(k, v, kv)
        outs.append(oracle.decode_attention(q, kc, vc, kv.block_table, kv.context_lens, 0.2))
    np.testing.assert_array_equal(outs[0], outs[1])
    # shortening the context by one equals attending over the first T-1 rows
    short = oracle.attention_contiguous(q, np.ascontiguousarray(k[:, :T - 1]), np.ascontiguousarray(v[:, :T - 1]), 0.2)
    kv = inputs.paged_kv(20, [T], Hkv=Hkv, D=D, page_size=8, spare_pages=2)
    kc, vc = _scatter(k, v, kv)
    ctx = np.array([T - 1], dtype=np.int32)
    np.testing.assert_array_equal(oracle.decode_attention(q, kc, vc, kv.block_table, ctx, 0.2), short)


def test_attention_peaked_score_selects_one_value():
    D, T = 128, 20
    k, v = inputs.contiguous_kv(17, 1, T, 1, D)
    q = k[:, 7].copy()  # q equals key 7; with a large scale key 7 dominates
    out = oracle.attention_contiguous(q, k, v, 50.0)
    np.testing.assert_allclose(out[0, 0], oracle.bf16_widen(v[0, 7, 0]), atol=1e-9)


def test_attention_empty_history_is_zero():
    kv = inputs.paged_kv(18, [0, 3], Hkv=1, D=16, page_size=4)
    q = inputs.query(18, 2, 1, 16)
    out = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, 0.25)
    assert np.all(out[0] == 0) and np.isfinite(out[1]).all()


# ---------------------------------------------------------------- A1 / A2 state
def _direct(scores, values):
    w = np.exp(scores - scores.max())
    return (w / w.sum()) @ values


def test_online_recurrence_equals_direct_softmax():
    gen = np.random.default_rng(21)
    for T in (1, 2, 7, 513):
        s = gen.standard_normal(T) * 4
        vals = gen.standard_normal((T, 16))
        st = oracle.state_update(oracle.state_init(16), s, vals)
        assert st[0] == s.max()
        np.testing.assert_allclose(oracle.state_finalize(st), _direct(s, vals), rtol=1e-12, atol=1e-13)
        # order of arrival does not matter
        perm = gen.permutation(T)
        st2 = oracle.state_update(oracle.state_init(16), s[perm], vals[perm])
        np.testing.assert_allclose(oracle.state_finalize(st2), _direct(s, vals), rtol=1e-12, atol=1e-13)


def test_init_state_values():
    m, l, acc = oracle.state_init(8)
    assert m == -1e30 and l == 0.0 and np.all(acc == 0)
    assert np.all(oracle.state_finalize((m, l, acc)) == 0)


@pytest.mark.parametrize("sizes", [[5, 5, 5], [1, 14], [0, 15], [15, 0], [3, 0, 0, 12], [15]])
def test_merge_of_any_split_equals_direct(sizes):
    gen = np.random.default_rng(22)
    T = sum(sizes)
    s = gen.standard_normal(T) * 6
    s[3] += 30.0  # one large score forces rescaling across partitions
    vals = gen.standard_normal((T, 8))
    ms, ls, accs = [], [], []
    start = 0
    for n in sizes:
        m, l, acc = oracle.state_update(oracle.state_init(8), s[start:start + n], vals[start:start + n])
        ms.append(m), ls.append(l), accs.append(acc)
        start += n
    merged = oracle.merge_partitions(np.array(ms), np.array(ls), np.array(accs))
    np.testing.assert_allclose(merged, _direct(s, vals), rtol=1e-12, atol=1e-13)


def test_merge_all_empty_is_zero():
    out = oracle.merge_partitions(np.full(3, -1e30), np.zeros(3), np.zeros((3, 4)))
    assert np.all(out == 0)


def test_tiled_state_matches_direct_attention():
    B, T, Hq, Hkv, D = 1, 70, 4, 2, 16
    k, v = inputs.contiguous_kv(23, B, T, Hkv, D)
    q = inputs.query(23, B, Hq, D)
    m, l, acc = oracle.tiled_state_reference(q, k, v, 0.3, tile=16)
    out = acc / l[..., None]
    np.testing.assert_allclose(out, oracle.attention_contiguous(q, k, v, 0.3), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- prologue
def test_prologue_writes_only_the_new_slots_and_copies_v():
    B, Hq, Hkv, D, P = 3, 4, 2, 128, 16
    ctx = [1, 16, 37]
    kv = inputs.paged_kv(24, ctx, Hkv=Hkv, D=D, page_size=P, fill_unused="normal")
    tok = inputs.new_token(24, B, Hq, Hkv, D)
    q_out, kc, vc = oracle.qk_norm_rope_append(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k, kv.context_lens,
                                               kv.block_table, kv.k_cache, kv.v_cache, P, 1e6)
    changed_k = np.argwhere(np.any(kc != kv.k_cache, axis=-1))
    changed_v = np.argwhere(np.any(vc != kv.v_cache, axis=-1))
    expect = set()
    for b, T in enumerate(ctx):
        for h in range(Hkv):
            off = oracle.cache_offset(kv.block_table, b, h, T - 1, Hkv, P, D, kv.num_pages)
            page, rest = divmod(off // D, Hkv * P)
            hh, o = divmod(rest, P)
            expect.add((page, hh, o))
            np.testing.assert_array_equal(vc[page, hh, o], tok.v[b, h])
    assert {tuple(x) for x in changed_k} <= expect
    assert {tuple(x) for x in changed_v} <= expect
    assert len({tuple(x) for x in changed_k}) == len(expect)


def test_prologue_position_zero_is_plain_rmsnorm_and_norm_is_kept():
    B, Hq, Hkv, D = 2, 4, 2, 128
    tok = inputs.new_token(25, B, Hq, Hkv, D)
    ones = np.full(D, 0x3F80, dtype=np.uint16)
    for T in (1, 5000):
        kv = inputs.paged_kv(25, [T, T], Hkv=Hkv, D=D, page_size=16, fill_unused="normal")
        q_out, kc, _ = oracle.qk_norm_rope_append(tok.q, tok.k, tok.v, ones, ones, kv.context_lens,
                                                  kv.block_table, kv.k_cache, kv.v_cache, 16, 1e6)
        qo = oracle.bf16_widen(q_out)
        # gamma = 1: each head leaves with RMS 1 (RoPE keeps the norm), up to bf16 rounding
        rms = np.sqrt(np.mean(qo**2, axis=-1))
        assert np.all(np.abs(rms - 1.0) < 4e-3)
        if T == 1:
            x = oracle.bf16_widen(tok.q[0, 0])
            want = x / np.sqrt(np.mean(x * x) + 1e-6)
            assert np.max(np.abs(qo[0, 0] - want)) <= 2.0**-8 * np.max(np.abs(want))


# --------------------------------------------------------------------------
# multi-query decode: M new tokens, token i at position T - M + i, causal
# --------------------------------------------------------------------------
def _multi_case(seed, ctx, M, Hq=16, Hkv=8):
    kv = inputs.paged_kv(seed, ctx, Hkv=Hkv, page_size=16)
    q = inputs.normal_bf16(inputs.generator(seed, 91), (len(ctx), M, Hq, 128))
    return kv, q


def test_multi_attention_with_one_token_is_the_decode_step():
    kv, q = _multi_case(700, [33, 200, 1], 1)
    multi = oracle.decode_attention_multi(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, 0.09)
    single = oracle.decode_attention(q[:, 0], kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, 0.09)
    assert np.array_equal(multi[:, 0], single)


@pytest.mark.parametrize("M", [2, 4, 7])
def test_multi_attention_token_i_is_a_decode_at_its_own_prefix(M):
    """Token i sees exactly the first T - M + i + 1 positions: the single-token
    oracle with the context shortened by M - 1 - i gives the same row."""
    kv, q = _multi_case(710 + M, [40, 17, 64], M)
    multi = oracle.decode_attention_multi(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, 0.09)
    for i in range(M):
        ctx_i = kv.context_lens - (M - 1 - i)
        single = oracle.decode_attention(q[:, i], kv.k_cache, kv.v_cache, kv.block_table, ctx_i, 0.09)
        assert np.allclose(multi[:, i], single, rtol=0, atol=1e-13), i


def test_multi_attention_first_token_of_a_fresh_sequence_returns_its_value():
    """T = M: token 0 sees only position 0, so its output is V[0] exactly."""
    M = 3
    kv, q = _multi_case(720, [M, M], M)
    multi = oracle.decode_attention_multi(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, 0.09)
    for b in range(2):
        page = kv.block_table[b, 0]
        for h in range(16):
            v0 = np.array([oracle.bf16_to_f64(x) for x in kv.v_cache[page, h // 2, 0]])
            assert np.array_equal(multi[b, 0, h], v0)


def test_multi_attention_refuses_context_shorter_than_m():
    kv, q = _multi_case(730, [2, 30], 3)
    with pytest.raises(oracle.OracleError):
        oracle.decode_attention_multi(q, kv.k_cache, kv.v_cache, kv.block_table, kv.context_lens, 0.09)


@pytest.mark.parametrize("M", [1, 3])
def test_multi_prologue_equals_single_token_prologues_in_order(M):
    """Token i of the multi prologue is the single-token prologue at context
    length T - M + i + 1; applying those one after the other gives the same
    rotated queries and the same cache bytes."""
    ctx = [40, 17, 64]
    kv = inputs.paged_kv(740 + M, ctx, Hkv=8, page_size=16)
    g = inputs.generator(740 + M, 92)
    q = inputs.normal_bf16(g, (3, M, 16, 128))
    k = inputs.normal_bf16(g, (3, M, 8, 128))
    v = inputs.normal_bf16(g, (3, M, 8, 128))
    tok = inputs.new_token(740 + M, 3, 16, 8)
    q_out, kc, vc = oracle.qk_norm_rope_append_multi(q, k, v, tok.gamma_q, tok.gamma_k, kv.context_lens,
                                                     kv.block_table, kv.k_cache, kv.v_cache, 16, 1e6)
    kc2, vc2 = kv.k_cache, kv.v_cache
    for i in range(M):
        qi, kc2, vc2 = oracle.qk_norm_rope_append(q[:, i], k[:, i], v[:, i], tok.gamma_q, tok.gamma_k,
                                                  kv.context_lens - (M - 1 - i), kv.block_table, kc2, vc2, 16, 1e6)
        assert np.array_equal(q_out[:, i], qi)
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)


# --------------------------------------------------------------------------
# INT8 KV rows: symmetric per-row quantization with an FP32 scale
# (Qwen3 runtime s0.1; RTX 5090 residency page, int8 note)
# --------------------------------------------------------------------------
def _bits(values) -> np.ndarray:
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_int8_row_amax_maps_to_127_and_error_is_half_a_step():
    rows = inputs.normal_bf16(inputs.generator(600, 1), (64, 128))
    codes, scales = oracle.quantize_rows_int8(rows)
    x = oracle.bf16_to_f64(rows)
    amax = np.abs(x).max(axis=1)
    assert np.allclose(scales, (amax / 127).astype(np.float32), rtol=0, atol=0)
    assert np.all(np.abs(codes).max(axis=1) == 127)
    err = np.abs(x - oracle.dequantize_int8(codes, scales))
    # half a step, plus the binary32 rounding of x / s (|x / s| <= 127, 2^-24 relative)
    assert np.all(err <= scales[:, None] * (0.5 + 127 * 2.0 ** -23))


def test_int8_row_ties_round_to_even_and_sign_is_symmetric():
    # amax = 127 makes the scale exactly 1, so x / s = x
    row = _bits([127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -126.5] + [0.0] * 120)
    codes, scales = oracle.quantize_rows_int8(row[None])
    assert scales[0] == 1.0
    assert list(codes[0, :8]) == [127, 2, 4, -2, -4, 0, 2, -126]
    neg = _bits(-oracle.bf16_to_f64(row))
    codes_n, scales_n = oracle.quantize_rows_int8(neg[None])
    assert scales_n[0] == scales[0] and np.array_equal(codes_n, -codes)


def test_int8_zero_row_has_zero_scale_and_codes():
    codes, scales = oracle.quantize_rows_int8(np.zeros((1, 128), dtype=np.uint16))
    assert scales[0] == 0.0 and not codes.any()


def test_int8_attention_equals_bf16_attention_when_dequantized_values_are_bf16():
    """With power-of-two scales every code * scale is a bf16 value (|code| <=
    127 < 256), so the INT8 attention must equal the bf16 oracle on that
    dequantized cache exactly."""
    kv = inputs.paged_kv(610, [40, 17, 3], Hkv=8, page_size=16, fill_unused="normal")
    g = np.random.default_rng(611)
    k8 = g.integers(-127, 128, kv.k_cache.shape, dtype=np.int8)
    v8 = g.integers(-127, 128, kv.v_cache.shape, dtype=np.int8)
    ks = (2.0 ** g.integers(-9, -4, kv.k_cache.shape[:-1])).astype(np.float32)
    vs = (2.0 ** g.integers(-9, -4, kv.v_cache.shape[:-1])).astype(np.float32)
    kb = _bits(oracle.dequantize_int8(k8, ks))
    vb = _bits(oracle.dequantize_int8(v8, vs))
    assert np.array_equal(oracle.bf16_to_f64(kb), oracle.dequantize_int8(k8, ks))  # exactly representable
    q = inputs.query(610, 3, 16)
    got = oracle.decode_attention_int8(q, k8, v8, ks, vs, kv.block_table, kv.context_lens, 0.09)
    ref = oracle.decode_attention(q, kb, vb, kv.block_table, kv.context_lens, 0.09)
    assert np.array_equal(got, ref)


def test_int8_prologue_quantizes_the_bf16_prologue_rows():
    """The INT8 prologue's K and V slots hold the per-row quantization of the
    bf16 prologue's K slot and of the V row; q_out is the same."""
    ctx = [40, 17, 64]
    kv = inputs.paged_kv(620, ctx, Hkv=8, page_size=16, fill_unused="normal")
    tok = inputs.new_token(620, 3, 16, 8)
    k8, ks = oracle.quantize_rows_int8(kv.k_cache)
    v8, vs = oracle.quantize_rows_int8(kv.v_cache)
    q_out, kc8, vc8, ks2, vs2 = oracle.qk_norm_rope_append_int8(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k,
                                                                 kv.context_lens, kv.block_table, k8, v8, ks, vs,
                                                                 16, 1e6)
    q_ref, kc_ref, vc_ref = oracle.qk_norm_rope_append(tok.q, tok.k, tok.v, tok.gamma_q, tok.gamma_k,
                                                       kv.context_lens, kv.block_table, kv.k_cache, kv.v_cache,
                                                       16, 1e6)
    assert np.array_equal(q_out, q_ref)
    k8_ref, ks_ref = oracle.quantize_rows_int8(kc_ref)
    v8_ref, vs_ref = oracle.quantize_rows_int8(vc_ref)
    assert np.array_equal(kc8, k8_ref) and np.array_equal(ks2, ks_ref)
    assert np.array_equal(vc8, v8_ref) and np.array_equal(vs2, vs_ref)
